"""Multi-token decode (steps of 1..16 query tokens per sequence, causal inside
the step) on the GPU against the fp64 oracle (TileInfer.jl "Performance"
page, "Attention for verify steps": 2-16-token steps run the split-KV decode
kernels).  The oracle is the same causal paged attention the prefill tests
use: token i of q_b new tokens in a sequence of L positions sees 0..L-q_b+i."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_flash_gb300 import workloads as W
from tests.helpers import check_lse, check_out, dev, dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pk():
    from paged_kv_flash_gb300 import pagedkv
    return pagedkv


def gpu_multi(pk, case: W.MultiCase, num_splits=0, max_q=None):
    pool = pk.Pool(dev_bf16(case.k_pool), dev_bf16(case.v_pool))
    mq = int(case.q_lens.max()) if max_q is None else max_q
    out, lse = pk.paged_attn_decode_multi(pool, dev_bf16(case.q), dev(case.cu_q),
                                          dev(case.layout.block_table), dev(case.seq_lens), mq,
                                          int(case.seq_lens.max()), case.scale,
                                          num_splits=num_splits)
    return out, lse


def oracle_multi(case: W.MultiCase, rows=None):
    return oracle.paged_attention(case.k_pool, case.v_pool, case.q, case.cu_q,
                                  case.layout.block_table, case.seq_lens, case.scale, rows=rows)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_ragged_steps_and_group_sizes(pk, G):
    """Steps of 1, 2, 5, 16 and 9 tokens; contexts from one page to several
    splits, a page boundary inside a step; every split count path."""
    rng = np.random.default_rng(300 + G)
    lens = np.array([40, 1024, 17, 777, 2000], np.int32)
    qlens = np.array([1, 2, 5, 16, 9], np.int32)
    case = W.multi_token_decode(rng, lens, qlens, Hq=2 * G, Hkv=2)
    ro, rl = oracle_multi(case)
    for splits in (0, 1, 3, 7):
        out, lse = gpu_multi(pk, case, splits)
        assert pk.poll_device_error() == pk.OK
        check_out(out, ro, f"G={G} splits={splits}")
        check_lse(lse, rl, f"G={G} splits={splits}")


def test_verify_step_16_tokens_1k(pk):
    """The pages' verify-step shape: 16 tokens against 1,024 positions, GQA 32/8."""
    rng = np.random.default_rng(310)
    case = W.multi_token_decode(rng, [1024], [16], Hq=32, Hkv=8)
    ro, rl = oracle_multi(case)
    out, lse = gpu_multi(pk, case)
    assert pk.poll_device_error() == pk.OK
    check_out(out, ro, "verify 16 x 1k")
    check_lse(lse, rl, "verify 16 x 1k")


def test_batched_verify_steps_sampled(pk):
    """8 sequences of 4k-8k positions with 16-token steps, sampled rows."""
    rng = np.random.default_rng(311)
    lens = rng.integers(4096, 8193, 8).astype(np.int32)
    case = W.multi_token_decode(rng, lens, [16] * 8, Hq=32, Hkv=8)
    out, lse = gpu_multi(pk, case)
    assert pk.poll_device_error() == pk.OK
    rows = np.sort(rng.choice(len(case.q), 24, replace=False)).astype(np.int32)
    ro, rl = oracle_multi(case, rows=rows)
    idx = torch.from_numpy(rows.astype(np.int64)).cuda()
    check_out(out[idx], ro, "batched verify")
    check_lse(lse[idx], rl, "batched verify")


def test_one_token_steps_match_the_decode_kernel(pk):
    """With one token per sequence the multi-token path is ordinary decode."""
    rng = np.random.default_rng(312)
    lens = np.array([1, 300, 4096, 65], np.int32)
    case = W.multi_token_decode(rng, lens, [1] * 4, Hq=32, Hkv=8)
    out, lse = gpu_multi(pk, case)
    pool = pk.Pool(dev_bf16(case.k_pool), dev_bf16(case.v_pool))
    out1, lse1 = pk.paged_attn_decode(pool, dev_bf16(case.q), dev(case.layout.block_table),
                                      dev(case.seq_lens), int(lens.max()), case.scale)
    assert pk.poll_device_error() == pk.OK
    ro, rl = oracle_multi(case)
    check_out(out, ro, "multi q=1")
    check_out(out1, ro, "decode")
    check_lse(lse, rl, "multi q=1")
    assert (out.float() - out1.float()).abs().max().item() <= 2e-2


def test_sequence_longer_than_max_q_is_flagged(pk):
    rng = np.random.default_rng(313)
    case = W.multi_token_decode(rng, [100, 200], [3, 5], Hq=8, Hkv=2)
    gpu_multi(pk, case, max_q=4)                 # sequence 1 has 5 tokens
    assert pk.poll_device_error() == pk.ERR_INVALID
    assert pk.poll_device_error() == pk.OK


def test_sequence_without_tokens_in_the_step(pk):
    """A batch where the middle sequence has no token in this step (an empty
    cu_q range): its cache is not read and the others are unaffected."""
    rng = np.random.default_rng(314)
    case = W.multi_token_decode(rng, [300, 500, 64], [3, 0, 5], Hq=8, Hkv=2)
    ro, rl = oracle_multi(case)
    for splits in (0, 3):
        out, lse = gpu_multi(pk, case, splits)
        assert pk.poll_device_error() == pk.OK
        check_out(out, ro, f"empty step splits={splits}")
        check_lse(lse, rl, f"empty step splits={splits}")
