"""The fused attention-input step (q/k RMSNorm, RoPE, KV write from the q/k/v
projection; TileInfer.jl "Performance" page, "Fused kernels, FlashAttention
and PagedAttention": the fused kernels are bit-identical to the chains of
kernels they replace) on the GPU against the oracle, bit for bit on every
path: norm and RoPE, norm only, RoPE only, neither.  The norm's mean square
is the exact sum rounded once to fp32 on both sides, so no summation order
enters; V and the untouched slots are compared bit for bit too.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_flash_gb300 import workloads as W
from tests.helpers import dev, dev_bf16, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pk():
    from paged_kv_flash_gb300 import pagedkv
    return pagedkv


def ordered(bits):
    """bf16 bit patterns -> integers in the order of their values."""
    b = bits.astype(np.int32)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def assert_bits_equal(got, want, what):
    """Bit-for-bit equality; on failure name the first differing elements."""
    bad = np.argwhere(got != want)
    if len(bad):
        show = [(tuple(int(i) for i in ix), float(W.bits_to_float(got[tuple(ix)])),
                 float(W.bits_to_float(want[tuple(ix)]))) for ix in bad[:6]]
        raise AssertionError(f"{what}: {len(bad)} of {got.size} differ; first "
                             f"(index, got, want): {show}")


def run(pk, case, norm=True, rope=True):
    kp, vp = W.empty_pool_bf16(case.layout.num_pages, case.Hkv)
    pool = pk.Pool(dev_bf16(kp), dev_bf16(vp))
    tw = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    q = pk.qkv_norm_rope_append(
        pool, dev_bf16(case.qkv), case.Hq, dev(case.cu_new), dev(case.layout.block_table),
        dev(case.seq_lens), q_norm_w=tw(case.q_w) if norm else None,
        k_norm_w=tw(case.k_w) if norm else None, eps=1e-6,
        rope_cos=tw(case.cos) if rope else None, rope_sin=tw(case.sin) if rope else None)
    assert pk.poll_device_error() == pk.OK
    ref = oracle.qkv_norm_rope_append(
        case.qkv, case.Hq, case.Hkv, case.q_w if norm else None, case.k_w if norm else None,
        1e-6, case.cos if rope else None, case.sin if rope else None, case.cu_new,
        case.layout.block_table, case.seq_lens, kp, vp)
    return (host_bits(q), host_bits(pool.k), host_bits(pool.v)), ref


@pytest.mark.parametrize("norm,rope", [(True, True), (True, False), (False, True)])
def test_small_batch_matches_oracle(pk, norm, rope):
    case = W.qkv_prep_case(90, [37, 5, 16], [37, 700, 130], Hq=32, Hkv=8)
    (q, k, v), (rq, rk, rv) = run(pk, case, norm, rope)
    what = f"norm={norm} rope={rope}"
    assert_bits_equal(q, rq, f"q_out {what}")
    assert_bits_equal(k, rk, f"K pool {what}")   # untouched slots: NaN sentinel on both sides
    assert_bits_equal(v, rv, f"V pool {what}")


def test_no_norm_no_rope_is_the_plain_append_bit_for_bit(pk):
    case = W.qkv_prep_case(91, [20, 3], [100, 3], Hq=16, Hkv=8)
    (q, k, v), (rq, rk, rv) = run(pk, case, norm=False, rope=False)
    assert_bits_equal(q, rq, "q_out")
    assert_bits_equal(k, rk, "K pool")
    assert_bits_equal(v, rv, "V pool")


def test_prefill_chunk_size(pk):
    """A 2,048-token chunk of one sequence at positions 14,336 .. 16,383:
    81,920 normed head vectors, every output bit-identical."""
    case = W.qkv_prep_case(92, [2048], [16384], Hq=32, Hkv=8)
    for norm, rope in ((True, True), (True, False)):
        (q, k, v), (rq, rk, rv) = run(pk, case, norm, rope)
        assert_bits_equal(q, rq, f"q_out chunk norm={norm} rope={rope}")
        assert_bits_equal(k, rk, f"K pool chunk norm={norm} rope={rope}")
        assert_bits_equal(v, rv, f"V pool chunk norm={norm} rope={rope}")


def test_norm_uses_the_exact_mean_square(pk):
    """A q head x = (16, 2^-8, 2^-15, 0, ...): the squares sum to 256 + 2^-16
    + 2^-30, so the mean 2 + 2^-23 + 2^-37 lies just above the fp32 midpoint
    2 + 2^-23 and rounds up to 2 + 2^-22, where a running fp32 sum would tie
    256 + 2^-16 back to 256 and give 2.  With eps = 0 the two means give
    different r, and the weight 1.0081796646... on channel 0 puts 16 r w
    exactly on the bf16 tie 11.40625 for the exact mean's r (-> 11.375 by
    ties to even) and one fp32 step above it for the running sum's (->
    11.4375).  Both q heads of
    the token and the k head carry the vector; values within 2^19 of each
    other, inside the range where the GPU's sum is exact."""
    case = W.qkv_prep_case(96, [3], [3], Hq=2, Hkv=1)
    x = np.zeros(W.HEAD_DIM, np.float32)
    x[:3] = (16.0, 2.0 ** -8, 2.0 ** -15)
    xb = W.to_bf16_bits(x)
    qkv = case.qkv.copy()
    qkv[1, 0] = xb
    qkv[1, 1] = xb
    qkv[1, 2] = xb
    w = np.ones(W.HEAD_DIM, np.float32)
    w[0] = np.uint32(1065421832).view(np.float32)
    kp, vp = W.empty_pool_bf16(case.layout.num_pages, case.Hkv)
    pool = pk.Pool(dev_bf16(kp), dev_bf16(vp))
    tw = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    q = pk.qkv_norm_rope_append(pool, dev_bf16(qkv), case.Hq, dev(case.cu_new),
                                dev(case.layout.block_table), dev(case.seq_lens),
                                q_norm_w=tw(w), k_norm_w=tw(w), eps=0.0)
    assert pk.poll_device_error() == pk.OK
    rq, rk, rv = oracle.qkv_norm_rope_append(qkv, case.Hq, case.Hkv, w, w, 0.0, None, None,
                                             case.cu_new, case.layout.block_table,
                                             case.seq_lens, kp, vp)
    assert W.bits_to_float(rq[1, 0, :1])[0] == np.float32(11.375)
    assert_bits_equal(host_bits(q), rq, "q_out, exact mean square")
    assert_bits_equal(host_bits(pool.k), rk, "K pool, exact mean square")
    assert_bits_equal(host_bits(pool.v), rv, "V pool, exact mean square")


def test_position_past_the_rope_table_is_flagged(pk):
    case = W.qkv_prep_case(93, [4], [40], Hq=8, Hkv=8, max_pos=38)
    kp, vp = W.empty_pool_bf16(case.layout.num_pages, case.Hkv)
    pool = pk.Pool(dev_bf16(kp), dev_bf16(vp))
    tw = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    pk.qkv_norm_rope_append(pool, dev_bf16(case.qkv), case.Hq, dev(case.cu_new),
                            dev(case.layout.block_table), dev(case.seq_lens),
                            rope_cos=tw(case.cos), rope_sin=tw(case.sin))
    assert pk.poll_device_error() == pk.ERR_INVALID
    assert pk.poll_device_error() == pk.OK                  # the flag is cleared once read


@pytest.mark.parametrize("Hq,Hkv", [(12, 3), (64, 8), (5, 5)])
def test_head_counts_that_split_a_warp_or_need_extra_passes(pk, Hq, Hkv):
    """q/k/v boundaries inside one warp's four heads (12/3, 5/5), and more
    heads than the loads issued ahead cover (64/8: 80 head vectors)."""
    case = W.qkv_prep_case(94, [19, 2], [19, 300], Hq=Hq, Hkv=Hkv)
    for norm, rope in ((True, True), (False, True)):
        (q, k, v), (rq, rk, rv) = run(pk, case, norm, rope)
        what = f"{Hq}/{Hkv} norm={norm} rope={rope}"
        assert_bits_equal(q, rq, f"q_out {what}")
        assert_bits_equal(k, rk, f"K pool {what}")
        assert_bits_equal(v, rv, f"V pool {what}")
