"""The fused attention-input step (q/k RMSNorm, RoPE, KV write from the q/k/v
projection; TileInfer.jl "Performance" page, "Fused kernels, FlashAttention
and PagedAttention") on the GPU against the fp64 oracle.

Both sides round to bf16 at the same points; the GPU's norm runs in fp32
(the oracle's in fp64), so a normed value may land one bf16 step from the
oracle's where the exact value sits at a rounding boundary.  Bounds: the norm
output within one bf16 step; a rotated output within one step of itself plus
one step of the larger of the two normed values it is made from (a one-step
difference there passes through the rotation, and cancellation can make it
many steps of a small output).  Nearly all elements must be bit-equal.  V and
the untouched slots are compared bit for bit.
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


def check_bf16(got, want, what, max_frac_off=1e-3):
    d = np.abs(ordered(got) - ordered(want))
    assert d.max() <= 1, f"{what}: {int(d.max())} bf16 steps off"
    assert (d != 0).mean() <= max_frac_off, f"{what}: {(d != 0).mean():.2e} of elements off"


def assert_bits_equal(got, want, what):
    """Bit-for-bit equality; on failure name the first differing elements."""
    bad = np.argwhere(got != want)
    if len(bad):
        show = [(tuple(int(i) for i in ix), float(W.bits_to_float(got[tuple(ix)])),
                 float(W.bits_to_float(want[tuple(ix)]))) for ix in bad[:6]]
        raise AssertionError(f"{what}: {len(bad)} of {got.size} differ; first "
                             f"(index, got, want): {show}")


def ulp(v):
    """One bf16 step at |v| (normal range)."""
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(a)) - 7)


def check_rotated(got, want, normed, what, max_frac_off=1e-3):
    """got/want: bf16 bits [..., 128] after norm and rotation; normed: the
    oracle's bf16 bits before the rotation."""
    g = W.bits_to_float(got).astype(np.float64)
    w = W.bits_to_float(want).astype(np.float64)
    n = np.abs(W.bits_to_float(normed).astype(np.float64))
    big = np.maximum(n[..., :64], n[..., 64:])
    big = np.concatenate([big, big], axis=-1)
    fin = np.isfinite(w)
    assert np.array_equal(np.isfinite(g), fin), f"{what}: finite pattern differs"
    err = np.abs(g - w)[fin]
    tol = (ulp(w) + ulp(big))[fin]
    assert (err <= tol).all(), f"{what}: {float((err / tol).max()):.2f} x the bound"
    assert (err != 0).mean() <= max_frac_off, f"{what}: {(err != 0).mean():.2e} of elements off"


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


def normed_ref(case):
    kp, vp = W.empty_pool_bf16(case.layout.num_pages, case.Hkv)
    nq, nk, _ = oracle.qkv_norm_rope_append(case.qkv, case.Hq, case.Hkv, case.q_w, case.k_w,
                                            1e-6, None, None, case.cu_new,
                                            case.layout.block_table, case.seq_lens, kp, vp)
    return nq, nk


@pytest.mark.parametrize("norm,rope", [(True, True), (True, False), (False, True)])
def test_small_batch_matches_oracle(pk, norm, rope):
    case = W.qkv_prep_case(90, [37, 5, 16], [37, 700, 130], Hq=32, Hkv=8)
    (q, k, v), (rq, rk, rv) = run(pk, case, norm, rope)
    if norm and rope:
        nq, nk = normed_ref(case)
        check_rotated(q, rq, nq, "q_out")
        check_rotated(k, rk, nk, "K pool")     # untouched slots: NaN sentinel on both sides
    elif not norm:
        # no norm: rotation of exact inputs, both sides round once
        assert_bits_equal(q, rq, "q_out rope only")
        assert_bits_equal(k, rk, "K pool rope only")
    else:
        check_bf16(q, rq, "q_out norm only")
        check_bf16(k, rk, "K pool norm only")
    assert np.array_equal(v, rv)


def test_no_norm_no_rope_is_the_plain_append_bit_for_bit(pk):
    case = W.qkv_prep_case(91, [20, 3], [100, 3], Hq=16, Hkv=8)
    (q, k, v), (rq, rk, rv) = run(pk, case, norm=False, rope=False)
    assert_bits_equal(q, rq, "q_out")
    assert_bits_equal(k, rk, "K pool")
    assert_bits_equal(v, rv, "V pool")


def test_prefill_chunk_size(pk):
    """A 2,048-token chunk of one sequence at positions 14,336 .. 16,383."""
    case = W.qkv_prep_case(92, [2048], [16384], Hq=32, Hkv=8)
    (q, k, v), (rq, rk, rv) = run(pk, case)
    nq, nk = normed_ref(case)
    check_rotated(q, rq, nq, "q_out chunk")
    check_rotated(k, rk, nk, "K pool chunk")
    assert np.array_equal(v, rv)


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
    (q, k, v), (rq, rk, rv) = run(pk, case)
    nq, nk = normed_ref(case)
    check_rotated(q, rq, nq, f"q_out {Hq}/{Hkv}")
    check_rotated(k, rk, nk, f"K pool {Hq}/{Hkv}")
    assert np.array_equal(v, rv)
    (q, k, v), (rq, rk, rv) = run(pk, case, norm=False, rope=True)
    assert_bits_equal(q, rq, f"q_out rope only {Hq}/{Hkv}")
    assert_bits_equal(k, rk, f"K pool rope only {Hq}/{Hkv}")
    assert_bits_equal(v, rv, f"V pool {Hq}/{Hkv}")
