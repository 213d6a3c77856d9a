"""paged_attn_decode on the GPU against the fp64 oracle, element by element
(TileInfer.jl "Performance" page: online softmax over the pages in place,
split-KV for decode plus a combine; "INT8 KV cache")."""
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


def gpu_decode(pk, case: W.DecodeCase, num_splits=0, int8_pools=None, smooth=None, fused=False):
    if int8_pools is None:
        pool = pk.Pool(dev_bf16(case.k_pool), dev_bf16(case.v_pool))
    else:
        pool = pk.Pool(*[dev(a) for a in int8_pools])
    out, lse = pk.paged_attn_decode(pool, dev_bf16(case.q), dev(case.layout.block_table),
                                    dev(case.seq_lens), int(case.seq_lens.max()), case.scale,
                                    k_smooth=dev(smooth) if smooth is not None else None,
                                    num_splits=num_splits, fused=fused)
    assert pk.poll_device_error() == pk.OK
    return out, lse


def oracle_decode(case: W.DecodeCase, rows=None, int8_pools=None, smooth=None):
    cu = np.arange(case.B + 1, dtype=np.int32)
    if int8_pools is None:
        return oracle.paged_attention(case.k_pool, case.v_pool, case.q, cu,
                                      case.layout.block_table, case.seq_lens, case.scale,
                                      rows=rows)
    k8, v8, ks, vs = int8_pools
    return oracle.paged_attention(k8, v8, case.q, cu, case.layout.block_table, case.seq_lens,
                                  case.scale, k_scale=ks, v_scale=vs, k_smooth=smooth, rows=rows)


@pytest.mark.parametrize("splits", [0, 1, 2, 3, 7, 64])
def test_single_sequence_1k(pk, splits):
    case = W.decode_1k()
    out, lse = gpu_decode(pk, case, splits)
    ro, rl = oracle_decode(case)
    check_out(out, ro, f"decode 1k splits={splits}")
    check_lse(lse, rl, f"decode 1k splits={splits}")


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_ragged_lengths_and_group_sizes(pk, G):
    rng = np.random.default_rng(30 + G)
    lens = [1, 15, 16, 17, 33, 100, 257, 1000, 63, 64, 65]
    case = W.decode_bf16(rng, lens, Hq=2 * G, Hkv=2)
    ro, rl = oracle_decode(case)
    for splits in (0, 1, 5):
        out, lse = gpu_decode(pk, case, splits)
        check_out(out, ro, f"G={G} splits={splits}")
        check_lse(lse, rl, f"G={G} splits={splits}")


def test_empty_context_row(pk):
    rng = np.random.default_rng(40)
    case = W.decode_bf16(rng, [0, 40, 0], Hq=8, Hkv=2)
    ro, rl = oracle_decode(case)
    for splits in (0, 1, 3):
        out, lse = gpu_decode(pk, case, splits)
        check_out(out, ro, "empty rows")
        check_lse(lse, rl, "empty rows")


def test_batched_decode_small(pk):
    case = W.batched_decode(B=8, lo=512, hi=2048)
    out, lse = gpu_decode(pk, case)
    ro, rl = oracle_decode(case)
    check_out(out, ro, "batched small")
    check_lse(lse, rl, "batched small")


def test_batched_decode_64_sequences_sampled(pk):
    """Full size (64 sequences, lengths 512..8192) in the bench's launch
    configuration; the oracle evaluates a seeded sample of 16 sequences."""
    case = W.batched_decode()
    out, lse = gpu_decode(pk, case)
    rows = np.sort(np.random.default_rng(41).choice(case.B, 16, replace=False)).astype(np.int32)
    ro, rl = oracle_decode(case, rows=rows)
    check_out(out[torch.from_numpy(rows).long().cuda()], ro, "batched full")
    check_lse(lse[torch.from_numpy(rows).long().cuda()], rl, "batched full")


def test_page_permutation_is_bit_identical(pk):
    rng = np.random.default_rng(42)
    case = W.decode_bf16(rng, [300, 77, 1024], Hq=32, Hkv=8)
    out1, lse1 = gpu_decode(pk, case)
    perm = rng.permutation(case.k_pool.shape[0])
    kp2 = np.empty_like(case.k_pool)
    vp2 = np.empty_like(case.v_pool)
    kp2[perm] = case.k_pool
    vp2[perm] = case.v_pool
    case2 = W.DecodeCase(case.Hq, case.Hkv, case.seq_lens,
                         W.Layout(case.layout.num_pages,
                                  perm[case.layout.block_table].astype(np.int32),
                                  int(perm[case.layout.sentinel_page])),
                         case.q, kp2, vp2)
    out2, lse2 = gpu_decode(pk, case2)
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


def int8_case(pk, B, smooth=True):
    """Fill an INT8 cache of B x 32,768 positions with kv_append, as the
    workload does, and return (decode case, int8 pools as numpy, w)."""
    app, q = W.int8_long_decode(B=B)
    w = app.k_smooth if smooth else None
    pool = pk.Pool.empty(app.layout.num_pages, app.Hkv, dtype=torch.int8)
    for t in (pool.k, pool.v):
        t.fill_(0x5A)
    for t in (pool.k_scale, pool.v_scale):
        t.fill_(float("nan"))
    pk.kv_append(pool, dev_bf16(app.k_new), dev_bf16(app.v_new), dev(app.cu_new),
                 dev(app.layout.block_table), dev(app.seq_lens),
                 k_smooth=dev(w) if w is not None else None)
    assert pk.poll_device_error() == pk.OK
    pools = tuple(t.cpu().numpy() for t in (pool.k, pool.v, pool.k_scale, pool.v_scale))
    case = W.DecodeCase(32, app.Hkv, app.seq_lens, app.layout, q, None, None)
    return case, pools, w


@pytest.mark.parametrize("smooth", [True, False])
def test_int8_32k_batch1(pk, smooth):
    case, pools, w = int8_case(pk, 1, smooth)
    ro, rl = oracle_decode(case, int8_pools=pools, smooth=w)
    for splits in (0, 1, 9):
        out, lse = gpu_decode(pk, case, splits, int8_pools=pools, smooth=w)
        check_out(out, ro, f"int8 32k smooth={smooth} splits={splits}")
        check_lse(lse, rl, f"int8 32k smooth={smooth} splits={splits}")


def test_int8_32k_batch8_sampled(pk):
    case, pools, w = int8_case(pk, 8, True)
    out, lse = gpu_decode(pk, case, int8_pools=pools, smooth=w)
    rows = np.array([0, 5], np.int32)
    ro, rl = oracle_decode(case, rows=rows, int8_pools=pools, smooth=w)
    idx = torch.from_numpy(rows).long().cuda()
    check_out(out[idx], ro, "int8 32k b8")
    check_lse(lse[idx], rl, "int8 32k b8")


def test_int8_key_smoothing_reduces_the_error_against_exact_attention(pk):
    """Keys whose channels carry scales w_c ~ U[0.5, 2] lose less to the INT8
    cache when they are quantised divided by w (the key smoothing of the
    "INT8 KV cache" section): at 32,768 positions the GPU's INT8 decode with
    smoothing is closer to the exact attention over the unquantised bf16
    keys and values (fp64 oracle) than without.  Both stay within the
    decode tolerance of it."""
    app, q = W.int8_long_decode(B=1)
    kp, vp = W.empty_pool_bf16(app.layout.num_pages, app.Hkv)
    kp, vp = oracle.kv_append_bf16(kp, vp, app.k_new, app.v_new, app.cu_new,
                                   app.layout.block_table, app.seq_lens)
    exact, _ = oracle_decode(W.DecodeCase(32, app.Hkv, app.seq_lens, app.layout, q, kp, vp))
    err = {}
    for smooth in (True, False):
        case, pools, w = int8_case(pk, 1, smooth)
        out, _ = gpu_decode(pk, case, int8_pools=pools, smooth=w)
        check_out(out, exact, f"int8 32k smooth={smooth} against unquantised K/V")
        o = out.float().cpu().numpy().astype(np.float64)
        err[smooth] = np.linalg.norm(o - exact) / np.linalg.norm(exact)
    assert err[True] < 0.95 * err[False], err


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_int8_group_sizes_ragged(pk, G):
    rng = np.random.default_rng(50 + G)
    lens = np.array([1, 17, 200, 513], np.int32)
    layout = W.scatter_pages(rng, lens)
    T = int(lens.sum())
    w = W.smoothing_weight(rng)
    app = W.AppendCase(2, W.cu_from_counts(lens), lens, layout,
                       W.keys_with_channel_weight(rng, (T, 2, W.HEAD_DIM), w),
                       W.normal_bf16(rng, (T, 2, W.HEAD_DIM)), k_smooth=w)
    pools = oracle.kv_append_int8(*W.empty_pool_int8(layout.num_pages, 2), app.k_new,
                                  app.v_new, app.cu_new, layout.block_table, lens, k_smooth=w)
    q = W.normal_bf16(rng, (4, 2 * G, W.HEAD_DIM))
    case = W.DecodeCase(2 * G, 2, lens, layout, q, None, None)
    ro, rl = oracle_decode(case, int8_pools=pools, smooth=w)
    for splits, fused in ((0, False), (3, False), (3, True), (1, False)):
        out, lse = gpu_decode(pk, case, splits, int8_pools=pools, smooth=w, fused=fused)
        check_out(out, ro, f"int8 G={G} splits={splits} fused={fused}")
        check_lse(lse, rl, f"int8 G={G} splits={splits} fused={fused}")


def test_fused_decode_workspace_reuse_is_exact():
    """The fused-merge decode: one workspace over a series of split calls
    gives the same bits as a fresh workspace per call and as the separate
    combine, and its part counters are zero after each call (the split that
    completes the count merges and resets it)."""
    from paged_kv_flash_gb300 import pagedkv as pk
    rng = np.random.default_rng(77)
    calls = []
    # batch 2, then 4, then 3: a later call may need more counters than an
    # earlier one wrote partials next to
    for lens in ([1, 4000], [3000, 17, 700, 2048], [5000, 5000, 5000]):
        case = W.decode_bf16(rng, np.array(lens, np.int32), 32, 8)
        pool = pk.Pool(dev_bf16(case.k_pool), dev_bf16(case.v_pool))
        args = (pool, dev_bf16(case.q), dev(case.layout.block_table), dev(case.seq_lens),
                int(max(lens)), case.scale)
        fresh = pk.paged_attn_decode(*args, num_splits=8, fused=True)
        assert pk.poll_device_error() == pk.OK
        sep = pk.paged_attn_decode(*args, num_splits=8)
        assert torch.equal(fresh[0], sep[0]) and torch.equal(fresh[1], sep[1])
        ro, rl = oracle.paged_attention(case.k_pool, case.v_pool, case.q,
                                        W.cu_from_counts([1] * len(lens)),
                                        case.layout.block_table, case.seq_lens, case.scale)
        check_out(fresh[0], ro, f"fused decode {lens}")
        check_lse(fresh[1], rl, f"fused decode {lens}")
        calls.append((args, fresh))
    plans = [pk.decode_plan(len(a[1]), 32, 8, a[4], 8) for a, _ in calls]
    ws = pk.decode_workspace(max(p[2] for p in plans), max(p[3] for p in plans))
    zero = max(p[3] for p in plans)
    for _ in range(2):
        for args, (o0, l0) in calls:
            o, l = pk.paged_attn_decode(*args, num_splits=8, workspace=ws, fused=True)
            assert torch.equal(o, o0) and torch.equal(l, l0)
            assert int(ws[:zero].count_nonzero()) == 0
    assert pk.poll_device_error() == pk.OK


def test_int8_empty_context_and_single_keys(pk):
    """INT8 rows with no cached position (out 0, lse -inf), one key, one page
    exactly, and one key into the next page, through the tensor-core path."""
    rng = np.random.default_rng(60)
    lens = np.array([0, 1, 16, 17], np.int32)
    layout = W.scatter_pages(rng, lens)
    T = int(lens.sum())
    w = W.smoothing_weight(rng)
    app = W.AppendCase(2, W.cu_from_counts(lens), lens, layout,
                       W.keys_with_channel_weight(rng, (T, 2, W.HEAD_DIM), w),
                       W.normal_bf16(rng, (T, 2, W.HEAD_DIM)), k_smooth=w)
    pools = oracle.kv_append_int8(*W.empty_pool_int8(layout.num_pages, 2), app.k_new,
                                  app.v_new, app.cu_new, layout.block_table, lens, k_smooth=w)
    q = W.normal_bf16(rng, (4, 8, W.HEAD_DIM))
    case = W.DecodeCase(8, 2, lens, layout, q, None, None)
    ro, rl = oracle_decode(case, int8_pools=pools, smooth=w)
    assert np.isneginf(rl[0]).all() and (ro[0] == 0).all()
    for splits in (0, 2):
        out, lse = gpu_decode(pk, case, splits, int8_pools=pools, smooth=w)
        check_out(out, ro, f"int8 edge splits={splits}")
        check_lse(lse, rl, f"int8 edge splits={splits}")


def scaled_bits(bits: np.ndarray, k: int) -> np.ndarray:
    """bf16 bit patterns of the values times 2^k (exact for these ranges:
    neither subnormal nor overflowing in bf16)."""
    x = W.bits_to_float(bits).astype(np.float64) * 2.0 ** k
    out = W.to_bf16_bits(x.astype(np.float32))
    assert np.array_equal(W.bits_to_float(out).astype(np.float64), x)
    return out


@pytest.mark.parametrize("k", [-16, 8])
def test_int8_decode_is_exact_under_power_of_two_v_scaling(pk, k):
    """V times 2^k gives the same INT8 codes and scales exactly 2^k times the
    originals (scale = max|v| / 127 and the quotient v / scale are exact
    under a power-of-two factor), so exact attention over the cache is 2^k
    times the unscaled one and the lse is unchanged ("INT8 KV cache" of the
    TileInfer.jl "Performance" page; the softmax weights do not depend on
    V).  The GPU output must follow at any V magnitude: at 2^-16 the
    products p * v_scale lie far below the smallest normal f16, at 2^8 far
    above the unit range.  The 32,768-position cache of the INT8 workload,
    batch 1, at the heuristic's split count and at 1 and 9 splits; the
    scaled output equals 2^k times the unscaled GPU output to a relative
    1e-2 per element, and matches the fp64 oracle within the decode
    tolerance once 2^k is divided out."""
    app, q = W.int8_long_decode(B=1)
    w = app.k_smooth
    outs = {}
    for kk in (0, k):
        v_new = app.v_new if kk == 0 else scaled_bits(app.v_new, kk)
        pool = pk.Pool.empty(app.layout.num_pages, app.Hkv, dtype=torch.int8)
        pk.kv_append(pool, dev_bf16(app.k_new), dev_bf16(v_new), dev(app.cu_new),
                     dev(app.layout.block_table), dev(app.seq_lens), k_smooth=dev(w))
        assert pk.poll_device_error() == pk.OK
        pools = tuple(t.cpu().numpy() for t in (pool.k, pool.v, pool.k_scale, pool.v_scale))
        case = W.DecodeCase(32, app.Hkv, app.seq_lens, app.layout, q, None, None)
        ro, rl = oracle_decode(case, int8_pools=pools, smooth=w)
        for splits in (0, 1, 9):
            out, lse = gpu_decode(pk, case, splits, int8_pools=pools, smooth=w)
            o = out.float().cpu().numpy().astype(np.float64) * 2.0 ** -kk
            check_out(torch.from_numpy(o), ro * 2.0 ** -kk,
                      f"int8 V x 2^{kk} splits={splits}, 2^{kk} divided out")
            check_lse(lse, rl, f"int8 V x 2^{kk} splits={splits}")
            outs[(kk, splits)] = (o, lse.cpu().numpy())
    for splits in (0, 1, 9):
        o0, l0 = outs[(0, splits)]
        ok, lk = outs[(k, splits)]
        rel = np.abs(ok - o0) / np.maximum(np.abs(o0), 1e-30)
        assert (rel <= 1e-2).all(), (k, splits, float(rel.max()))
        assert np.array_equal(l0, lk), (k, splits)
