"""Pins for the fp64 oracle, independent of the oracle's own code.

Each test checks the oracle against something the pages or the mathematics
fix -- closed forms, invariants, a library routine on special cases, brute
force on tiny inputs, hand-worked values -- chosen so that a dropped term, a
wrong index or sign, or a transposed operand fails at least one of them.

The method (TileInfer.jl "Performance" page, section "Fused kernels,
FlashAttention and PagedAttention"): softmax attention over pages read in
place through a block table; split-KV decode plus a combine; GQA heads.
INT8 cache: one scale per cached vector ("INT8 KV cache" section).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_flash_gb300 import workloads as W

D = W.HEAD_DIM
P = W.PAGE
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def make_pool_from_dense(rng, dense_k, dense_v, extra_pages=3):
    """Scatter dense per-sequence K/V ([L_b][Hkv][D] uint16 bits) into a pool
    through a random block table -- the inverse of the oracle's gather.
    Unused pages and slots hold NaN, so a wrong gather shows."""
    B = len(dense_k)
    Hkv = dense_k[0].shape[1]
    lens = np.array([k.shape[0] for k in dense_k], np.int32)
    npg = (lens + P - 1) // P
    num_pages = int(npg.sum()) + extra_pages
    perm = rng.permutation(num_pages)
    maxp = max(int(npg.max()), 1)
    bt = np.full((B, maxp), num_pages - 1, np.int32)
    kp = np.full((num_pages, Hkv, P, D), W.BF16_NAN, np.uint16)
    vp = kp.copy()
    off = 0
    for b in range(B):
        for j in range(npg[b]):
            bt[b, j] = perm[off]
            off += 1
        for p in range(lens[b]):
            kp[bt[b, p // P], :, p % P, :] = dense_k[b][p]
            vp[bt[b, p // P], :, p % P, :] = dense_v[b][p]
    return kp, vp, bt, lens


def f(bits):
    return W.bits_to_float(bits).astype(np.float64)


def decode_cu(B):
    return np.arange(B + 1, dtype=np.int32)


# ------------------------------------------------------------ closed forms

def test_single_key_returns_its_value_row():
    rng = np.random.default_rng(1)
    k = W.normal_bf16(rng, (1, 2, D))
    v = W.normal_bf16(rng, (1, 2, D))
    q = W.normal_bf16(rng, (1, 4, D))
    kp, vp, bt, lens = make_pool_from_dense(rng, [k], [v])
    s = 0.0883883
    out, lse = oracle.paged_attention(kp, vp, q, decode_cu(1), bt, lens, s)
    for h in range(4):
        hk = h // 2
        assert np.array_equal(out[0, h], f(v[0, hk]))           # exactly V
        dot = math.fsum(f(q[0, h]) * f(k[0, hk]))
        assert abs(lse[0, h] - s * dot) <= 1e-12 * max(1.0, abs(s * dot))


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(2)
    L = 37                                              # 3 pages, ragged tail
    k1 = W.normal_bf16(rng, (1, 1, D))
    k = np.repeat(k1, L, axis=0)
    v = W.normal_bf16(rng, (L, 1, D))
    q = W.normal_bf16(rng, (1, 3, D))
    kp, vp, bt, lens = make_pool_from_dense(rng, [k], [v])
    s = 1 / math.sqrt(D)
    out, lse = oracle.paged_attention(kp, vp, q, decode_cu(1), bt, lens, s)
    mean = f(v[:, 0]).mean(axis=0)
    for h in range(3):
        np.testing.assert_allclose(out[0, h], mean, rtol=0, atol=1e-13)
        dot = math.fsum(f(q[0, h]) * f(k1[0, 0]))
        assert abs(lse[0, h] - (s * dot + math.log(L))) < 1e-12


def test_zero_query_gives_uniform_weights():
    rng = np.random.default_rng(3)
    L = 50
    k = W.normal_bf16(rng, (L, 2, D))
    v = W.normal_bf16(rng, (L, 2, D))
    q = np.zeros((1, 2, D), np.uint16)                 # bf16 +0
    kp, vp, bt, lens = make_pool_from_dense(rng, [k], [v])
    out, lse = oracle.paged_attention(kp, vp, q, decode_cu(1), bt, lens, 0.125)
    for h in range(2):
        np.testing.assert_allclose(out[0, h], f(v[:, h]).mean(axis=0), rtol=0, atol=1e-13)
        assert abs(lse[0, h] - math.log(L)) < 1e-13


def test_two_keys_logistic_weight():
    rng = np.random.default_rng(4)
    k = W.normal_bf16(rng, (2, 1, D))
    v = W.normal_bf16(rng, (2, 1, D))
    q = W.normal_bf16(rng, (1, 1, D))
    kp, vp, bt, lens = make_pool_from_dense(rng, [k], [v])
    s = 0.3
    out, lse = oracle.paged_attention(kp, vp, q, decode_cu(1), bt, lens, s)
    s1 = s * math.fsum(f(q[0, 0]) * f(k[0, 0]))
    s2 = s * math.fsum(f(q[0, 0]) * f(k[1, 0]))
    w1 = 1.0 / (1.0 + math.exp(s2 - s1))
    np.testing.assert_allclose(out[0, 0], w1 * f(v[0, 0]) + (1 - w1) * f(v[1, 0]),
                               rtol=0, atol=1e-13)
    # lse of two terms: max + log1p(exp(-|s1 - s2|))
    assert abs(lse[0, 0] - (max(s1, s2) + math.log1p(math.exp(-abs(s1 - s2))))) < 1e-13


def test_gqa_grouping_is_consecutive():
    """V constant per KV head: query head h must return the constant of KV head h // G."""
    rng = np.random.default_rng(5)
    Hkv, G, L = 4, 3, 20
    consts = [1.0, -2.0, 0.5, 4.0]
    k = W.normal_bf16(rng, (L, Hkv, D))
    v = np.zeros((L, Hkv, D), np.uint16)
    for h in range(Hkv):
        v[:, h, :] = W.to_bf16_bits(np.full(D, consts[h], np.float32))
    q = W.normal_bf16(rng, (1, Hkv * G, D))
    kp, vp, bt, lens = make_pool_from_dense(rng, [k], [v])
    out, _ = oracle.paged_attention(kp, vp, q, decode_cu(1), bt, lens, 0.1)
    for hq in range(Hkv * G):
        np.testing.assert_allclose(out[0, hq], consts[hq // G], rtol=0, atol=1e-13)


# ------------------------------------------------------------- invariants

def test_page_permutation_leaves_output_bit_identical():
    rng = np.random.default_rng(6)
    case = W.decode_bf16(rng, [40, 71, 16, 1], Hq=4, Hkv=2)
    cu = decode_cu(case.B)
    out1, lse1 = oracle.paged_attention(case.k_pool, case.v_pool, case.q, cu,
                                        case.layout.block_table, case.seq_lens, case.scale)
    perm = rng.permutation(case.k_pool.shape[0])       # physical page p moves to perm[p]
    kp2 = np.empty_like(case.k_pool)
    vp2 = np.empty_like(case.v_pool)
    kp2[perm] = case.k_pool
    vp2[perm] = case.v_pool
    bt2 = perm[case.layout.block_table].astype(np.int32)
    out2, lse2 = oracle.paged_attention(kp2, vp2, case.q, cu, bt2, case.seq_lens, case.scale)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)


@pytest.mark.parametrize("S", [1, 2, 3, 7, "pages"])
def test_split_plus_combine_equals_unsplit(S):
    rng = np.random.default_rng(7)
    case = W.decode_bf16(rng, [200, 33, 16, 97], Hq=8, Hkv=2)
    cu = decode_cu(case.B)
    args = (case.k_pool, case.v_pool, case.q, cu, case.layout.block_table, case.seq_lens,
            case.scale)
    ref, lref = oracle.paged_attention(*args)
    nsplit = int((case.seq_lens.max() + P - 1) // P) if S == "pages" else S
    out, lse = oracle.paged_attention(*args, num_splits=nsplit)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lref, rtol=0, atol=1e-12)


def test_keys_after_the_causal_edge_do_not_matter():
    rng = np.random.default_rng(8)
    L, qlen = 45, 12
    k = W.normal_bf16(rng, (L, 2, D))
    v = W.normal_bf16(rng, (L, 2, D))
    q = W.normal_bf16(rng, (qlen, 4, D))
    kp, vp, bt, lens = make_pool_from_dense(rng, [k], [v])
    cu = np.array([0, qlen], np.int32)
    out1, lse1 = oracle.paged_attention(kp, vp, q, cu, bt, lens, 0.09)
    # change K/V at positions > pos(row 5) = L - qlen + 5
    edge = L - qlen + 5
    k2, v2 = k.copy(), v.copy()
    k2[edge + 1:] = W.normal_bf16(rng, k2[edge + 1:].shape)
    v2[edge + 1:] = W.normal_bf16(rng, v2[edge + 1:].shape)
    kp2, vp2 = kp.copy(), vp.copy()
    for p in range(L):
        kp2[bt[0, p // P], :, p % P] = k2[p]
        vp2[bt[0, p // P], :, p % P] = v2[p]
    out2, lse2 = oracle.paged_attention(kp2, vp2, q, cu, bt, lens, 0.09)
    assert np.array_equal(out1[:6], out2[:6]) and np.array_equal(lse1[:6], lse2[:6])
    assert not np.array_equal(out1[6:], out2[6:])


# ------------------------------------------------ library routine: SDPA

def _sdpa_reference(q, k, v, scale, qlen, L, G):
    """torch's scaled_dot_product_attention in float64 with a bottom-right
    causal mask, GQA by repeating KV heads; lse via torch.logsumexp."""
    return _sdpa_f64(f(q), f(k), f(v), scale, qlen, L, G)


def _sdpa_f64(q, k, v, scale, qlen, L, G):
    """_sdpa_reference on float64 arrays q [qlen][Hq][D], k, v [L][Hkv][D]."""
    qt = torch.from_numpy(q).permute(1, 0, 2)                     # [Hq][qlen][D]
    kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(G, dim=0)
    vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(G, dim=0)
    i = torch.arange(qlen)[:, None]
    j = torch.arange(L)[None, :]
    mask = j <= (L - qlen + i)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask,
                                                         scale=scale)
    scores = (qt @ kt.transpose(1, 2)) * scale
    lse = torch.logsumexp(scores.masked_fill(~mask, float("-inf")), dim=-1)
    return o.permute(1, 0, 2).numpy(), lse.permute(1, 0).numpy()


@pytest.mark.parametrize("shape", [[(5, 37), (40, 40), (1, 1), (17, 33)],
                                   [(16, 16), (3, 70)]])
def test_causal_prefill_matches_sdpa(shape):
    rng = np.random.default_rng(9)
    Hkv, G = 2, 3
    ks, vs, qs = [], [], []
    for qlen, L in shape:
        ks.append(W.normal_bf16(rng, (L, Hkv, D)))
        vs.append(W.normal_bf16(rng, (L, Hkv, D)))
        qs.append(W.normal_bf16(rng, (qlen, Hkv * G, D)))
    kp, vp, bt, lens = make_pool_from_dense(rng, ks, vs)
    cu = W.cu_from_counts([s[0] for s in shape])
    scale = 1 / math.sqrt(D)
    out, lse = oracle.paged_attention(kp, vp, np.concatenate(qs), cu, bt, lens, scale)
    for b, (qlen, L) in enumerate(shape):
        ro, rl = _sdpa_reference(qs[b], ks[b], vs[b], scale, qlen, L, G)
        np.testing.assert_allclose(out[cu[b]:cu[b + 1]], ro, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[cu[b]:cu[b + 1]], rl, rtol=0, atol=1e-12)


def _int8_cache(rng, shape, Hkv, G, w):
    """Sequences (qlen, L) of N(0,1) bf16 keys and values quantised into an
    INT8 cache by the oracle's append (key smoothing w, or None); returns the
    pools, scales, layout, queries and the bf16 inputs."""
    ks = [W.normal_bf16(rng, (L, Hkv, D)) for _, L in shape]
    vs = [W.normal_bf16(rng, (L, Hkv, D)) for _, L in shape]
    qs = np.concatenate([W.normal_bf16(rng, (qlen, Hkv * G, D)) for qlen, _ in shape])
    kp, _, bt, lens = make_pool_from_dense(rng, ks, vs)
    k8, v8, kscale, vscale = W.empty_pool_int8(kp.shape[0], Hkv)
    k8, v8, kscale, vscale = oracle.kv_append_int8(
        k8, v8, kscale, vscale, np.concatenate(ks), np.concatenate(vs),
        W.cu_from_counts([L for _, L in shape]), bt, lens, k_smooth=w)
    return k8, v8, kscale, vscale, bt, lens, qs


def test_int8_attention_matches_sdpa_on_the_dequantised_cache():
    """Causal rows over an INT8 cache with per-vector scales and key
    smoothing equal torch's SDPA in float64 on the dequantised vectors, key
    = code * scale * w and value = code * scale: each scale and the smoothing
    weight enter once, on their own operand."""
    rng = np.random.default_rng(31)
    Hkv, G = 2, 2
    shape = [(3, 45), (1, 20), (16, 16)]
    w = rng.uniform(0.5, 2.0, D).astype(np.float32)
    k8, v8, kscale, vscale, bt, lens, q = _int8_cache(rng, shape, Hkv, G, w)
    cu = W.cu_from_counts([qlen for qlen, _ in shape])
    scale = 1 / math.sqrt(D)
    out, lse = oracle.paged_attention(k8, v8, q, cu, bt, lens, scale, k_scale=kscale,
                                      v_scale=vscale, k_smooth=w)
    for b, (qlen, L) in enumerate(shape):
        pg, sl = bt[b, np.arange(L) // P], np.arange(L) % P
        kd = (k8[pg, :, sl].astype(np.float64) * kscale[pg, :, sl][:, :, None].astype(np.float64)
              * w.astype(np.float64))
        vd = v8[pg, :, sl].astype(np.float64) * vscale[pg, :, sl][:, :, None].astype(np.float64)
        ro, rl = _sdpa_f64(f(q[cu[b]:cu[b + 1]]), kd, vd, scale, qlen, L, G)
        np.testing.assert_allclose(out[cu[b]:cu[b + 1]], ro, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[cu[b]:cu[b + 1]], rl, rtol=0, atol=1e-12)


@pytest.mark.parametrize("S", [2, 5, 13])
def test_int8_split_plus_combine_equals_unsplit(S):
    rng = np.random.default_rng(32)
    Hkv, G = 2, 4
    shape = [(1, 200), (1, 33), (1, 16), (1, 97)]
    w = rng.uniform(0.5, 2.0, D).astype(np.float32)
    k8, v8, kscale, vscale, bt, lens, q = _int8_cache(rng, shape, Hkv, G, w)
    args = (k8, v8, q, decode_cu(len(shape)), bt, lens, 1 / math.sqrt(D))
    kw = dict(k_scale=kscale, v_scale=vscale, k_smooth=w)
    ref, lref = oracle.paged_attention(*args, **kw)
    out, lse = oracle.paged_attention(*args, num_splits=S, **kw)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lref, rtol=0, atol=1e-12)


def test_row_subset_matches_full_evaluation():
    rng = np.random.default_rng(10)
    case = W.decode_bf16(rng, [30, 64, 5], Hq=4, Hkv=4)
    cu = decode_cu(case.B)
    args = (case.k_pool, case.v_pool, case.q, cu, case.layout.block_table, case.seq_lens,
            case.scale)
    full, lfull = oracle.paged_attention(*args)
    sub, lsub = oracle.paged_attention(*args, rows=[2, 0])
    assert np.array_equal(sub, full[[2, 0]]) and np.array_equal(lsub, lfull[[2, 0]])


def test_empty_context_gives_zero_and_minus_inf():
    rng = np.random.default_rng(11)
    case = W.decode_bf16(rng, [0, 9], Hq=2, Hkv=1)
    out, lse = oracle.paged_attention(case.k_pool, case.v_pool, case.q, decode_cu(2),
                                      case.layout.block_table, case.seq_lens, case.scale)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(out[1]))


# ----------------------------------------------------------------- INT8

def _golden_cases():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "int8_half_even.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("case "):
                cur = {"name": line[5:]}
                cases.append(cur)
            else:
                key, vals = line.split(":", 1)
                cur[key] = [float(x) for x in vals.split()]
    return cases


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_int8_golden_vectors(case):
    x = np.zeros(D, np.float32)
    x[:len(case["x"])] = case["x"]
    bits = W.to_bf16_bits(x)
    assert np.array_equal(W.bits_to_float(bits), x)     # exactly representable
    w = None
    if "w" in case:
        w = np.ones(D, np.float32)
        w[:len(case["w"])] = case["w"]
    codes, scale = oracle.quantize_row_int8(bits, w)
    assert scale == np.float32(case["scale"][0])
    exp = np.zeros(D, np.int8)
    exp[:len(case["codes"])] = np.array(case["codes"], np.int8)
    assert np.array_equal(codes, exp)


def test_int8_random_vectors_match_numpy_float32_ieee():
    """numpy's float32 division is IEEE round-to-nearest and np.rint rounds
    half to even: the same fp32 steps, from an independent library."""
    rng = np.random.default_rng(12)
    for trial in range(200):
        x = W.normal_bf16(rng, (D,))
        w = W.smoothing_weight(rng) if trial % 2 else None
        codes, scale = oracle.quantize_row_int8(x, w)
        xf = W.bits_to_float(x)
        if w is not None:
            xf = (xf / w).astype(np.float32)
        amax = np.float32(np.max(np.abs(xf)))
        s = np.float32(amax / np.float32(127.0))
        assert scale.view(np.uint32) == s.view(np.uint32)
        ref = np.clip(np.rint((xf / s).astype(np.float32)), -127, 127).astype(np.int8)
        assert np.array_equal(codes, ref)
        assert np.abs(codes.astype(np.int32)).max() == 127       # amax maps to +-127


def test_int8_requantising_dequantised_codes_is_idempotent():
    rng = np.random.default_rng(13)
    for _ in range(100):
        x = W.normal_bf16(rng, (D,))
        codes, scale = oracle.quantize_row_int8(x)
        xd = (codes.astype(np.float32) * scale)
        xb = W.to_bf16_bits(xd)
        # dequantised values rounded back to bf16 keep their codes
        codes2, _ = oracle.quantize_row_int8(xb)
        assert np.array_equal(codes, codes2)


def test_int8_cache_with_exact_codes_equals_bf16_cache():
    """K/V chosen so that quantisation is exact (integer entries, max|x| = 127,
    power-of-two smoothing weights): the INT8 attention must equal the bf16
    attention bit for bit, which pins the dequantisation (code * scale * w)."""
    rng = np.random.default_rng(14)
    Hkv, G, L = 2, 2, 35
    w = rng.choice([0.5, 1.0, 2.0], D).astype(np.float32)
    xk = rng.integers(-127, 128, (L, Hkv, D)).astype(np.float32)
    xk[:, :, 0] = 127.0
    xv = rng.integers(-127, 128, (L, Hkv, D)).astype(np.float32)
    xv[:, :, 1] = -127.0
    kb = W.to_bf16_bits(xk * w)            # k = x * w, so k / w = x exactly
    vb = W.to_bf16_bits(xv)
    q = W.normal_bf16(rng, (1, Hkv * G, D))
    kp, vp, bt, lens = make_pool_from_dense(rng, [kb], [vb])
    cu_new = np.array([0, L], np.int32)
    k8, v8, ks, vs = W.empty_pool_int8(kp.shape[0], Hkv)
    k8, v8, ks, vs = oracle.kv_append_int8(k8, v8, ks, vs, kb, vb, cu_new, bt, lens, k_smooth=w)
    for p in range(L):
        assert np.all(ks[bt[0, p // P], :, p % P] == 1.0)
        assert np.all(vs[bt[0, p // P], :, p % P] == 1.0)
    o_bf, l_bf = oracle.paged_attention(kp, vp, q, decode_cu(1), bt, lens, 0.1)
    o_i8, l_i8 = oracle.paged_attention(k8, v8, q, decode_cu(1), bt, lens, 0.1,
                                        k_scale=ks, v_scale=vs, k_smooth=w)
    assert np.array_equal(o_bf, o_i8) and np.array_equal(l_bf, l_i8)


# ----------------------------------------------------------------- appends

def test_bf16_append_writes_exactly_the_named_slots():
    rng = np.random.default_rng(15)
    Hkv = 3
    lens_before = np.array([0, 14, 31], np.int32)
    n_new = np.array([20, 5, 1], np.int32)
    lens = lens_before + n_new
    layout = W.scatter_pages(rng, lens)
    kp, vp = W.empty_pool_bf16(layout.num_pages, Hkv)
    T = int(n_new.sum())
    k_new = W.normal_bf16(rng, (T, Hkv, D))
    v_new = W.normal_bf16(rng, (T, Hkv, D))
    cu = W.cu_from_counts(n_new)
    k2, v2 = oracle.kv_append_bf16(kp, vp, k_new, v_new, cu, layout.block_table, lens)
    touched = np.zeros(kp.shape[:3], bool)
    for b in range(3):
        for i in range(n_new[b]):
            p = lens_before[b] + i
            page = layout.block_table[b, p // P]
            assert np.array_equal(k2[page, :, p % P], k_new[cu[b] + i])
            assert np.array_equal(v2[page, :, p % P], v_new[cu[b] + i])
            touched[page, :, p % P] = True
    assert np.all(k2[~touched] == W.BF16_NAN) and np.all(v2[~touched] == W.BF16_NAN)


def test_int8_append_rows_are_quantised_rows():
    rng = np.random.default_rng(16)
    Hkv = 2
    lens = np.array([19], np.int32)
    layout = W.scatter_pages(rng, lens)
    w = W.smoothing_weight(rng)
    k_new = W.keys_with_channel_weight(rng, (19, Hkv, D), w)
    v_new = W.normal_bf16(rng, (19, Hkv, D))
    k8, v8, ks, vs = W.empty_pool_int8(layout.num_pages, Hkv)
    k8, v8, ks, vs = oracle.kv_append_int8(k8, v8, ks, vs, k_new, v_new,
                                           W.cu_from_counts([19]), layout.block_table, lens,
                                           k_smooth=w)
    touched = np.zeros(k8.shape[:3], bool)
    for p in range(19):
        page = layout.block_table[0, p // P]
        for h in range(Hkv):
            ck, sk = oracle.quantize_row_int8(k_new[p, h], w)
            cv, sv = oracle.quantize_row_int8(v_new[p, h])
            assert np.array_equal(k8[page, h, p % P], ck) and ks[page, h, p % P] == sk
            assert np.array_equal(v8[page, h, p % P], cv) and vs[page, h, p % P] == sv
            touched[page, h, p % P] = True
    assert np.all(np.isnan(ks[~touched])) and np.all(k8[~touched] == 0x5A)


# ------------------------------------------------ fused attention inputs

def _bits(vals):
    return np.asarray(W.to_bf16_bits(np.asarray(vals, np.float32)), np.uint16).reshape(-1)


def _one_token_case(D, x, Hq=1, Hkv=1):
    """One token of one sequence at position 0: qkv rows q = x, k = x, v = x."""
    qkv = np.stack([np.stack([x] * (Hq + 2 * Hkv))])            # [1][H][D]
    kp = np.full((2, Hkv, P, D), W.BF16_NAN, np.uint16)
    vp = kp.copy()
    return qkv, kp, vp, np.array([0, 1], np.int32), np.array([[1]], np.int32), \
        np.array([1], np.int32)


def test_bf16_rounding_ties_to_even_and_subnormals():
    assert oracle.bf16_from_double(1.0) == 0x3F80
    assert oracle.bf16_from_double(1 + 2 ** -8) == 0x3F80        # tie -> even
    assert oracle.bf16_from_double(1 + 3 * 2 ** -8) == 0x3F82    # tie -> even
    assert oracle.bf16_from_double(1 + 2 ** -8 + 2 ** -30) == 0x3F81
    assert oracle.bf16_from_double(-2.5) == 0xC020
    assert oracle.bf16_from_double(2 ** -133) == 0x0001          # smallest subnormal
    assert oracle.bf16_from_double(3.4e38) == 0x7F80             # past the largest finite
    # against torch's bf16 conversion on a spread of exactly-fp32 values
    rng = np.random.default_rng(11)
    v = (rng.standard_normal(4000) * np.exp2(rng.integers(-40, 40, 4000))).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([oracle.bf16_from_double(float(t)) for t in v], np.uint16)
    assert np.array_equal(got, ref)
    # around the smallest normal (2^-126) and through the subnormals
    v = (rng.uniform(1.0, 2.0, 2000) * np.exp2(rng.integers(-134, -120, 2000))).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([oracle.bf16_from_double(float(t)) for t in v], np.uint16)
    assert np.array_equal(got, ref)


def _golden_rows():
    with open(os.path.join(GOLDEN, "qkv_norm_rope_d4.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = [np.array([float(t) for t in p.split()]) for p in line.split("|")]
            yield parts


@pytest.mark.parametrize("row", list(range(4)))
def test_norm_rope_golden_d4(row):
    x, w, c, s, want = list(_golden_rows())[row]
    D = 4
    qkv, kp, vp, cu, bt, sl = _one_token_case(D, _bits(x))
    q, k, v = oracle.qkv_norm_rope_append(qkv, 1, 1, w.astype(np.float32), w.astype(np.float32),
                                          0.0, c[None].astype(np.float32),
                                          s[None].astype(np.float32), cu, bt, sl, kp, vp)
    assert np.array_equal(q[0, 0], _bits(want))
    assert np.array_equal(k[bt[0, 0], 0, 0], _bits(want))       # K gets the same steps
    assert np.array_equal(v[bt[0, 0], 0, 0], _bits(x))          # V is copied


def test_no_norm_no_rope_is_the_plain_append():
    rng = np.random.default_rng(12)
    Hq, Hkv = 4, 2
    lens, news = np.array([37, 5], np.int32), np.array([7, 5], np.int32)
    lay = W.scatter_pages(rng, lens)
    T = int(news.sum())
    qkv = W.normal_bf16(rng, (T, Hq + 2 * Hkv, D))
    kp, vp = W.empty_pool_bf16(lay.num_pages, Hkv)
    cu = W.cu_from_counts(news)
    q, k, v = oracle.qkv_norm_rope_append(qkv, Hq, Hkv, None, None, 0.0, None, None, cu,
                                          lay.block_table, lens, kp, vp)
    assert np.array_equal(q, qkv[:, :Hq])
    k2, v2 = oracle.kv_append_bf16(kp, vp, qkv[:, Hq:Hq + Hkv], qkv[:, Hq + Hkv:], cu,
                                   lay.block_table, lens)
    assert np.array_equal(k, k2) and np.array_equal(v, v2)


def test_rmsnorm_is_scale_free_and_unit_rms():
    rng = np.random.default_rng(13)
    x = W.normal_bf16(rng, (D,))
    x2 = _bits(2.0 * W.bits_to_float(x))                        # exact doubling
    ones = np.ones(D, np.float32)
    outs = []
    for xx in (x, x2):
        qkv, kp, vp, cu, bt, sl = _one_token_case(D, xx)
        q, _, _ = oracle.qkv_norm_rope_append(qkv, 1, 1, ones, ones, 0.0, None, None, cu, bt,
                                              sl, kp, vp)
        outs.append(q[0, 0])
    assert np.array_equal(outs[0], outs[1])
    n = W.bits_to_float(outs[0]).astype(np.float64)
    assert abs(np.mean(n * n) - 1.0) < 4 * 2.0 ** -8             # unit RMS up to bf16 rounding
    # the weight multiplies channel by channel
    w = rng.uniform(0.5, 2.0, D).astype(np.float32)
    qkv, kp, vp, cu, bt, sl = _one_token_case(D, x)
    qw, _, _ = oracle.qkv_norm_rope_append(qkv, 1, 1, w, w, 0.0, None, None, cu, bt, sl, kp, vp)
    assert np.allclose(W.bits_to_float(qw[0, 0]), n * w, rtol=2 * 2.0 ** -8, atol=0)


def _rope_table(max_pos, base=1.0e6):
    inv = base ** (-np.arange(0, D, 2, dtype=np.float64) / D)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def test_rope_rotates_pairs_and_keeps_relative_position():
    rng = np.random.default_rng(14)
    cos_t, sin_t = _rope_table(64)
    q0, k0 = W.normal_bf16(rng, (D,)), W.normal_bf16(rng, (D,))

    def rot(x, p):
        qkv, kp, vp, _, bt, _ = _one_token_case(D, x)
        sl = np.array([p + 1], np.int32)
        bt = np.zeros((1, 8), np.int32)
        bt[0, p // P] = 1
        q, _, _ = oracle.qkv_norm_rope_append(qkv, 1, 1, None, None, 0.0, cos_t, sin_t,
                                              np.array([0, 1], np.int32), bt, sl, kp, vp)
        return W.bits_to_float(q[0, 0]).astype(np.float64)

    # position 0 is the identity
    assert np.array_equal(rot(q0, 0), W.bits_to_float(q0).astype(np.float64))
    # each (i, i + D/2) pair keeps its length
    x = W.bits_to_float(q0).astype(np.float64)
    r = rot(q0, 37)
    half = D // 2
    assert np.allclose(np.hypot(r[:half], r[half:]), np.hypot(x[:half], x[half:]),
                       rtol=3 * 2.0 ** -8, atol=1e-6)
    # <rot(q, m), rot(k, n)> depends only on m - n
    dots = [rot(q0, m) @ rot(k0, m - 5) for m in (5, 20, 50)]
    assert np.allclose(dots, dots[0], rtol=0, atol=0.05 * np.sqrt(D))
    # ... and does change with m - n
    assert abs(rot(q0, 40) @ rot(k0, 0) - dots[0]) > 0.05 * np.sqrt(D)


def test_rope_quarter_turn_swaps_halves_exactly():
    rng = np.random.default_rng(15)
    x = W.normal_bf16(rng, (D,))
    cos_t = np.zeros((1, D // 2), np.float32)
    sin_t = np.ones((1, D // 2), np.float32)
    qkv, kp, vp, cu, bt, sl = _one_token_case(D, x)
    q, _, _ = oracle.qkv_norm_rope_append(qkv, 1, 1, None, None, 0.0, cos_t, sin_t, cu, bt, sl,
                                          kp, vp)
    xf = W.bits_to_float(x)
    half = D // 2
    want = np.concatenate([-xf[half:], xf[:half]])
    assert np.array_equal(W.bits_to_float(q[0, 0]), want)


def test_q_and_k_take_their_own_weights():
    rng = np.random.default_rng(16)
    x = W.normal_bf16(rng, (D,))
    qw = np.full(D, 1.0, np.float32)
    kw = np.full(D, 0.5, np.float32)
    qkv, kp, vp, cu, bt, sl = _one_token_case(D, x)
    q, k, _ = oracle.qkv_norm_rope_append(qkv, 1, 1, qw, kw, 0.0, None, None, cu, bt, sl, kp, vp)
    qf = W.bits_to_float(q[0, 0])
    kf = W.bits_to_float(k[bt[0, 0], 0, 0])
    assert np.array_equal(kf, qf * np.float32(0.5))      # halving is exact in bf16


def _nearest_float_to_rsqrt(z):
    """Brute force in exact rational arithmetic: among the floats around
    1/sqrt(z), the one whose rounding interval (the midpoints with its two
    neighbours) holds 1/sqrt(z); y lies above a midpoint m iff m^2 z < 1."""
    from fractions import Fraction
    zq = Fraction(float(z))
    r = np.float32(1.0 / np.sqrt(np.float64(z)))
    down, up = np.float32(0), np.float32(np.inf)
    cands = [np.nextafter(np.nextafter(r, down), down), np.nextafter(r, down), r,
             np.nextafter(r, up), np.nextafter(np.nextafter(r, up), up)]
    for c in cands:
        cq = Fraction(float(c))
        lo = (Fraction(float(np.nextafter(c, down))) + cq) / 2
        hi = (Fraction(float(np.nextafter(c, up))) + cq) / 2
        if lo * lo * zq <= 1 <= hi * hi * zq:
            return np.float32(c)
    raise AssertionError(f"no candidate for z = {float(z)}")


def test_rsqrt_rn_is_the_nearest_float():
    """The RMSNorm's reciprocal square root (fused attention inputs, TileInfer.jl
    "Performance" page, "Fused kernels, FlashAttention and PagedAttention":
    the chain's fp32 norm) is the correctly rounded 1/sqrt(z): checked in
    exact rational arithmetic on seeded floats spread over the normal range,
    on both sides of powers of two, and on powers of four (exact results)."""
    rng = np.random.default_rng(5)
    zs = list((rng.uniform(0.5, 1.0, 300) * np.exp2(rng.integers(-120, 120, 300)))
              .astype(np.float32))
    for e in range(-60, 61, 7):
        p = np.float32(2.0 ** e)
        zs += [p, np.nextafter(p, np.float32(0)), np.nextafter(p, np.float32(np.inf))]
    zs += [np.float32(x) for x in (1.0, 6.25, 3.0, 1e-6, 1.0 + 1e-6)]
    for z in zs:
        got, want = oracle.rsqrt_rn(z), _nearest_float_to_rsqrt(z)
        assert got == want, (float(z), float(got), float(want))
    for k in range(-30, 31):
        assert oracle.rsqrt_rn(np.float32(4.0 ** k)) == np.float32(2.0 ** -k)


def test_norm_mean_square_rounds_once_from_the_exact_sum():
    """The RMSNorm's mean square is the exact sum of squares rounded once to
    fp32.  x = (2, 2^-11, 2^-23, 0), D = 4: the squares sum to 4 + 2^-22 +
    2^-46, so the mean 1 + 2^-24 + 2^-48 lies just above the midpoint of 1
    and 1 + 2^-23 and rounds up; r = 1/sqrt(1 + 2^-23) rounds to 1 - 2^-24.
    (A running fp32 sum ties 4 + 2^-22 to 4 and gives r = 1.)  The weight
    w0 = 1 + 3 * 2^-8 puts 2 r w0 next to the bf16 tie 2 + 3 * 2^-7: with
    r = 1 - 2^-24 the fp32 product 2 + 3 * 2^-7 - 2^-22 rounds down to
    2.015625 (r = 1 would tie to even, 2.03125)."""
    D = 4
    x = np.array([2.0, 2.0 ** -11, 2.0 ** -23, 0.0], np.float32)
    w = np.array([1.0 + 3 * 2.0 ** -8, 1.0, 1.0, 1.0], np.float32)
    assert oracle.rsqrt_rn(np.float32(1.0 + 2.0 ** -23)) == np.float32(1.0 - 2.0 ** -24)
    qkv, kp, vp, cu, bt, sl = _one_token_case(D, _bits(x))
    q, _, _ = oracle.qkv_norm_rope_append(qkv, 1, 1, w, w, 0.0, None, None, cu, bt, sl, kp, vp)
    assert W.bits_to_float(q[0, 0])[0] == np.float32(2.015625)
