"""Host-only checks of the C ABI: the library builds and loads, exports every
symbol include/pagedkv.h declares, and rejects bad arguments before any
launch (no GPU needed: these paths never reach the device)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_flash_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "pagedkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_three_calls():
    syms = declared_symbols()
    for name in ("pkv_kv_append", "pkv_paged_attn_decode", "pkv_paged_attn_prefill"):
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), f"{name} not exported"


def test_binding_covers_every_declared_symbol():
    import importlib.util
    spec = importlib.util.find_spec("paged_kv_flash_gb300.pagedkv")
    src = open(spec.origin).read()
    for name in declared_symbols():
        assert f'"{name}"' in src, f"{name} has no binding signature"


class Pool(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("num_pages", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


FAKE = 1 << 20          # a non-null, 256-aligned address that is never dereferenced


def good_pool(**kw):
    p = dict(k=FAKE, v=FAKE * 2, k_scale=None, v_scale=None, num_pages=4, num_kv_heads=2,
             page_size=16, head_dim=128, dtype=0)
    p.update(kw)
    return Pool(**p)


def decode(lib, pool, **kw):
    a = dict(q=FAKE, B=1, Hq=4, bt=FAKE, max_pages=4, sl=FAKE, max_seq_len=64, scale=0.1,
             smooth=None, splits=0, ws=None, ws_bytes=0, out=FAKE, lse=None)
    a.update(kw)
    f = lib.pkv_paged_attn_decode
    f.restype = ctypes.c_int32
    return f(ctypes.byref(pool), ctypes.c_void_p(a["q"]), a["B"], a["Hq"],
             ctypes.c_void_p(a["bt"]), a["max_pages"], ctypes.c_void_p(a["sl"]),
             a["max_seq_len"], ctypes.c_float(a["scale"]), ctypes.c_void_p(a["smooth"]),
             a["splits"], ctypes.c_void_p(a["ws"]), ctypes.c_size_t(a["ws_bytes"]),
             ctypes.c_void_p(a["out"]), ctypes.c_void_p(a["lse"]), None)


INVALID, UNSUPPORTED = -1, -2


@pytest.mark.parametrize("bad", [dict(head_dim=64), dict(page_size=32), dict(num_kv_heads=0),
                                 dict(k=None), dict(k=FAKE + 8), dict(dtype=7),
                                 dict(k_scale=FAKE), dict(dtype=1)])
def test_decode_rejects_bad_pool(lib, bad):
    assert decode(lib, good_pool(**bad)) == INVALID


@pytest.mark.parametrize("bad", [dict(Hq=3), dict(q=None), dict(out=None), dict(B=-1),
                                 dict(max_seq_len=65), dict(scale=float("nan")),
                                 dict(splits=-2), dict(smooth=FAKE)])
def test_decode_rejects_bad_arguments(lib, bad):
    assert decode(lib, good_pool(), **bad) == INVALID


def test_decode_rejects_short_workspace(lib):
    # four splits of one page each need a workspace; none given
    assert decode(lib, good_pool(), splits=4) == INVALID
    s, c, w, z = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.pkv_decode_plan(1, 4, 2, 64, 0, 4, ctypes.byref(s), ctypes.byref(c),
                               ctypes.byref(w), ctypes.byref(z)) == 0
    assert (s.value, c.value) == (4, 1) and w.value > 0
    assert z.value == 65536 * 4                 # fixed counter region
    assert decode(lib, good_pool(), splits=4, ws=FAKE, ws_bytes=w.value - 1) == INVALID
    assert decode(lib, good_pool(), splits=4, ws=FAKE + 16, ws_bytes=w.value) == INVALID


def test_forced_split_beyond_counter_region_is_rejected(lib):
    s, c, w, z = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_size_t(), ctypes.c_size_t()
    # 8,193 sequences x 8 KV heads > 65,536 counters
    assert lib.pkv_decode_plan(8193, 32, 8, 4096, 0, 4, ctypes.byref(s), ctypes.byref(c),
                               ctypes.byref(w), ctypes.byref(z)) == INVALID
    # the heuristic does not split them
    assert lib.pkv_decode_plan(8193, 32, 8, 4096, 0, 0, ctypes.byref(s), ctypes.byref(c),
                               ctypes.byref(w), ctypes.byref(z)) == 0
    assert s.value == 1 and w.value == 0 and z.value == 0


def test_decode_unsupported_group_size(lib):
    assert decode(lib, good_pool(num_kv_heads=1), Hq=3) == UNSUPPORTED


def test_decode_empty_batch_is_a_no_op(lib):
    assert decode(lib, good_pool(), B=0) == 0


def test_plan_heuristic_bounds(lib):
    s, c, w, z = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_size_t(), ctypes.c_size_t()
    for B, Hkv, L in [(1, 8, 1024), (64, 8, 8192), (1, 8, 32768), (8, 8, 32768), (32, 8, 16398)]:
        for dtype, cap in ((0, 96), (1, 128)):
            assert lib.pkv_decode_plan(B, 4 * Hkv, Hkv, L, dtype, 0, ctypes.byref(s),
                                       ctypes.byref(c), ctypes.byref(w), ctypes.byref(z)) == 0
            pages = (L + 15) // 16
            assert 1 <= c.value <= cap and s.value == -(-pages // c.value)
            if s.value > 1:
                assert z.value == 65536 * 4
                assert w.value >= z.value + B * 4 * Hkv * s.value * 129 * 4
            else:
                assert w.value == 0 and z.value == 0


def test_plan_rejects_unknown_dtype(lib):
    s, c, w, z = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_size_t(), ctypes.c_size_t()
    for dtype in (-1, 2):
        assert lib.pkv_decode_plan(1, 4, 2, 64, dtype, 0, ctypes.byref(s), ctypes.byref(c),
                                   ctypes.byref(w), ctypes.byref(z)) == INVALID


def test_append_rejects_bad_arguments(lib):
    f = lib.pkv_kv_append
    f.restype = ctypes.c_int32
    p = good_pool()
    args = [ctypes.byref(p), ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), 8,
            ctypes.c_void_p(FAKE), 1, ctypes.c_void_p(FAKE), 4, ctypes.c_void_p(FAKE), None, None]
    assert f(*args[:1], None, *args[2:]) == INVALID            # no k_new
    bad = list(args)
    bad[9] = ctypes.c_void_p(FAKE)                              # smoothing on a bf16 pool
    assert f(*bad) == INVALID
    zero = list(args)
    zero[3] = 0
    assert f(*zero) == 0                                        # nothing to append


def test_prefill_rejects_int8_pool_and_bad_arguments(lib):
    f = lib.pkv_paged_attn_prefill
    f.restype = ctypes.c_int32
    i8 = good_pool(dtype=1, k_scale=FAKE, v_scale=FAKE)
    V = ctypes.c_void_p
    plan = lib.pkv_prefill_plan
    plan.restype = ctypes.c_int32
    ctas, ws, zb = ctypes.c_int32(), ctypes.c_size_t(), ctypes.c_size_t()
    assert plan(ctypes.byref(ctas), ctypes.byref(ws), ctypes.byref(zb)) == 0
    assert ctas.value > 0
    # counters (2 per CTA, whole 256-byte lines), then one slot per CTA of
    # 256 rows x (128 + 1) fp32
    assert zb.value == (8 * ctas.value + 255) // 256 * 256
    assert ws.value == zb.value + ctas.value * 256 * 129 * 4
    args = [V(FAKE), 16, V(FAKE), 1, 4, V(FAKE), 4, V(FAKE), 16, ctypes.c_float(0.1), V(FAKE),
            ctypes.c_size_t(ws.value), 0, V(FAKE), None, None]
    assert f(ctypes.byref(i8), *args) == UNSUPPORTED
    bf = good_pool()
    bad = list(args)
    bad[4] = 3                                                  # Hq not a multiple of Hkv
    assert f(ctypes.byref(bf), *bad) == INVALID
    small = list(args)
    small[11] = ctypes.c_size_t(ws.value - 16)                  # workspace too small
    assert f(ctypes.byref(bf), *small) == INVALID
    nows = list(args)
    nows[10] = None                                             # no workspace
    assert f(ctypes.byref(bf), *nows) == INVALID
    odd = list(args)
    odd[10] = V(FAKE + 8)                                       # workspace not 16-byte aligned
    assert f(ctypes.byref(bf), *odd) == INVALID
    neg = list(args)
    neg[1] = -1                                                 # negative total_q
    assert f(ctypes.byref(bf), *neg) == INVALID
    none = list(args)
    none[1] = 0                                                 # no query rows: nothing to do
    assert f(ctypes.byref(bf), *none) == 0
    negc = list(args)
    negc[12] = -1                                               # negative CTA count
    assert f(ctypes.byref(bf), *negc) == INVALID


def test_overlap_split_bounds_and_order(lib):
    f = lib.pkv_overlap_prefill_ctas
    f.restype = ctypes.c_int32
    f.argtypes = [ctypes.c_double, ctypes.c_double, ctypes.POINTER(ctypes.c_int32)]
    all_ = ctypes.c_int32()
    assert lib.pkv_prefill_plan(ctypes.byref(all_), None, None) == 0
    n = ctypes.c_int32()
    got = []
    for flops in (0.0, 1e10, 1e11, 1e12, 1e13, 1e15):
        assert f(flops, 1.26e9, ctypes.byref(n)) == 0
        assert max(1, all_.value // 3) <= n.value <= all_.value
        got.append(n.value)
    assert got == sorted(got)                   # more prefill work: more of the SMs
    assert got[-1] > got[0]
    assert f(1e12, 0.0, ctypes.byref(n)) == 0 and n.value == all_.value   # no decode: all SMs
    for bad in ((-1.0, 1e9), (1e12, -1.0), (float("nan"), 1e9), (1e12, float("inf"))):
        assert f(*bad, ctypes.byref(n)) == INVALID
    assert f(1e12, 1e9, None) == INVALID


def test_status_strings(lib):
    f = lib.pkv_status_string
    f.restype = ctypes.c_char_p
    for s in (0, -1, -2, -3, -4):
        assert f(s)


def test_qkv_prep_rejects_bad_arguments(lib):
    f = lib.pkv_qkv_norm_rope_append
    f.restype = ctypes.c_int32
    V = ctypes.c_void_p
    bf = good_pool()
    #       qkv     T  Hq  q_w   k_w   eps                 cos     sin     maxpos cu
    args = [V(FAKE), 4, 4, None, None, ctypes.c_float(1e-6), V(FAKE), V(FAKE), 64, V(FAKE),
            1, V(FAKE), 4, V(FAKE), V(FAKE), None]
    i8 = good_pool(dtype=1, k_scale=FAKE, v_scale=FAKE)
    assert f(ctypes.byref(i8), *args) == UNSUPPORTED
    bad = list(args)
    bad[2] = 3                                        # Hq not a multiple of Hkv
    assert f(ctypes.byref(bf), *bad) == INVALID
    bad = list(args)
    bad[7] = None                                     # cos without sin
    assert f(ctypes.byref(bf), *bad) == INVALID
    bad = list(args)
    bad[5] = ctypes.c_float(-1.0)                     # negative eps
    assert f(ctypes.byref(bf), *bad) == INVALID
    bad = list(args)
    bad[0] = V(FAKE + 2)                              # unaligned qkv
    assert f(ctypes.byref(bf), *bad) == INVALID
    none = list(args)
    none[1] = 0                                       # no tokens: nothing to do
    assert f(ctypes.byref(bf), *none) == 0


def test_decode_multi_plan_and_argument_checks(lib):
    plan = lib.pkv_decode_multi_plan
    plan.restype = ctypes.c_int32
    s, c, w = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_size_t()
    out = (ctypes.byref(s), ctypes.byref(c), ctypes.byref(w))
    assert plan(2, 20, 8, 2, 16, 1000, 0, *out) == 0
    assert s.value * c.value * 16 >= 1000 and s.value >= 1
    assert (w.value == 0) == (s.value == 1)
    assert plan(2, 20, 8, 2, 16, 1000, 3, *out) == 0 and s.value == 3
    assert plan(2, 20, 8, 2, 17, 1000, 0, *out) == UNSUPPORTED          # > 16 tokens
    assert plan(2, 20, 8, 3, 4, 1000, 0, *out) == INVALID               # Hq % Hkv
    assert plan(2, 20, 8, 2, 0, 1000, 0, *out) == INVALID               # no tokens

    f = lib.pkv_paged_attn_decode_multi
    f.restype = ctypes.c_int32
    V = ctypes.c_void_p
    bf = good_pool()
    #       q       total cu      B  Hq  bt      maxp sl      maxq maxL scale              splits
    args = [V(FAKE), 4, V(FAKE), 2, 4, V(FAKE), 4, V(FAKE), 2, 64, ctypes.c_float(0.1), 1,
            None, 0, V(FAKE), None, None]
    i8 = good_pool(dtype=1, k_scale=FAKE, v_scale=FAKE)
    assert f(ctypes.byref(i8), *args) == UNSUPPORTED                    # bf16 pools only
    bad = list(args)
    bad[8] = 17                                                         # max_q_len > 16
    assert f(ctypes.byref(bf), *bad) == UNSUPPORTED
    bad = list(args)
    bad[9] = 65                                                         # past the block table
    assert f(ctypes.byref(bf), *bad) == INVALID
    bad = list(args)
    bad[0] = V(FAKE + 4)                                                # unaligned q
    assert f(ctypes.byref(bf), *bad) == INVALID
    bad = list(args)
    bad[11] = 2                                                         # 2 splits, no workspace
    assert f(ctypes.byref(bf), *bad) == INVALID
    none = list(args)
    none[1] = 0                                                         # no tokens
    assert f(ctypes.byref(bf), *none) == 0


def test_wait_selftest_rejects_a_null_counter(lib):
    """Checked on the host before any launch (no GPU needed)."""
    assert lib.pkv_selftest_bounded_wait(None, 1, None) == -1
