"""fp64 CPU oracle for attention over a paged KV cache -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The CUDA library never calls it and the two
share no code: this wrapper only marshals numpy arrays into ``liborc.so``,
built from ``pkv_oracle.c`` by ``oracle/build.py``.

Every function follows the plain definition stated in ``pkv_oracle.c``
(TileInfer.jl "Performance" page: the reference-ops attention that gathers
pages into dense K/V, the split-KV decode with a separate combine, and the
"INT8 KV cache" section's one-scale-per-vector cache).

Pins: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, invariants, a library routine on special cases, hand-worked
golden values); none is "parity unpinned".
"""
import ctypes
import os

import numpy as np

from . import build as _build

BF16, INT8 = 0, 1


class _Pool(ctypes.Structure):
    _fields_ = [
        ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
        ("k_smooth", ctypes.c_void_p),
        ("num_pages", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
        ("page_size", ctypes.c_int), ("head_dim", ctypes.c_int), ("dtype", ctypes.c_int),
    ]


_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.orc_paged_attention.argtypes = [ctypes.POINTER(_Pool), P, P, I, I, P, I, P,
                                            ctypes.c_double, P, I, I, P, P, I]
        lib.orc_paged_attention.restype = I
        lib.orc_kv_append_bf16.argtypes = [P, P, I, I, I, I, P, P, P, I, P, I, P]
        lib.orc_kv_append_bf16.restype = I
        lib.orc_kv_append_int8.argtypes = [P, P, P, P, I, I, I, I, P, P, P, P, I, P, I, P]
        lib.orc_kv_append_int8.restype = I
        lib.orc_quantize_row_int8.argtypes = [P, P, I, P, P]
        lib.orc_quantize_row_int8.restype = None
        lib.orc_qkv_norm_rope_append.argtypes = [P, I, I, I, P, P, ctypes.c_double, P, P, I, P,
                                                 I, P, I, P, P, P, P, I, I]
        lib.orc_qkv_norm_rope_append.restype = I
        lib.orc_bf16_from_double.argtypes = [ctypes.c_double]
        lib.orc_bf16_from_double.restype = ctypes.c_uint16
        lib.orc_rsqrt_rn.argtypes = [ctypes.c_float]
        lib.orc_rsqrt_rn.restype = ctypes.c_float
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _threads(n):
    return int(n) if n else (os.cpu_count() or 1)


def paged_attention(k_pool, v_pool, q, cu_q, block_table, seq_lens, scale, *,
                    k_scale=None, v_scale=None, k_smooth=None, rows=None,
                    num_splits=0, nthreads=0):
    """Attention of query rows over the paged cache, fp64.

    k_pool, v_pool: uint16 bf16 bits or int8 codes, [num_pages][Hkv][P][D].
    q: uint16 bf16 bits [total_q][Hq][D]; cu_q: int32 [B+1];
    block_table: int32 [B][max_pages]; seq_lens: int32 [B] (cached positions,
    the rows' own included).  rows: which of the total_q rows to evaluate
    (default all).  num_splits > 0 evaluates through split-KV partials and
    the log-sum-exp combine instead of one softmax.
    Returns (out [nrows][Hq][D] float64, lse [nrows][Hq] float64).
    """
    lib = _load()
    int8 = k_pool.dtype == np.int8
    k_pool = np.ascontiguousarray(k_pool)
    v_pool = np.ascontiguousarray(v_pool)
    num_pages, Hkv, P, D = k_pool.shape
    q = _c(q, np.uint16)
    total_q, Hq, Dq = q.shape
    assert Dq == D
    cu_q = _c(cu_q, np.int32)
    bt = _c(block_table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    B = seq_lens.shape[0]
    rows = np.arange(total_q, dtype=np.int32) if rows is None else _c(rows, np.int32)
    ks, vs, sm = _c(k_scale, np.float32), _c(v_scale, np.float32), _c(k_smooth, np.float32)
    pool = _Pool(_ptr(k_pool), _ptr(v_pool), _ptr(ks), _ptr(vs), _ptr(sm),
                 num_pages, Hkv, P, D, INT8 if int8 else BF16)
    out = np.zeros((rows.shape[0], Hq, D), np.float64)
    lse = np.zeros((rows.shape[0], Hq), np.float64)
    rc = lib.orc_paged_attention(ctypes.byref(pool), _ptr(q), _ptr(cu_q), B, Hq, _ptr(bt),
                                 bt.shape[1], _ptr(seq_lens), float(scale), _ptr(rows),
                                 rows.shape[0], int(num_splits), _ptr(out), _ptr(lse),
                                 _threads(nthreads))
    if rc != 0:
        raise ValueError("oracle: invalid arguments")
    return out, lse


def kv_append_bf16(k_pool, v_pool, k_new, v_new, cu_new, block_table, seq_lens):
    """Write new bf16 K/V rows [T][Hkv][D] into copies of the pools; returns them."""
    lib = _load()
    k_pool = np.array(k_pool, dtype=np.uint16, copy=True)
    v_pool = np.array(v_pool, dtype=np.uint16, copy=True)
    num_pages, Hkv, P, D = k_pool.shape
    k_new, v_new = _c(k_new, np.uint16), _c(v_new, np.uint16)
    cu_new, bt, sl = _c(cu_new, np.int32), _c(block_table, np.int32), _c(seq_lens, np.int32)
    rc = lib.orc_kv_append_bf16(_ptr(k_pool), _ptr(v_pool), num_pages, Hkv, P, D, _ptr(k_new),
                                _ptr(v_new), _ptr(cu_new), sl.shape[0], _ptr(bt), bt.shape[1],
                                _ptr(sl))
    if rc != 0:
        raise ValueError("oracle: position outside the block table")
    return k_pool, v_pool


def kv_append_int8(k_pool, v_pool, k_scale, v_scale, k_new, v_new, cu_new, block_table,
                   seq_lens, k_smooth=None):
    """Quantise new bf16 K/V rows into copies of the int8 pools and scale pools."""
    lib = _load()
    k_pool = np.array(k_pool, dtype=np.int8, copy=True)
    v_pool = np.array(v_pool, dtype=np.int8, copy=True)
    k_scale = np.array(k_scale, dtype=np.float32, copy=True)
    v_scale = np.array(v_scale, dtype=np.float32, copy=True)
    num_pages, Hkv, P, D = k_pool.shape
    k_new, v_new = _c(k_new, np.uint16), _c(v_new, np.uint16)
    sm = _c(k_smooth, np.float32)
    cu_new, bt, sl = _c(cu_new, np.int32), _c(block_table, np.int32), _c(seq_lens, np.int32)
    rc = lib.orc_kv_append_int8(_ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale),
                                num_pages, Hkv, P, D, _ptr(k_new), _ptr(v_new), _ptr(sm),
                                _ptr(cu_new), sl.shape[0], _ptr(bt), bt.shape[1], _ptr(sl))
    if rc != 0:
        raise ValueError("oracle: position outside the block table")
    return k_pool, v_pool, k_scale, v_scale


def quantize_row_int8(x_bits, w=None):
    """One bf16 vector (uint16 bits) -> (int8 codes, fp32 scale)."""
    lib = _load()
    x = _c(x_bits, np.uint16)
    w = _c(w, np.float32)
    codes = np.zeros(x.shape[0], np.int8)
    scale = np.zeros(1, np.float32)
    lib.orc_quantize_row_int8(_ptr(x), _ptr(w), x.shape[0], _ptr(codes), _ptr(scale))
    return codes, scale[0]


def bf16_from_double(v):
    """v rounded to the nearest bf16 (ties to even), as uint16 bits."""
    return int(_load().orc_bf16_from_double(float(v)))


def qkv_norm_rope_append(qkv, Hq, Hkv, q_w, k_w, eps, cos_tab, sin_tab, cu_new, block_table,
                         seq_lens, k_pool, v_pool):
    """Fused attention inputs: qkv uint16 bf16 bits [T][Hq + 2 Hkv][D] -> q_out
    bits [T][Hq][D] and copies of the bf16 pools with the new tokens' K
    (normed, rotated) and V written.  q_w / k_w: fp32 [D] or None (no norm);
    cos_tab / sin_tab: fp32 [max_pos][D/2] or None (no RoPE)."""
    lib = _load()
    qkv = _c(qkv, np.uint16)
    T, H, D = qkv.shape
    assert H == Hq + 2 * Hkv
    k_pool = np.array(k_pool, dtype=np.uint16, copy=True)
    v_pool = np.array(v_pool, dtype=np.uint16, copy=True)
    num_pages, hkv_pool, P, Dp = k_pool.shape
    assert hkv_pool == Hkv and Dp == D
    qw, kw = _c(q_w, np.float32), _c(k_w, np.float32)
    ct, st = _c(cos_tab, np.float32), _c(sin_tab, np.float32)
    max_pos = 0 if ct is None else ct.shape[0]
    cu_new, bt, sl = _c(cu_new, np.int32), _c(block_table, np.int32), _c(seq_lens, np.int32)
    q_out = np.zeros((T, Hq, D), np.uint16)
    rc = lib.orc_qkv_norm_rope_append(_ptr(qkv), Hq, Hkv, D, _ptr(qw), _ptr(kw), float(eps),
                                      _ptr(ct), _ptr(st), max_pos, _ptr(cu_new), sl.shape[0],
                                      _ptr(bt), bt.shape[1], _ptr(sl), _ptr(q_out),
                                      _ptr(k_pool), _ptr(v_pool), num_pages, P)
    if rc != 0:
        raise ValueError("oracle: position outside the block table or the RoPE table")
    return q_out, k_pool, v_pool


def rsqrt_rn(z: float) -> np.float32:
    """The float nearest to 1 / sqrt(z) (ties to even) for a positive normal
    float z: the RMSNorm's reciprocal square root in the fused attention
    inputs."""
    return np.float32(_load().orc_rsqrt_rn(float(np.float32(z))))
