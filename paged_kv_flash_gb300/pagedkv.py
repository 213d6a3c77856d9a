"""ctypes binding over libpagedkv.so (C ABI in include/pagedkv.h).

Argument marshalling only: every step of the attention path runs in the
library's CUDA kernels.  Tensors are torch CUDA tensors (PyTorch supplies
device memory and streams); the library itself allocates nothing, so where a
call needs an output or a workspace and none is given, this binding
allocates it with torch before the call.

There is no fallback: if the library is missing or fails to load, importing
this module raises.
"""
import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpagedkv.so")

OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = 0, -1, -2, -3, -4
BF16, INT8 = 0, 1
HEAD_DIM, PAGE_SIZE = 128, 16


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_lib.pkv_status_string(status).decode()} ({status})")


class _Pool(ctypes.Structure):
    _fields_ = [
        ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
        ("num_pages", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32),
    ]


# Every symbol include/pagedkv.h declares, with its ctypes signature.
_P, _I, _F, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
_POOLP = ctypes.POINTER(_Pool)
SIGNATURES = {
    "pkv_kv_append": (_I, [_POOLP, _P, _P, _I, _P, _I, _P, _I, _P, _P, _P]),
    "pkv_decode_plan": (_I, [_I, _I, _I, _I, _I, _I, ctypes.POINTER(_I), ctypes.POINTER(_I),
                             ctypes.POINTER(_SZ), ctypes.POINTER(_SZ)]),
    "pkv_paged_attn_decode": (_I, [_POOLP, _P, _I, _I, _P, _I, _P, _I, _F, _P, _I, _P, _SZ,
                                   _P, _P, _P]),
    "pkv_paged_attn_decode_fused": (_I, [_POOLP, _P, _I, _I, _P, _I, _P, _I, _F, _P, _I, _P,
                                         _SZ, _P, _P, _P]),
    "pkv_paged_attn_decode_noalloc": (_I, [_POOLP, _P, _I, _I, _P, _I, _P, _I, _F, _P, _I, _P,
                                           _P, _P]),
    "pkv_prefill_plan": (_I, [ctypes.POINTER(_I), ctypes.POINTER(_SZ), ctypes.POINTER(_SZ)]),
    "pkv_paged_attn_prefill": (_I, [_POOLP, _P, _I, _P, _I, _I, _P, _I, _P, _I, _F, _P, _SZ, _I,
                                    _P, _P, _P]),
    "pkv_overlap_prefill_ctas": (_I, [ctypes.c_double, ctypes.c_double, ctypes.POINTER(_I)]),
    "pkv_decode_multi_plan": (_I, [_I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(_I),
                                   ctypes.POINTER(_I), ctypes.POINTER(_SZ)]),
    "pkv_paged_attn_decode_multi": (_I, [_POOLP, _P, _I, _P, _I, _I, _P, _I, _P, _I, _I, _F, _I,
                                         _P, _SZ, _P, _P, _P]),
    "pkv_qkv_norm_rope_append": (_I, [_POOLP, _P, _I, _I, _P, _P, _F, _P, _P, _I, _P, _I, _P,
                                      _I, _P, _P, _P]),
    "pkv_selftest_bounded_wait": (_I, [_P, ctypes.c_uint32, _P]),
    "pkv_poll_device_error": (_I, [_P]),
    "pkv_status_string": (ctypes.c_char_p, [_I]),
    "pkv_device_sm_count": (_I, []),
}


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"{_LIB_PATH} is not built; run paged_kv_flash_gb300.build.build()")
    lib = ctypes.CDLL(_LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def lib_path() -> str:
    return _LIB_PATH


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status: int, what: str):
    if status != OK:
        raise PkvError(status, what)


def _need(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous CUDA {dtype} tensor, got "
                         f"{t.dtype} on {t.device} (contiguous={t.is_contiguous()})")


@dataclass
class Pool:
    """A paged KV pool: k, v [num_pages][Hkv][16][128] (bf16 or int8) and, for
    int8, fp32 scales [num_pages][Hkv][16]."""
    k: torch.Tensor
    v: torch.Tensor
    k_scale: Optional[torch.Tensor] = None
    v_scale: Optional[torch.Tensor] = None

    @property
    def dtype(self) -> int:
        return INT8 if self.k.dtype == torch.int8 else BF16

    @property
    def num_pages(self) -> int:
        return self.k.shape[0]

    @property
    def num_kv_heads(self) -> int:
        return self.k.shape[1]

    def c(self) -> _Pool:
        """The C struct of the pool, rebuilt (and the tensors checked) only
        when a tensor has changed (it is passed on every call, and a serving
        loop makes many)."""
        key = (self.k.data_ptr(), self.v.data_ptr(),
               self.k_scale.data_ptr() if self.k_scale is not None else None,
               self.v_scale.data_ptr() if self.v_scale is not None else None,
               tuple(self.k.shape), tuple(self.v.shape), self.k.device, self.dtype)
        cached = self.__dict__.get("_c")
        if cached is None or cached[0] != key:
            self._validate()
            cached = (key, _Pool(key[0], key[1], key[2], key[3], *key[4], key[7]))
            self.__dict__["_c"] = cached
        return cached[1]

    def _validate(self):
        """The kernels take the pool's pointers as they are: host memory or a
        wrong layout must be refused here, before any launch."""
        want = torch.int8 if self.k.dtype == torch.int8 else torch.bfloat16
        _need(self.k, want, "pool.k")
        _need(self.v, want, "pool.v")
        if (self.k.dim() != 4 or tuple(self.k.shape[2:]) != (PAGE_SIZE, HEAD_DIM)
                or self.v.shape != self.k.shape or self.v.device != self.k.device):
            raise ValueError(f"pool: k and v must be [num_pages][Hkv][{PAGE_SIZE}][{HEAD_DIM}] "
                             f"on one device, got {tuple(self.k.shape)} on {self.k.device} "
                             f"and {tuple(self.v.shape)} on {self.v.device}")
        scales = (("pool.k_scale", self.k_scale), ("pool.v_scale", self.v_scale))
        if want == torch.int8:
            for name, t in scales:
                if t is None:
                    raise ValueError(f"{name}: an INT8 pool needs fp32 scales")
                _need(t, torch.float32, name)
                if tuple(t.shape) != tuple(self.k.shape[:3]) or t.device != self.k.device:
                    raise ValueError(f"{name}: expected {tuple(self.k.shape[:3])} on "
                                     f"{self.k.device}, got {tuple(t.shape)} on {t.device}")
        elif self.k_scale is not None or self.v_scale is not None:
            raise ValueError("a bf16 pool has no scales")

    @staticmethod
    def empty(num_pages: int, num_kv_heads: int, dtype=torch.bfloat16, device="cuda"):
        shape = (num_pages, num_kv_heads, PAGE_SIZE, HEAD_DIM)
        if dtype == torch.int8:
            return Pool(torch.empty(shape, dtype=torch.int8, device=device),
                        torch.empty(shape, dtype=torch.int8, device=device),
                        torch.empty(shape[:3], dtype=torch.float32, device=device),
                        torch.empty(shape[:3], dtype=torch.float32, device=device))
        return Pool(torch.empty(shape, dtype=torch.bfloat16, device=device),
                    torch.empty(shape, dtype=torch.bfloat16, device=device))


def kv_append(pool: Pool, k_new, v_new, cu_new, block_table, seq_lens, k_smooth=None,
              stream=None):
    """Write k_new/v_new [T][Hkv][128] bf16 into the pool (see pkv_kv_append)."""
    _need(k_new, torch.bfloat16, "k_new")
    _need(v_new, torch.bfloat16, "v_new")
    for t, n in ((cu_new, "cu_new"), (block_table, "block_table"), (seq_lens, "seq_lens")):
        _need(t, torch.int32, n)
    if k_smooth is not None:
        _need(k_smooth, torch.float32, "k_smooth")
    pc = pool.c()
    st = _lib.pkv_kv_append(ctypes.byref(pc), _ptr(k_new), _ptr(v_new), k_new.shape[0],
                            _ptr(cu_new), seq_lens.shape[0], _ptr(block_table),
                            block_table.shape[1], _ptr(seq_lens), _ptr(k_smooth),
                            _stream(stream))
    _check(st, "pkv_kv_append")


def decode_plan(batch, num_q_heads, num_kv_heads, max_seq_len, num_splits=0, dtype=BF16):
    """(splits, pages_per_split, workspace_bytes, zero_bytes) of a decode call
    on a pool of the given dtype (BF16 or INT8)."""
    s, c, w, z = _I(), _I(), _SZ(), _SZ()
    st = _lib.pkv_decode_plan(batch, num_q_heads, num_kv_heads, max_seq_len, int(dtype),
                              num_splits, ctypes.byref(s), ctypes.byref(c), ctypes.byref(w),
                              ctypes.byref(z))
    _check(st, "pkv_decode_plan")
    return s.value, c.value, w.value, z.value


def decode_workspace(nbytes, zero_bytes, device="cuda"):
    """A decode workspace of nbytes (at least 256) ready for its first call:
    the leading zero_bytes (part counters) zeroed.  Calls leave it ready
    again, so it is meant to be kept and reused."""
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
    if zero_bytes:
        ws[:zero_bytes].zero_()
    return ws


def paged_attn_decode(pool: Pool, q, block_table, seq_lens, max_seq_len, softmax_scale,
                      k_smooth=None, num_splits=0, workspace=None, out=None, lse=None,
                      want_lse=True, stream=None, fused=False):
    """One query token per sequence: q [B][Hq][128] bf16 -> (out bf16, lse fp32).
    fused=True merges the splits inside the split kernel
    (pkv_paged_attn_decode_fused; its workspace's counters must start zeroed,
    as decode_workspace() leaves them)."""
    _need(q, torch.bfloat16, "q")
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    B, Hq, _ = q.shape
    if workspace is None:                   # (a given workspace's size is checked by the call)
        _, _, ws_bytes, zero_bytes = decode_plan(B, Hq, pool.num_kv_heads, max_seq_len,
                                                 num_splits, pool.dtype)
        if ws_bytes:
            workspace = decode_workspace(ws_bytes, zero_bytes, q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    pc = pool.c()
    fn = _lib.pkv_paged_attn_decode_fused if fused else _lib.pkv_paged_attn_decode
    st = fn(
        ctypes.byref(pc), _ptr(q), B, Hq, _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), int(max_seq_len), float(softmax_scale), _ptr(k_smooth),
        int(num_splits), _ptr(workspace), workspace.numel() if workspace is not None else 0,
        _ptr(out), _ptr(lse), _stream(stream))
    _check(st, "pkv_paged_attn_decode_fused" if fused else "pkv_paged_attn_decode")
    return out, lse


def paged_attn_decode_noalloc(pool: Pool, q, block_table, seq_lens, max_seq_len, softmax_scale,
                              k_smooth=None, num_splits=0, out=None, lse=None, want_lse=True,
                              stream=None):
    """Decode for callers that cannot allocate device memory: the split
    partials live in the library's fixed 16 MiB device array instead of a
    workspace (see pkv_paged_attn_decode_noalloc).  Calls on one device share
    that array, so they must not overlap on the GPU."""
    _need(q, torch.bfloat16, "q")
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    B, Hq, _ = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    pc = pool.c()
    st = _lib.pkv_paged_attn_decode_noalloc(
        ctypes.byref(pc), _ptr(q), B, Hq, _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), int(max_seq_len), float(softmax_scale), _ptr(k_smooth),
        int(num_splits), _ptr(out), _ptr(lse), _stream(stream))
    _check(st, "pkv_paged_attn_decode_noalloc")
    return out, lse


def prefill_plan():
    """(persistent CTAs, workspace bytes, leading bytes that must start zero)
    of a prefill call on the current device."""
    n, w, z = _I(), _SZ(), _SZ()
    _check(_lib.pkv_prefill_plan(ctypes.byref(n), ctypes.byref(w), ctypes.byref(z)),
           "pkv_prefill_plan")
    return n.value, w.value, z.value


def prefill_workspace(device="cuda"):
    """A prefill workspace ready for its first call (counters zeroed).  Calls
    leave it ready again, so it is meant to be kept and reused."""
    _, nbytes, zbytes = prefill_plan()
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    ws[:zbytes].zero_()
    return ws


def paged_attn_prefill(pool: Pool, q, cu_q, block_table, seq_lens, max_q_len, softmax_scale,
                       workspace=None, out=None, lse=None, want_lse=True, stream=None,
                       num_ctas=0):
    """Causal chunk attention: q [total_q][Hq][128] bf16 -> (out bf16, lse fp32).
    `workspace` (from prefill_workspace()) is allocated when not given.
    num_ctas: persistent CTAs, 0 = one per SM (see overlap_prefill_ctas)."""
    _need(q, torch.bfloat16, "q")
    for t, n in ((cu_q, "cu_q"), (block_table, "block_table"), (seq_lens, "seq_lens")):
        _need(t, torch.int32, n)
    T, Hq, _ = q.shape
    if workspace is None:
        workspace = prefill_workspace(q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device)
    pc = pool.c()
    st = _lib.pkv_paged_attn_prefill(
        ctypes.byref(pc), _ptr(q), T, _ptr(cu_q), seq_lens.shape[0], Hq, _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), int(max_q_len), float(softmax_scale),
        _ptr(workspace), workspace.numel() * workspace.element_size(), int(num_ctas), _ptr(out),
        _ptr(lse), _stream(stream))
    _check(st, "pkv_paged_attn_prefill")
    return out, lse


def overlap_prefill_ctas(prefill_flops, decode_bytes):
    """num_ctas for a prefill that runs beside a decode on another stream
    (see pkv_overlap_prefill_ctas)."""
    n = _I()
    _check(_lib.pkv_overlap_prefill_ctas(float(prefill_flops), float(decode_bytes),
                                         ctypes.byref(n)), "pkv_overlap_prefill_ctas")
    return n.value


def decode_multi_plan(batch, total_q, num_q_heads, num_kv_heads, max_q_len, max_seq_len,
                      num_splits=0):
    """(splits, pages_per_split, workspace_bytes) of a multi-token decode."""
    s, c, w = _I(), _I(), _SZ()
    st = _lib.pkv_decode_multi_plan(batch, total_q, num_q_heads, num_kv_heads, max_q_len,
                                    max_seq_len, num_splits, ctypes.byref(s), ctypes.byref(c),
                                    ctypes.byref(w))
    _check(st, "pkv_decode_multi_plan")
    return s.value, c.value, w.value


def paged_attn_decode_multi(pool: Pool, q, cu_q, block_table, seq_lens, max_q_len, max_seq_len,
                            softmax_scale, num_splits=0, workspace=None, out=None, lse=None,
                            want_lse=True, stream=None):
    """1..16 query tokens per sequence, causal inside the step (verify steps):
    q [total_q][Hq][128] bf16 -> (out bf16, lse fp32).  The workspace is
    allocated when not given."""
    _need(q, torch.bfloat16, "q")
    for t, n in ((cu_q, "cu_q"), (block_table, "block_table"), (seq_lens, "seq_lens")):
        _need(t, torch.int32, n)
    T, Hq, _ = q.shape
    B = seq_lens.shape[0]
    if workspace is None:
        _, _, wsb = decode_multi_plan(B, T, Hq, pool.k.shape[1], int(max_q_len),
                                      int(max_seq_len), num_splits)
        workspace = torch.empty(max(wsb, 256), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device)
    pc = pool.c()
    st = _lib.pkv_paged_attn_decode_multi(
        ctypes.byref(pc), _ptr(q), T, _ptr(cu_q), B, Hq, _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), int(max_q_len), int(max_seq_len), float(softmax_scale), int(num_splits),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out), _ptr(lse),
        _stream(stream))
    _check(st, "pkv_paged_attn_decode_multi")
    return out, lse


def qkv_norm_rope_append(pool: Pool, qkv, num_q_heads, cu_new, block_table, seq_lens,
                         q_norm_w=None, k_norm_w=None, eps=1e-6, rope_cos=None, rope_sin=None,
                         q_out=None, stream=None):
    """Fused attention inputs (see pkv_qkv_norm_rope_append): qkv bf16
    [T][Hq + 2 Hkv][128] -> q_out bf16 [T][Hq][128]; K (normed, rotated) and
    V are written into the pool."""
    _need(qkv, torch.bfloat16, "qkv")
    for t, n in ((cu_new, "cu_new"), (block_table, "block_table"), (seq_lens, "seq_lens")):
        _need(t, torch.int32, n)
    for t, n in ((q_norm_w, "q_norm_w"), (k_norm_w, "k_norm_w"), (rope_cos, "rope_cos"),
                 (rope_sin, "rope_sin")):
        if t is not None:
            _need(t, torch.float32, n)
    T = qkv.shape[0]
    if q_out is None:
        q_out = torch.empty((T, num_q_heads, HEAD_DIM), dtype=torch.bfloat16, device=qkv.device)
    pc = pool.c()
    st = _lib.pkv_qkv_norm_rope_append(
        ctypes.byref(pc), _ptr(qkv), T, num_q_heads, _ptr(q_norm_w), _ptr(k_norm_w), float(eps),
        _ptr(rope_cos), _ptr(rope_sin), rope_cos.shape[0] if rope_cos is not None else 0,
        _ptr(cu_new), seq_lens.shape[0], _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
        _ptr(q_out), _stream(stream))
    _check(st, "pkv_qkv_norm_rope_append")
    return q_out


def selftest_bounded_wait(counter, target, stream=None):
    """One device thread waits (bounded, one second) for the int32 tensor
    `counter` (read as uint32) to reach `target`; a wait that runs out shows
    as ERR_TIMEOUT at the next poll_device_error."""
    _need(counter, torch.int32, "counter")
    _check(_lib.pkv_selftest_bounded_wait(_ptr(counter), int(target), _stream(stream)),
           "pkv_selftest_bounded_wait")


def poll_device_error(stream=None) -> int:
    """Synchronise and return the status of the kernels' device-side checks."""
    return _lib.pkv_poll_device_error(_stream(stream))


def sm_count() -> int:
    return _lib.pkv_device_sm_count()


def status_string(status: int) -> str:
    return _lib.pkv_status_string(status).decode()


def raw():
    """The loaded ctypes library (for tests that exercise the C ABI directly)."""
    return _lib
