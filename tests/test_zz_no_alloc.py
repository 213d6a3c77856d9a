"""pkv_paged_attn_decode_noalloc: decode for callers that cannot allocate.

Some users of this library cannot hand it a workspace: a plain C host
program with no device allocator of its own, a plugin inside a runtime that
owns all device memory and forbids cudaMalloc on its threads, or code that
cannot afford an allocation's implicit synchronisation.  For them the
library keeps the split partials in a fixed 16 MiB device array of its own.
These tests call that entry point through the C ABI and compare it with the
workspace entry point, on consecutive calls that share the array, and with
the fp64 oracle.

The file name sorts last so that a run that stops at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest

import oracle
from paged_kv_flash_gb300 import workloads as W
from tests.helpers import check_lse, check_out, dev, dev_bf16, host_f32


class _Pool(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("num_pages", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


def _noalloc_fn(lib):
    f = lib.pkv_paged_attn_decode_noalloc
    f.restype = ctypes.c_int32
    V, I = ctypes.c_void_p, ctypes.c_int32
    f.argtypes = [ctypes.POINTER(_Pool), V, I, I, V, I, V, I, ctypes.c_float, V, I, V, V, V]
    return f


def test_noalloc_rejects_forced_splits_beyond_the_fixed_array():
    """A forced split count whose partials exceed 16 MiB is refused on the
    host, before any launch (no GPU needed)."""
    from paged_kv_flash_gb300 import build
    lib = ctypes.CDLL(build.build())
    f = _noalloc_fn(lib)
    fake = 1 << 20
    pool = _Pool(fake, 2 * fake, None, None, 4, 8, 16, 128, 0)
    # 1024 rows x 32 heads x 2 splits x 516 B = 33.8 MB > 16 MiB
    st = f(ctypes.byref(pool), fake, 1024, 32, fake, 4, fake, 32, ctypes.c_float(0.1), None, 2,
           fake, None, None)
    assert st == -1


@pytest.mark.gpu
def test_noalloc_decode_matches_workspace_decode_on_consecutive_calls():
    import torch
    from paged_kv_flash_gb300 import pagedkv as pk
    f = _noalloc_fn(pk.raw())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    cases = []
    # 64 sequences of 512..8192 positions: the heuristic's partials (about
    # 17 MB) do not fit in 16 MiB, so this call runs with fewer splits
    c = W.batched_decode()
    cases.append((c, pk.Pool(dev_bf16(c.k_pool), dev_bf16(c.v_pool)), 0))
    # one 1,024-position sequence, forced 7 splits
    c = W.decode_1k()
    cases.append((c, pk.Pool(dev_bf16(c.k_pool), dev_bf16(c.v_pool)), 7))

    for case, pool, splits in cases + cases[:1]:          # three calls in a row
        q = dev_bf16(case.q)
        bt, sl = dev(case.layout.block_table), dev(case.seq_lens)
        ms = int(case.seq_lens.max())
        ref_out, ref_lse = pk.paged_attn_decode(pool, q, bt, sl, ms, case.scale,
                                                num_splits=splits)
        out = torch.full_like(q, float("nan"))
        lse = torch.full((case.B, case.Hq), float("nan"), dtype=torch.float32, device="cuda")
        pc = pool.c()
        cpool = _Pool(pc.k, pc.v, pc.k_scale, pc.v_scale, pc.num_pages, pc.num_kv_heads,
                      pc.page_size, pc.head_dim, pc.dtype)
        st = f(ctypes.byref(cpool), q.data_ptr(), case.B, case.Hq, bt.data_ptr(),
               bt.shape[1], sl.data_ptr(), ms, ctypes.c_float(case.scale), None, splits,
               out.data_ptr(), lse.data_ptr(), stream)
        assert st == 0, pk.status_string(st)
        assert pk.poll_device_error() == pk.OK
        check_out(out, host_f32(ref_out).astype(np.float64), "noalloc vs workspace decode")
        check_lse(lse, ref_lse.cpu().numpy().astype(np.float64), "noalloc vs workspace decode")
        # and against the fp64 oracle: every row of the single sequence, a
        # seeded sample of 16 of the 64 sequences (the lowered-split call)
        rows = np.arange(case.B, dtype=np.int32) if case.B <= 16 else np.sort(
            np.random.default_rng(70).choice(case.B, 16, replace=False)).astype(np.int32)
        ro, rl = oracle.paged_attention(case.k_pool, case.v_pool, case.q,
                                        np.arange(case.B + 1, dtype=np.int32),
                                        case.layout.block_table, case.seq_lens, case.scale,
                                        rows=rows)
        idx = torch.from_numpy(rows).long().cuda()
        check_out(out[idx], ro, "noalloc vs oracle")
        check_lse(lse[idx], rl, "noalloc vs oracle")
