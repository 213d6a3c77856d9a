"""The mixed continuous-batching step end to end on the GPU against the fp64
oracle: the bench's own step sequence (one 26,926-token prompt prefilled in
2,048-row chunks against its cached prefix, plus 32 decode rows with contexts
~ U[128, 16384] that gain one token per step, in one shared pool of 16-token
pages), all 14 steps: append (chunk rows and one row per decode sequence,
one call), then prefill of the chunk and decode of the 32 rows -- one after
the other on one stream, and overlapped (the prefill on part of the SMs, the
decode beside it on a second stream, as the bench times it) (TileInfer.jl
"Performance" page, "Fused kernels, FlashAttention and PagedAttention":
split-KV decode over the pages in place; "What is left to gain": chunked
prefill).

At the first, a middle and the last step every decode row (contexts past
8,192 positions, the split heuristic's plan for 32 rows) and a seeded sample
of prefill rows are compared element by element with the oracle run on a
pool that the oracle's own append built; after the last step the GPU pool
must equal that pool byte for byte."""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import check_lse, check_out

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("overlap", [True, False], ids=["overlapped", "sequential"])
def test_mixed_step_all_fourteen_steps_against_the_oracle(overlap):
    import bench
    from paged_kv_flash_gb300 import pagedkv as pk
    from paged_kv_flash_gb300 import workloads as W

    mixed = bench.Mixed(torch, pk, overlap=overlap)
    if overlap:
        all_ctas = pk.prefill_plan()[0]
        ctas = [st["ctas"] for st in mixed.steps]
        assert all(1 <= n <= all_ctas for n in ctas) and min(ctas) < all_ctas
    wl = mixed.wl
    assert len(wl.steps) == 14 and len(wl.decode_lens0) == 32
    assert int(wl.steps[0].decode_lens.max()) > 8192
    bt = wl.layout.block_table
    kp, vp = wl.k_pool, wl.v_pool
    scale = float(bench.SCALE)
    rng = np.random.default_rng(71)
    checked = {0, 7, 13}
    R = len(wl.decode_lens0)
    for c, s in enumerate(wl.steps):
        mixed.step(c)                              # append, then prefill and decode
        cu_app, lens_app = wl.step_append(s)
        kp, vp = oracle.kv_append_bf16(kp, vp, s.k_new, s.v_new, cu_app, bt, lens_app)
        if c not in checked:
            continue
        torch.cuda.synchronize()
        assert pk.poll_device_error() == pk.OK
        # every decode row
        ro, rl = oracle.paged_attention(kp, vp, s.q_decode, np.arange(R + 1, dtype=np.int32),
                                        bt[1:], s.decode_lens, scale)
        check_out(mixed.out_d, ro, f"mixed step {c}: decode rows")
        check_lse(mixed.lse_d, rl, f"mixed step {c}: decode rows")
        # prefill rows: the chunk's first and last rows and a seeded sample
        n = s.chunk_len
        rows = np.unique(np.concatenate([[0, n - 1], rng.choice(n, 24, replace=False)]))
        rows = rows.astype(np.int32)
        ro, rl = oracle.paged_attention(kp, vp, s.q_chunk, W.cu_from_counts([n]), bt[:1],
                                        np.array([s.prefill_len], np.int32), scale, rows=rows)
        idx = torch.from_numpy(rows).long().cuda()
        check_out(mixed.out_p[:n][idx], ro, f"mixed step {c}: prefill rows")
        check_lse(mixed.lse_p[:n][idx], rl, f"mixed step {c}: prefill rows")
    # every page write of the 14 appends, and nothing else
    gk = mixed.pool.k.cpu().view(torch.int16).numpy().view(np.uint16)
    gv = mixed.pool.v.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(gk, kp) and np.array_equal(gv, vp)
