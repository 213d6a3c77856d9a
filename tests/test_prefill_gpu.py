"""paged_attn_prefill (tcgen05) on the GPU against the fp64 oracle, element
by element: causal, chunked against the cached prefix, bottom-right aligned
(TileInfer.jl "Performance" page: paged flash attention over the pages in
place; a block per head over every page; chunked prefill)."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_flash_gb300 import workloads as W
from tests.helpers import check_lse, check_out, dev, dev_bf16

pytestmark = pytest.mark.gpu
D = W.HEAD_DIM


@pytest.fixture(scope="module")
def pk():
    from paged_kv_flash_gb300 import pagedkv
    return pagedkv


def chunk_case(rng, shapes, Hq, Hkv):
    """Sequences with (q_len, L): L cached positions of which the last q_len
    are this chunk's rows.  The pool holds all L positions (NaN elsewhere)."""
    lens = np.array([L for _, L in shapes], np.int32)
    case = W.decode_bf16(rng, lens, Hq, Hkv)
    qlens = [q for q, _ in shapes]
    q = W.normal_bf16(rng, (sum(qlens), Hq, D))
    return case, q, W.cu_from_counts(qlens), max(qlens)


def run(pk, case, q, cu, max_q):
    pool = pk.Pool(dev_bf16(case.k_pool), dev_bf16(case.v_pool))
    out, lse = pk.paged_attn_prefill(pool, dev_bf16(q), dev(cu), dev(case.layout.block_table),
                                     dev(case.seq_lens), max_q, case.scale)
    assert pk.poll_device_error() == pk.OK
    return out, lse


def ref(case, q, cu, rows=None):
    return oracle.paged_attention(case.k_pool, case.v_pool, q, cu, case.layout.block_table,
                                  case.seq_lens, case.scale, rows=rows)


def test_tiny_causal_brute_force(pk):
    """q_len, L <= 40 with page edges inside the chunk, several sequences."""
    rng = np.random.default_rng(60)
    shapes = [(5, 37), (40, 40), (1, 1), (17, 33), (16, 16), (3, 19)]
    case, q, cu, mq = chunk_case(rng, shapes, Hq=8, Hkv=2)
    out, lse = run(pk, case, q, cu, mq)
    ro, rl = ref(case, q, cu)
    check_out(out, ro, "tiny causal")
    check_lse(lse, rl, "tiny causal")


def test_a_bounded_wait_that_runs_out_reports_timeout_and_the_context_stays_usable(pk):
    """The bounded wait a merging CTA uses, on a counter that nothing raises:
    it gives up after about a second, the poll reports the timeout once, a
    reached target returns at once, and the next prefill is still correct."""
    import time
    ctr = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.monotonic()
    pk.selftest_bounded_wait(ctr, 1)
    assert pk.poll_device_error() == pk.ERR_TIMEOUT
    assert 0.9 < time.monotonic() - t0 < 60
    assert pk.poll_device_error() == pk.OK        # the word is cleared once read
    pk.selftest_bounded_wait(ctr, 0)              # already reached: no wait, no error
    assert pk.poll_device_error() == pk.OK
    test_tiny_causal_brute_force(pk)


def test_short_chunk_over_long_context_cuts_units(pk):
    """A 300-row chunk against 6,000 cached positions, GQA 32/8: 64 long units
    for more CTAs than that, so the work is cut between CTAs and the parts
    merged, although each CTA's share is small."""
    rng = np.random.default_rng(66)
    case, q, cu, mq = chunk_case(rng, [(300, 6000)], Hq=32, Hkv=8)
    out, lse = run(pk, case, q, cu, mq)
    rows = np.r_[0:8, 120:136, 250:300].astype(np.int32)   # both tiles, both pairs, the tail
    ro, rl = ref(case, q, cu, rows=rows)
    idx = torch.from_numpy(rows).long().cuda()
    check_out(out[idx], ro, "short chunk over a long context")
    check_lse(lse[idx], rl, "short chunk over a long context")


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (4, 4), (16, 2)])
def test_ragged_chunks_against_prefix(pk, Hq, Hkv):
    """Chunks spanning several 128-row tiles and 128-key blocks, ragged tails."""
    rng = np.random.default_rng(61 + Hq)
    shapes = [(300, 1000), (129, 129), (128, 700), (257, 260)]
    case, q, cu, mq = chunk_case(rng, shapes, Hq=Hq, Hkv=Hkv)
    out, lse = run(pk, case, q, cu, mq)
    ro, rl = ref(case, q, cu)
    check_out(out, ro, f"ragged {Hq}/{Hkv}")
    check_lse(lse, rl, f"ragged {Hq}/{Hkv}")


def test_prompt_1024_tokens_after_append(pk):
    """The 1,024-token prompt: kv_append into seeded pages, then prefill."""
    app, q = W.prefill_prompt()
    kp, vp = W.empty_pool_bf16(app.layout.num_pages, app.Hkv)
    pool = pk.Pool(dev_bf16(kp), dev_bf16(vp))
    bt, sl = dev(app.layout.block_table), dev(app.seq_lens)
    pk.kv_append(pool, dev_bf16(app.k_new), dev_bf16(app.v_new), dev(app.cu_new), bt, sl)
    scale = 1.0 / np.sqrt(D)
    out, lse = pk.paged_attn_prefill(pool, dev_bf16(q), dev(app.cu_new), bt, sl, 1024, scale)
    assert pk.poll_device_error() == pk.OK
    kr, vr = oracle.kv_append_bf16(kp, vp, app.k_new, app.v_new, app.cu_new,
                                   app.layout.block_table, app.seq_lens)
    ro, rl = oracle.paged_attention(kr, vr, q, app.cu_new, app.layout.block_table,
                                    app.seq_lens, scale)
    check_out(out, ro, "prompt 1024")
    check_lse(lse, rl, "prompt 1024")


def test_page_permutation_is_bit_identical(pk):
    rng = np.random.default_rng(62)
    case, q, cu, mq = chunk_case(rng, [(200, 500)], Hq=8, Hkv=2)
    out1, lse1 = run(pk, case, q, cu, mq)
    perm = rng.permutation(case.k_pool.shape[0])
    kp2 = np.empty_like(case.k_pool)
    vp2 = np.empty_like(case.v_pool)
    kp2[perm] = case.k_pool
    vp2[perm] = case.v_pool
    case2 = W.DecodeCase(case.Hq, case.Hkv, case.seq_lens,
                         W.Layout(case.layout.num_pages,
                                  perm[case.layout.block_table].astype(np.int32), 0),
                         case.q, kp2, vp2)
    out2, lse2 = run(pk, case2, q, cu, mq)
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


def test_mixed_step_chunks_sampled(pk):
    """The 26,926-token prompt in 2,048-row chunks at full size: append every
    chunk; check all rows of the first chunk and seeded samples of the middle
    and last (302-row) chunks against the oracle."""
    wl = W.mixed_step(R=1, lo=128, hi=256)
    pool = pk.Pool(dev_bf16(wl.k_pool), dev_bf16(wl.v_pool))
    bt_all = wl.layout.block_table
    bt = dev(bt_all[:1])
    kp, vp = wl.k_pool, wl.v_pool
    scale = 1.0 / np.sqrt(D)
    rng = np.random.default_rng(63)
    checks = {0: None, 6: 24, len(wl.steps) - 1: 24}
    for c, s in enumerate(wl.steps):
        cu = W.cu_from_counts([s.chunk_len])
        lens = np.array([s.prefill_len], np.int32)
        k_new, v_new = s.k_new[:s.chunk_len], s.v_new[:s.chunk_len]
        pk.kv_append(pool, dev_bf16(k_new), dev_bf16(v_new), dev(cu), bt, dev(lens))
        kp, vp = oracle.kv_append_bf16(kp, vp, k_new, v_new, cu, bt_all[:1], lens)
        if c not in checks:
            continue
        out, lse = pk.paged_attn_prefill(pool, dev_bf16(s.q_chunk), dev(cu), bt, dev(lens),
                                         s.chunk_len, scale)
        assert pk.poll_device_error() == pk.OK
        n = checks[c]
        rows = np.arange(s.chunk_len, dtype=np.int32) if n is None else \
            np.sort(rng.choice(s.chunk_len, n, replace=False)).astype(np.int32)
        if c == len(wl.steps) - 1:
            rows = np.unique(np.concatenate([rows, [0, s.chunk_len - 1]])).astype(np.int32)
        ro, rl = oracle.paged_attention(kp, vp, s.q_chunk, cu, bt_all[:1], lens, scale,
                                        rows=rows)
        idx = torch.from_numpy(rows).long().cuda()
        check_out(out[idx], ro, f"mixed chunk {c}")
        check_lse(lse[idx], rl, f"mixed chunk {c}")


def test_empty_chunk_is_a_no_op(pk):
    rng = np.random.default_rng(64)
    case, q, cu, mq = chunk_case(rng, [(0, 40), (8, 40)], Hq=4, Hkv=2)
    out, lse = run(pk, case, q, cu, mq)
    ro, rl = ref(case, q, cu)
    check_out(out, ro, "empty chunk")
    check_lse(lse, rl, "empty chunk")


def test_one_unit_split_over_many_ctas(pk):
    """A single (sequence, tile pair, head) unit long enough to be cut over
    about thirty CTAs: every part is merged by the log-sum-exp rule."""
    rng = np.random.default_rng(65)
    case, q, cu, mq = chunk_case(rng, [(256, 8192)], Hq=1, Hkv=1)
    out, lse = run(pk, case, q, cu, mq)
    ro, rl = ref(case, q, cu)
    check_out(out, ro, "one unit, many parts")
    check_lse(lse, rl, "one unit, many parts")


def test_many_short_sequences(pk):
    """Forty sequences of 1-300 rows: many segments per CTA, pairs whose
    second tile is past the chunk, units cut anywhere."""
    rng = np.random.default_rng(66)
    qlens = rng.integers(1, 301, size=40)
    shapes = [(int(n), int(n + rng.integers(0, 700))) for n in qlens]
    case, q, cu, mq = chunk_case(rng, shapes, Hq=8, Hkv=2)
    out, lse = run(pk, case, q, cu, mq)
    ro, rl = ref(case, q, cu)
    check_out(out, ro, "many short")
    check_lse(lse, rl, "many short")


def test_workspace_reuse_is_exact(pk):
    """One workspace over a series of different calls gives the same bits as
    a fresh workspace per call (the part counters return to zero), and the
    same call twice gives the same bits (the merge order is fixed, whichever
    CTA finishes last)."""
    rng = np.random.default_rng(67)
    calls = []
    for shapes in ([(700, 3000)], [(256, 4096), (33, 90)], [(1000, 1000)]):
        case, q, cu, mq = chunk_case(rng, shapes, Hq=8, Hkv=2)
        pool = pk.Pool(dev_bf16(case.k_pool), dev_bf16(case.v_pool))
        args = (pool, dev_bf16(q), dev(cu), dev(case.layout.block_table), dev(case.seq_lens),
                mq, case.scale)
        fresh = pk.paged_attn_prefill(*args)
        assert pk.poll_device_error() == pk.OK
        ro, rl = ref(case, q, cu)
        check_out(fresh[0], ro, f"reuse {shapes}")
        check_lse(fresh[1], rl, f"reuse {shapes}")
        calls.append((args, fresh))
    ws = pk.prefill_workspace()
    zero_bytes = pk.prefill_plan()[2]
    for _ in range(2):
        for args, (o0, l0) in calls:
            o, l = pk.paged_attn_prefill(*args, workspace=ws)
            assert torch.equal(o, o0) and torch.equal(l, l0)
    assert pk.poll_device_error() == pk.OK
    assert int(ws[:zero_bytes].count_nonzero()) == 0


@pytest.mark.parametrize("num_ctas", [1, 7, 61])
def test_fewer_persistent_ctas(pk, num_ctas):
    """num_ctas below the SM count (the prefill beside a decode on another
    stream): the same work in fewer persistent CTAs -- whole units, cut
    units and a head-pair chunk tail -- matches the oracle and leaves the
    workspace's part counters at zero; a call on every SM with units cut
    over many CTAs then shares that workspace and still matches (the
    partial results of the first call never sit where its counters go)."""
    rng = np.random.default_rng(68 + num_ctas)
    ws = pk.prefill_workspace()
    zero_bytes = pk.prefill_plan()[2]
    for shapes, n in (([(1000, 3000), (130, 4100), (33, 90), (1, 700)], num_ctas),
                      ([(256, 8192), (700, 2000)], 0)):
        case, q, cu, mq = chunk_case(rng, shapes, Hq=8, Hkv=2)
        pool = pk.Pool(dev_bf16(case.k_pool), dev_bf16(case.v_pool))
        out, lse = pk.paged_attn_prefill(pool, dev_bf16(q), dev(cu),
                                         dev(case.layout.block_table), dev(case.seq_lens), mq,
                                         case.scale, workspace=ws, num_ctas=n)
        assert pk.poll_device_error() == pk.OK
        ro, rl = ref(case, q, cu)
        check_out(out, ro, f"{n} CTAs")
        check_lse(lse, rl, f"{n} CTAs")
        assert int(ws[:zero_bytes].count_nonzero()) == 0
