"""kv_append on the GPU against the oracle: every byte of the pool (bf16) or
every code and scale bit (INT8) must match; slots not named stay untouched.
(TileInfer.jl "Performance" page: the KV cache write; "INT8 KV cache".)"""
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


def run_bf16(pk, app: W.AppendCase, k_pool, v_pool):
    pool = pk.Pool(dev_bf16(k_pool), dev_bf16(v_pool))
    pk.kv_append(pool, dev_bf16(app.k_new), dev_bf16(app.v_new), dev(app.cu_new),
                 dev(app.layout.block_table), dev(app.seq_lens))
    assert pk.poll_device_error() == pk.OK
    return host_bits(pool.k), host_bits(pool.v)


def run_int8(pk, app: W.AppendCase, pools):
    k8, v8, ks, vs = pools
    pool = pk.Pool(dev(k8), dev(v8), dev(ks), dev(vs))
    smooth = dev(app.k_smooth) if app.k_smooth is not None else None
    pk.kv_append(pool, dev_bf16(app.k_new), dev_bf16(app.v_new), dev(app.cu_new),
                 dev(app.layout.block_table), dev(app.seq_lens), k_smooth=smooth)
    assert pk.poll_device_error() == pk.OK
    return (pool.k.cpu().numpy(), pool.v.cpu().numpy(), pool.k_scale.cpu().numpy(),
            pool.v_scale.cpu().numpy())


def test_bf16_prompt_1024_tokens(pk):
    app, _ = W.prefill_prompt()
    kp, vp = W.empty_pool_bf16(app.layout.num_pages, app.Hkv)
    gk, gv = run_bf16(pk, app, kp, vp)
    rk, rv = oracle.kv_append_bf16(kp, vp, app.k_new, app.v_new, app.cu_new,
                                   app.layout.block_table, app.seq_lens)
    assert np.array_equal(gk, rk) and np.array_equal(gv, rv)


def ragged_case(rng, Hkv=3, smooth=False):
    before = np.array([0, 14, 31, 100, 7, 0], np.int32)
    n_new = np.array([20, 5, 1, 33, 0, 16], np.int32)
    lens = before + n_new
    layout = W.scatter_pages(rng, lens)
    T = int(n_new.sum())
    w = W.smoothing_weight(rng) if smooth else None
    k_new = W.keys_with_channel_weight(rng, (T, Hkv, W.HEAD_DIM), w) if smooth else \
        W.normal_bf16(rng, (T, Hkv, W.HEAD_DIM))
    v_new = W.normal_bf16(rng, (T, Hkv, W.HEAD_DIM))
    return W.AppendCase(Hkv, W.cu_from_counts(n_new), lens, layout, k_new, v_new, k_smooth=w)


def test_bf16_ragged_sequences(pk):
    app = ragged_case(np.random.default_rng(21))
    kp, vp = W.empty_pool_bf16(app.layout.num_pages, app.Hkv)
    gk, gv = run_bf16(pk, app, kp, vp)
    rk, rv = oracle.kv_append_bf16(kp, vp, app.k_new, app.v_new, app.cu_new,
                                   app.layout.block_table, app.seq_lens)
    assert np.array_equal(gk, rk) and np.array_equal(gv, rv)


def test_bf16_mixed_step_rows(pk):
    """One step of the mixed workload: a 2,048-row chunk plus one row for each
    of 32 decode sequences (shrunk prompt, same structure)."""
    wl = W.mixed_step(prompt_len=2048 + 300, chunk=2048, R=32, lo=128, hi=2000, steps=2)
    kp, vp = wl.k_pool, wl.v_pool
    for s in wl.steps:
        cu, lens = wl.step_append(s)
        app = W.AppendCase(wl.Hkv, cu, lens, wl.layout, s.k_new, s.v_new)
        gk, gv = run_bf16(pk, app, kp, vp)
        kp, vp = oracle.kv_append_bf16(kp, vp, s.k_new, s.v_new, cu, wl.layout.block_table,
                                       lens)
        assert np.array_equal(gk, kp) and np.array_equal(gv, vp)


@pytest.mark.parametrize("smooth", [False, True])
def test_int8_ragged_sequences(pk, smooth):
    app = ragged_case(np.random.default_rng(22), smooth=smooth)
    pools = W.empty_pool_int8(app.layout.num_pages, app.Hkv)
    got = run_int8(pk, app, pools)
    ref = oracle.kv_append_int8(*pools, app.k_new, app.v_new, app.cu_new,
                                app.layout.block_table, app.seq_lens, k_smooth=app.k_smooth)
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])
    # scales bit for bit (NaN sentinels of untouched slots compare as equal bits)
    assert np.array_equal(got[2].view(np.uint32), ref[2].view(np.uint32))
    assert np.array_equal(got[3].view(np.uint32), ref[3].view(np.uint32))


@pytest.mark.parametrize("smooth", [True, False])
def test_int8_32k_context(pk, smooth):
    app, _ = W.int8_long_decode(B=1)
    if not smooth:
        app.k_smooth = None
    pools = W.empty_pool_int8(app.layout.num_pages, app.Hkv)
    got = run_int8(pk, app, pools)
    ref = oracle.kv_append_int8(*pools, app.k_new, app.v_new, app.cu_new,
                                app.layout.block_table, app.seq_lens, k_smooth=app.k_smooth)
    for g, r in zip(got, ref):
        assert np.array_equal(g.view(np.uint8), r.view(np.uint8))


def test_int8_zero_and_tie_vectors(pk):
    """All-zero vectors store scale 0 and codes 0; exact .5 quotients round to even."""
    Hkv = 1
    x = np.zeros((3, Hkv, W.HEAD_DIM), np.float32)
    x[1, 0, :6] = [127, -63.5, 0.5, 1.5, 2.5, -2.5]
    x[2, 0, :3] = [254, 3, 5]
    bits = W.to_bf16_bits(x)
    lens = np.array([3], np.int32)
    layout = W.scatter_pages(np.random.default_rng(23), lens)
    app = W.AppendCase(Hkv, W.cu_from_counts([3]), lens, layout, bits, bits)
    pools = W.empty_pool_int8(layout.num_pages, Hkv)
    got = run_int8(pk, app, pools)
    page = layout.block_table[0, 0]
    assert got[2][page, 0, 0] == 0.0 and not got[0][page, 0, 0].any()
    assert list(got[0][page, 0, 1, :6]) == [127, -64, 0, 2, 2, -2]
    assert got[2][page, 0, 2] == 2.0 and list(got[0][page, 0, 2, :3]) == [127, 2, 2]


def test_device_check_flags_a_position_past_the_block_table(pk):
    """seq_lens beyond the block table: the row is skipped and the poll reports it."""
    app, _ = W.prefill_prompt(T=32)
    kp, vp = W.empty_pool_bf16(app.layout.num_pages, app.Hkv)
    pool = pk.Pool(dev_bf16(kp), dev_bf16(vp))
    bad_lens = app.seq_lens + 10**6
    pk.kv_append(pool, dev_bf16(app.k_new), dev_bf16(app.v_new), dev(app.cu_new),
                 dev(app.layout.block_table), dev(bad_lens))
    assert pk.poll_device_error() == pk.ERR_INVALID
    assert np.array_equal(host_bits(pool.k), kp)          # nothing written
    assert pk.poll_device_error() == pk.OK                # cleared
