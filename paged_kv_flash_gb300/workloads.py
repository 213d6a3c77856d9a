"""Seeded synthetic inputs for the paged-KV attention workloads.

This module only draws random numbers and lays them out (pool pages, block
tables, sequence lengths, query rows).  It holds none of the attention or
quantisation arithmetic, so the CUDA path and the CPU oracle can both be fed
from it without sharing any of the method.

Shapes follow the workloads the pages run (TileInfer.jl "Performance" page:
Qwen3-4B / Qwen3-0.6B decode and 1,024-token prefill, the INT8 KV cache at
32,768 positions; Qml-engine landing page: Llama-3.1-8B with a 26,926-token
prompt): head_dim 128, 16-token pages, GQA 16/8 or 32/8 heads.

Conventions shared by every generator:
  * bf16 values are carried as uint16 bit patterns (round-to-nearest-even
    from float32 draws); the same bits go to the GPU and to the oracle.
  * Pools are [num_pages][Hkv][page_size][head_dim]; K and V separate.
  * Pages that no sequence owns, and slots past a sequence's length, hold a
    NaN sentinel (bf16) or a NaN scale (int8) so that a stray read shows.
  * Block-table entries past a sequence's last page name a sentinel page.
"""
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

PAGE = 16
HEAD_DIM = 128
BF16_NAN = np.uint16(0x7FC0)
BASE_SEED = 1000


def rng_for(workload_index: int, salt: int = 0) -> np.random.Generator:
    """Generator seeded 1000 + workload index (+ salt for extra streams)."""
    return np.random.default_rng(BASE_SEED + workload_index + 7919 * salt)


def to_bf16_bits(x) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even.  Inputs are finite,
    so the 32-bit sum below cannot wrap (largest: 0xFF7FFFFF + 0x8000)."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32)
    r = (u >> 16) & np.uint32(1)
    r += np.uint32(0x7FFF)
    r += u
    r >>= 16
    return r.astype(np.uint16)


def bits_to_float(b) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


@dataclass
class Layout:
    """Pages of a shared pool handed out to sequences."""
    num_pages: int
    block_table: np.ndarray          # int32 [B][max_pages]
    sentinel_page: int               # never owned; block-table filler


def scatter_pages(rng, lens, max_len=None, slack=0.10, min_pages=0) -> Layout:
    """Give each sequence ceil(len/16) pages (room for max_len) drawn without
    replacement from a random permutation of a pool with `slack` spare pages.
    The last pool page is a sentinel that no sequence owns."""
    lens = np.asarray(lens, dtype=np.int64)
    cap = lens if max_len is None else np.maximum(lens, np.asarray(max_len, dtype=np.int64))
    need = (cap + PAGE - 1) // PAGE
    total = int(need.sum())
    num_pages = max(int(np.ceil(total * (1.0 + slack))) + 1, min_pages, total + 1)
    perm = rng.permutation(num_pages - 1).astype(np.int32)
    sentinel = num_pages - 1
    max_pages = int(need.max()) if len(need) else 1
    bt = np.full((len(lens), max(max_pages, 1)), sentinel, dtype=np.int32)
    off = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[off:off + n]
        off += int(n)
    return Layout(num_pages, bt, sentinel)


def empty_pool_bf16(num_pages, Hkv):
    shape = (num_pages, Hkv, PAGE, HEAD_DIM)
    return np.full(shape, BF16_NAN, np.uint16), np.full(shape, BF16_NAN, np.uint16)


def empty_pool_int8(num_pages, Hkv, code_fill=0x5A):
    shape = (num_pages, Hkv, PAGE, HEAD_DIM)
    k = np.full(shape, code_fill, np.int8)
    v = np.full(shape, code_fill, np.int8)
    ks = np.full(shape[:3], np.nan, np.float32)
    vs = np.full(shape[:3], np.nan, np.float32)
    return k, v, ks, vs


def fill_pool_bf16(rng, layout: Layout, lens, Hkv, k_pool, v_pool):
    """Write N(0,1) bf16 K and V at every cached position of every sequence."""
    for b, L in enumerate(np.asarray(lens)):
        npg = (int(L) + PAGE - 1) // PAGE
        if npg == 0:
            continue
        pages = layout.block_table[b, :npg]
        kk = normal_bf16(rng, (npg, Hkv, PAGE, HEAD_DIM))
        vv = normal_bf16(rng, (npg, Hkv, PAGE, HEAD_DIM))
        tail = npg * PAGE - int(L)
        if tail:
            kk[-1, :, PAGE - tail:, :] = BF16_NAN
            vv[-1, :, PAGE - tail:, :] = BF16_NAN
        k_pool[pages] = kk
        v_pool[pages] = vv


def cu_from_counts(counts) -> np.ndarray:
    c = np.zeros(len(counts) + 1, np.int32)
    c[1:] = np.cumsum(np.asarray(counts, dtype=np.int64))
    return c


@dataclass
class DecodeCase:
    """q_b = 1 per sequence, the pool already holds every position."""
    Hq: int
    Hkv: int
    seq_lens: np.ndarray             # int32 [B]
    layout: Layout
    q: np.ndarray                    # uint16 [B][Hq][D]
    k_pool: np.ndarray
    v_pool: np.ndarray
    k_scale: Optional[np.ndarray] = None
    v_scale: Optional[np.ndarray] = None
    k_smooth: Optional[np.ndarray] = None
    scale: float = 1.0 / np.sqrt(HEAD_DIM)

    @property
    def B(self):
        return int(self.seq_lens.shape[0])


def decode_bf16(rng, lens, Hq, Hkv, slack=0.10, layout=None) -> DecodeCase:
    lens = np.asarray(lens, dtype=np.int32)
    layout = layout or scatter_pages(rng, lens, slack=slack)
    k_pool, v_pool = empty_pool_bf16(layout.num_pages, Hkv)
    fill_pool_bf16(rng, layout, lens, Hkv, k_pool, v_pool)
    q = normal_bf16(rng, (len(lens), Hq, HEAD_DIM))
    return DecodeCase(Hq, Hkv, lens, layout, q, k_pool, v_pool)


@dataclass
class MultiCase:
    """A step of q_lens[b] new tokens per sequence (1..16, e.g. a speculative
    verify step) over a bf16 cache of seq_lens[b] positions that already holds
    them; q rows cu_q[b]..cu_q[b+1]-1 belong to sequence b."""
    Hq: int
    Hkv: int
    seq_lens: np.ndarray             # int32 [B]
    q_lens: np.ndarray               # int32 [B]
    cu_q: np.ndarray                 # int32 [B+1]
    layout: Layout
    q: np.ndarray                    # uint16 bf16 bits [T][Hq][D]
    k_pool: np.ndarray
    v_pool: np.ndarray
    scale: float = 1.0 / np.sqrt(HEAD_DIM)


def multi_token_decode(rng, lens, q_lens, Hq, Hkv) -> MultiCase:
    """Scattered pages filled with N(0,1) K/V for `lens` positions, and
    N(0,1) queries for the last q_lens[b] positions of each sequence."""
    dc = decode_bf16(rng, lens, Hq, Hkv)
    q_lens = np.asarray(q_lens, np.int32)
    q = normal_bf16(rng, (int(q_lens.sum()), Hq, HEAD_DIM))
    return MultiCase(Hq, Hkv, dc.seq_lens, q_lens, cu_from_counts(q_lens), dc.layout, q,
                     dc.k_pool, dc.v_pool)


def smoothing_weight(rng) -> np.ndarray:
    """Per-channel key weight w_c ~ U[0.5, 2] (float32), shared by all heads."""
    return rng.uniform(0.5, 2.0, HEAD_DIM).astype(np.float32)


def keys_with_channel_weight(rng, shape, w) -> np.ndarray:
    """K = N(0,1) * w_c rounded to bf16 (channel = last axis)."""
    x = rng.standard_normal(shape, dtype=np.float32) * w.astype(np.float32)
    return to_bf16_bits(x)


@dataclass
class AppendCase:
    """New K/V rows for several sequences: rows cu_new[b]..cu_new[b+1]-1 belong to
    sequence b and land at positions seq_lens[b] - n_b .. seq_lens[b] - 1."""
    Hkv: int
    cu_new: np.ndarray               # int32 [B+1]
    seq_lens: np.ndarray             # int32 [B], after the append
    layout: Layout
    k_new: np.ndarray                # uint16 [T][Hkv][D]
    v_new: np.ndarray
    k_smooth: Optional[np.ndarray] = None


# ---------------------------------------------------------------- configs
# The five workloads, by what they are.  Each returns plain numpy arrays.

def decode_1k(seed_index=1, L=1024, Hq=16, Hkv=8) -> DecodeCase:
    """Single-sequence decode, Qwen3-0.6B-like GQA 16/8, 1,024 positions in 64
    pages; the block table is a random permutation of the pool's 64 pages."""
    rng = rng_for(seed_index)
    npg = (L + PAGE - 1) // PAGE
    perm = rng.permutation(npg).astype(np.int32)
    bt = np.full((1, npg), npg, np.int32)
    bt[0, :] = perm
    layout = Layout(npg + 1, bt, npg)    # +1: the sentinel page
    return decode_bf16(rng, [L], Hq, Hkv, layout=layout)


def prefill_prompt(seed_index=2, T=1024, Hq=32, Hkv=8):
    """One causal prompt of T tokens, Qwen3-4B-like GQA 32/8: the K/V rows to
    append (into pages of a seeded random block table) and the T query rows."""
    rng = rng_for(seed_index)
    layout = scatter_pages(rng, [T], slack=0.0)
    k_new = normal_bf16(rng, (T, Hkv, HEAD_DIM))
    v_new = normal_bf16(rng, (T, Hkv, HEAD_DIM))
    q = normal_bf16(rng, (T, Hq, HEAD_DIM))
    app = AppendCase(Hkv, cu_from_counts([T]), np.array([T], np.int32), layout, k_new, v_new)
    return app, q


def batched_decode(seed_index=3, B=64, Hq=32, Hkv=8, lo=512, hi=8192) -> DecodeCase:
    """Llama-3.1-8B-like GQA 32/8, B sequences with lengths ~ U{lo..hi}, pages
    scattered across one shared pool (10 % spare pages)."""
    rng = rng_for(seed_index)
    lens = rng.integers(lo, hi + 1, size=B).astype(np.int32)
    return decode_bf16(rng, lens, Hq, Hkv)


def int8_long_decode(seed_index=4, B=1, L=32768, Hq=32, Hkv=8):
    """Qwen3-4B-like GQA 32/8 at L positions with an INT8 cache: returns the
    append case that fills the whole context (K = N(0,1) * w_c, V = N(0,1)),
    the decode queries and the smoothing weight w."""
    rng = rng_for(seed_index, salt=B)
    lens = np.full(B, L, np.int32)
    layout = scatter_pages(rng, lens, slack=0.0)
    w = smoothing_weight(rng)
    k_new = keys_with_channel_weight(rng, (B * L, Hkv, HEAD_DIM), w)
    v_new = normal_bf16(rng, (B * L, Hkv, HEAD_DIM))
    q = normal_bf16(rng, (B, Hq, HEAD_DIM))
    app = AppendCase(Hkv, cu_from_counts(lens), lens, layout, k_new, v_new, k_smooth=w)
    return app, q


@dataclass
class MixedStep:
    """Step c of the mixed continuous-batching workload: append the chunk's
    K/V plus one token per decode row, prefill the chunk, decode the rows."""
    chunk_lo: int
    chunk_len: int
    prefill_len: int                 # cached positions of the prompt after the chunk
    decode_lens: np.ndarray          # int32 [R], after this step's token
    q_chunk: np.ndarray              # uint16 [chunk_len][Hq][D]
    q_decode: np.ndarray             # uint16 [R][Hq][D]
    k_new: np.ndarray                # uint16 [chunk_len + R][Hkv][D]
    v_new: np.ndarray


@dataclass
class MixedWorkload:
    Hq: int
    Hkv: int
    prompt_len: int
    chunk: int
    layout: Layout                   # row 0: the prompt; rows 1..R: decode rows
    k_pool: np.ndarray
    v_pool: np.ndarray
    decode_lens0: np.ndarray         # positions cached before step 0
    steps: list = field(default_factory=list)

    def step_append(self, s: MixedStep):
        """(cu_new, seq_lens) of the step's append over sequences 0..R."""
        R = len(self.decode_lens0)
        cu = cu_from_counts([s.chunk_len] + [1] * R)
        lens = np.concatenate([[s.prefill_len], s.decode_lens]).astype(np.int32)
        return cu, lens


def mixed_step(seed_index=5, prompt_len=26926, chunk=2048, R=32, Hq=32, Hkv=8,
               lo=128, hi=16384, steps=None) -> MixedWorkload:
    """Llama-3.1-8B-like GQA 32/8: one prompt prefilled in `chunk`-token chunks
    against its own cached prefix, plus R decode rows with contexts ~ U{lo..hi}
    that each gain one token per step; one shared pool of 16-token pages."""
    rng = rng_for(seed_index)
    nsteps_all = (prompt_len + chunk - 1) // chunk
    nsteps = nsteps_all if steps is None else min(steps, nsteps_all)
    lens0 = rng.integers(lo, hi + 1, size=R).astype(np.int32)
    final = np.concatenate([[prompt_len], lens0 + nsteps_all]).astype(np.int64)
    layout = scatter_pages(rng, np.zeros(R + 1, np.int64), max_len=final)
    k_pool, v_pool = empty_pool_bf16(layout.num_pages, Hkv)
    # decode rows' initial contexts
    sub = Layout(layout.num_pages, layout.block_table[1:], layout.sentinel_page)
    fill_pool_bf16(rng, sub, lens0, Hkv, k_pool, v_pool)
    wl = MixedWorkload(Hq, Hkv, prompt_len, chunk, layout, k_pool, v_pool, lens0)
    for c in range(nsteps):
        lo_c = c * chunk
        n = min(chunk, prompt_len - lo_c)
        dl = (lens0 + c + 1).astype(np.int32)
        wl.steps.append(MixedStep(
            chunk_lo=lo_c, chunk_len=n, prefill_len=lo_c + n, decode_lens=dl,
            q_chunk=normal_bf16(rng, (n, Hq, HEAD_DIM)),
            q_decode=normal_bf16(rng, (R, Hq, HEAD_DIM)),
            k_new=normal_bf16(rng, (n + R, Hkv, HEAD_DIM)),
            v_new=normal_bf16(rng, (n + R, Hkv, HEAD_DIM))))
    return wl


# ------------------------------------------------ fused attention inputs

def rope_tables(max_pos, base=1.0e6, D=HEAD_DIM):
    """A model's RoPE cos/sin table, fp32 [max_pos][D/2]: angle p * base^(-2i/D)
    (Qwen3-style base 1e6).  An input of the fused step, like its weights."""
    inv = base ** (-np.arange(0, D, 2, dtype=np.float64) / D)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


@dataclass
class QkvPrepCase:
    Hq: int
    Hkv: int
    qkv: np.ndarray          # uint16 bf16 bits [T][Hq + 2 Hkv][D]
    q_w: np.ndarray          # fp32 [D] (bf16-representable, like stored weights)
    k_w: np.ndarray
    cos: np.ndarray          # fp32 [max_pos][D/2]
    sin: np.ndarray
    cu_new: np.ndarray       # int32 [B+1]
    seq_lens: np.ndarray     # int32 [B], new tokens included
    layout: Layout


def qkv_prep_case(seed, new_counts, totals, Hq=32, Hkv=8, max_pos=None):
    """Seeded inputs of the fused attention-input step: a projection output
    with N(0, 1) bf16 entries, norm weights U[0.5, 1.5] rounded to bf16, the
    RoPE table, and scattered pages for sequences of `totals` positions whose
    last `new_counts` are the new tokens."""
    rng = np.random.default_rng(seed)
    new_counts = np.asarray(new_counts, np.int32)
    totals = np.asarray(totals, np.int32)
    T = int(new_counts.sum())
    qkv = normal_bf16(rng, (T, Hq + 2 * Hkv, HEAD_DIM))
    q_w = bits_to_float(to_bf16_bits(rng.uniform(0.5, 1.5, HEAD_DIM).astype(np.float32)))
    k_w = bits_to_float(to_bf16_bits(rng.uniform(0.5, 1.5, HEAD_DIM).astype(np.float32)))
    cos, sin = rope_tables(int(totals.max()) if max_pos is None else max_pos)
    layout = scatter_pages(rng, totals)
    return QkvPrepCase(Hq, Hkv, qkv, q_w.astype(np.float32), k_w.astype(np.float32), cos, sin,
                       cu_from_counts(new_counts), totals, layout)
