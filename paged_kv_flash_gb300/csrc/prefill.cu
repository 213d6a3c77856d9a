// prefill.cu -- causal chunked prefill attention over the paged cache on the
// 5th-generation tensor cores (tcgen05 MMAs, TMEM accumulators, TMA loads).
//
// The method: TileInfer.jl "Performance" page -- paged flash attention runs
// an online softmax over the pages read in place through the block table
// ("Fused kernels, FlashAttention and PagedAttention"); the prefill kernel
// runs a block per head over every page ("Attention for verify steps");
// chunked prefill attends a chunk of new rows to the cached prefix ("What is
// left to gain").  Rows sit bottom-right: row i of a chunk of q rows in a
// sequence of L cached positions is position L - q + i and sees keys 0..it.
//
// One CTA per (query head, 128-row query tile, sequence); 6 warps:
//   warp 0     TMA producer: 128-key K and V blocks, each gathered as eight
//              16-row page boxes (one per page named by the block table) per
//              64-channel half, 128-byte swizzled, 2-stage ring per operand;
//   warp 1     MMA issuer (one thread): S = Q K^T into TMEM (double
//              buffered, 2 x 128 columns), O += P V into TMEM (128 columns);
//   warps 2-5  softmax: thread = query row = TMEM lane; reads S with
//              tcgen05.ld, keeps the running max and sum of its row, rescales
//              O in TMEM only when its max grows by more than 2^8 (exact: the
//              final normalisation uses the same stale max), writes P as bf16
//              into shared memory in the swizzled K-major layout the PV MMA
//              reads, and finally normalises O and writes out and lse.
// Q is loaded once by the softmax warps (rows past the chunk are zero) into
// the same swizzled layout.  V rows at positions >= L in the last block are
// zeroed by the MMA warp before the PV MMA, so stale or poisoned pool slots
// can never reach the accumulator (P is 0 there, but 0 * NaN is NaN).
//
// Every wait is bounded (wall clock, one second); a wait that runs out sets
// the device error word and an abort flag that makes every role leave its
// loop; the MMA warp drains its issued MMAs and the producer its loads
// before TMEM is freed and the CTA exits.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"

namespace {

using namespace pkv;

__device__ uint32_t g_err_prefill;

constexpr int BM = 128;                       // query rows per tile (= TMEM lanes)
constexpr int BN = 128;                       // keys per block (8 pages)
constexpr int NSTAGE = 2;                     // K and V ring depth
constexpr int HALF = 16384;                   // one 128 x 64 bf16 swizzled half-tile
constexpr int TILE = 2 * HALF;                // 128 x 128 bf16
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_O = 256;                // O accumulator columns 256..383

// Shared-memory map (offsets from a 1024-byte aligned base).
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + TILE;
constexpr int OFF_V = OFF_K + NSTAGE * TILE;
constexpr int OFF_P = OFF_V + NSTAGE * TILE;
constexpr int OFF_BAR = OFF_P + TILE;
// barriers: q_full, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2],
// s_free[2], p_full, pv_done, drain
constexpr int BAR_Q = 0, BAR_KF = 1, BAR_KE = 3, BAR_VF = 5, BAR_VE = 7, BAR_SF = 9,
              BAR_SR = 11, BAR_PF = 13, BAR_PV = 14, BAR_DR = 15, NUM_BARS = 16;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;   // + alignment slack

// kind::f16 instruction descriptor: D fp32, A and B bf16, M = N = 128.
// bits 4-5 D format, 7-9 A format, 10-12 B format, 15/16 A/B major
// (0 = K-major, 1 = MN-major), 17-22 N >> 3, 24-28 M >> 4.
constexpr uint32_t IDESC_QK =
    (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
constexpr uint32_t IDESC_PV = IDESC_QK | (1u << 16);   // B (= V) is MN-major

// Shared-memory matrix descriptor, 128-byte swizzle: start address >> 4
// (bits 0-13), leading byte offset >> 4 (16-29), stride byte offset >> 4
// (32-45), descriptor version 1 (bit 46), swizzle mode 2 = 128B (61-63).
// K-major tiles: 8-row groups 1024 B apart (SBO); the leading offset is
// unused.  MN-major V tiles: 64-channel halves 16 KiB apart (LBO), 8-key
// groups 1024 B apart (SBO).
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)(HALF >> 4) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

#define PKV_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                  "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define PKV_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
                  "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : PKV_R8(0), PKV_R8(8), PKV_R8(16), PKV_R8(24)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      ::"r"(taddr), PKV_W8(0), PKV_W8(8), PKV_W8(16), PKV_W8(24)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Bounded wait shared by all roles; the result is uniform across the warp.
// Gives up when another role raised the abort flag or after kWaitLimitNs.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t* abort) {
  bool ok = mbar_try_wait(bar, parity);
  if (!ok) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
      if (mbar_try_wait(bar, parity)) { ok = true; break; }
      if ((it & 63u) == 0) {
        if (*abort) break;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          *abort = 1u;
          atomicOr(&g_err_prefill, kErrTimeout);
          break;
        }
      }
    }
  }
  return __all_sync(0xffffffffu, ok);
}

struct PrefillParams {
  pkv_host::PrefillLaunch a;
  int n_tiles;                  // tiles of the longest chunk
};

__global__ void __launch_bounds__(NUM_THREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                   const __grid_constant__ PrefillParams prm) {
  const pkv_host::PrefillLaunch& a = prm.a;
  const int hq = blockIdx.x;
  const int t = prm.n_tiles - 1 - (int)blockIdx.y;      // heaviest tiles first
  const int b = blockIdx.z;
  const int Hq = a.num_q_heads;
  const int G = Hq / a.num_kv_heads;
  const int hkv = hq / G;

  const int q0 = a.cu_q[b];
  const int q_len = a.cu_q[b + 1] - q0;
  if (q_len > prm.n_tiles * BM && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
    atomicOr(&g_err_prefill, kErrBadIndex);             // chunk longer than max_q_len
  if (t * BM >= q_len) return;                          // no rows in this tile
  const int L = a.seq_lens[b];
  if (L < q_len || L > a.max_pages * kPageSize) {
    if (threadIdx.x == 0) atomicOr(&g_err_prefill, kErrBadIndex);
    return;
  }
  const int pos_min = L - q_len + t * BM;                     // position of tile row 0
  const int rows = min(BM, q_len - t * BM);
  const int pos_max = pos_min + rows - 1;
  const int n_blk = pos_max / BN + 1;
  const int npages = (L + kPageSize - 1) / kPageSize;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_s - raw_s);
  auto bar = [&](int i) -> uint32_t { return base_s + OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(base + OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(bar(BAR_Q), 128);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(bar(BAR_KF + s), 1);
      mbar_init(bar(BAR_KE + s), 1);
      mbar_init(bar(BAR_VF + s), 1);
      mbar_init(bar(BAR_VE + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(BAR_SF + s), 1);
      mbar_init(bar(BAR_SR + s), 128);
    }
    mbar_init(bar(BAR_PF), 128);
    mbar_init(bar(BAR_PV), 1);
    mbar_init(bar(BAR_DR), 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(tmem_slot)), "r"(TMEM_COLS) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  int last_k[NSTAGE], last_v[NSTAGE];            // producer: last block issued per stage
  for (int s = 0; s < NSTAGE; ++s) last_k[s] = last_v[s] = -1;
  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    const int32_t* bt_row = a.block_table + (size_t)b * a.max_pages;
    bool ok = true;
    for (int j = 0; j < n_blk && ok; ++j) {
      const int st = j % NSTAGE;
      const int lp = j * (BN / kPageSize) + (lane & 7);
      int pg = 0;
      if (lane < 8 && lp < npages) {
        pg = __ldg(bt_row + lp);
        if (pg < 0 || pg >= a.num_pages) {
          atomicOr(&g_err_prefill, kErrBadIndex);
          pg = 0;
        }
      }
      int pgs[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) pgs[i] = __shfl_sync(0xffffffffu, pg, i);
      const int nload = min(BN / kPageSize, npages - j * (BN / kPageSize));
      const uint32_t bytes = (uint32_t)nload * 2u * (kPageSize * 64 * 2);
      if (j >= NSTAGE && !(ok = wait_bar(bar(BAR_KE + st), ((j / NSTAGE) - 1) & 1, abort_flag)))
        break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(BAR_KF + st), bytes);
        const uint32_t dst = base_s + OFF_K + st * TILE;
        for (int i = 0; i < nload; ++i) {
          const int row = (pgs[i] * a.num_kv_heads + hkv) * kPageSize;
          tma_load_2d(dst + i * 2048, &tk, 0, row, bar(BAR_KF + st));
          tma_load_2d(dst + HALF + i * 2048, &tk, 64, row, bar(BAR_KF + st));
        }
      }
      last_k[st] = j;
      if (j >= NSTAGE && !(ok = wait_bar(bar(BAR_VE + st), ((j / NSTAGE) - 1) & 1, abort_flag)))
        break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(BAR_VF + st), bytes);
        const uint32_t dst = base_s + OFF_V + st * TILE;
        for (int i = 0; i < nload; ++i) {
          const int row = (pgs[i] * a.num_kv_heads + hkv) * kPageSize;
          tma_load_2d(dst + i * 2048, &tv, 0, row, bar(BAR_VF + st));
          tma_load_2d(dst + HALF + i * 2048, &tv, 64, row, bar(BAR_VF + st));
        }
      }
      last_v[st] = j;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    auto pv = [&](int jj) -> bool {
      const int st = jj % NSTAGE;
      if (!wait_bar(bar(BAR_PF), jj & 1, abort_flag)) return false;
      if (!wait_bar(bar(BAR_VF + st), (jj / NSTAGE) & 1, abort_flag)) return false;
      const int kbase = jj * BN;
      if (kbase + BN > L) {
        // zero V rows at positions >= L (both 64-channel halves of each row)
        const int first = L - kbase;
        uint8_t* vt = base + OFF_V + st * TILE;
        for (int idx = lane; idx < (BN - first) * 16; idx += 32) {
          const int row = first + (idx >> 4), c = idx & 15;
          *reinterpret_cast<uint4*>(vt + (c >> 3) * HALF + row * 128 + (c & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_async_smem();
        __syncwarp();
      }
      tc_fence_after();
      if (lane == 0) {
        const uint32_t p_s = base_s + OFF_P, v_s = base_s + OFF_V + st * TILE;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_bf16(tmem + TM_O, desc_kmajor(p_s + (kk >> 2) * HALF + (kk & 3) * 32),
                   desc_mnmajor(v_s + kk * 2048), IDESC_PV, (jj > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(BAR_PV));
        mma_commit(bar(BAR_VE + st));
      }
      __syncwarp();
      return true;
    };
    bool ok = wait_bar(bar(BAR_Q), 0, abort_flag);
    for (int j = 0; j < n_blk && ok; ++j) {
      const int st = j % NSTAGE;
      if (!(ok = wait_bar(bar(BAR_KF + st), (j / NSTAGE) & 1, abort_flag))) break;
      if (j >= 2 && !(ok = wait_bar(bar(BAR_SR + (j & 1)), ((j - 2) >> 1) & 1, abort_flag))) break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t q_s = base_s + OFF_Q, k_s = base_s + OFF_K + st * TILE;
#pragma unroll
        for (int kk = 0; kk < kHeadDim / 16; ++kk) {
          const uint32_t off = (kk >> 2) * HALF + (kk & 3) * 32;
          mma_bf16(tmem + (j & 1) * BN, desc_kmajor(q_s + off), desc_kmajor(k_s + off), IDESC_QK,
                   kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(BAR_SF + (j & 1)));
        mma_commit(bar(BAR_KE + st));
      }
      __syncwarp();
      if (j >= 1) ok = pv(j - 1);
    }
    if (ok) ok = pv(n_blk - 1);
    // drain: every MMA issued above completes before TMEM is released
    if (lane == 0) mma_commit(bar(BAR_DR));
    __syncwarp();
    (void)mbar_wait(bar(BAR_DR), 0);
  } else {
    // ---------------------------------------------------------- softmax
    const int quarter = warp & 3;                 // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane;            // row of the tile
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    const int pos_r = min(pos_min + r, L - 1);    // padding rows clamp to the last key
    const bool row_valid = r < rows;

    // Q tile -> swizzled shared memory (rows past the chunk are zero).
    {
      const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(a.q);
      uint8_t* qs = base + OFF_Q;
      for (int it = 0; it < 16; ++it) {
        const int row = quarter * 32 + 2 * it + (lane >> 4);
        const int c = lane & 15;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row < rows)
          v = __ldg(reinterpret_cast<const uint4*>(
                        qg + ((size_t)(q0 + t * BM + row) * Hq + hq) * kHeadDim) + c);
        *reinterpret_cast<uint4*>(qs + (c >> 3) * HALF + row * 128 + (((c & 7) ^ (row & 7)) << 4)) =
            v;
      }
      fence_async_smem();
      mbar_arrive(bar(BAR_Q));
    }

    const float sl2 = a.softmax_scale * kLog2e;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_blk; ++j) {
      if (!(ok = wait_bar(bar(BAR_SF + (j & 1)), (j >> 1) & 1, abort_flag))) break;
      tc_fence_after();
      float s[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(t_lane + (j & 1) * BN + 32 * c, rr);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) s[32 * c + i] = __uint_as_float(rr[i]);
      }
      tc_fence_before();
      mbar_arrive(bar(BAR_SR + (j & 1)));

      const int kbase = j * BN;
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (kbase + BN - 1 > pos_min) {               // block crosses the causal edge
        const int lim = pos_r - kbase;
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          s[c] = (c > lim) ? -INFINITY : s[c] * sl2;
          mx[c & 3] = fmaxf(mx[c & 3], s[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          s[c] *= sl2;
          mx[c & 3] = fmaxf(mx[c & 3], s[c]);
        }
      }
      const float m_blk = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      const float m_new = fmaxf(m_run, m_blk);
      const bool need = m_new > m_run + 8.0f;       // lazy rescale threshold (2^8)
      const float m_use = need ? m_new : m_run;
      const float alpha = need ? fast_exp2(m_run - m_use) : 1.0f;
      uint32_t pk[BN / 2];
      float sum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < BN / 2; ++c) {
        const float p0 = fast_exp2(s[2 * c] - m_use);
        const float p1 = fast_exp2(s[2 * c + 1] - m_use);
        sum[c & 3] += p0 + p1;
        pk[c] = pack_bf16(p0, p1);
      }
      l_run = l_run * alpha + ((sum[0] + sum[1]) + (sum[2] + sum[3]));
      m_run = m_use;

      if (j > 0) {
        // PV of the previous block must be done: the P buffer is free and O
        // holds every earlier block.
        if (!(ok = wait_bar(bar(BAR_PV), (j - 1) & 1, abort_flag))) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, need)) {
#pragma unroll
          for (int c = 0; c < kHeadDim / 32; ++c) {
            uint32_t rr[32];
            tmem_ld32(t_lane + TM_O + 32 * c, rr);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
            tmem_st32(t_lane + TM_O + 32 * c, rr);
          }
          tmem_wait_st();
        }
      }
      // P row -> swizzled K-major shared tile (16-byte chunk c of a 128-byte
      // row lands at chunk c ^ (row & 7)).
      uint8_t* ps = base + OFF_P;
#pragma unroll
      for (int ch = 0; ch < BN / 8; ++ch) {
        *reinterpret_cast<uint4*>(ps + (ch >> 3) * HALF + r * 128 + (((ch & 7) ^ (r & 7)) << 4)) =
            make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(bar(BAR_PF));
    }

    if (ok && wait_bar(bar(BAR_PV), (n_blk - 1) & 1, abort_flag)) {
      tc_fence_after();
      const float inv = 1.0f / l_run;
      const size_t orow = ((size_t)(q0 + t * BM + r) * Hq + hq) * kHeadDim;
      uint4* og = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + orow);
#pragma unroll
      for (int c = 0; c < kHeadDim / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(t_lane + TM_O + 32 * c, rr);
        tmem_wait_ld();
        if (row_valid) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 v;
            v.x = pack_bf16(__uint_as_float(rr[8 * k + 0]) * inv, __uint_as_float(rr[8 * k + 1]) * inv);
            v.y = pack_bf16(__uint_as_float(rr[8 * k + 2]) * inv, __uint_as_float(rr[8 * k + 3]) * inv);
            v.z = pack_bf16(__uint_as_float(rr[8 * k + 4]) * inv, __uint_as_float(rr[8 * k + 5]) * inv);
            v.w = pack_bf16(__uint_as_float(rr[8 * k + 6]) * inv, __uint_as_float(rr[8 * k + 7]) * inv);
            og[4 * c + k] = v;
          }
        }
      }
      if (row_valid && a.lse)
        a.lse[(size_t)(q0 + t * BM + r) * Hq + hq] = (m_run + fast_log2(l_run)) * kLn2;
    }
  }

  // Every role has left its loop.  After an abort, loads may still be in
  // flight: the producer lets each one land before the CTA can exit.
  __syncthreads();
  if (warp == 0 && *abort_flag) {
    for (int s = 0; s < NSTAGE; ++s) {
      if (last_k[s] >= 0) (void)mbar_wait(bar(BAR_KF + s), (last_k[s] / NSTAGE) & 1);
      if (last_v[s] >= 0) (void)mbar_wait(bar(BAR_VF + s), (last_v[s] / NSTAGE) & 1);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS)
                 : "memory");
  }
}

// cuTensorMapEncodeTiled, fetched through the runtime (no libcuda link).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// The pool as a 2-D bf16 tensor of (num_pages * Hkv * 16) rows of 128
// channels; a box is one page slab (16 rows) by 64 channels, 128B-swizzled.
bool encode_pool_map(CUtensorMap* m, const void* base, int num_pages, int hkv) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)num_pages * hkv * kPageSize};
  cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kPageSize};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace pkv_host {

cudaError_t launch_prefill(const PrefillLaunch& a, cudaStream_t s) {
  if ((long long)a.num_pages * a.num_kv_heads * kPageSize >= (1ll << 31))
    return cudaErrorNotSupported;
  CUtensorMap tk, tv;
  if (!encode_pool_map(&tk, a.k, a.num_pages, a.num_kv_heads) ||
      !encode_pool_map(&tv, a.v, a.num_pages, a.num_kv_heads))
    return cudaErrorInvalidValue;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  PrefillParams prm{a, (a.max_q_len + BM - 1) / BM};
  dim3 grid(a.num_q_heads, prm.n_tiles, a.batch);
  prefill_kernel<<<grid, NUM_THREADS, SMEM_BYTES, s>>>(tk, tv, prm);
  return cudaGetLastError();
}

uint32_t take_prefill_error(cudaStream_t s) {
  uint32_t h = 0, zero = 0;
  if (cudaMemcpyFromSymbolAsync(&h, g_err_prefill, sizeof h, 0, cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return ~0u;
  cudaStreamSynchronize(s);
  if (h) cudaMemcpyToSymbolAsync(g_err_prefill, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s);
  cudaStreamSynchronize(s);
  return h;
}

}  // namespace pkv_host
