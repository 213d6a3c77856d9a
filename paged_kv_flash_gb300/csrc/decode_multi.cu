// decode_multi.cu -- split-KV decode for steps of 2..16 query tokens per
// sequence (TileInfer.jl "Performance" page, "Attention for verify steps":
// steps of 2-16 tokens, such as speculative-decoding verify steps, run the
// split-KV decode kernels instead of the prefill kernel).  Causal inside the
// step, bottom-right aligned: token i of q_b new tokens in a sequence of L_b
// cached positions (the step's tokens included) sees positions 0 .. L_b -
// q_b + i.  bf16 pools.
//
// One CTA per (split, KV head x row group, sequence).  The rows of a
// (sequence, KV head) are its q_b x G (token, query head) pairs, row = i G +
// g; a CTA takes up to 64 of them, 16 per consumer warp.  A producer warp
// streams the split's pages through a ring of shared-memory stages (TMA
// tensor copies of the 16 x 64-channel halves of the K and V slabs, 128-byte
// swizzle); every consumer warp runs flash attention on warp-level tensor
// core MMAs (mma.sync.m16n8k16, bf16 in, fp32 accumulate), FA2 layout:
//   S = Q K^T: A = 16 query rows (bf16, exact, from registers), B = K^T by
//       ldmatrix from the stage; two 8-key tiles x 8 channel steps;
//   O += P V:  A = P (the QK accumulators rounded to bf16, no data
//       movement between lanes), B = V by ldmatrix.trans; 16 channel tiles.
// When a CTA has fewer than four row tiles, warps with the same rows take
// alternate pages and are merged at the end (log-sum-exp rule), so a 1-row
// decode still keeps four warps busy.
#include <type_traits>

#include <cuda.h>

#include "common.cuh"
#include "internal.h"

namespace {

using namespace pkv;

__device__ uint32_t g_err_multi;

constexpr int kConsumers = 4;                       // warps with rows
constexpr int kThreads = (kConsumers + 1) * 32;     // + the producer warp
constexpr int NS = 8;                               // page stages
constexpr int HALF = kPageSize * 128;               // one TMA box: 16 keys x 64 bf16
constexpr int STAGE = 4 * HALF;                     // K halves 0, 1, then V halves 0, 1
constexpr int SMEM = 1024 + NS * STAGE;
static_assert(kConsumers * (32 + 16 * kHeadDim) * 4 <= NS * STAGE,
              "the warps' (m, l) and O fit in the ring");
constexpr float kNoKey = -1.0e30f;                  // running max before any visible key

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// Shared-memory address of the 16-byte chunk holding channels ch .. ch + 7
// of key row `key` in a stage half-pair (base = K or V half 0): the halves
// are 64 channels wide and 128-byte swizzled (chunk c of row k at c ^ (k & 7)).
__device__ __forceinline__ uint32_t chunk_addr(uint32_t base, int key, int ch) {
  const int half = ch >> 6, c = (ch & 63) >> 3;
  return base + half * HALF + key * 128 + ((c ^ (key & 7)) << 4);
}

__device__ __forceinline__ void tma_box(uint32_t dst, const CUtensorMap* map, int x, int row,
                                        uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(row), "r"(bar), "l"(policy)
      : "memory");
}

// Bounded wait that also gives up when another warp raised the abort flag.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile uint32_t* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        *abort = 1u;
        atomicOr(&g_err_multi, kErrTimeout);
        return false;
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads, 3)
    decode_multi_kernel(const __grid_constant__ CUtensorMap tk,
                        const __grid_constant__ CUtensorMap tv,
                        const __grid_constant__ pkv_host::MultiLaunch a) {
  constexpr uint32_t FULL = 0xffffffffu;
  pdl_trigger();                                // the combine may be placed now
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);          // full [NS], empty [NS]
  volatile uint32_t* abort = reinterpret_cast<volatile uint32_t*>(smem + 1016);
  uint8_t* ring = smem + 1024;
  const uint32_t ring_s = smem_u32(ring);
  const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * NS;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hq = a.num_q_heads, G = Hq / a.num_kv_heads;
  const int split = blockIdx.x;
  const int h = blockIdx.y / a.row_groups, rg = blockIdx.y % a.row_groups;
  const int b = blockIdx.z;

  // The producer's first 32 page ids go out with the lengths (any entry of
  // the table row is in bounds; those past the sequence are not used).
  const int32_t* bt_row = a.block_table + (size_t)b * a.max_pages + split * a.pages_per_split;
  int bt_first = 0;
  if (warp == kConsumers && split * a.pages_per_split + lane < a.max_pages)
    bt_first = __ldg(bt_row + lane);
  const int q0 = a.cu_q[b], qn = a.cu_q[b + 1] - q0;
  const int L = a.seq_lens[b];
  if (qn < 0 || qn > a.max_q || L < qn || L > a.max_pages * kPageSize) {
    if (threadIdx.x == 0 && (qn != 0 || L < 0 || L > a.max_pages * kPageSize))
      atomicOr(&g_err_multi, kErrBadIndex);
    return;
  }
  const int R = qn * G;                                         // rows of (b, h)
  const int row0 = rg * 16 * kConsumers;
  if (row0 >= R) return;
  const int Rc = min(16 * kConsumers, R - row0);                // rows of this CTA
  const int T = (Rc + 15) >> 4;                                 // row tiles
  const int Tp = T == 1 ? 1 : (T == 2 ? 2 : 4);                 // warps per page
  const int P = kConsumers / Tp;                                // page subsets
  const int npages = (L + kPageSize - 1) / kPageSize;
  const int C = a.pages_per_split;
  const int p_begin = split * C;
  if (split > 0 && p_begin >= npages) return;                   // empty split
  const int nvs = max(1, (npages + C - 1) / C);                 // splits holding keys
  const bool direct = a.splits == 1 || nvs == 1;
  const int n_pages = max(0, min(npages, p_begin + C) - p_begin);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, Tp);
    }
    *abort = 0u;
    fence_mbar_init();
  }
  __syncthreads();

  // consumer state (the producer warp carries it unused)
  const int r = lane >> 2, qd = lane & 3;
  const int tile = warp % Tp, sub = warp / Tp;
  const bool has_rows = warp < kConsumers && tile < T;
  float o[16][4];
#pragma unroll
  for (int nt = 0; nt < 16; ++nt)
#pragma unroll
    for (int j = 0; j < 4; ++j) o[nt][j] = 0.f;
  float m[2] = {kNoKey, kNoKey}, l[2] = {0.f, 0.f};

  if (warp == kConsumers) {
    // ---------------------------------------------------------- producer
    const uint64_t policy = l2_policy_evict_first();
    int bt_cache = 0, issued = 0;
    for (int i = 0; i < n_pages; ++i) {
      if ((i & 31) == 0)
        bt_cache = (i + lane < n_pages) ? (i == 0 ? bt_first : __ldg(bt_row + i + lane)) : 0;
      int pg = __shfl_sync(FULL, bt_cache, i & 31);
      if (pg < 0 || pg >= a.num_pages) {
        if (lane == 0) atomicOr(&g_err_multi, kErrBadIndex);
        pg = 0;
      }
      const int s = i % NS;
      bool ok = true;
      if (i >= NS) ok = wait_or_abort(empty0 + 8 * s, (uint32_t)((i / NS) - 1) & 1u, abort);
      ok = __shfl_sync(FULL, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      if (lane == 0) {
        const uint32_t st = ring_s + s * STAGE, bar = full0 + 8 * s;
        const int row = (pg * a.num_kv_heads + h) * kPageSize;
        mbar_arrive_expect_tx(bar, STAGE);
        tma_box(st, &tk, 0, row, bar, policy);
        tma_box(st + HALF, &tk, 64, row, bar, policy);
        tma_box(st + 2 * HALF, &tv, 0, row, bar, policy);
        tma_box(st + 3 * HALF, &tv, 64, row, bar, policy);
      }
      ++issued;
    }
    // the last copies of each stage have landed before the ring is reused
    // below or the CTA exits (immediate when the consumers have seen them)
    if (lane == 0)
      for (int i = max(0, issued - NS); i < issued; ++i)
        (void)mbar_wait(full0 + 8 * (i % NS), (uint32_t)(i / NS) & 1u);
    __syncwarp();
  } else {
    // ---------------------------------------------------------- consumers
    // this lane's two rows (r, r + 8 of the tile): query row and causal limit
    int lim[2];
    uint32_t qa[8][4];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int rho = row0 + 16 * tile + r + 8 * hr;          // row within (b, h)
      const bool valid = has_rows && rho < R;
      const int i = valid ? rho / G : 0, g = valid ? rho % G : 0;
      lim[hr] = valid ? L - qn + i : L - 1;                   // padding rows: the sequence
      const __nv_bfloat16* qrow = static_cast<const __nv_bfloat16*>(a.q) +
                                  ((size_t)(q0 + i) * Hq + h * G + g) * kHeadDim;
#pragma unroll
      for (int kb = 0; kb < 8; ++kb) {
        uint32_t lo = 0, hi = 0;
        if (valid) {
          lo = __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * kb + 2 * qd));
          hi = __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * kb + 8 + 2 * qd));
        }
        qa[kb][hr] = lo;          // a0a1 (row r) / a2a3 (row r + 8)
        qa[kb][2 + hr] = hi;      // a4a5 / a6a7
      }
    }
    // the earliest limit of the warp's rows: pages wholly at or before it
    // need no causal mask (a padding row's limit is the sequence's end)
    int lim_min = min(lim[0], lim[1]);
#pragma unroll
    for (int x = 16; x >= 1; x >>= 1) lim_min = min(lim_min, __shfl_xor_sync(FULL, lim_min, x));
    const float qs = a.softmax_scale * kLog2e;

    // One page: S = Q K^T, online softmax, O += P V.  MASKED: the page holds
    // the causal edge or the end of the sequence.
    auto page = [&](uint32_t kst, int key0, auto masked_tag) {
      constexpr bool MASKED = decltype(masked_tag)::value;
      const uint32_t vst = kst + 2 * HALF;
      // S for keys 8 nt + (0..7); even and odd channel steps in separate
      // accumulators: four independent MMA chains of four
      float d[2][2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int j = 0; j < 4; ++j) d[nt][u][j] = 0.f;
#pragma unroll
      for (int kb2 = 0; kb2 < 4; ++kb2)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          uint32_t bk[4];
          ldsm_x4(chunk_addr(kst, 8 * nt + (lane & 7), 32 * kb2 + 8 * (lane >> 3)), bk);
          mma_bf16(d[nt][0], qa[2 * kb2], bk[0], bk[1]);
          mma_bf16(d[nt][1], qa[2 * kb2 + 1], bk[2], bk[3]);
        }
      // scores (log2 domain), causal mask, running max per row
      float sc[2][2][2];                                         // [row half][tile][e]
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        float mx = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float v = (d[nt][0][2 * hr + e] + d[nt][1][2 * hr + e]) * qs;
            if constexpr (MASKED) {
              if (key0 + 8 * nt + 2 * qd + e > lim[hr]) v = -INFINITY;
            }
            sc[hr][nt][e] = v;
            mx = fmaxf(mx, v);
          }
        mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 2));
        // the max the exponentials use moves only when a page passes it by
        // more than 8 (p <= 256); O and l are rescaled then
        if (mx > m[hr] + 8.f) {
          const float alpha = fast_exp2(m[hr] - mx);
          m[hr] = mx;
          l[hr] *= alpha;
#pragma unroll
          for (int nt = 0; nt < 16; ++nt) {
            o[nt][2 * hr] *= alpha;
            o[nt][2 * hr + 1] *= alpha;
          }
        }
      }
      uint32_t pa[4];                                            // P as the A operand
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const float p0 = fast_exp2(sc[hr][nt][0] - m[hr]);
          const float p1 = fast_exp2(sc[hr][nt][1] - m[hr]);
          l[hr] += p0 + p1;
          pa[2 * nt + hr] = pack_bf16(p0, p1);
        }
      // V rows of slots past the sequence (only in its last page) may hold
      // anything, NaN included, and 0 x NaN would reach O: zero this lane's
      // halves of keys 2qd, 2qd + 1 (vm0) and 2qd + 8, 2qd + 9 (vm1)
      uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
      if constexpr (MASKED) {
        const int nvalid = L - key0;
        vm0 = (2 * qd < nvalid ? 0x0000ffffu : 0u) | (2 * qd + 1 < nvalid ? 0xffff0000u : 0u);
        vm1 = (2 * qd + 8 < nvalid ? 0x0000ffffu : 0u) | (2 * qd + 9 < nvalid ? 0xffff0000u : 0u);
      }
      // O += P V for channels 16 cg .. 16 cg + 15
#pragma unroll
      for (int cg = 0; cg < 8; ++cg) {
        uint32_t bv[4];
        ldsm_x4_t(chunk_addr(vst, (lane & 7) + 8 * ((lane >> 3) & 1), 16 * cg + 8 * (lane >> 4)),
                  bv);
        if constexpr (MASKED) {
          bv[0] &= vm0;
          bv[1] &= vm1;
          bv[2] &= vm0;
          bv[3] &= vm1;
        }
        mma_bf16(o[2 * cg], pa, bv[0], bv[1]);
        mma_bf16(o[2 * cg + 1], pa, bv[2], bv[3]);
      }
    };

    for (int i = sub; i < n_pages; i += P) {
      const int s = i % NS;
      const bool ok = wait_or_abort(full0 + 8 * s, (uint32_t)(i / NS) & 1u, abort);
      if (!__all_sync(FULL, ok)) break;          // uniform: the MMAs below need the whole warp
      if (has_rows) {
        const int key0 = (p_begin + i) * kPageSize;              // position of the page's key 0
        if (key0 + kPageSize - 1 <= lim_min)
          page(ring_s + s * STAGE, key0, std::false_type{});
        else
          page(ring_s + s * STAGE, key0, std::true_type{});
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * s);
    }
    // row sums over the quad's lanes
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      l[hr] += __shfl_xor_sync(FULL, l[hr], 1);
      l[hr] += __shfl_xor_sync(FULL, l[hr], 2);
    }
  }
  __syncthreads();                   // every warp is done with the ring

  // ------------------------------------------------- merge warps, store
  // Warps with the same rows (P of them) merge by the log-sum-exp rule:
  // (m, l) of every warp go to shared memory; each warp scales its O by
  // 2^(m - M) / L_sum; with P > 1 the warps of page subsets 1.. park their
  // scaled O and the subset-0 warp adds them.  Results leave from the MMA
  // fragment registers (row r / r + 8, channels 8 nt + 2 qd, + 1).
  float* ml = reinterpret_cast<float*>(ring);                     // [warp][m 16 | l 16]
  float* po = ml + kConsumers * 32;                               // [warp][16][128]
  if (has_rows && qd == 0) {
    ml[warp * 32 + r] = m[0];
    ml[warp * 32 + r + 8] = m[1];
    ml[warp * 32 + 16 + r] = l[0];
    ml[warp * 32 + 16 + r + 8] = l[1];
  }
  __syncthreads();
  const bool bad = *abort != 0u;
  float f[2] = {0.f, 0.f}, lse2[2] = {-INFINITY, -INFINITY};
  if (has_rows) {
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int ir = r + 8 * hr;
      float M = kNoKey;
      for (int j = 0; j < P; ++j) M = fmaxf(M, ml[(tile + Tp * j) * 32 + ir]);
      float Ls = 0.f;
      for (int j = 0; j < P; ++j) {
        const int w = tile + Tp * j;
        Ls += fast_exp2(ml[w * 32 + ir] - M) * ml[w * 32 + 16 + ir];
      }
      if (Ls > 0.f && !bad) {
        f[hr] = fast_exp2(m[hr] - M) / Ls;
        lse2[hr] = M + fast_log2(Ls);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      o[nt][0] *= f[0];
      o[nt][1] *= f[0];
      o[nt][2] *= f[1];
      o[nt][3] *= f[1];
    }
  }
  if (P > 1) {                                                    // CTA-uniform
    if (has_rows && sub > 0) {
      float* mine = po + (size_t)warp * 16 * kHeadDim;
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        const int ch = 8 * nt + 2 * qd;
        *reinterpret_cast<float2*>(mine + r * kHeadDim + ch) = make_float2(o[nt][0], o[nt][1]);
        *reinterpret_cast<float2*>(mine + (r + 8) * kHeadDim + ch) =
            make_float2(o[nt][2], o[nt][3]);
      }
    }
    __syncthreads();
    if (has_rows && sub == 0) {
      for (int j = 1; j < P; ++j) {
        const float* other = po + (size_t)(tile + Tp * j) * 16 * kHeadDim;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
          const int ch = 8 * nt + 2 * qd;
          const float2 x0 = *reinterpret_cast<const float2*>(other + r * kHeadDim + ch);
          const float2 x1 = *reinterpret_cast<const float2*>(other + (r + 8) * kHeadDim + ch);
          o[nt][0] += x0.x;
          o[nt][1] += x0.y;
          o[nt][2] += x1.x;
          o[nt][3] += x1.y;
        }
      }
    }
  }
  if (has_rows && sub == 0) {
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int rho = row0 + 16 * tile + r + 8 * hr;
      if (rho >= R) continue;
      const size_t bh = (size_t)(q0 + rho / G) * Hq + h * G + rho % G;
      if (direct) {
        uint32_t* dst = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(a.out) +
                                                    bh * kHeadDim);
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
          dst[4 * nt + qd] = pack_bf16(o[nt][2 * hr], o[nt][2 * hr + 1]);
        if (a.lse && qd == 0) a.lse[bh] = lse2[hr] * kLn2;
      } else {
        const size_t slot = bh * a.splits + split;
        float* dst = a.ws_o + slot * kHeadDim;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
          *reinterpret_cast<float2*>(dst + 8 * nt + 2 * qd) =
              make_float2(o[nt][2 * hr], o[nt][2 * hr + 1]);
        if (qd == 0) a.ws_lse[slot] = lse2[hr];
      }
    }
  }
}

// Combine of the split partials of one (token, query head): the token's
// sequence is found in cu_q; its splits that hold keys are merged with the
// log-sum-exp rule (a split with no key visible to the row has lse -inf and
// weight 0).  Rows whose sequence fits one split were written directly.
__global__ void __launch_bounds__(128)
    decode_multi_combine_kernel(const __grid_constant__ pkv_host::MultiLaunch a) {
  __shared__ float wsm[128], red[4];
  pdl_wait();                                   // the split kernel's partials
  const int bh = blockIdx.x;
  const int t = bh / a.num_q_heads;
  const int b = owner_seq(a.cu_q, a.batch, t);
  int L = a.seq_lens[b];
  if (L < 0 || L > a.max_pages * kPageSize) L = 0;
  const int npages = (L + kPageSize - 1) / kPageSize;
  const int n = min(a.splits, (npages + a.pages_per_split - 1) / a.pages_per_split);
  if (n <= 1) return;
  const float2 res = merge_splits(a.ws_lse + (size_t)bh * a.splits,
                                  a.ws_o + (size_t)bh * a.splits * kHeadDim, n, wsm, red);
  const int d = threadIdx.x;
  static_cast<__nv_bfloat16*>(a.out)[(size_t)bh * kHeadDim + d] = __float2bfloat16_rn(res.x);
  if (a.lse && d == 0) a.lse[bh] = res.y * kLn2;
}

}  // namespace

namespace pkv_host {

cudaError_t launch_decode_multi(const MultiLaunch& a, cudaStream_t s) {
  if (a.batch == 0 || a.total_q == 0) return cudaSuccess;
  cudaError_t e = pkv_host::set_max_dynamic_smem(
      reinterpret_cast<const void*>(decode_multi_kernel), SMEM);
  if (e != cudaSuccess) return e;
  if ((long long)a.num_pages * a.num_kv_heads * kPageSize >= (1ll << 31))
    return cudaErrorNotSupported;
  CUtensorMap tk, tv;
  if (!encode_bf16_pool_map(&tk, a.k, a.num_pages, a.num_kv_heads) ||
      !encode_bf16_pool_map(&tv, a.v, a.num_pages, a.num_kv_heads))
    return cudaErrorInvalidValue;
  dim3 grid(a.splits, a.num_kv_heads * a.row_groups, a.batch);
  decode_multi_kernel<<<grid, kThreads, SMEM, s>>>(tk, tv, a);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.splits == 1) return e;
  // placed while the split kernel's last CTAs run; waits for its partials
  return pkv_host::launch_dependent(decode_multi_combine_kernel, dim3(a.total_q * a.num_q_heads),
                                    dim3(128), s, a);
}

uint32_t take_multi_error(cudaStream_t s) { return take_error_word(&g_err_multi, s); }

}  // namespace pkv_host
