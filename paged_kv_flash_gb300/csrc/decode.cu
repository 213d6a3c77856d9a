// decode.cu -- split-KV paged decode attention and the log-sum-exp combine
// (TileInfer.jl "Performance" page, "Fused kernels, FlashAttention and
// PagedAttention": online softmax over the pages in place through the block
// table, split-KV for decode, and a combine kernel kept separate from the
// split kernel; "INT8 KV cache": dequantisation inside attention).
//
// Two split kernels: decode_split_kernel (bf16 pools) and
// decode_split_i8mma_kernel (INT8 pools), both on warp-level tensor-core
// MMAs (see their own comments further down).  Both run one CTA per (split,
// KV head, sequence); a split is a run of consecutive logical pages of one
// sequence, its warps take the pages round-robin and each warp streams its
// pages through a private ring of shared-memory page buffers filled by the
// TMA engine (L2 evict-first), so no CTA-wide barrier sits in the page loop.
// Every warp serves all G query heads of the KV head, so each K/V byte is
// read from HBM once per decode step.
//
// The split's result is normalised (O / l) and written with its log2-domain
// lse; with a single split the kernel writes the bf16 output directly and
// the combine is skipped.
#include <algorithm>
#include <mutex>

#include <cuda.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"

namespace {

using namespace pkv;

__device__ uint32_t g_err_decode;

// ------------------------------------------------------------------------
// bf16 split kernel on tensor cores (mma.sync m16n8k16, bf16 in, fp32 out).
//
// A warp takes whole 16-key pages of its split (round-robin over the CTA's
// warps) from a private ring of shared-memory buffers that the TMA engine
// fills (K and V slabs as 16-row x 64-channel boxes, 128-byte swizzled, L2
// evict-first), so no CTA-wide barrier sits in the page loop.  Per page:
//   S^T = K Q^T: A = the page's 16 keys (ldmatrix), B = the G query rows of
//        the KV head as columns (bf16, exact, in registers); 8 channel steps
//        in two accumulators.  Lane (r, qd) gets keys r and r + 8 of heads
//        2qd and 2qd + 1, so the running max, sum and the O columns of a
//        head live in the lanes that own it (no shuffles but the page max);
//   O^T += V^T P^T: A = V^T (ldmatrix.trans), B = P (rounded to bf16) moved
//        from the key-major layout of S^T to the head-major B fragment by
//        two register transposes (movmatrix); 8 channel tiles.
// 16 MMAs per page instead of ~1,000 FMAs and shuffles on CUDA cores.  Slots
// past the sequence's end get p = 0 and their V values are zeroed before
// the MMA (0 x NaN would reach O).
namespace bfmma {

// Three CTAs of 4 warps per SM, 2 page buffers per warp: as many bytes in
// flight per SM as two CTAs with 3 buffers per warp, and half again as many
// warps to work on the pages that have landed.  On the whole GPU the kernel
// is HBM-bound either way; on a few SMs beside a prefill (a continuous-
// batching step) the work per page sets its pace, and there the extra warps
// took the mixed step from 424 to 402 us (the decode alone: unchanged).
constexpr int W = pkv_host::kDecodeWarps;               // warps per CTA, pages round-robin
constexpr int NB = 2;                                   // page buffers per warp
constexpr int CTAS_PER_SM = 3;                          // resident CTAs (shared memory)
constexpr int HALF = kPageSize * 128;                   // one box: 16 keys x 64 bf16
constexpr int SLAB = 2 * HALF;                          // K or V of one (page, head)
constexpr int PAGE = 2 * SLAB;                          // K, then V
constexpr int WARP_BYTES = NB * PAGE;
constexpr int SMEM = 1024 + W * WARP_BYTES;
static_assert(W * NB * 8 <= 1016, "barriers fit the header");
static_assert(CTAS_PER_SM * (SMEM + 1024) <= 228 * 1024, "resident CTAs fit shared memory");

// The 16-byte chunk holding channels ch .. ch + 7 of key row `key` of a slab:
// two 64-channel halves, chunk c of row k at c ^ (k & 7).
__device__ __forceinline__ uint32_t slab_chunk(uint32_t slab, int key, int ch) {
  const int half = ch >> 6, c = (ch & 63) >> 3;
  return slab + half * HALF + key * 128 + ((c ^ (key & 7)) << 4);
}

// An 8 x 8 b16 matrix held one row per 4 lanes, transposed across the warp.
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ void tma_box(uint32_t dst, const CUtensorMap* map, int x, int row,
                                        uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(row), "r"(bar), "l"(policy)
      : "memory");
}

}  // namespace bfmma

// The CTA's merge of its warps: each warp has parked (O [G][128], m [G],
// l [G]) at the start of its buffer area (bufs + w * warp_stride, log2
// domain, O unnormalised); combine them, then write the bf16 output (one
// split) or the split's partial, and with FUSED let the last split of the
// (sequence, KV head) merge the partials.
template <int G, bool FUSED, int W = pkv_host::kDecodeWarps>
__device__ __forceinline__ void merge_warps(const pkv_host::DecodeLaunch& a, uint8_t* smem,
                                            const uint8_t* bufs, size_t warp_stride, int split,
                                            int h, int b, int nv, bool direct) {
  const int Hq = a.num_q_heads;
  for (int t = threadIdx.x; t < G * kHeadDim; t += W * 32) {
    const int g = t / kHeadDim, d = t % kHeadDim;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      const float* wmw = reinterpret_cast<const float*>(bufs + w * warp_stride) + G * kHeadDim;
      M = fmaxf(M, wmw[g]);
    }
    float Lsum = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const float* wow = reinterpret_cast<const float*>(bufs + w * warp_stride);
        const float* wmw = wow + G * kHeadDim;
        const float f = fast_exp2(wmw[g] - M);
        Lsum += f * wmw[G + g];
        O += f * wow[g * kHeadDim + d];
      }
      O = O / Lsum;
    }
    const float lse2 = (M == -INFINITY) ? -INFINITY : M + fast_log2(Lsum);
    const int hq = h * G + g;
    if (direct) {
      static_cast<__nv_bfloat16*>(a.out)[((size_t)b * Hq + hq) * kHeadDim + d] =
          __float2bfloat16_rn(O);
      if (a.lse && d == 0) a.lse[(size_t)b * Hq + hq] = lse2 * kLn2;
    } else {
      const size_t row = ((size_t)b * Hq + hq) * a.splits + split;
      a.ws_o[row * kHeadDim + d] = O;
      if (d == 0) a.ws_lse[row] = lse2;
    }
  }
  if (direct || !FUSED) return;                 // separate combine kernel

  // Fused merge: count this split's part; the split that completes the count merges the
  // nv parts of (b, KV head) (log-sum-exp rule, splits in order, so the
  // result does not depend on which split merges) and resets the count.
  // the flag sits in the unused end of the barrier header (no static shared
  // memory: it would pad the 1024-byte aligned dynamic allocation)
  volatile uint32_t& s_last = *reinterpret_cast<volatile uint32_t*>(smem + 1020);
  static_assert(W * 5 * 8 <= 1020, "barrier header");
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t* ctr = a.ws_ctr + (size_t)b * a.num_kv_heads + h;
    uint32_t old;
    asm volatile("fence.acq_rel.gpu;\n\tatom.relaxed.gpu.global.add.u32 %0, [%1], 1;"
                 : "=r"(old) : "l"(ctr) : "memory");
    const bool last = old == (uint32_t)(nv - 1);
    if (last) {
      asm volatile("fence.acq_rel.gpu;" ::: "memory");
      *ctr = 0u;                                  // ready for the next call
    }
    s_last = last ? 1u : 0u;
  }
  __syncthreads();
  if (!s_last) return;
  // the warps' buffers are free now: weights and the block reduction use them
  float* wsm = reinterpret_cast<float*>(const_cast<uint8_t*>(bufs));
  float* red = wsm + 128;
  for (int g = 0; g < G; ++g) {
    const size_t bh = (size_t)b * Hq + h * G + g;
    const float2 r = merge_splits(a.ws_lse + bh * a.splits, a.ws_o + bh * a.splits * kHeadDim,
                                  nv, wsm, red);
    const int d = threadIdx.x;
    if (d < kHeadDim) {
      static_cast<__nv_bfloat16*>(a.out)[bh * kHeadDim + d] = __float2bfloat16_rn(r.x);
      if (a.lse && d == 0) a.lse[bh] = r.y * kLn2;
    }
  }
}

// FUSED: the split that completes a (sequence, KV head) merges its splits
// (a.ws_ctr counts them); otherwise a separate combine kernel does.  A
// template parameter, so that the default kernel carries none of that code.
template <int G, bool FUSED>
__global__ void __launch_bounds__(bfmma::W * 32, bfmma::CTAS_PER_SM)
    decode_split_kernel(const __grid_constant__ CUtensorMap tk,
                        const __grid_constant__ CUtensorMap tv,
                        const __grid_constant__ pkv_host::DecodeLaunch a) {
  using namespace bfmma;
  constexpr uint32_t FULL = 0xffffffffu;
  pdl_trigger();                                // the combine may be placed now
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint8_t* bufs = smem + 1024;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, qd = lane & 3;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int Hq = a.num_q_heads;

  // Every load that needs nothing else goes out first, so that their
  // latencies overlap: the length, this warp's first 32 page ids (any entry
  // of the table row is in bounds; those past the sequence are not used)
  // and the query rows as B fragments (column r = head r of the group, zero
  // for r >= G; rows = channels 16 ks + 2qd, + 1 (qb[ks][0]) and + 8, + 9).
  const int32_t* bt_row = a.block_table + (size_t)b * a.max_pages;
  const int p_begin = split * a.pages_per_split;
  int L = a.seq_lens[b];
  const int lp0 = p_begin + warp + lane * W;
  const int bt_first = lp0 < a.max_pages ? __ldg(bt_row + lp0) : 0;
  uint32_t qb[8][2];
  {
    const bool valid = r < G;
    const __nv_bfloat16* qrow = static_cast<const __nv_bfloat16*>(a.q) +
                                ((size_t)b * Hq + h * G + (valid ? r : 0)) * kHeadDim;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qb[ks][0] = valid ? __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * qd)) : 0u;
      qb[ks][1] = valid ? __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 8 + 2 * qd))
                        : 0u;
    }
  }
  if (L < 0 || L > a.max_pages * kPageSize) {
    if (threadIdx.x == 0) atomicOr(&g_err_decode, kErrBadIndex);
    L = 0;
  }
  const int npages = (L + kPageSize - 1) / kPageSize;
  if (split > 0 && p_begin >= npages) return;   // empty split: the merge skips it
  // splits holding keys (split 0 always runs); with one, it writes the output
  const int nv = max(1, (npages + a.pages_per_split - 1) / a.pages_per_split);
  const bool direct = a.splits == 1 || nv == 1;
  const int p_end = min(npages, p_begin + a.pages_per_split);
  const int n_w = max(0, (p_end - p_begin - warp + W - 1) / W);   // pages of this warp

  const uint32_t bar0 = smem_u32(bars + warp * NB);
  uint8_t* wbuf = bufs + (size_t)warp * WARP_BYTES;
  const uint32_t wbuf_s = smem_u32(wbuf);
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < NB; ++k) mbar_init(bar0 + 8 * k, 1);
    fence_mbar_init();
  }
  __syncwarp();

  // Page ids of this warp's pages, 32 at a time, one per lane (the first 32
  // loaded above).
  const uint64_t policy = l2_policy_evict_first();
  int bt_cache = 0;
  auto page_id = [&](int i) -> int {
    if ((i & 31) == 0) {
      const int lp = p_begin + warp + (i + lane) * W;
      bt_cache = (i + lane < n_w) ? (i == 0 ? bt_first : __ldg(bt_row + lp)) : 0;
    }
    int pg = __shfl_sync(FULL, bt_cache, i & 31);
    if (pg < 0 || pg >= a.num_pages) {
      if (lane == 0) atomicOr(&g_err_decode, kErrBadIndex);
      pg = 0;
    }
    return pg;
  };
  auto issue = [&](int i, int pg) {
    if (lane == 0) {
      const int k = i % NB;
      const uint32_t bar = bar0 + 8 * k, dst = wbuf_s + k * PAGE;
      const int row = (pg * a.num_kv_heads + h) * kPageSize;
      // the warp's generic-proxy reads of this buffer are done (__syncwarp);
      // order them before the async-proxy refill
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive_expect_tx(bar, PAGE);
      tma_box(dst, &tk, 0, row, bar, policy);
      tma_box(dst + HALF, &tk, 64, row, bar, policy);
      tma_box(dst + SLAB, &tv, 0, row, bar, policy);
      tma_box(dst + SLAB + HALF, &tv, 64, row, bar, policy);
    }
  };
  const int pro = min(NB, n_w);
  for (int i = 0; i < pro; ++i) issue(i, page_id(i));
  int issued = pro;
  const float sl2 = a.softmax_scale * kLog2e;
  // O^T: channels 16 mt + r (o[mt][0..1]) and + 8 (o[mt][2..3]) of heads 2qd
  // (o[mt][0], o[mt][2]) and 2qd + 1 (o[mt][1], o[mt][3])
  float o[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int j = 0; j < 4; ++j) o[mt][j] = 0.f;
  // per head 2qd + e: the max the exponentials are taken against (log2
  // domain) and this lane's part of the sum
  float mu[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  // this lane's ldmatrix rows: K (keys, non-transposed) and V (transposed)
  const int k_key = (lane & 7) + 8 * ((lane >> 3) & 1), k_ch = 8 * (lane >> 4);
  const int v_key = (lane & 7) + 8 * (lane >> 4), v_ch = 8 * ((lane >> 3) & 1);

  bool failed = false;
  int i_fail = 0;
  for (int i = 0; i < n_w; ++i) {
    const int k = i % NB;
    if (!mbar_wait(bar0 + 8 * k, (uint32_t)(i / NB) & 1u)) {
      failed = true;
      i_fail = i;
      break;
    }
    const int lp = p_begin + warp + i * W;
    const int nvalid = min(kPageSize, L - lp * kPageSize);
    const uint32_t kst = wbuf_s + k * PAGE, vst = kst + SLAB;

    float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 8; ks += 2) {
      uint32_t ka[4], kb[4];
      ldsm_x4(slab_chunk(kst, k_key, 16 * ks + k_ch), ka);
      ldsm_x4(slab_chunk(kst, k_key, 16 * ks + 16 + k_ch), kb);
      mma_bf16(d0, ka, qb[ks][0], qb[ks][1]);
      mma_bf16(d1, kb, qb[ks + 1][0], qb[ks + 1][1]);
    }
    // scores (unscaled): key r of heads 2qd, 2qd + 1 (s[0], s[1]), key r + 8 (s[2], s[3])
    float s[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) s[e] = d0[e] + d1[e];
    if (nvalid < kPageSize) {
      if (r >= nvalid) s[0] = s[1] = -INFINITY;
      if (r + 8 >= nvalid) s[2] = s[3] = -INFINITY;
    }
    float pm[2] = {fmaxf(s[0], s[2]), fmaxf(s[1], s[3])};
#pragma unroll
    for (int x = 4; x <= 16; x <<= 1) {
      pm[0] = fmaxf(pm[0], __shfl_xor_sync(FULL, pm[0], x));
      pm[1] = fmaxf(pm[1], __shfl_xor_sync(FULL, pm[1], x));
    }
    // the max moves only when the page max passes it by more than 2^8
    // (p <= 256; exact: l and O share it)
    float alpha[2] = {1.f, 1.f};
    bool grow = false;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float m_pg = pm[e] * sl2;
      if (m_pg > mu[e] + 8.f) {
        alpha[e] = fast_exp2(mu[e] - m_pg);
        mu[e] = m_pg;
        l[e] *= alpha[e];
        grow = true;
      }
    }
    if (__any_sync(FULL, grow)) {
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        o[mt][0] *= alpha[0];
        o[mt][2] *= alpha[0];
        o[mt][1] *= alpha[1];
        o[mt][3] *= alpha[1];
      }
    }
    const float p0 = fast_exp2(fmaf(s[0], sl2, -mu[0])), p1 = fast_exp2(fmaf(s[1], sl2, -mu[1]));
    const float p2 = fast_exp2(fmaf(s[2], sl2, -mu[0])), p3 = fast_exp2(fmaf(s[3], sl2, -mu[1]));
    l[0] += p0 + p2;
    l[1] += p1 + p3;
    // P as the B fragment of O^T += V^T P^T: head r, keys 2qd, 2qd + 1 (+ 8)
    const uint32_t pb0 = movm_t(pack_bf16x2(p0, p1));
    const uint32_t pb1 = movm_t(pack_bf16x2(p2, p3));
    uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;   // V of slots past the sequence -> 0
    if (nvalid < kPageSize) {
      mlo = (2 * qd < nvalid ? 0x0000ffffu : 0u) | (2 * qd + 1 < nvalid ? 0xffff0000u : 0u);
      mhi = (2 * qd + 8 < nvalid ? 0x0000ffffu : 0u) | (2 * qd + 9 < nvalid ? 0xffff0000u : 0u);
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      uint32_t va[4];
      ldsm_x4_t(slab_chunk(vst, v_key, 16 * mt + v_ch), va);
      va[0] &= mlo;
      va[1] &= mlo;
      va[2] &= mhi;
      va[3] &= mhi;
      mma_bf16(o[mt], va, pb0, pb1);
    }
    __syncwarp();
    if (issued < n_w) {
      issue(issued, page_id(issued));
      ++issued;
    }
  }
  if (failed) {
    if (lane == 0) atomicOr(&g_err_decode, kErrTimeout);
    // let every copy this warp issued land (bounded) before the buffers are
    // reused or the CTA exits
    for (int i = i_fail; i < issued; ++i)
      (void)mbar_wait(bar0 + 8 * (i % NB), (uint32_t)(i / NB) & 1u);
  }
  __syncwarp();

  // Park (O unnormalised, m, l) of the warp's G heads in its buffers (all of
  // its copies have landed), then merge the warps.
#pragma unroll
  for (int x = 4; x <= 16; x <<= 1) {
    l[0] += __shfl_xor_sync(FULL, l[0], x);
    l[1] += __shfl_xor_sync(FULL, l[1], x);
  }
  float* wo = reinterpret_cast<float*>(wbuf);              // [G][128]
  float* wm = wo + G * kHeadDim;                           // [G]
  float* wl = wm + G;                                      // [G]
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int g = 2 * qd + e;
    if (g < G) {
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        wo[g * kHeadDim + 16 * mt + r] = failed ? 0.f : o[mt][e];
        wo[g * kHeadDim + 16 * mt + r + 8] = failed ? 0.f : o[mt][2 + e];
      }
      if (r == 0) {
        wm[g] = failed ? -INFINITY : mu[e];
        wl[g] = failed ? 0.f : l[e];
      }
    }
  }
  __syncthreads();
  merge_warps<G, FUSED, W>(a, smem, bufs, (size_t)WARP_BYTES, split, h, b, nv, direct);
}

// ------------------------------------------------------------------------
// INT8 split kernel on tensor cores (mma.sync m16n8k16, f16 in, f32 out).
//
// On CUDA cores the INT8 page loop is bound by instruction issue: widening
// 4 KB of codes and the G-head dot products and reductions cost ~700 warp
// instructions per page.  Here both products of a page run as warp MMAs:
//   QK: A = the query rows (16 x 16 channels per k-step), B = the page's
//       keys (16 channels x 8 keys), two key tiles x 8 k-steps = 16 MMAs;
//   PV: A = V^T (16 channels x 16 keys), B = P' = p * v_scale (16 keys x
//       8 heads), 8 channel tiles = 8 MMAs.
// int8 codes become f16 exactly with a byte permute: 0x64XX is the f16
// 1024 + XX, and XX = code ^ 0x80 = code + 128.  K subtracts the 1152 bias
// in f16 (exact); V keeps it and the epilogue removes 1152 * sum(P'), using
// the f16 P' values the MMAs saw.  The query is split into an f16 high part
// and an f16 low part (q' = hi + lo to ~22 bits) placed in rows 0..G-1 and
// G..2G-1 of A; the two rows' scores are added after the MMA, so the scores
// keep fp32-like precision.  Rows 2G..15 are zero.
//
// Layouts follow the m16n8k16 fragments: lane = 4 r + qd.  In QK, B's k
// index 2qd + e (+8) of k-step kb is channel 32 qd + 4 kb + e (+2), so a
// lane converts whole 4-byte words of its 32-byte chunk of a key row; D
// leaves lane (r, qd) with the scores of row r for keys 8t + 2qd + {0, 1},
// which is exactly the B fragment PV needs (column r, those keys): P never
// moves between lanes.  In PV, rows r and r + 8 of channel tile 2i + m are
// channels 16 r + 4 i + 2 m and + 1.  K and V slabs arrive by TMA with
// 128-byte swizzle (16-byte chunk c of row k at c ^ (k & 7)), which makes
// every fragment load conflict-free.
namespace i8mma {

constexpr int W = 8;                                    // warps per CTA, pages round-robin
constexpr int NB = 3;                                   // page buffers per warp
constexpr int SLAB = kPageSize * kHeadDim;              // 2 KiB: K or V of one (page, head)
constexpr int KV = 2 * SLAB;                            // one page buffer (1 KiB aligned)
constexpr int SC = 2 * kPageSize * 4;                   // K and V scales of one page
constexpr int WARP_BYTES = NB * KV;
constexpr int SMEM = 1024 + W * NB * (KV + SC);
constexpr uint32_t kMagic = 0x64646464u;                // f16 exponent byte of 1024
constexpr uint32_t kBias2 = 0x64806480u;                // f16x2 (1152, 1152)
constexpr float kBias = 1152.0f;

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two f16 pairs (exact codes) from a word of four int8 codes: bytes (0, 1)
// and (2, 3).
__device__ __forceinline__ void codes_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(__byte_perm(u, kMagic, 0x4140)), "r"(kBias2));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(__byte_perm(u, kMagic, 0x4342)), "r"(kBias2));
}

// Two keys' words of the same four channels -> four f16 pairs (key a low,
// key b high) of 1152 + code, one per channel byte.
__device__ __forceinline__ void codes_pair_f16(uint32_t wa, uint32_t wb, uint32_t (&c)[4]) {
  const uint32_t tl = __byte_perm(wa, wb, 0x5140) ^ 0x80808080u;
  const uint32_t th = __byte_perm(wa, wb, 0x7362) ^ 0x80808080u;
  c[0] = __byte_perm(tl, kMagic, 0x4140);
  c[1] = __byte_perm(tl, kMagic, 0x4342);
  c[2] = __byte_perm(th, kMagic, 0x4140);
  c[3] = __byte_perm(th, kMagic, 0x4342);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ float2 unpack_f16x2(uint32_t v) {
  const __half2 h = *reinterpret_cast<const __half2*>(&v);
  return __half22float2(h);
}

__device__ __forceinline__ uint4 lds128(const uint8_t* p) {
  return *reinterpret_cast<const uint4*>(p);
}

__device__ __forceinline__ void tma_slab(uint32_t dst, const CUtensorMap* map, int row,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row), "r"(bar), "l"(policy)
      : "memory");
}

}  // namespace i8mma

template <int G, bool FUSED>
__global__ void __launch_bounds__(i8mma::W * 32, 2)
    decode_split_i8mma_kernel(const __grid_constant__ CUtensorMap tk,
                              const __grid_constant__ CUtensorMap tv,
                              const __grid_constant__ pkv_host::DecodeLaunch a) {
  using namespace i8mma;
  constexpr uint32_t FULL = 0xffffffffu;
  pdl_trigger();                                // the combine may be placed now
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint8_t* bufs = smem + 1024;
  float* scales = reinterpret_cast<float*>(bufs + W * WARP_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, qd = lane & 3;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int Hq = a.num_q_heads;

  // Every load that needs nothing else goes out first, so that their
  // latencies overlap: the length, this warp's first 32 page ids (any entry
  // of the table row is in bounds; those past the sequence are not used),
  // and the query channels and smoothing weights of this lane's A fragments
  // (row rr < G is head rr's high part, G <= rr < 2G head rr - G's low part;
  // per k-step kb, channels 32 qd + 4 kb + {0..3} of rows r and r + 8).
  const int32_t* bt_row = a.block_table + (size_t)b * a.max_pages;
  const int p_begin = split * a.pages_per_split;
  int L = a.seq_lens[b];
  const int lp0 = p_begin + warp + lane * W;
  const int bt_first = lp0 < a.max_pages ? __ldg(bt_row + lp0) : 0;
  int qg[2];
  bool qlow[2];
  uint2 qraw[2][8];
  float4 qw[8];
  {
    const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(a.q);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int rr = r + 8 * half;
      int g = -1;
      bool low = false;
      if (half == 0 || G == 8) {
        if (rr < G) {
          g = rr;
        } else if (rr < 2 * G) {
          g = rr - G;
          low = true;
        }
      }
      qg[half] = g;
      qlow[half] = low;
#pragma unroll
      for (int kb = 0; kb < 8; ++kb)
        qraw[half][kb] = g >= 0 ? __ldg(reinterpret_cast<const uint2*>(
                                      qb + ((size_t)b * Hq + h * G + g) * kHeadDim +
                                      32 * qd + 4 * kb))
                                : make_uint2(0u, 0u);
    }
#pragma unroll
    for (int kb = 0; kb < 8; ++kb)
      qw[kb] = a.k_smooth ? __ldg(reinterpret_cast<const float4*>(a.k_smooth + 32 * qd + 4 * kb))
                          : make_float4(1.f, 1.f, 1.f, 1.f);
  }
  if (L < 0 || L > a.max_pages * kPageSize) {
    if (threadIdx.x == 0) atomicOr(&g_err_decode, kErrBadIndex);
    L = 0;
  }
  const int npages = (L + kPageSize - 1) / kPageSize;
  if (split > 0 && p_begin >= npages) return;   // empty split: the merge skips it
  const int nv = max(1, (npages + a.pages_per_split - 1) / a.pages_per_split);
  const bool direct = a.splits == 1 || nv == 1;
  const int p_end = min(npages, p_begin + a.pages_per_split);
  const int n_w = max(0, (p_end - p_begin - warp + W - 1) / W);   // pages of this warp

  const uint32_t bar0 = smem_u32(bars + warp * NB);
  uint8_t* wbuf = bufs + (size_t)warp * WARP_BYTES;
  const uint32_t wbuf_s = smem_u32(wbuf);
  const float* wsc = scales + warp * NB * (SC / 4);
  const uint32_t wsc_s = smem_u32(wsc);
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < NB; ++k) mbar_init(bar0 + 8 * k, 1);
    fence_mbar_init();
  }
  __syncwarp();

  const uint64_t policy = l2_policy_evict_first();
  int bt_cache = 0;
  auto page_id = [&](int i) -> int {
    if ((i & 31) == 0) {
      const int lp = p_begin + warp + (i + lane) * W;
      bt_cache = (i + lane < n_w) ? (i == 0 ? bt_first : __ldg(bt_row + lp)) : 0;
    }
    int pg = __shfl_sync(FULL, bt_cache, i & 31);
    if (pg < 0 || pg >= a.num_pages) {
      if (lane == 0) atomicOr(&g_err_decode, kErrBadIndex);
      pg = 0;
    }
    return pg;
  };
  auto issue = [&](int i, int pg) {
    if (lane == 0) {
      const int k = i % NB;
      const uint32_t bar = bar0 + 8 * k;
      const int row = (pg * a.num_kv_heads + h) * kPageSize;
      // the warp's generic-proxy reads of this buffer are done (__syncwarp);
      // order them before the async-proxy refill
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive_expect_tx(bar, KV + SC);
      tma_slab(wbuf_s + k * KV, &tk, row, bar, policy);
      tma_slab(wbuf_s + k * KV + SLAB, &tv, row, bar, policy);
      bulk_g2s(wsc_s + k * SC, a.k_scale + row, SC / 2, bar);
      bulk_g2s(wsc_s + k * SC + SC / 2, a.v_scale + row, SC / 2, bar);
    }
  };
  const int pro = min(NB, n_w);
  for (int i = 0; i < pro; ++i) issue(i, page_id(i));
  int issued = pro;

  // A fragments of the query (the loads above): lane (r, qd) holds channels
  // 32 qd + 4 kb + {0, 1} (a0a1 / a2a3) and + {2, 3} (a4a5 / a6a7) of rows
  // r and r + 8, pre-scaled by softmax_scale * log2(e) and the key smoothing
  // weight.
  uint32_t qa[8][4];
  {
    const float qs = a.softmax_scale * kLog2e;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
#pragma unroll
      for (int kb = 0; kb < 8; ++kb) {
        uint32_t v01 = 0, v23 = 0;
        if (qg[half] >= 0) {
          const uint2 raw = qraw[half][kb];
          float x[4] = {bf16lo(raw.x) * qs, bf16hi(raw.x) * qs, bf16lo(raw.y) * qs,
                        bf16hi(raw.y) * qs};
          if (a.k_smooth) {
            x[0] *= qw[kb].x;
            x[1] *= qw[kb].y;
            x[2] *= qw[kb].z;
            x[3] *= qw[kb].w;
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float hi = __half2float(__float2half_rn(x[e]));
            x[e] = qlow[half] ? x[e] - hi : hi;
          }
          v01 = pack_f16x2(x[0], x[1]);
          v23 = pack_f16x2(x[2], x[3]);
        }
        qa[kb][half] = v01;
        qa[kb][2 + half] = v23;
      }
    }
  }

  float o[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int j = 0; j < 4; ++j) o[mt][j] = 0.f;
  float m_used = -INFINITY, l = 0.f, cs = 0.f;
  float pc = 0.f;                     // power-of-two multiplier of P' (head row r)

  bool failed = false;
  int i_fail = 0;
  for (int i = 0; i < n_w; ++i) {
    const int k = i % NB;
    if (!mbar_wait(bar0 + 8 * k, (uint32_t)(i / NB) & 1u)) {
      failed = true;
      i_fail = i;
      break;
    }
    const int lp = p_begin + warp + i * W;
    const int nvalid = min(kPageSize, L - lp * kPageSize);
    const uint8_t* kbuf = wbuf + k * KV;
    const uint8_t* vbuf = kbuf + SLAB;
    const float* sc = wsc + k * (SC / 4);

    // QK: two tiles of 8 keys; key 8t + r's row, chunks 2qd and 2qd + 1
    float d[2][4];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
#pragma unroll
      for (int j = 0; j < 4; ++j) d[t][j] = 0.f;
      const uint8_t* row = kbuf + (8 * t + r) * kHeadDim;
      const uint4 x0 = lds128(row + (((2 * qd) ^ r) << 4));
      const uint4 x1 = lds128(row + (((2 * qd + 1) ^ r) << 4));
      const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
      for (int kb = 0; kb < 8; ++kb) {
        uint32_t blo, bhi;
        codes_f16(w[kb], blo, bhi);
        mma16816(d[t], qa[kb][0], qa[kb][1], qa[kb][2], qa[kb][3], blo, bhi);
      }
    }
    // scores of head row r for keys 8t + 2qd + e: high + low rows, times the
    // key scale; keys past the sequence are masked
    const float2 ksc[2] = {*reinterpret_cast<const float2*>(sc + 2 * qd),
                           *reinterpret_cast<const float2*>(sc + 8 + 2 * qd)};
    const float2 vsc[2] = {*reinterpret_cast<const float2*>(sc + 16 + 2 * qd),
                           *reinterpret_cast<const float2*>(sc + 24 + 2 * qd)};
    float s[2][2];
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float v = d[t][e];
        if constexpr (G == 8)
          v += d[t][e + 2];
        else
          v += __shfl_xor_sync(FULL, d[t][e], 4 * G);
        v *= e ? ksc[t].y : ksc[t].x;
        s[t][e] = (8 * t + 2 * qd + e < nvalid) ? v : -INFINITY;
      }
    float pm = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
    pm = fmaxf(pm, __shfl_xor_sync(FULL, pm, 1));
    pm = fmaxf(pm, __shfl_xor_sync(FULL, pm, 2));
    // the max the exponentials are taken against moves only when the page
    // max passes it by more than 2^8 (p <= 256; exact: l and O share it)
    const bool grow = pm > m_used + 8.f;
    float alpha = 1.f;
    if (grow) {
      alpha = fast_exp2(m_used - pm);
      m_used = pm;
      l *= alpha;
    }
    float pv[2][2];
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float p = fast_exp2(s[t][e] - m_used);
        l += p;
        // masked keys: p = 0, and their (unwritten) scale must not reach the MMA
        pv[t][e] = (8 * t + 2 * qd + e < nvalid) ? p * (e ? vsc[t].y : vsc[t].x) : 0.f;
      }
    // P' = p * v_scale goes to the MMA in f16, whose range (2^-24 .. 65504)
    // is far narrower than the V scales' (amax / 127 of any bf16 vector).  The
    // head carries a power-of-two multiplier pc (0 until a nonzero P' is
    // seen): it is lowered so that the page's largest P' * pc stays below
    // 2^14 and set, when first needed, so that it lands in [2^13, 2^14).  O
    // and the bias sum hold P' * pc units, rescaled exactly when pc moves, and
    // the epilogue divides pc out.  Scaling every V by 2^k scales pc by 2^-k
    // and leaves the f16 values unchanged.
    float pvm = fmaxf(fmaxf(pv[0][0], pv[0][1]), fmaxf(pv[1][0], pv[1][1]));
    pvm = fmaxf(pvm, __shfl_xor_sync(FULL, pvm, 1));
    pvm = fmaxf(pvm, __shfl_xor_sync(FULL, pvm, 2));
    const int pve = __float_as_int(pvm) >> 23;               // biased exponent (pvm >= 0)
    const float pc_want = __int_as_float(min(254, 267 - pve) << 23);   // 2^(13 - floor(log2 pvm))
    float f = alpha;
    if (pve > 0 && (pc == 0.f || pc_want < pc)) {             // unset, or P' * pc >= 2^14
      if (pc != 0.f) f *= pc_want / pc;                       // exact: powers of two
      pc = pc_want;
    }
    cs *= f;
    if (__any_sync(FULL, f != 1.f)) {
      const float a0 = __shfl_sync(FULL, f, 8 * qd);           // head 2qd's row
      const float a1 = __shfl_sync(FULL, f, 8 * qd + 4);       // head 2qd + 1's row
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        o[mt][0] *= a0;
        o[mt][1] *= a1;
        o[mt][2] *= a0;
        o[mt][3] *= a1;
      }
    }
    const uint32_t pb0 = pack_f16x2(pv[0][0] * pc, pv[0][1] * pc);
    const uint32_t pb1 = pack_f16x2(pv[1][0] * pc, pv[1][1] * pc);
    {
      const float2 f0 = unpack_f16x2(pb0), f1 = unpack_f16x2(pb1);
      cs += (f0.x + f0.y) + (f1.x + f1.y);
    }

    // PV: chunk r of keys 2qd, 2qd + 1, 2qd + 8, 2qd + 9
    const int k0 = 2 * qd;
    const uint4 va = lds128(vbuf + k0 * kHeadDim + ((r ^ k0) << 4));
    const uint4 vb = lds128(vbuf + (k0 + 1) * kHeadDim + ((r ^ (k0 + 1)) << 4));
    const uint4 vc = lds128(vbuf + (k0 + 8) * kHeadDim + ((r ^ k0) << 4));
    const uint4 vd = lds128(vbuf + (k0 + 9) * kHeadDim + ((r ^ (k0 + 1)) << 4));
    const uint32_t wa[4] = {va.x, va.y, va.z, va.w}, wb[4] = {vb.x, vb.y, vb.z, vb.w};
    const uint32_t wc[4] = {vc.x, vc.y, vc.z, vc.w}, wd[4] = {vd.x, vd.y, vd.z, vd.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t c[4], e[4];
      codes_pair_f16(wa[j], wb[j], c);
      codes_pair_f16(wc[j], wd[j], e);
      mma16816(o[2 * j], c[0], c[1], e[0], e[1], pb0, pb1);
      mma16816(o[2 * j + 1], c[2], c[3], e[2], e[3], pb0, pb1);
    }
    __syncwarp();
    if (issued < n_w) {
      issue(issued, page_id(issued));
      ++issued;
    }
  }
  if (failed) {
    if (lane == 0) atomicOr(&g_err_decode, kErrTimeout);
    for (int i = i_fail; i < issued; ++i)
      (void)mbar_wait(bar0 + 8 * (i % NB), (uint32_t)(i / NB) & 1u);
  }
  __syncwarp();

  // Park (O - 1152 sum P', m, l) of the warp's G heads in its buffers (all of
  // its copies have landed), then merge the warps.
  l += __shfl_xor_sync(FULL, l, 1);
  l += __shfl_xor_sync(FULL, l, 2);
  cs += __shfl_xor_sync(FULL, cs, 1);
  cs += __shfl_xor_sync(FULL, cs, 2);
  const float bA = kBias * __shfl_sync(FULL, cs, 8 * qd);
  const float bB = kBias * __shfl_sync(FULL, cs, 8 * qd + 4);
  // O and the bias sum are in units of pc: divide it out (pc = 0: no P' was
  // nonzero, O is 0)
  const float ipc = pc != 0.f ? 1.f / pc : 1.f;
  const float iA = __shfl_sync(FULL, ipc, 8 * qd), iB = __shfl_sync(FULL, ipc, 8 * qd + 4);
  float* wo = reinterpret_cast<float*>(wbuf);              // [G][128]
  float* wm = wo + G * kHeadDim;                           // [G]
  float* wl = wm + G;                                      // [G]
  const int c0 = 2 * qd, c1 = 2 * qd + 1;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const int ch = 16 * r + 4 * (mt >> 1) + 2 * (mt & 1);
    if (c0 < G)
      *reinterpret_cast<float2*>(wo + c0 * kHeadDim + ch) =
          failed ? make_float2(0.f, 0.f)
                 : make_float2((o[mt][0] - bA) * iA, (o[mt][2] - bA) * iA);
    if (c1 < G)
      *reinterpret_cast<float2*>(wo + c1 * kHeadDim + ch) =
          failed ? make_float2(0.f, 0.f)
                 : make_float2((o[mt][1] - bB) * iB, (o[mt][3] - bB) * iB);
  }
  if (qd == 0 && r < G) {
    wm[r] = failed ? -INFINITY : m_used;
    wl[r] = failed ? 0.f : l;
  }
  __syncthreads();
  merge_warps<G, FUSED, W>(a, smem, bufs, (size_t)WARP_BYTES, split, h, b, nv, direct);
}

// Combine (separate kernel): out = sum_s 2^(lse_s - lse) * O_s, lse = log2
// sum_s 2^lse_s, over the splits that hold keys (ceil(pages / pages_per_split)
// of them); rows whose keys fit one split were finished by that split.
__global__ void __launch_bounds__(128) decode_combine_kernel(const __grid_constant__
                                                             pkv_host::DecodeLaunch a) {
  __shared__ float wsm[128], red[4];
  pdl_wait();                                   // the split kernel's partials
  const int bh = blockIdx.x;
  const int b = bh / a.num_q_heads;
  const int d = threadIdx.x;
  int L = a.seq_lens[b];
  if (L < 0 || L > a.max_pages * kPageSize) L = 0;
  const int npages = (L + kPageSize - 1) / kPageSize;
  const int n = min(a.splits, (npages + a.pages_per_split - 1) / a.pages_per_split);
  if (n <= 1) return;                           // one split: it wrote the output itself
  const float2 r = merge_splits(a.ws_lse + (size_t)bh * a.splits,
                                a.ws_o + (size_t)bh * a.splits * kHeadDim, n, wsm, red);
  static_cast<__nv_bfloat16*>(a.out)[(size_t)bh * kHeadDim + d] = __float2bfloat16_rn(r.x);
  if (a.lse && d == 0) a.lse[bh] = r.y * kLn2;
}

template <int G, bool FUSED>
cudaError_t launch_split_as(const pkv_host::DecodeLaunch& a, cudaStream_t s) {
  cudaError_t e = pkv_host::set_max_dynamic_smem(
      reinterpret_cast<const void*>(decode_split_kernel<G, FUSED>), bfmma::SMEM);
  if (e != cudaSuccess) return e;
  if ((long long)a.num_pages * a.num_kv_heads * kPageSize >= (1ll << 31))
    return cudaErrorNotSupported;
  CUtensorMap tk, tv;
  if (!pkv_host::encode_bf16_pool_map(&tk, a.k, a.num_pages, a.num_kv_heads) ||
      !pkv_host::encode_bf16_pool_map(&tv, a.v, a.num_pages, a.num_kv_heads))
    return cudaErrorInvalidValue;
  dim3 grid(a.splits, a.num_kv_heads, a.batch);
  decode_split_kernel<G, FUSED><<<grid, bfmma::W * 32, bfmma::SMEM, s>>>(tk, tv, a);
  return cudaGetLastError();
}

template <int G>
cudaError_t launch_split(const pkv_host::DecodeLaunch& a, cudaStream_t s) {
  return a.ws_ctr ? launch_split_as<G, true>(a, s) : launch_split_as<G, false>(a, s);
}

template <int G, bool FUSED>
cudaError_t launch_i8mma_as(const pkv_host::DecodeLaunch& a, cudaStream_t s) {
  cudaError_t e = pkv_host::set_max_dynamic_smem(
      reinterpret_cast<const void*>(decode_split_i8mma_kernel<G, FUSED>), i8mma::SMEM);
  if (e != cudaSuccess) return e;
  if ((long long)a.num_pages * a.num_kv_heads * kPageSize >= (1ll << 31))
    return cudaErrorNotSupported;
  CUtensorMap tk, tv;
  if (!pkv_host::encode_int8_slab_map(&tk, a.k, a.num_pages, a.num_kv_heads) ||
      !pkv_host::encode_int8_slab_map(&tv, a.v, a.num_pages, a.num_kv_heads))
    return cudaErrorInvalidValue;
  dim3 grid(a.splits, a.num_kv_heads, a.batch);
  decode_split_i8mma_kernel<G, FUSED>
      <<<grid, i8mma::W * 32, i8mma::SMEM, s>>>(tk, tv, a);
  return cudaGetLastError();
}

template <int G>
cudaError_t launch_i8mma(const pkv_host::DecodeLaunch& a, cudaStream_t s) {
  return a.ws_ctr ? launch_i8mma_as<G, true>(a, s) : launch_i8mma_as<G, false>(a, s);
}

cudaError_t dispatch_i8mma(const pkv_host::DecodeLaunch& a, cudaStream_t s) {
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_i8mma<1>(a, s);
    case 2: return launch_i8mma<2>(a, s);
    case 4: return launch_i8mma<4>(a, s);
    case 8: return launch_i8mma<8>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t dispatch_group(const pkv_host::DecodeLaunch& a, cudaStream_t s) {
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_split<1>(a, s);
    case 2: return launch_split<2>(a, s);
    case 4: return launch_split<4>(a, s);
    case 8: return launch_split<8>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

namespace pkv_host {

bool decode_supports_group(int g) { return g == 1 || g == 2 || g == 4 || g == 8; }

cudaError_t launch_decode(const DecodeLaunch& a, bool int8, cudaStream_t s) {
  if (a.batch == 0) return cudaSuccess;
  cudaError_t e = int8 ? dispatch_i8mma(a, s) : dispatch_group(a, s);
  if (e != cudaSuccess || a.splits == 1 || a.ws_ctr) return e;
  // the combine's CTAs are placed while the split kernel's last ones run and
  // wait on the device for its partials, instead of a launch after it
  return launch_dependent(decode_combine_kernel, dim3(a.batch * a.num_q_heads), dim3(128), s, a);
}

uint32_t take_decode_error(cudaStream_t s) { return take_error_word(&g_err_decode, s); }

}  // namespace pkv_host

// ------------------------------------------------------------------------
// Fixed scratch for callers that cannot allocate (pkv_paged_attn_decode_noalloc).
// It holds the split partials that pkv_paged_attn_decode keeps in the
// caller's workspace.  In host code the name below is only a stand-in for
// the device array, never a device address: the kernels receive the address
// that cudaGetSymbolAddress returns for the current device.

static constexpr size_t kFixedScratchBytes = size_t(16) << 20;   // 16 MiB
static __device__ __align__(256) unsigned char g_decode_fixed_scratch[kFixedScratchBytes];

namespace pkv_host {

size_t decode_fixed_scratch_bytes() { return kFixedScratchBytes; }

cudaError_t decode_fixed_scratch(void** ptr) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_fixed_scratch);
    if (e != cudaSuccess) return e;
    if (!p) return cudaErrorInvalidSymbol;
    addr[dev] = p;
  }
  *ptr = addr[dev];
  return cudaSuccess;
}

}  // namespace pkv_host
