// decode.cu -- split-KV paged decode attention and the log-sum-exp combine
// (TileInfer.jl "Performance" page, "Fused kernels, FlashAttention and
// PagedAttention": online softmax over the pages in place through the block
// table, split-KV for decode, and a combine kernel kept separate from the
// split kernel; "INT8 KV cache": dequantisation inside attention).
//
// Split kernel: one CTA per (split, KV head, sequence), 4 warps.  A split is
// a run of consecutive logical pages of one sequence; the warps take its
// pages round-robin and each warp streams its pages through a private ring
// of shared-memory page buffers filled by the TMA engine (cp.async.bulk of
// the contiguous 4 KiB (page, head) slabs, L2 evict-first), so no CTA-wide
// barrier sits in the page loop.  Every warp serves all G query heads of
// the KV head, so each K/V byte is read from HBM once per decode step.
//
// Lane layout inside a warp: DL lanes cover one key's 128 channels (DPL
// channels each), KG = 32 / DL keys per pass, 16 / KG passes per page.
// Partial dot products are reduced across the DL lanes with a reduce-scatter
// (each stage halves the heads a lane carries), so after log2(DL) shuffle
// stages every lane holds one head's score of its key.  The online-softmax
// state of a head lives in the lanes that own it; p and the rescale factor
// reach the other lanes by shuffles.  Shared-memory reads rotate their
// 16-byte chunk order by key so that a warp's 32 loads hit all 32 banks.
//
// The split's result is normalised (O / l) and written with its log2-domain
// lse; with a single split the kernel writes the bf16 output directly and
// the combine is skipped.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

using namespace pkv;

__device__ uint32_t g_err_decode;

template <int G, bool INT8>
struct Cfg {
  // lanes per key: INT8 with G = 4 uses 16 lanes (8 channels each), which
  // halves the query/accumulator registers so more warps fit per SM
  static constexpr int DL = (G <= 2) ? 4 : ((G == 4 && !INT8) ? 8 : 16);
  static constexpr int KG = 32 / DL;                              // keys per pass
  static constexpr int PASSES = kPageSize / KG;
  static constexpr int DPL = kHeadDim / DL;                       // channels per lane
  static constexpr int ESZ = INT8 ? 1 : 2;
  static constexpr int LDB = (DPL * ESZ >= 16) ? 16 : DPL * ESZ;  // bytes per shared load
  static constexpr int EPL = LDB / ESZ;                           // elements per load
  static constexpr int NLD = DPL / EPL;                           // loads per lane per key
  static constexpr int ROWB = kHeadDim * ESZ;                     // bytes per key row
  static constexpr int SLAB = kPageSize * ROWB;                   // K or V slab bytes
  static constexpr int SCB = INT8 ? kPageSize * 4 : 0;            // scale bytes per slab
  static constexpr int BUF = 2 * SLAB + 2 * SCB;                  // one page of K, V (+scales)
  static constexpr int HL = DL / G;                               // lanes per head after scatter
  static constexpr int NBUF = INT8 ? (DL == 16 ? 3 : 5) : 3;      // page buffers per warp
  static_assert(NLD >= 1 && (NLD & (NLD - 1)) == 0, "loads per key must be a power of two");
  static_assert(BUF % 128 == 0, "page buffers stay 128-byte aligned");
};

struct SplitArgs {
  pkv_host::DecodeLaunch a;
};

// Loads EPL consecutive elements at a shared address and widens them to fp32
// pairs.  int8 codes are widened exactly (no scale applied here).
template <bool INT8, int EPL>
__device__ __forceinline__ void load_widen(const uint8_t* p, float2 (&x)[EPL / 2]) {
  if constexpr (!INT8) {
    static_assert(EPL == 8, "bf16 loads are 16 bytes");
    const uint4 r = *reinterpret_cast<const uint4*>(p);
    x[0] = make_float2(bf16lo(r.x), bf16hi(r.x));
    x[1] = make_float2(bf16lo(r.y), bf16hi(r.y));
    x[2] = make_float2(bf16lo(r.z), bf16hi(r.z));
    x[3] = make_float2(bf16lo(r.w), bf16hi(r.w));
  } else {
    constexpr int NW = EPL / 4;
    uint32_t w[NW];
    if constexpr (EPL == 16) {
      const uint4 r = *reinterpret_cast<const uint4*>(p);
      w[0] = r.x; w[1] = r.y; w[2] = r.z; w[3] = r.w;
    } else {
      static_assert(EPL == 8, "int8 loads are 8 or 16 bytes");
      const uint2 r = *reinterpret_cast<const uint2*>(p);
      w[0] = r.x; w[1] = r.y;
    }
    const float2 bias = make_float2(-kI8Bias, -kI8Bias);
#pragma unroll
    for (int k = 0; k < NW; ++k) {
      const uint32_t u = w[k] ^ 0x80808080u;
      x[2 * k] = add2(make_float2(__uint_as_float(i8_biased_bits<0>(u)),
                                  __uint_as_float(i8_biased_bits<1>(u))), bias);
      x[2 * k + 1] = add2(make_float2(__uint_as_float(i8_biased_bits<2>(u)),
                                      __uint_as_float(i8_biased_bits<3>(u))), bias);
    }
  }
}

// Sum of v[g] over the DL lanes of a key, scattered: afterwards lane dl holds
// the full sum of head dl / (DL / G).
template <int G, int DL>
__device__ __forceinline__ float reduce_scatter(float (&v)[G], int dl) {
  int nv = G;
#pragma unroll
  for (int m = DL / 2; m >= 1; m >>= 1) {
    const bool upper = (dl & m) != 0;
    if (nv > 1) {
#pragma unroll
      for (int i = 0; i < G / 2; ++i) {
        if (i < nv / 2) {
          const float send = upper ? v[i] : v[i + nv / 2];
          const float keep = upper ? v[i + nv / 2] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
      }
      nv >>= 1;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], m);
    }
  }
  return v[0];
}

template <int G, bool INT8>
struct WarpState {
  using C = Cfg<G, INT8>;
  float2 q[C::NLD][C::EPL / 2][G];   // pre-scaled query, in this lane's chunk order
  float2 o[C::NLD][C::EPL / 2][G];   // unnormalised output accumulators
  float m = -INFINITY;               // running max (log2 domain) of head dl / HL
  float l = 0.f;                     // partial sum of head dl / HL over this lane's keys
};

// One page of 16 keys (nvalid of them real) from shared memory.
template <int G, bool INT8, bool PARTIAL>
__device__ __forceinline__ void process_page(WarpState<G, INT8>& st, const uint8_t* buf,
                                             int nvalid, int kg, int dl) {
  using C = Cfg<G, INT8>;
  const uint8_t* kbuf = buf;
  const uint8_t* vbuf = buf + C::SLAB;
  const float* ksc = reinterpret_cast<const float*>(buf + 2 * C::SLAB);
  const float* vsc = ksc + kPageSize;
  const int lane = kg * C::DL + dl;

  float s[C::PASSES];
#pragma unroll
  for (int ps = 0; ps < C::PASSES; ++ps) {
    const int key = ps * C::KG + kg;
    const uint8_t* row = kbuf + key * C::ROWB + dl * C::DPL * C::ESZ;
    float2 acc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) acc[g] = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < C::NLD; ++j) {
      const int jj = (j + kg) & (C::NLD - 1);
      float2 x[C::EPL / 2];
      load_widen<INT8, C::EPL>(row + jj * C::LDB, x);
#pragma unroll
      for (int i = 0; i < C::EPL / 2; ++i)
#pragma unroll
        for (int g = 0; g < G; ++g) acc[g] = fma2(st.q[j][i][g], x[i], acc[g]);
    }
    float part[G];
#pragma unroll
    for (int g = 0; g < G; ++g) part[g] = acc[g].x + acc[g].y;
    float sc = reduce_scatter<G, C::DL>(part, dl);
    if constexpr (INT8) sc *= ksc[key];
    s[ps] = (PARTIAL && key >= nvalid) ? -INFINITY : sc;
  }

  float pm = s[0];
#pragma unroll
  for (int ps = 1; ps < C::PASSES; ++ps) pm = fmaxf(pm, s[ps]);
#pragma unroll
  for (int m = C::DL; m < 32; m <<= 1) pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, m));
  const float m_new = fmaxf(st.m, pm);
  const float alpha = fast_exp2(st.m - m_new);
  float p[C::PASSES];
  float lsum = 0.f;
#pragma unroll
  for (int ps = 0; ps < C::PASSES; ++ps) {
    p[ps] = fast_exp2(s[ps] - m_new);
    lsum += p[ps];
  }
  st.l = st.l * alpha + lsum;
  st.m = m_new;

  if (__any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float ag = __shfl_sync(0xffffffffu, alpha, g * C::HL);
      const float2 a2 = make_float2(ag, ag);
#pragma unroll
      for (int j = 0; j < C::NLD; ++j)
#pragma unroll
        for (int i = 0; i < C::EPL / 2; ++i) st.o[j][i][g] = mul2(st.o[j][i][g], a2);
    }
  }

#pragma unroll
  for (int ps = 0; ps < C::PASSES; ++ps) {
    const int key = ps * C::KG + kg;
    float pg[G];
#pragma unroll
    for (int g = 0; g < G; ++g)
      pg[g] = __shfl_sync(0xffffffffu, p[ps], (lane & ~(C::DL - 1)) | (g * C::HL));
    if (!PARTIAL || key < nvalid) {
      if constexpr (INT8) {
        const float vs = vsc[key];
#pragma unroll
        for (int g = 0; g < G; ++g) pg[g] *= vs;
      }
      const uint8_t* row = vbuf + key * C::ROWB + dl * C::DPL * C::ESZ;
#pragma unroll
      for (int j = 0; j < C::NLD; ++j) {
        const int jj = (j + kg) & (C::NLD - 1);
        float2 x[C::EPL / 2];
        load_widen<INT8, C::EPL>(row + jj * C::LDB, x);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float2 p2 = make_float2(pg[g], pg[g]);
#pragma unroll
          for (int i = 0; i < C::EPL / 2; ++i) st.o[j][i][g] = fma2(p2, x[i], st.o[j][i][g]);
        }
      }
    }
  }
}

// FUSED: the split that completes a (sequence, KV head) merges its splits
// (a.ws_ctr counts them); otherwise a separate combine kernel does.  A
// template parameter, so that the default kernel carries none of that code.
template <int G, bool INT8, bool FUSED>
__global__ void __launch_bounds__(pkv_host::kDecodeWarps * 32)
    decode_split_kernel(const __grid_constant__ pkv_host::DecodeLaunch a) {
  using C = Cfg<G, INT8>;
  constexpr int W = pkv_host::kDecodeWarps;
  constexpr int NBUF = C::NBUF;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint8_t* bufs = smem + 1024;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kg = lane / C::DL, dl = lane % C::DL;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int Hq = a.num_q_heads;

  int L = a.seq_lens[b];
  if (L < 0 || L > a.max_pages * kPageSize) {
    if (threadIdx.x == 0) atomicOr(&g_err_decode, kErrBadIndex);
    L = 0;
  }
  const int npages = (L + kPageSize - 1) / kPageSize;
  const int p_begin = split * a.pages_per_split;
  if (split > 0 && p_begin >= npages) return;   // empty split: the merge skips it
  // splits holding keys (split 0 always runs); with one, it writes the output
  const int nv = max(1, (npages + a.pages_per_split - 1) / a.pages_per_split);
  const bool direct = a.splits == 1 || nv == 1;
  const int p_end = min(npages, p_begin + a.pages_per_split);
  const int n_w = max(0, (p_end - p_begin - warp + W - 1) / W);   // pages of this warp

  const uint32_t bar0 = smem_u32(bars + warp * NBUF);
  uint8_t* wbuf = bufs + (size_t)warp * NBUF * C::BUF;
  const uint32_t wbuf_s = smem_u32(wbuf);
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < NBUF; ++k) mbar_init(bar0 + 8 * k, 1);
    fence_mbar_init();
  }
  __syncwarp();

  const int32_t* bt_row = a.block_table + (size_t)b * a.max_pages;
  const size_t Hkv = (size_t)a.num_kv_heads;
  const uint8_t* kpool = static_cast<const uint8_t*>(a.k);
  const uint8_t* vpool = static_cast<const uint8_t*>(a.v);
  const uint64_t policy = l2_policy_evict_first();

  // Page ids of this warp's pages, 32 at a time, one per lane.
  int bt_cache = 0;
  auto page_id = [&](int i) -> int {
    if ((i & 31) == 0) {
      const int lp = p_begin + warp + (i + lane) * W;
      bt_cache = (i + lane < n_w) ? __ldg(bt_row + lp) : 0;
    }
    int pg = __shfl_sync(0xffffffffu, bt_cache, i & 31);
    if (pg < 0 || pg >= a.num_pages) {
      if (lane == 0) atomicOr(&g_err_decode, kErrBadIndex);
      pg = 0;
    }
    return pg;
  };
  auto issue = [&](int i, int pg) {
    if (lane == 0) {
      const int k = i % NBUF;
      const uint32_t bar = bar0 + 8 * k;
      const uint32_t dst = wbuf_s + k * C::BUF;
      const size_t slab = (size_t)pg * Hkv + h;
      // the warp's generic-proxy reads of this buffer are done (__syncwarp);
      // order them before the async-proxy refill
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive_expect_tx(bar, C::BUF);
      bulk_g2s_hint(dst, kpool + slab * C::SLAB, C::SLAB, bar, policy);
      bulk_g2s_hint(dst + C::SLAB, vpool + slab * C::SLAB, C::SLAB, bar, policy);
      if constexpr (INT8) {
        bulk_g2s(dst + 2 * C::SLAB, a.k_scale + slab * kPageSize, C::SCB, bar);
        bulk_g2s(dst + 2 * C::SLAB + C::SCB, a.v_scale + slab * kPageSize, C::SCB, bar);
      }
    }
  };

  // Page ids are needed in issue order 0, 1, 2, ...; the prologue issues the
  // first NBUF pages, the loop refills buffer k after consuming page i.
  const int pro = min(NBUF, n_w);
  for (int i = 0; i < pro; ++i) issue(i, page_id(i));
  int issued = pro;
  // Query rows of the group, pre-scaled by softmax_scale * log2(e) (and by
  // the key smoothing weight, which the dequantised keys carry).  Loaded
  // after the first page copies are in flight, so their latency overlaps.
  WarpState<G, INT8> st;
  {
    const float qs = a.softmax_scale * kLog2e;
    const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(a.q);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const __nv_bfloat16* qrow = qb + ((size_t)b * Hq + h * G + g) * kHeadDim;
#pragma unroll
      for (int j = 0; j < C::NLD; ++j) {
        const int jj = (j + kg) & (C::NLD - 1);
        const int d0 = dl * C::DPL + jj * C::EPL;      // EPL is 8 or 16: whole 16-byte chunks
#pragma unroll
        for (int c8 = 0; c8 < C::EPL / 8; ++c8) {
          const uint4 raw = __ldg(reinterpret_cast<const uint4*>(qrow + d0 + 8 * c8));
          const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float x0 = bf16lo(w[e]) * qs, x1 = bf16hi(w[e]) * qs;
            if (INT8 && a.k_smooth) {
              const float2 ww = __ldg(reinterpret_cast<const float2*>(a.k_smooth + d0 + 8 * c8 + 2 * e));
              x0 *= ww.x;
              x1 *= ww.y;
            }
            st.q[j][4 * c8 + e][g] = make_float2(x0, x1);
            st.o[j][4 * c8 + e][g] = make_float2(0.f, 0.f);
          }
        }
      }
    }
  }

  bool failed = false;
  int i_fail = 0;
  for (int i = 0; i < n_w; ++i) {
    const int k = i % NBUF;
    if (!mbar_wait(bar0 + 8 * k, (uint32_t)(i / NBUF) & 1u)) {
      failed = true;
      i_fail = i;
      break;
    }
    const int lp = p_begin + warp + i * W;
    const int nvalid = min(kPageSize, L - lp * kPageSize);
    const uint8_t* buf = wbuf + k * C::BUF;
    if (nvalid == kPageSize)
      process_page<G, INT8, false>(st, buf, nvalid, kg, dl);
    else
      process_page<G, INT8, true>(st, buf, nvalid, kg, dl);
    __syncwarp();
    if (issued < n_w) {
      issue(issued, page_id(issued));
      ++issued;
    }
  }
  if (failed) {
    if (lane == 0) atomicOr(&g_err_decode, kErrTimeout);
    // Let every copy this warp issued land (bounded) before the buffers are
    // reused or the CTA exits.
    for (int i = i_fail; i < issued; ++i)
      (void)mbar_wait(bar0 + 8 * (i % NBUF), (uint32_t)(i / NBUF) & 1u);
    st.m = -INFINITY;
    st.l = 0.f;
  }

  // Warp merge: lanes of different key groups hold the same channels, but
  // in rotated chunk order (slot j holds chunk (j + kg) mod NLD); put every
  // lane back in natural order, then sum over the key groups.
  float l = st.l;
#pragma unroll
  for (int m = C::DL; m < 32; m <<= 1) l += __shfl_xor_sync(0xffffffffu, l, m);
  if constexpr (C::NLD > 1) {
    float2 nat[C::NLD][C::EPL / 2][G];
#pragma unroll
    for (int c = 0; c < C::NLD; ++c)
#pragma unroll
      for (int i = 0; i < C::EPL / 2; ++i)
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float2 v = st.o[0][i][g];
#pragma unroll
          for (int j = 1; j < C::NLD; ++j)
            if (((j + kg) & (C::NLD - 1)) == c) v = st.o[j][i][g];
          nat[c][i][g] = v;
        }
#pragma unroll
    for (int c = 0; c < C::NLD; ++c)
#pragma unroll
      for (int i = 0; i < C::EPL / 2; ++i)
#pragma unroll
        for (int g = 0; g < G; ++g) st.o[c][i][g] = nat[c][i][g];
  }
#pragma unroll
  for (int j = 0; j < C::NLD; ++j)
#pragma unroll
    for (int i = 0; i < C::EPL / 2; ++i)
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float2 v = st.o[j][i][g];
#pragma unroll
        for (int m = C::DL; m < 32; m <<= 1) {
          v.x += __shfl_xor_sync(0xffffffffu, v.x, m);
          v.y += __shfl_xor_sync(0xffffffffu, v.y, m);
        }
        st.o[j][i][g] = v;
      }

  // Each warp parks (m, l, O) of its G heads in its own buffers (all of its
  // copies have landed), then the CTA merges the warps.
  float* wo = reinterpret_cast<float*>(wbuf);              // [G][128]
  float* wm = wo + G * kHeadDim;                           // [G]
  float* wl = wm + G;                                      // [G]
  if (kg == 0) {
#pragma unroll
    for (int j = 0; j < C::NLD; ++j)
#pragma unroll
      for (int i = 0; i < C::EPL / 2; ++i)
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const int d = dl * C::DPL + j * C::EPL + 2 * i;   // natural chunk order
          *reinterpret_cast<float2*>(wo + g * kHeadDim + d) =
              failed ? make_float2(0.f, 0.f) : st.o[j][i][g];
        }
    if (dl % C::HL == 0) {
      wm[dl / C::HL] = st.m;
      wl[dl / C::HL] = failed ? 0.f : l;
    }
  }
  __syncthreads();

  for (int t = threadIdx.x; t < G * kHeadDim; t += W * 32) {
    const int g = t / kHeadDim, d = t % kHeadDim;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      const float* wmw = reinterpret_cast<const float*>(bufs + (size_t)w * NBUF * C::BUF) +
                         G * kHeadDim;
      M = fmaxf(M, wmw[g]);
    }
    float Lsum = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const float* wow = reinterpret_cast<const float*>(bufs + (size_t)w * NBUF * C::BUF);
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
  static_assert(pkv_host::kDecodeWarps * 5 * 8 <= 1020, "barrier header");
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
  for (int t = threadIdx.x; t < G * kHeadDim; t += W * 32) {
    const int g = t / kHeadDim, d = t % kHeadDim;
    const size_t bh = (size_t)b * Hq + h * G + g;
    const float* lp = a.ws_lse + bh * a.splits;
    const float* op = a.ws_o + bh * a.splits * kHeadDim;
    float M = -INFINITY;
    for (int sp = 0; sp < nv; ++sp) M = fmaxf(M, __ldcg(lp + sp));
    float sum = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int sp = 0; sp < nv; ++sp) {
        const float f = fast_exp2(__ldcg(lp + sp) - M);
        sum += f;
        O += f * __ldcg(op + (size_t)sp * kHeadDim + d);
      }
      O = O / sum;
    }
    static_cast<__nv_bfloat16*>(a.out)[bh * kHeadDim + d] = __float2bfloat16_rn(O);
    if (a.lse && d == 0) a.lse[bh] = (M == -INFINITY) ? -INFINITY : (M + fast_log2(sum)) * kLn2;
  }
}

// Combine (separate kernel): out = sum_s 2^(lse_s - lse) * O_s, lse = log2
// sum_s 2^lse_s, over the splits that hold keys (ceil(pages / pages_per_split)
// of them); rows whose keys fit one split were finished by that split.
__global__ void __launch_bounds__(128) decode_combine_kernel(const __grid_constant__
                                                             pkv_host::DecodeLaunch a) {
  const int bh = blockIdx.x;
  const int b = bh / a.num_q_heads;
  const int d = threadIdx.x;
  int L = a.seq_lens[b];
  if (L < 0 || L > a.max_pages * kPageSize) L = 0;
  const int npages = (L + kPageSize - 1) / kPageSize;
  const int n = min(a.splits, (npages + a.pages_per_split - 1) / a.pages_per_split);
  if (n <= 1) return;                           // one split: it wrote the output itself
  const float* lp = a.ws_lse + (size_t)bh * a.splits;
  const float* op = a.ws_o + (size_t)bh * a.splits * kHeadDim;
  float M = -INFINITY;
  for (int s = 0; s < n; ++s) M = fmaxf(M, lp[s]);
  float sum = 0.f, O = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < n; ++s) {
      const float f = fast_exp2(lp[s] - M);
      sum += f;
      O += f * op[(size_t)s * kHeadDim + d];
    }
    O = O / sum;
  }
  static_cast<__nv_bfloat16*>(a.out)[(size_t)bh * kHeadDim + d] = __float2bfloat16_rn(O);
  if (a.lse && d == 0)
    a.lse[bh] = (M == -INFINITY) ? -INFINITY : (M + fast_log2(sum)) * kLn2;
}

template <int G, bool INT8, bool FUSED>
cudaError_t launch_split_as(const pkv_host::DecodeLaunch& a, cudaStream_t s) {
  using C = Cfg<G, INT8>;
  constexpr int smem = 1024 + pkv_host::kDecodeWarps * C::NBUF * C::BUF;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<G, INT8, FUSED>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(a.splits, a.num_kv_heads, a.batch);
  decode_split_kernel<G, INT8, FUSED><<<grid, pkv_host::kDecodeWarps * 32, smem, s>>>(a);
  return cudaGetLastError();
}

template <int G, bool INT8>
cudaError_t launch_split(const pkv_host::DecodeLaunch& a, cudaStream_t s) {
  return a.ws_ctr ? launch_split_as<G, INT8, true>(a, s) : launch_split_as<G, INT8, false>(a, s);
}

template <bool INT8>
cudaError_t dispatch_group(const pkv_host::DecodeLaunch& a, cudaStream_t s) {
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_split<1, INT8>(a, s);
    case 2: return launch_split<2, INT8>(a, s);
    case 4: return launch_split<4, INT8>(a, s);
    case 8: return launch_split<8, INT8>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

namespace pkv_host {

bool decode_supports_group(int g) { return g == 1 || g == 2 || g == 4 || g == 8; }

cudaError_t launch_decode(const DecodeLaunch& a, bool int8, cudaStream_t s) {
  if (a.batch == 0) return cudaSuccess;
  cudaError_t e = int8 ? dispatch_group<true>(a, s) : dispatch_group<false>(a, s);
  if (e != cudaSuccess || a.splits == 1 || a.ws_ctr) return e;
  decode_combine_kernel<<<a.batch * a.num_q_heads, 128, 0, s>>>(a);
  return cudaGetLastError();
}

uint32_t take_decode_error(cudaStream_t s) {
  uint32_t h = 0, zero = 0;
  if (cudaMemcpyFromSymbolAsync(&h, g_err_decode, sizeof h, 0, cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return ~0u;
  cudaStreamSynchronize(s);
  if (h) cudaMemcpyToSymbolAsync(g_err_decode, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s);
  cudaStreamSynchronize(s);
  return h;
}

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
