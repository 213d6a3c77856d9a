// qkv_prep.cu -- the fused attention-input step: from the fused q/k/v
// projection output, per-head RMSNorm of q and k, RoPE, and the KV cache
// write, in one pass (TileInfer.jl "Performance" page, section "Fused
// kernels, FlashAttention and PagedAttention": the attention-input kernel
// that replaces 3 copies, 2 norms, 2 RoPE and 1 write).
//
// Steps per head vector x (128 bf16 channels), as the unfused chain would
// run them: RMSNorm n_c = bf16(x_c * r * w_c), r = 1/sqrt(z) correctly
// rounded, z = fp32(ms + eps), ms = the exact mean of x^2 rounded once to
// fp32 (each step one fp32 rounding, so no summation order enters); RoPE by halves with the caller's cos/sin
// table at the token's position, o_i = bf16(n_i cos - n_{i+64} sin),
// o_{i+64} = bf16(n_{i+64} cos + n_i sin) (fp32, each product and sum
// rounded once); V copied.  A NULL weight skips that norm, a NULL table
// skips RoPE.
//
// One CTA of 4 warps per token; 8 lanes per head vector, 16-byte loads and
// stores, packed f32x2 arithmetic for the norm (the layout is described
// above finish_head).  HBM-bound: per token (Hq + 2 Hkv) x 256 bytes read and as
// many written.  Each warp issues the loads of its first three passes (12
// head vectors) before the position/page lookup, so the projection row is
// in flight while the dependent index loads resolve.
#include "common.cuh"
#include "internal.h"

namespace {

using namespace pkv;

__device__ uint32_t g_err_qkv;

__device__ __forceinline__ uint32_t bf16x2_rn(float2 v) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(v.y), "f"(v.x));
  return d;
}

__device__ __forceinline__ float2 unpack2(uint32_t w) { return make_float2(bf16lo(w), bf16hi(w)); }

constexpr int kWarps = 4;       // warps per CTA; one CTA per token
constexpr int kHeadsPerPass = kWarps * 4;
constexpr int kPassesAhead = 3; // passes whose loads are issued before the index chain

// Lane layout: 8 lanes per head vector, 4 heads per warp.  Lane l8 of a group
// holds channels 8 l8 .. 8 l8 + 7 (word a) and 64 + 8 l8 .. 64 + 8 l8 + 7
// (word b), so every RoPE pair (i, i + 64) sits in one lane and each warp
// access moves four 128-byte half rows.
struct Rope {
  float2 c[4], s[4];  // cos/sin of this lane's channel pairs at the token's position
};

// The mean of the squares of one head vector's 128 bf16 values, rounded once
// to fp32 from the exact sum, so that the result does not depend on the
// order of summation.  Each lane holds 16 of the values (words wa, wb); the
// 8 lanes of the head reduce by shuffles.  A bf16 magnitude is m 2^(E - 134)
// with an 8-bit integer m (E the biased exponent, 1 for subnormals), so its
// square is m^2 2^(2E - 268) with m^2 < 2^16.  The squares are added as
// integers in units of 2^(2 Emax - 308), Emax the head's largest exponent:
// m^2 << (2 (E - Emax) + 40), at most 2^56 each, 2^63 for all 128.  Exact
// while the values span at most 2^20 in magnitude (smaller squares are
// dropped below 2^-40 of the largest); the one rounding is the conversion
// of the 64-bit sum to fp32.  Caller contract: finite inputs.
__device__ __forceinline__ float mean_square_rn(const uint32_t (&wa)[4],
                                                const uint32_t (&wb)[4]) {
  uint32_t mx = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) mx = __vmaxu2(__vmaxu2(mx, wa[e] & 0x7fff7fffu), wb[e] & 0x7fff7fffu);
  mx = max(mx & 0xffffu, mx >> 16);
#pragma unroll
  for (int o = 4; o >= 1; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const int emax = max(1, (int)(mx >> 7));
  unsigned long long acc = 0;
  // m^2 << (2 (E - Emax) + 40) = (m << (E - Emax + 20))^2: a 32-bit shift
  // (below 2^28) and one widening multiply-add instead of 64-bit shifts
  const auto add = [&](uint32_t h) {
    h &= 0x7fffu;
    const int E = (int)(h >> 7);
    const uint32_t m = (h & 0x7fu) | (E ? 0x80u : 0u);
    const int s = max(E, 1) - emax + 20;
    const uint32_t v = s >= 0 ? m << s : 0u;
    acc += (unsigned long long)v * v;
  };
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    add(wa[e]);
    add(wa[e] >> 16);
    add(wb[e]);
    add(wb[e] >> 16);
  }
#pragma unroll
  for (int o = 4; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  // sum / 128 = acc 2^(2 emax - 315): scaling by a power of two is exact
  // while the result is a normal float
  return ldexpf(__ull2float_rn(acc), 2 * emax - 315);
}

// Norm, rotate (or copy) head h of token t and store it.  Every lane of the
// warp calls this together (the sum of squares is reduced with shuffles);
// lanes of a head past H compute on zeros and store nothing.
__device__ __forceinline__ void finish_head(const pkv_host::QkvPrepLaunch& a, int t, int h, int H,
                                            const uint4& xa, const uint4& xb, size_t slot0,
                                            bool rope, const Rope& rp, int l8) {
  const int Hq = a.num_q_heads, Hkv = a.num_kv_heads;
  const int kind = h < Hq ? 0 : h < Hq + Hkv ? 1 : h < H ? 2 : 3;  // q, k, v, none
  const uint32_t wa[4] = {xa.x, xa.y, xa.z, xa.w}, wb[4] = {xb.x, xb.y, xb.z, xb.w};
  float2 A[4], B[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    A[e] = unpack2(wa[e]);
    B[e] = unpack2(wb[e]);
  }
  const float ms = mean_square_rn(wa, wb);

  const float* w = kind == 0 ? a.q_w : kind == 1 ? a.k_w : nullptr;
  uint32_t oa[4], ob[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    oa[e] = wa[e];
    ob[e] = wb[e];
  }
  if (w) {
    // the chain's fp32 norm: z = fp32(mean + eps), r = 1/sqrt(z) correctly
    // rounded; it stores bf16
    const float r = __frsqrt_rn(__fadd_rn(ms, a.eps));
    const float2 rr = make_float2(r, r);
    const float4* w4 = reinterpret_cast<const float4*>(w) + 2 * l8;
    const float4 w0 = __ldg(w4), w1 = __ldg(w4 + 1), w2 = __ldg(w4 + 16), w3 = __ldg(w4 + 17);
    const float2 WA[4] = {{w0.x, w0.y}, {w0.z, w0.w}, {w1.x, w1.y}, {w1.z, w1.w}};
    const float2 WB[4] = {{w2.x, w2.y}, {w2.z, w2.w}, {w3.x, w3.y}, {w3.z, w3.w}};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      oa[e] = bf16x2_rn(mul2(mul2(A[e], rr), WA[e]));
      ob[e] = bf16x2_rn(mul2(mul2(B[e], rr), WB[e]));
      A[e] = unpack2(oa[e]);
      B[e] = unpack2(ob[e]);
    }
  }
  if (rope && kind < 2) {
    // Scalar round-to-nearest products and sums: ptxas may fuse a packed
    // f32x2 multiply into the packed add that consumes it, which changes
    // the rounding the chain's RoPE kernel performs.
    const auto rot_lo = [](float2 x, float2 y, float2 c, float2 s) {
      return make_float2(__fsub_rn(__fmul_rn(x.x, c.x), __fmul_rn(y.x, s.x)),
                         __fsub_rn(__fmul_rn(x.y, c.y), __fmul_rn(y.y, s.y)));
    };
    const auto rot_hi = [](float2 x, float2 y, float2 c, float2 s) {
      return make_float2(__fadd_rn(__fmul_rn(y.x, c.x), __fmul_rn(x.x, s.x)),
                         __fadd_rn(__fmul_rn(y.y, c.y), __fmul_rn(x.y, s.y)));
    };
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      oa[e] = bf16x2_rn(rot_lo(A[e], B[e], rp.c[e], rp.s[e]));
      ob[e] = bf16x2_rn(rot_hi(A[e], B[e], rp.c[e], rp.s[e]));
    }
  }
  uint4* dst;
  if (kind == 0)
    dst = static_cast<uint4*>(a.q_out) + ((size_t)t * Hq + h) * 16;
  else if (kind == 1)
    dst = static_cast<uint4*>(a.k) + (slot0 + (size_t)(h - Hq) * kPageSize) * 16;
  else if (kind == 2)
    dst = static_cast<uint4*>(a.v) + (slot0 + (size_t)(h - Hq - Hkv) * kPageSize) * 16;
  else
    return;
  dst[l8] = make_uint4(oa[0], oa[1], oa[2], oa[3]);
  dst[8 + l8] = make_uint4(ob[0], ob[1], ob[2], ob[3]);
}

__global__ void __launch_bounds__(kWarps * 32) qkv_prep_kernel(const __grid_constant__ pkv_host::QkvPrepLaunch a) {
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 3, l8 = lane & 7;
  const int H = a.num_q_heads + 2 * a.num_kv_heads;
  const uint4* row = static_cast<const uint4*>(a.qkv) + (size_t)t * H * 16;
  // The projection row needs nothing from the index chain below: put this
  // warp's first passes in flight before walking it.
  uint4 xa[kPassesAhead], xb[kPassesAhead];
#pragma unroll
  for (int j = 0; j < kPassesAhead; ++j) {
    const int h = j * kHeadsPerPass + warp * 4 + g;
    xa[j] = xb[j] = make_uint4(0, 0, 0, 0);
    if (h < H) {
      xa[j] = __ldg(row + (size_t)h * 16 + l8);
      xb[j] = __ldg(row + (size_t)h * 16 + 8 + l8);
    }
  }
  const int b = owner_seq(a.cu_new, a.batch, t);
  const int first = __ldg(a.cu_new + b);
  const int n = __ldg(a.cu_new + b + 1) - first;
  const int p = __ldg(a.seq_lens + b) - n + (t - first);
  bool bad = p < 0 || p >= a.max_pages * kPageSize || (a.cos && p >= a.max_pos);
  int page = 0;
  if (!bad) {
    page = __ldg(a.block_table + (size_t)b * a.max_pages + (p >> 4));
    bad = page < 0 || page >= a.num_pages;
  }
  if (bad) {
    if (threadIdx.x == 0) atomicOr(&g_err_qkv, kErrBadIndex);
    return;
  }
  const bool rope = a.cos != nullptr;
  Rope rp;
  if (rope) {
    const float4* c4 = reinterpret_cast<const float4*>(a.cos + (size_t)p * 64) + 2 * l8;
    const float4* s4 = reinterpret_cast<const float4*>(a.sin + (size_t)p * 64) + 2 * l8;
    const float4 c0 = __ldg(c4), c1 = __ldg(c4 + 1), s0 = __ldg(s4), s1 = __ldg(s4 + 1);
    rp.c[0] = make_float2(c0.x, c0.y); rp.c[1] = make_float2(c0.z, c0.w);
    rp.c[2] = make_float2(c1.x, c1.y); rp.c[3] = make_float2(c1.z, c1.w);
    rp.s[0] = make_float2(s0.x, s0.y); rp.s[1] = make_float2(s0.z, s0.w);
    rp.s[2] = make_float2(s1.x, s1.y); rp.s[3] = make_float2(s1.z, s1.w);
  }
  const size_t slot0 = (size_t)page * a.num_kv_heads * kPageSize + (p & 15);
#pragma unroll
  for (int j = 0; j < kPassesAhead; ++j) {
    if (j * kHeadsPerPass >= H) break;  // warp-uniform
    finish_head(a, t, j * kHeadsPerPass + warp * 4 + g, H, xa[j], xb[j], slot0, rope, rp, l8);
  }
  for (int base = kPassesAhead * kHeadsPerPass; base < H; base += kHeadsPerPass) {
    const int h = base + warp * 4 + g;
    uint4 ya = make_uint4(0, 0, 0, 0), yb = ya;
    if (h < H) {
      ya = __ldg(row + (size_t)h * 16 + l8);
      yb = __ldg(row + (size_t)h * 16 + 8 + l8);
    }
    finish_head(a, t, h, H, ya, yb, slot0, rope, rp, l8);
  }
}

}  // namespace

namespace pkv_host {

cudaError_t launch_qkv_prep(const QkvPrepLaunch& a, cudaStream_t s) {
  if (a.num_tokens == 0) return cudaSuccess;
  qkv_prep_kernel<<<a.num_tokens, kWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

uint32_t take_qkv_error(cudaStream_t s) { return take_error_word(&g_err_qkv, s); }

}  // namespace pkv_host
