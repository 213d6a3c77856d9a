// kv_append.cu -- write new K/V vectors into the pages named by the block
// table (TileInfer.jl "Performance" page, "Fused kernels, FlashAttention and
// PagedAttention": the KV cache write; "INT8 KV cache": one scale per cached
// vector, keys smoothed by the key norm's weight).
//
// bf16: a bit-for-bit copy, one thread per 16-byte chunk, 16 threads per
// 256-byte row, so every warp writes two full rows (coalesced 16-byte
// stores).  int8: one warp per (token, head) vector; each lane holds 4
// channels, the max |x| is a warp-shuffle reduction and every step of the
// quantiser is IEEE fp32 (round-to-nearest division, round-half-even to
// integer), so the codes and scales are bit-exact against any IEEE fp32
// implementation of the same steps.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace {

using namespace pkv;

__device__ uint32_t g_err_append;

// Flat slot (page * 16 + slot) of new row t, or -1 (and the error word set)
// when the position or the page id falls outside the caller's arrays.
__device__ __forceinline__ long long slot_of_row(const pkv_host::AppendLaunch& a, int t) {
  const int b = owner_seq(a.cu_new, a.batch, t);
  const int first = __ldg(a.cu_new + b);
  const int n = __ldg(a.cu_new + b + 1) - first;
  const int p = __ldg(a.seq_lens + b) - n + (t - first);
  if (p < 0 || p >= a.max_pages * kPageSize) {
    atomicOr(&g_err_append, kErrBadIndex);
    return -1;
  }
  const int page = __ldg(a.block_table + (size_t)b * a.max_pages + (p >> 4));
  if (page < 0 || page >= a.num_pages) {
    atomicOr(&g_err_append, kErrBadIndex);
    return -1;
  }
  return (long long)page * kPageSize + (p & 15);
}

__global__ void __launch_bounds__(256) append_bf16_kernel(pkv_host::AppendLaunch a) {
  const long long total = (long long)a.num_tokens * a.num_kv_heads * 16;
  const long long stride = (long long)gridDim.x * blockDim.x;
  uint4* __restrict__ kp = static_cast<uint4*>(a.k);
  uint4* __restrict__ vp = static_cast<uint4*>(a.v);
  const uint4* __restrict__ kn = static_cast<const uint4*>(a.k_new);
  const uint4* __restrict__ vn = static_cast<const uint4*>(a.v_new);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int c = (int)(i & 15);
    const long long row = i >> 4;                 // (token, head)
    const int h = (int)(row % a.num_kv_heads);
    const int t = (int)(row / a.num_kv_heads);
    // the new vectors need nothing from the slot lookup: load them first, so
    // that their latency overlaps the lookup's chain of dependent loads
    const uint4 kx = __ldg(kn + i);
    const uint4 vx = __ldg(vn + i);
    const long long fs = slot_of_row(a, t);
    if (fs < 0) continue;
    const long long page = fs >> 4, slot = fs & 15;
    const long long dst = (((page * a.num_kv_heads + h) << 4) + slot) * 16 + c;
    kp[dst] = kx;
    vp[dst] = vx;
  }
}

// Quantises the 128-channel vector spread over the warp (4 channels per
// lane) and stores the lane's 4 codes plus, from lane 0, the scale.
__device__ __forceinline__ void quantize_store(float x0, float x1, float x2, float x3,
                                               int8_t* __restrict__ dst_row,
                                               float* __restrict__ dst_scale, int lane) {
  float amax = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
  const float scale = __fdiv_rn(amax, 127.0f);
  uint32_t packed = 0;
  if (scale != 0.0f) {
    const float xs[4] = {x0, x1, x2, x3};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      int c = __float2int_rn(__fdiv_rn(xs[e], scale));   // nearest, ties to even
      c = max(-127, min(127, c));
      packed |= (uint32_t)(c & 0xff) << (8 * e);
    }
  }
  reinterpret_cast<uint32_t*>(dst_row)[lane] = packed;
  if (lane == 0) *dst_scale = scale;
}

__global__ void __launch_bounds__(256) append_int8_kernel(pkv_host::AppendLaunch a) {
  const int lane = threadIdx.x & 31;
  const long long rows = (long long)a.num_tokens * a.num_kv_heads;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  int8_t* __restrict__ kp = static_cast<int8_t*>(a.k);
  int8_t* __restrict__ vp = static_cast<int8_t*>(a.v);
  const uint2* __restrict__ kn = static_cast<const uint2*>(a.k_new);
  const uint2* __restrict__ vn = static_cast<const uint2*>(a.v_new);
  float4 w = make_float4(1.f, 1.f, 1.f, 1.f);
  if (a.k_smooth) w = __ldg(reinterpret_cast<const float4*>(a.k_smooth) + lane);
  for (long long row = (((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5); row < rows;
       row += nwarps) {
    const int h = (int)(row % a.num_kv_heads);
    const int t = (int)(row / a.num_kv_heads);
    const uint2 kr = __ldg(kn + row * 32 + lane);     // before the slot lookup (see above)
    const uint2 vr = __ldg(vn + row * 32 + lane);
    const long long fs = slot_of_row(a, t);
    if (fs < 0) continue;
    const long long page = fs >> 4, slot = fs & 15;
    const long long dst = ((page * a.num_kv_heads + h) << 4) + slot;   // vector index
    float k0 = bf16lo(kr.x), k1 = bf16hi(kr.x), k2 = bf16lo(kr.y), k3 = bf16hi(kr.y);
    if (a.k_smooth) {
      k0 = __fdiv_rn(k0, w.x);
      k1 = __fdiv_rn(k1, w.y);
      k2 = __fdiv_rn(k2, w.z);
      k3 = __fdiv_rn(k3, w.w);
    }
    quantize_store(k0, k1, k2, k3, kp + dst * kHeadDim, a.k_scale + dst, lane);
    quantize_store(bf16lo(vr.x), bf16hi(vr.x), bf16lo(vr.y), bf16hi(vr.y),
                   vp + dst * kHeadDim, a.v_scale + dst, lane);
  }
}

}  // namespace

namespace pkv_host {

cudaError_t launch_append(const AppendLaunch& a, bool int8, cudaStream_t s) {
  if (a.num_tokens == 0) return cudaSuccess;
  const int sms = sm_count();
  if (!int8) {
    const long long threads = (long long)a.num_tokens * a.num_kv_heads * 16;
    const long long blocks = (threads + 255) / 256;
    const int grid = (int)std::min<long long>(blocks, (long long)sms * 16);
    append_bf16_kernel<<<grid, 256, 0, s>>>(a);
  } else {
    const long long warps = (long long)a.num_tokens * a.num_kv_heads;
    const long long blocks = (warps + 7) / 8;
    const int grid = (int)std::min<long long>(blocks, (long long)sms * 16);
    append_int8_kernel<<<grid, 256, 0, s>>>(a);
  }
  return cudaGetLastError();
}

uint32_t take_append_error(cudaStream_t s) { return take_error_word(&g_err_append, s); }

}  // namespace pkv_host
