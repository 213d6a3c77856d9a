// common.cuh -- device helpers shared by the sm_103a kernels of libpagedkv.
//
// Everything here is plain PTX for sm_103a: mbarriers with bounded waits,
// bulk (TMA-engine) copies, bf16 unpacking, packed f32x2 arithmetic and the
// log-sum-exp merge of split partials.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "pagedkv.h"

namespace pkv {

constexpr int kHeadDim = 128;
constexpr int kPageSize = 16;

// Bits of the device error word (one word per translation unit, read and
// cleared by pkv_poll_device_error).
constexpr uint32_t kErrTimeout = 1u;       // a bounded wait ran out
constexpr uint32_t kErrBadIndex = 2u;      // a block-table / position check failed

// Wall-clock limit of every spin-wait in these kernels (nanoseconds).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Sequence b that owns packed row t of a batch whose rows are laid out by
// prefix sums cu[0..batch] (cu non-decreasing, cu[0] = 0): the last b with
// cu[b] <= t, by binary search.
__device__ __forceinline__ int owner_seq(const int32_t* __restrict__ cu, int batch, int t) {
  int lo = 0, hi = batch;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(cu + mid) <= t) lo = mid; else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------- mbarriers

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Programmatic dependent launch.  A kernel calls pdl_trigger() to let the
// next kernel of its stream, when that one is launched with
// launch_dependent(), be scheduled before it has finished (the trigger takes
// effect once every CTA has issued it or exited); that kernel calls
// pdl_wait() before it touches memory: it returns once the previous kernel
// has completed and its writes are visible.  Both are no-ops without such a
// launch.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete.  Gives up after
// kWaitLimitNs of wall-clock time and returns false; never spins forever.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// --------------------------------------------------------- bulk copies

// One contiguous global -> shared copy by the TMA engine; completion is
// signalled as transaction bytes on the mbarrier.  Addresses 16-byte aligned,
// size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Same, with an L2 eviction-priority hint (streamed data: evict first).
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ------------------------------------------------------------ unpacking

// Two bf16 packed in a 32-bit word -> (low, high) as fp32 (exact).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }


// ------------------------------------------------- packed f32x2 helpers

union F2 {
  float2 f;
  unsigned long long u;
};

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  F2 x, y, z, r;
  x.f = a;
  y.f = b;
  z.f = c;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.u) : "l"(x.u), "l"(y.u), "l"(z.u));
  return r.f;
}

__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  F2 x, y, r;
  x.f = a;
  y.f = b;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.u) : "l"(x.u), "l"(y.u));
  return r.f;
}

__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  F2 x, y, r;
  x.f = a;
  y.f = b;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.u) : "l"(x.u), "l"(y.u));
  return r.f;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ------------------------------------------- warp-level bf16 tensor MMAs

// D += A B, m16n8k16, bf16 inputs, fp32 accumulate.  Fragments (r = lane / 4,
// qd = lane % 4): A rows r and r + 8, columns 2qd, 2qd + 1 (a0, a1) and
// 2qd + 8, 2qd + 9 (a2, a3); B rows 2qd, 2qd + 1 (b0) and + 8 (b1) of column
// r; D rows r (d0, d1) and r + 8 (d2, d3), columns 2qd, 2qd + 1.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four 8 x 8 b16 matrices from shared memory; lanes 8i .. 8i + 7 give the
// row addresses of matrix i (16 bytes each).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

// The same, each matrix transposed.
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

// ------------------------------------------------- split merge

// Log-sum-exp merge of n split partials of one (row, head) by a CTA of 128
// or more threads; threads 0..127 take one channel each, the others only
// join the barriers.  lp = the partials' log2-domain lse [n], op = their
// normalised O [n][128] (written by other CTAs: read through L2).
// Block-wide max, weights staged 128 splits at a time in shared memory
// (wsm, 128 floats; red, 4 floats), 8 partial rows in flight per thread.
// Every thread of the CTA must call it.  Returns (O, lse2) of channel
// threadIdx.x (threads 0..127); lse2 = -inf and O = 0 when no split holds a
// key.
__device__ __forceinline__ float2 merge_splits(const float* lp, const float* op, int n,
                                               float* wsm, float* red) {
  const int d = threadIdx.x;
  const bool act = d < 128;
  float M = -INFINITY;
  if (act)
    for (int s = d; s < n; s += 128) M = fmaxf(M, __ldcg(lp + s));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  __syncthreads();                                   // red / wsm free (earlier use done)
  if (act && (d & 31) == 0) red[d >> 5] = M;
  __syncthreads();
  M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  if (M == -INFINITY) return make_float2(0.f, -INFINITY);   // uniform over the CTA
  float sum = 0.f, O = 0.f;
  for (int base = 0; base < n; base += 128) {
    const int cnt = min(128, n - base);
    __syncthreads();                                 // the previous chunk's weights are used
    if (d < cnt) wsm[d] = fast_exp2(__ldcg(lp + base + d) - M);
    __syncthreads();
    if (!act) continue;
    const float* ob = op + (size_t)base * kHeadDim + d;
    int j = 0;
    for (; j + 8 <= cnt; j += 8) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = __ldcg(ob + (size_t)(j + u) * kHeadDim);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        sum += wsm[j + u];
        O += wsm[j + u] * v[u];
      }
    }
    for (; j < cnt; ++j) {
      sum += wsm[j];
      O += wsm[j] * __ldcg(ob + (size_t)j * kHeadDim);
    }
  }
  return act ? make_float2(O / sum, M + fast_log2(sum)) : make_float2(0.f, -INFINITY);
}

}  // namespace pkv

// Host-side helpers shared by the translation units.
namespace pkv_host {

// Reads a translation unit's device error word (its address is passed, from
// that unit) and clears it when it is set; ~0 if the copy fails.
inline uint32_t take_error_word(const void* symbol, cudaStream_t s) {
  uint32_t h = 0, zero = 0;
  if (cudaMemcpyFromSymbolAsync(&h, symbol, sizeof h, 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return ~0u;
  cudaStreamSynchronize(s);
  if (h) cudaMemcpyToSymbolAsync(symbol, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s);
  cudaStreamSynchronize(s);
  return h;
}
int sm_count();                 // cached SM count of the current device

// Raises a kernel's dynamic shared-memory limit to `bytes` once per (kernel,
// current device): the attribute belongs to the device's context, so a
// process flag would skip a second device.  Thread-safe.
cudaError_t set_max_dynamic_smem(const void* kernel, int bytes);

// Launches kernel k (no dynamic shared memory) after the work queued on s,
// allowed to start before the previous kernel has finished (programmatic
// stream serialization): k must call pdl_wait() before it reads what that
// kernel wrote.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*k)(Params...), dim3 grid, dim3 block, cudaStream_t s,
                             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, static_cast<Args&&>(args)...);
}
}
