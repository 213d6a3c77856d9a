// api.cu -- the extern "C" entry points of libpagedkv.so (declared in
// include/pagedkv.h): host-side argument checks, the split-count heuristic
// and kernel dispatch.  Nothing here allocates device or host memory.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace pkv_host {

namespace {
constexpr int kMaxDevices = 64;
}

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  static std::atomic<int> cached[kMaxDevices];     // 0: not looked up yet
  const bool slot = dev >= 0 && dev < kMaxDevices;
  int n = slot ? cached[dev].load(std::memory_order_relaxed) : 0;
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 152;
  if (slot) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

cudaError_t set_max_dynamic_smem(const void* kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  // (kernel, device) pairs already raised; a fixed table, no allocation
  // (when it is full the attribute is simply set on every launch)
  struct Entry {
    const void* kernel;
    int dev;
  };
  static std::mutex mu;
  static Entry done[512];
  static int n_done = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_done; ++i)
    if (done[i].kernel == kernel && done[i].dev == dev) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && n_done < 512) done[n_done++] = {kernel, dev};
  return e;
}

}  // namespace pkv_host

namespace {

using pkv_host::sm_count;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

pkv_status check_pool(const pkv_pool* pool) {
  if (!pool || !pool->k || !pool->v) return PKV_ERR_INVALID;
  if (pool->head_dim != pkv::kHeadDim || pool->page_size != pkv::kPageSize)
    return PKV_ERR_INVALID;
  if (pool->num_pages <= 0 || pool->num_kv_heads <= 0) return PKV_ERR_INVALID;
  if (!aligned(pool->k, 16) || !aligned(pool->v, 16)) return PKV_ERR_INVALID;
  if (pool->dtype == PKV_BF16) {
    if (pool->k_scale || pool->v_scale) return PKV_ERR_INVALID;
  } else if (pool->dtype == PKV_INT8) {
    if (!pool->k_scale || !pool->v_scale) return PKV_ERR_INVALID;
    if (!aligned(pool->k_scale, 16) || !aligned(pool->v_scale, 16)) return PKV_ERR_INVALID;
  } else {
    return PKV_ERR_INVALID;
  }
  return PKV_OK;
}

// Split plan: pages per split C and split count S for a decode call.
//
// The split kernel runs one CTA per (split, KV head, sequence) with 4 warps
// (bf16, three CTAs resident per SM) or 8 (INT8, two); the plan counts two
// resident CTAs per SM for both.  A CTA pays a few microseconds of start-up
// (query and block-table loads, the first page copies), so splits are made
// as long as the machine allows: about 0.8 CTAs per resident slot for bf16
// (bound by HBM) and one for INT8 (bound by the work per page, which an SM
// with one CTA does not share: one 32k sequence, 248 CTAs -> 296), estimated
// from the longest sequence, with 8 to 96 bf16 pages or 8 to 128 INT8 pages
// (half the bytes) per split, a multiple of the 4 warps so that they get
// equal work.  Measured on GB300: 64 sequences of 512..8,192 positions and
// the 32 decode rows of the mixed step (contexts up to 16,384) run best at
// 64..96 bf16 pages per split, 8 bf16 sequences of 32,768 positions at 64..96;
// one 32k-position INT8 sequence with one full wave of CTAs (37 splits of 56
// pages; 31 splits, 0.8 per slot, were 8 % slower), eight of them at 128
// pages.  A forced split count S gives C = ceil(pages / S).
constexpr long long kPlanSlotsNum = 4, kPlanSlotsDen = 5;   // 0.8 CTAs per slot (bf16)
constexpr long long kPlanMinPages = 8, kPlanMaxPages = 128, kPlanMaxPagesBf16 = 96;

// Workspace (splits > 1): part counters u32 [kDecodeCounters] indexed by
// b * Hkv + h (a fixed region, so that a workspace reused by calls of any
// shape never finds partials where counters go; zero between calls), then
// normalised partial O fp32 [B][Hq][S][128], then log2 lse fp32 [B][Hq][S],
// each 256-byte aligned.  With more than kDecodeCounters (sequence, KV head)
// pairs the heuristic does not split (there is parallelism enough).
constexpr long long kDecodeCounters = 65536;
struct Plan {
  int splits, pages_per_split;
  size_t ws_bytes, ws_zero_bytes, ws_o_offset, ws_lse_offset;
};

// int8: the pool's dtype (longer splits, a full wave of CTAs).
Plan make_plan(int batch, int num_q_heads, int num_kv_heads, int max_seq_len, int num_splits,
               bool int8) {
  const int mp = std::max(1, (max_seq_len + pkv::kPageSize - 1) / pkv::kPageSize);
  int C;
  if (num_splits > 0) {
    C = (mp + num_splits - 1) / num_splits;
  } else {
    const long long slots = (long long)sm_count() * pkv_host::kDecodeCtasPerSm;
    const long long page_heads = (long long)batch * num_kv_heads * mp;
    const long long target =
        std::max<long long>(1, int8 ? slots : slots * kPlanSlotsNum / kPlanSlotsDen);
    long long c = (page_heads + target - 1) / target;
    c = std::max<long long>(kPlanMinPages,
                            std::min<long long>(int8 ? kPlanMaxPages : kPlanMaxPagesBf16, c));
    c = (c + pkv_host::kDecodeWarps - 1) / pkv_host::kDecodeWarps * pkv_host::kDecodeWarps;
    C = (int)std::min<long long>(c, mp);
  }
  C = std::max(1, C);
  if (num_splits == 0 && (long long)batch * num_kv_heads > kDecodeCounters) C = mp;
  Plan p;
  p.splits = (mp + C - 1) / C;
  p.pages_per_split = C;
  if (p.splits == 1) {
    p.ws_bytes = p.ws_zero_bytes = p.ws_o_offset = p.ws_lse_offset = 0;
  } else {
    const size_t rows = (size_t)batch * num_q_heads * p.splits;
    const size_t o_bytes = rows * pkv::kHeadDim * sizeof(float);
    p.ws_zero_bytes = (size_t)kDecodeCounters * sizeof(uint32_t);
    p.ws_o_offset = p.ws_zero_bytes;
    p.ws_lse_offset = p.ws_o_offset + (o_bytes + 255) / 256 * 256;
    p.ws_bytes = p.ws_lse_offset + (rows * sizeof(float) + 255) / 256 * 256;
  }
  return p;
}

pkv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }

void set_workspace(pkv_host::DecodeLaunch& a, const Plan& p, void* ws, bool fused) {
  char* base = static_cast<char*>(ws);
  a.ws_ctr = p.ws_bytes && fused ? reinterpret_cast<uint32_t*>(base) : nullptr;
  a.ws_o = p.ws_bytes ? reinterpret_cast<float*>(base + p.ws_o_offset) : nullptr;
  a.ws_lse = p.ws_bytes ? reinterpret_cast<float*>(base + p.ws_lse_offset) : nullptr;
}

// Plan of a multi-token decode.  Its kernel fits three CTAs per SM; a CTA
// of T row tiles (16 rows each, T <= 4) puts Tp = 1, 2 or 4 warps on every
// page, so a page costs it more as the step grows.  Pages per split: the
// single-token rule (about 0.8 CTAs per resident slot, 8..128 pages) on
// three slots per SM, divided by Tp / 2 (at least 4 pages), a multiple of
// 4; a plan between one and two waves of CTAs becomes one wave of longer
// splits.  A GB300 sweep of forced split counts put the optimum there for
// steps of 1, 8 and 16 tokens.  Workspace: total_q x Hq rows of split
// partials.
constexpr int kMultiMaxQ = 16;
constexpr int kMultiRowsPerCta = 64;
constexpr int kMultiCtasPerSm = 3;

struct MultiPlan {
  Plan p;
  int row_groups;
};

MultiPlan make_multi_plan(int batch, int total_q, int num_q_heads, int num_kv_heads, int max_q,
                          int max_seq_len, int num_splits) {
  MultiPlan m;
  const int G = num_q_heads / num_kv_heads;
  const int rows = max_q * G;
  m.row_groups = std::max(1, (rows + kMultiRowsPerCta - 1) / kMultiRowsPerCta);
  const int T = (std::min(rows, kMultiRowsPerCta) + 15) / 16;
  const int Tp = T <= 1 ? 1 : (T == 2 ? 2 : 4);
  const int mp = std::max(1, (max_seq_len + pkv::kPageSize - 1) / pkv::kPageSize);
  int C;
  if (num_splits > 0) {
    C = (mp + num_splits - 1) / num_splits;
  } else {
    const long long slots = (long long)sm_count() * kMultiCtasPerSm;
    const long long target = std::max<long long>(1, slots * kPlanSlotsNum / kPlanSlotsDen);
    const long long units = (long long)batch * m.row_groups * num_kv_heads;
    long long c = (units * mp + target - 1) / target;
    c = std::max<long long>(kPlanMinPages, std::min<long long>(kPlanMaxPages, c));
    c = std::max<long long>(4, c / std::max(1, Tp / 2));
    c = (c + 3) / 4 * 4;
    C = (int)std::min<long long>(c, mp);
    // between one and two waves of CTAs: take one wave of longer splits
    // (the second, partial wave would leave most SMs idle)
    const long long ctas = units * ((mp + C - 1) / C);
    if (ctas > slots && ctas < 2 * slots && units <= slots) {
      const long long s1 = slots / units;                     // splits that fit one wave
      const long long c1 = (mp + s1 - 1) / s1;
      if (c1 <= kPlanMaxPages) C = (int)std::min<long long>(c1, mp);
    }
  }
  C = std::max(1, C);
  Plan& p = m.p;
  p.splits = (mp + C - 1) / C;
  p.pages_per_split = C;
  p.ws_zero_bytes = 0;
  if (p.splits == 1) {
    p.ws_bytes = p.ws_o_offset = p.ws_lse_offset = 0;
  } else {
    const size_t n = (size_t)total_q * num_q_heads * p.splits;
    p.ws_o_offset = 0;
    p.ws_lse_offset = (n * pkv::kHeadDim * sizeof(float) + 255) / 256 * 256;
    p.ws_bytes = p.ws_lse_offset + (n * sizeof(float) + 255) / 256 * 256;
  }
  return m;
}

}  // namespace

extern "C" {

pkv_status pkv_kv_append(const pkv_pool* pool, const void* k_new, const void* v_new,
                         int32_t num_tokens, const int32_t* cu_new, int32_t batch,
                         const int32_t* block_table, int32_t max_pages,
                         const int32_t* seq_lens, const float* k_smooth, void* stream) {
  pkv_status st = check_pool(pool);
  if (st != PKV_OK) return st;
  if (num_tokens < 0 || batch < 0 || max_pages < 0) return PKV_ERR_INVALID;
  if (num_tokens == 0) return PKV_OK;
  if (batch == 0 || max_pages == 0) return PKV_ERR_INVALID;
  if (!k_new || !v_new || !cu_new || !block_table || !seq_lens) return PKV_ERR_INVALID;
  if (!aligned(k_new, 16) || !aligned(v_new, 16)) return PKV_ERR_INVALID;
  if (pool->dtype == PKV_BF16 && k_smooth) return PKV_ERR_INVALID;
  if (k_smooth && !aligned(k_smooth, 16)) return PKV_ERR_INVALID;
  pkv_host::AppendLaunch a{pool->k, pool->v, pool->k_scale, pool->v_scale, pool->num_pages,
                           pool->num_kv_heads, k_new, v_new, num_tokens, cu_new, batch,
                           block_table, max_pages, seq_lens, k_smooth};
  return cuda_status(pkv_host::launch_append(a, pool->dtype == PKV_INT8,
                                             static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_decode_plan(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                           int32_t max_seq_len, int32_t dtype, int32_t num_splits,
                           int32_t* splits_out, int32_t* pages_per_split_out,
                           size_t* workspace_bytes_out, size_t* zero_bytes_out) {
  if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads ||
      max_seq_len < 0 || num_splits < 0 || (dtype != PKV_BF16 && dtype != PKV_INT8))
    return PKV_ERR_INVALID;
  if (num_splits > 1 && (long long)batch * num_kv_heads > kDecodeCounters) return PKV_ERR_INVALID;
  const Plan p = make_plan(batch, num_q_heads, num_kv_heads, max_seq_len, num_splits,
                           dtype == PKV_INT8);
  if (splits_out) *splits_out = p.splits;
  if (pages_per_split_out) *pages_per_split_out = p.pages_per_split;
  if (workspace_bytes_out) *workspace_bytes_out = p.ws_bytes;
  if (zero_bytes_out) *zero_bytes_out = p.ws_zero_bytes;
  return PKV_OK;
}

static pkv_status decode_call(const pkv_pool* pool, const void* q, int32_t batch,
                              int32_t num_q_heads, const int32_t* block_table, int32_t max_pages,
                              const int32_t* seq_lens, int32_t max_seq_len, float softmax_scale,
                              const float* k_smooth, int32_t num_splits, void* workspace,
                              size_t workspace_bytes, void* out, float* lse, void* stream,
                              bool fused) {
  pkv_status st = check_pool(pool);
  if (st != PKV_OK) return st;
  if (batch < 0 || num_q_heads <= 0 || num_q_heads % pool->num_kv_heads || max_pages <= 0 ||
      max_seq_len < 0 || (long long)max_seq_len > (long long)max_pages * pkv::kPageSize ||
      num_splits < 0 || !std::isfinite(softmax_scale))
    return PKV_ERR_INVALID;
  if (!pkv_host::decode_supports_group(num_q_heads / pool->num_kv_heads))
    return PKV_ERR_UNSUPPORTED;
  if (batch == 0) return PKV_OK;
  if (!q || !block_table || !seq_lens || !out) return PKV_ERR_INVALID;
  if (pool->dtype == PKV_BF16 && k_smooth) return PKV_ERR_INVALID;
  if (num_splits > 1 && (long long)batch * pool->num_kv_heads > kDecodeCounters)
    return PKV_ERR_INVALID;
  const Plan p = make_plan(batch, num_q_heads, pool->num_kv_heads, max_seq_len, num_splits,
                           pool->dtype == PKV_INT8);
  if (p.ws_bytes > 0 && (!workspace || workspace_bytes < p.ws_bytes || !aligned(workspace, 256)))
    return PKV_ERR_INVALID;
  if ((long long)batch > 65535 || p.splits > 2147483647 / 2) return PKV_ERR_UNSUPPORTED;
  pkv_host::DecodeLaunch a{};
  a.k = pool->k;
  a.v = pool->v;
  a.k_scale = pool->k_scale;
  a.v_scale = pool->v_scale;
  a.num_pages = pool->num_pages;
  a.num_kv_heads = pool->num_kv_heads;
  a.q = q;
  a.batch = batch;
  a.num_q_heads = num_q_heads;
  a.block_table = block_table;
  a.max_pages = max_pages;
  a.seq_lens = seq_lens;
  a.softmax_scale = softmax_scale;
  a.k_smooth = k_smooth;
  a.splits = p.splits;
  a.pages_per_split = p.pages_per_split;
  set_workspace(a, p, workspace, fused);
  a.out = out;
  a.lse = lse;
  return cuda_status(pkv_host::launch_decode(a, pool->dtype == PKV_INT8,
                                             static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_paged_attn_decode(const pkv_pool* pool, const void* q, int32_t batch,
                                 int32_t num_q_heads, const int32_t* block_table,
                                 int32_t max_pages, const int32_t* seq_lens,
                                 int32_t max_seq_len, float softmax_scale,
                                 const float* k_smooth, int32_t num_splits, void* workspace,
                                 size_t workspace_bytes, void* out, float* lse, void* stream) {
  return decode_call(pool, q, batch, num_q_heads, block_table, max_pages, seq_lens, max_seq_len,
                     softmax_scale, k_smooth, num_splits, workspace, workspace_bytes, out, lse,
                     stream, false);
}

pkv_status pkv_paged_attn_decode_fused(const pkv_pool* pool, const void* q, int32_t batch,
                                       int32_t num_q_heads, const int32_t* block_table,
                                       int32_t max_pages, const int32_t* seq_lens,
                                       int32_t max_seq_len, float softmax_scale,
                                       const float* k_smooth, int32_t num_splits,
                                       void* workspace, size_t workspace_bytes, void* out,
                                       float* lse, void* stream) {
  return decode_call(pool, q, batch, num_q_heads, block_table, max_pages, seq_lens, max_seq_len,
                     softmax_scale, k_smooth, num_splits, workspace, workspace_bytes, out, lse,
                     stream, true);
}

pkv_status pkv_paged_attn_decode_noalloc(const pkv_pool* pool, const void* q, int32_t batch,
                                         int32_t num_q_heads, const int32_t* block_table,
                                         int32_t max_pages, const int32_t* seq_lens,
                                         int32_t max_seq_len, float softmax_scale,
                                         const float* k_smooth, int32_t num_splits, void* out,
                                         float* lse, void* stream) {
  // Same checks as pkv_paged_attn_decode; the split partials go to the
  // library's fixed device array instead of a caller workspace.
  pkv_status st = check_pool(pool);
  if (st != PKV_OK) return st;
  if (batch < 0 || num_q_heads <= 0 || num_q_heads % pool->num_kv_heads || max_pages <= 0 ||
      max_seq_len < 0 || (long long)max_seq_len > (long long)max_pages * pkv::kPageSize ||
      num_splits < 0 || !std::isfinite(softmax_scale))
    return PKV_ERR_INVALID;
  if (!pkv_host::decode_supports_group(num_q_heads / pool->num_kv_heads))
    return PKV_ERR_UNSUPPORTED;
  if (batch == 0) return PKV_OK;
  if (!q || !block_table || !seq_lens || !out) return PKV_ERR_INVALID;
  if (pool->dtype == PKV_BF16 && k_smooth) return PKV_ERR_INVALID;
  if (num_splits > 1 && (long long)batch * pool->num_kv_heads > kDecodeCounters)
    return PKV_ERR_INVALID;
  const size_t cap = pkv_host::decode_fixed_scratch_bytes();
  const bool int8 = pool->dtype == PKV_INT8;
  Plan p = make_plan(batch, num_q_heads, pool->num_kv_heads, max_seq_len, num_splits, int8);
  if (p.ws_bytes > cap) {
    if (num_splits > 0) return PKV_ERR_INVALID;       // forced split count does not fit
    int s = p.splits;
    while (s > 1 && p.ws_bytes > cap) {
      --s;
      p = make_plan(batch, num_q_heads, pool->num_kv_heads, max_seq_len, s, int8);
    }
    if (p.ws_bytes > cap) return PKV_ERR_INVALID;
  }
  if ((long long)batch > 65535) return PKV_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if (p.ws_bytes > 0 && pkv_host::decode_fixed_scratch(&scratch) != cudaSuccess)
    return PKV_ERR_CUDA;
  pkv_host::DecodeLaunch a{};
  a.k = pool->k;
  a.v = pool->v;
  a.k_scale = pool->k_scale;
  a.v_scale = pool->v_scale;
  a.num_pages = pool->num_pages;
  a.num_kv_heads = pool->num_kv_heads;
  a.q = q;
  a.batch = batch;
  a.num_q_heads = num_q_heads;
  a.block_table = block_table;
  a.max_pages = max_pages;
  a.seq_lens = seq_lens;
  a.softmax_scale = softmax_scale;
  a.k_smooth = k_smooth;
  a.splits = p.splits;
  a.pages_per_split = p.pages_per_split;
  set_workspace(a, p, scratch, false);
  a.out = out;
  a.lse = lse;
  return cuda_status(pkv_host::launch_decode(a, pool->dtype == PKV_INT8,
                                             static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_prefill_plan(int32_t* ctas, size_t* workspace_bytes, size_t* zero_bytes) {
  const int n = pkv_host::prefill_ctas(sm_count());
  if (ctas) *ctas = n;
  if (workspace_bytes) *workspace_bytes = pkv_host::prefill_workspace_bytes(n);
  if (zero_bytes) *zero_bytes = pkv_host::prefill_workspace_zero_bytes(n);
  return PKV_OK;
}

// Overlap of a prefill with a decode on another stream: the prefill's time
// scales with its SMs; the decode, HBM-bound on the whole GPU, draws about
// twice the average per-SM bandwidth when it has few SMs (measured on GB300:
// ~85 GB/s per SM against 6.5 TB/s / 152).  Both finish together when the
// decode holds N_d SMs with N_d / (SMs - N_d) = t_d / (kOverlapDecodeGain *
// t_p), t_p and t_d the two calls' times alone on the whole GPU.  On the
// mixed step (a 26,926-token prompt in 2,048-row chunks beside 32 decode
// rows) this picks within a few percent of the best of a sweep per chunk,
// and the factor 2 was the best of 1.6..4.0 (a larger prefill share pushes
// the decode's CTAs into a further wave).
constexpr double kOverlapPrefillFlopsPerSec = 1.45e15, kOverlapPrefillFixedSec = 10e-6;
constexpr double kOverlapDecodeBytesPerSec = 6.5e12, kOverlapDecodeGain = 2.0;

pkv_status pkv_overlap_prefill_ctas(double prefill_flops, double decode_bytes, int32_t* ctas) {
  if (!ctas || !std::isfinite(prefill_flops) || !std::isfinite(decode_bytes) ||
      prefill_flops < 0 || decode_bytes < 0)
    return PKV_ERR_INVALID;
  const int all = pkv_host::prefill_ctas(sm_count());
  const double tp = prefill_flops / kOverlapPrefillFlopsPerSec + kOverlapPrefillFixedSec;
  const double r = decode_bytes / kOverlapDecodeBytesPerSec / (kOverlapDecodeGain * tp);
  const int nd = (int)std::lround((double)all * r / (1.0 + r));
  *ctas = std::max(std::max(1, all / 3), std::min(all, all - nd));
  return PKV_OK;
}

pkv_status pkv_paged_attn_prefill(const pkv_pool* pool, const void* q, int32_t total_q,
                                  const int32_t* cu_q,
                                  int32_t batch, int32_t num_q_heads,
                                  const int32_t* block_table, int32_t max_pages,
                                  const int32_t* seq_lens, int32_t max_q_len,
                                  float softmax_scale, void* workspace, size_t workspace_bytes,
                                  int32_t num_ctas, void* out, float* lse, void* stream) {
  pkv_status st = check_pool(pool);
  if (st != PKV_OK) return st;
  if (batch < 0 || total_q < 0 || num_q_heads <= 0 || num_q_heads % pool->num_kv_heads ||
      max_pages <= 0 || max_q_len < 0 || !std::isfinite(softmax_scale) || num_ctas < 0)
    return PKV_ERR_INVALID;
  if (pool->dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
  if (batch == 0 || max_q_len == 0 || total_q == 0) return PKV_OK;
  if (!q || !cu_q || !block_table || !seq_lens || !out) return PKV_ERR_INVALID;
  if (!aligned(q, 16) || !aligned(out, 16)) return PKV_ERR_INVALID;
  if (batch > 65535 || num_q_heads > 65535) return PKV_ERR_UNSUPPORTED;
  const int all = pkv_host::prefill_ctas(sm_count());
  const int ctas = num_ctas > 0 && num_ctas < all ? num_ctas : all;
  // the workspace is laid out for every SM whatever num_ctas is
  if (!workspace || !aligned(workspace, 16) ||
      workspace_bytes < pkv_host::prefill_workspace_bytes(all))
    return PKV_ERR_INVALID;
  pkv_host::PrefillLaunch a{pool->k, pool->v, pool->num_pages, pool->num_kv_heads, q, total_q,
                            cu_q, batch, num_q_heads, block_table, max_pages, seq_lens, max_q_len,
                            softmax_scale, out, lse, ctas, workspace, all};
  cudaError_t e = pkv_host::launch_prefill(a, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return PKV_ERR_UNSUPPORTED;
  return cuda_status(e);
}

pkv_status pkv_qkv_norm_rope_append(const pkv_pool* pool, const void* qkv, int32_t num_tokens,
                                    int32_t num_q_heads, const float* q_norm_w,
                                    const float* k_norm_w, float eps, const float* rope_cos,
                                    const float* rope_sin, int32_t max_pos, const int32_t* cu_new,
                                    int32_t batch, const int32_t* block_table, int32_t max_pages,
                                    const int32_t* seq_lens, void* q_out, void* stream) {
  pkv_status st = check_pool(pool);
  if (st != PKV_OK) return st;
  if (num_tokens < 0 || batch < 0 || max_pages < 0 || num_q_heads <= 0 ||
      num_q_heads % pool->num_kv_heads || !std::isfinite(eps) || eps < 0.f)
    return PKV_ERR_INVALID;
  if (pool->dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (batch == 0 || max_pages == 0) return PKV_ERR_INVALID;
  if (!qkv || !cu_new || !block_table || !seq_lens || !q_out) return PKV_ERR_INVALID;
  if (!rope_cos != !rope_sin || (rope_cos && max_pos <= 0)) return PKV_ERR_INVALID;
  if (!aligned(qkv, 16) || !aligned(q_out, 16)) return PKV_ERR_INVALID;
  for (const void* p : {(const void*)q_norm_w, (const void*)k_norm_w, (const void*)rope_cos,
                        (const void*)rope_sin})
    if (p && !aligned(p, 16)) return PKV_ERR_INVALID;
  if (num_tokens > 2147483647 / (num_q_heads + 2 * pool->num_kv_heads) / 64)
    return PKV_ERR_UNSUPPORTED;
  pkv_host::QkvPrepLaunch a{qkv,       num_tokens, num_q_heads,  pool->num_kv_heads,
                            q_norm_w,  k_norm_w,   eps,          rope_cos,
                            rope_sin,  max_pos,    cu_new,       batch,
                            block_table, max_pages, seq_lens,    pool->k,
                            pool->v,   pool->num_pages, q_out};
  return cuda_status(pkv_host::launch_qkv_prep(a, static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_decode_multi_plan(int32_t batch, int32_t total_q, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t max_q_len, int32_t max_seq_len,
                                 int32_t num_splits, int32_t* splits_out,
                                 int32_t* pages_per_split_out, size_t* workspace_bytes_out) {
  if (batch < 0 || total_q < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      num_q_heads % num_kv_heads || max_q_len < 1 || max_seq_len < 0 || num_splits < 0)
    return PKV_ERR_INVALID;
  if (max_q_len > kMultiMaxQ) return PKV_ERR_UNSUPPORTED;
  const MultiPlan m = make_multi_plan(batch, total_q, num_q_heads, num_kv_heads, max_q_len,
                                      max_seq_len, num_splits);
  if (splits_out) *splits_out = m.p.splits;
  if (pages_per_split_out) *pages_per_split_out = m.p.pages_per_split;
  if (workspace_bytes_out) *workspace_bytes_out = m.p.ws_bytes;
  return PKV_OK;
}

pkv_status pkv_paged_attn_decode_multi(const pkv_pool* pool, const void* q, int32_t total_q,
                                       const int32_t* cu_q, int32_t batch, int32_t num_q_heads,
                                       const int32_t* block_table, int32_t max_pages,
                                       const int32_t* seq_lens, int32_t max_q_len,
                                       int32_t max_seq_len, float softmax_scale,
                                       int32_t num_splits, void* workspace,
                                       size_t workspace_bytes, void* out, float* lse,
                                       void* stream) {
  pkv_status st = check_pool(pool);
  if (st != PKV_OK) return st;
  if (batch < 0 || total_q < 0 || num_q_heads <= 0 || num_q_heads % pool->num_kv_heads ||
      max_pages <= 0 || max_q_len < 1 || max_seq_len < 0 ||
      (long long)max_seq_len > (long long)max_pages * pkv::kPageSize || num_splits < 0 ||
      !std::isfinite(softmax_scale))
    return PKV_ERR_INVALID;
  if (pool->dtype != PKV_BF16 || max_q_len > kMultiMaxQ) return PKV_ERR_UNSUPPORTED;
  if (batch == 0 || total_q == 0) return PKV_OK;
  if (!q || !cu_q || !block_table || !seq_lens || !out) return PKV_ERR_INVALID;
  if (!aligned(q, 16) || !aligned(out, 16)) return PKV_ERR_INVALID;
  const MultiPlan m = make_multi_plan(batch, total_q, num_q_heads, pool->num_kv_heads, max_q_len,
                                      max_seq_len, num_splits);
  if (m.p.ws_bytes > 0 &&
      (!workspace || workspace_bytes < m.p.ws_bytes || !aligned(workspace, 256)))
    return PKV_ERR_INVALID;
  if ((long long)batch > 65535 || (long long)pool->num_kv_heads * m.row_groups > 65535 ||
      (long long)total_q * num_q_heads > 2147483647ll / 2 || m.p.splits > 2147483647 / 2)
    return PKV_ERR_UNSUPPORTED;
  pkv_host::MultiLaunch a{};
  a.k = pool->k;
  a.v = pool->v;
  a.num_pages = pool->num_pages;
  a.num_kv_heads = pool->num_kv_heads;
  a.q = q;
  a.total_q = total_q;
  a.cu_q = cu_q;
  a.batch = batch;
  a.num_q_heads = num_q_heads;
  a.block_table = block_table;
  a.max_pages = max_pages;
  a.seq_lens = seq_lens;
  a.max_q = max_q_len;
  a.softmax_scale = softmax_scale;
  a.splits = m.p.splits;
  a.pages_per_split = m.p.pages_per_split;
  a.row_groups = m.row_groups;
  char* base = static_cast<char*>(workspace);
  a.ws_o = m.p.ws_bytes ? reinterpret_cast<float*>(base + m.p.ws_o_offset) : nullptr;
  a.ws_lse = m.p.ws_bytes ? reinterpret_cast<float*>(base + m.p.ws_lse_offset) : nullptr;
  a.out = out;
  a.lse = lse;
  return cuda_status(pkv_host::launch_decode_multi(a, static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_selftest_bounded_wait(const uint32_t* counter, uint32_t target, void* stream) {
  if (!counter) return PKV_ERR_INVALID;
  return cuda_status(
      pkv_host::launch_wait_selftest(counter, target, static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_poll_device_error(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return PKV_ERR_CUDA;
  const uint32_t e = pkv_host::take_append_error(s) | pkv_host::take_decode_error(s) |
                     pkv_host::take_prefill_error(s) | pkv_host::take_qkv_error(s) |
                     pkv_host::take_multi_error(s);
  if (e == ~0u) return PKV_ERR_CUDA;
  if (e & pkv::kErrTimeout) return PKV_ERR_TIMEOUT;
  return e ? PKV_ERR_INVALID : PKV_OK;
}

const char* pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_TIMEOUT: return "a device-side bounded wait ran out";
  }
  return "unknown status";
}

int32_t pkv_device_sm_count(void) { return sm_count(); }

}  // extern "C"
