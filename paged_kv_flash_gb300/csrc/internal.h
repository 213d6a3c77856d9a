// internal.h -- host-side interface between the C ABI (api.cu) and the
// kernel translation units.  Not installed; not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace pkv_host {

struct AppendLaunch {
  void* k;                 // pool K (bf16 or int8)
  void* v;
  float* k_scale;          // int8 only
  float* v_scale;
  int num_pages, num_kv_heads;
  const void* k_new;       // bf16 [T][Hkv][128]
  const void* v_new;
  int num_tokens;
  const int32_t* cu_new;   // [B+1]
  int batch;
  const int32_t* block_table;
  int max_pages;
  const int32_t* seq_lens;
  const float* k_smooth;   // int8 only, may be null
};

cudaError_t launch_append(const AppendLaunch& a, bool int8, cudaStream_t s);
uint32_t take_append_error(cudaStream_t s);

struct DecodeLaunch {
  const void* k;
  const void* v;
  const float* k_scale;
  const float* v_scale;
  int num_pages, num_kv_heads;
  const void* q;           // bf16 [B][Hq][128]
  int batch, num_q_heads;
  const int32_t* block_table;
  int max_pages;
  const int32_t* seq_lens;
  float softmax_scale;
  const float* k_smooth;
  int splits, pages_per_split;
  uint32_t* ws_ctr;        // fused merge: parts counted per b * Hkv + h (zero between
                           // calls); null: a separate combine kernel merges
  float* ws_o;             // [B][Hq][splits][128] when splits > 1
  float* ws_lse;           // [B][Hq][splits]
  void* out;               // bf16 [B][Hq][128]
  float* lse;              // [B][Hq] or null
};

// Kernel geometry the split heuristic needs.
constexpr int kDecodeWarps = 4;          // warps per split CTA
constexpr int kDecodeCtasPerSm = 2;      // split CTAs per SM the plan counts on

// cuTensorMapEncodeTiled of an INT8 pool (K or V) as 2-D uint8 rows of 128
// bytes, one box per (page, head) slab of 16 rows, 128B-swizzled; `map`
// points to a CUtensorMap.  False if the driver entry point is missing or
// rejects the arguments.
bool encode_int8_slab_map(void* map, const void* base, int num_pages, int hkv);

bool decode_supports_group(int group);
cudaError_t launch_decode(const DecodeLaunch& a, bool int8, cudaStream_t s);
uint32_t take_decode_error(cudaStream_t s);

// Fixed device scratch for pkv_paged_attn_decode_noalloc (decode.cu).
size_t decode_fixed_scratch_bytes();
// Device address of that scratch on the current device (looked up once per
// device with cudaGetSymbolAddress).
cudaError_t decode_fixed_scratch(void** ptr);

// Split-KV decode of 1..16 query tokens per sequence (decode_multi.cu).
struct MultiLaunch {
  const void* k;           // bf16 pool
  const void* v;
  int num_pages, num_kv_heads;
  const void* q;           // bf16 [total_q][Hq][128]
  int total_q;
  const int32_t* cu_q;     // [B+1]
  int batch, num_q_heads;
  const int32_t* block_table;
  int max_pages;
  const int32_t* seq_lens; // [B], the step's tokens included
  int max_q;               // tokens per sequence at most (<= 16)
  float softmax_scale;
  int splits, pages_per_split;
  int row_groups;          // ceil(max_q * G / 64): CTAs per (split, KV head, sequence)
  float* ws_o;             // [total_q * Hq][splits][128] when splits > 1
  float* ws_lse;           // [total_q * Hq][splits]
  void* out;               // bf16 [total_q][Hq][128]
  float* lse;              // [total_q][Hq] or null
};

cudaError_t launch_decode_multi(const MultiLaunch& a, cudaStream_t s);
uint32_t take_multi_error(cudaStream_t s);
// cuTensorMapEncodeTiled of a bf16 pool (K or V) as 2-D rows of 128
// channels, one box per 16-row x 64-channel half slab, 128B-swizzled
// (prefill.cu); `map` points to a CUtensorMap.
bool encode_bf16_pool_map(void* map, const void* base, int num_pages, int hkv);

struct PrefillLaunch {
  const void* k;
  const void* v;
  int num_pages, num_kv_heads;
  const void* q;           // bf16 [total_q][Hq][128]
  int total_q;
  const int32_t* cu_q;     // [B+1]
  int batch, num_q_heads;
  const int32_t* block_table;
  int max_pages;
  const int32_t* seq_lens;
  int max_q_len;
  float softmax_scale;
  void* out;
  float* lse;
  int ctas;                // persistent CTAs (at most one per SM)
  void* workspace;         // prefill_workspace_bytes(ws_ctas) bytes, 16-byte aligned
  int ws_ctas;             // the CTA count the workspace is laid out for (>= ctas): the
                           // same for every call, whatever its ctas, so that one call's
                           // partial results never sit where another's counters go
};

constexpr int kMaxPrefillCtas = 1024;
// Workspace of a prefill launch with `ctas` persistent CTAs: part counters,
// then per CTA two partial-result slots of 256 rows x 128 fp32 plus 256 fp32
// lse.  Its first prefill_workspace_zero_bytes(ctas) bytes (the counters)
// must be zero before the first launch; a launch that completes leaves them
// zero.
size_t prefill_workspace_bytes(int ctas);
size_t prefill_workspace_zero_bytes(int ctas);
// Persistent CTAs of a prefill launch on a device with `sms` SMs.
int prefill_ctas(int sms);
cudaError_t launch_prefill(const PrefillLaunch& a, cudaStream_t s);
uint32_t take_prefill_error(cudaStream_t s);
// One thread waits (bounded, as a merging prefill CTA does) for *counter >= target.
cudaError_t launch_wait_selftest(const uint32_t* counter, uint32_t target, cudaStream_t s);

struct QkvPrepLaunch {
  const void* qkv;         // bf16 [T][Hq + 2 Hkv][128]
  int num_tokens, num_q_heads, num_kv_heads;
  const float* q_w;        // fp32 [128] or null
  const float* k_w;
  float eps;
  const float* cos;        // fp32 [max_pos][64] or null
  const float* sin;
  int max_pos;
  const int32_t* cu_new;   // [B+1]
  int batch;
  const int32_t* block_table;
  int max_pages;
  const int32_t* seq_lens;
  void* k;                 // bf16 pool
  void* v;
  int num_pages;
  void* q_out;             // bf16 [T][Hq][128]
};

cudaError_t launch_qkv_prep(const QkvPrepLaunch& a, cudaStream_t s);
uint32_t take_qkv_error(cudaStream_t s);

int sm_count();

}  // namespace pkv_host
