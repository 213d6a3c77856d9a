/*
 * pagedkv.h -- C ABI of libpagedkv.so: attention over a paged KV cache on one
 * GB300 (sm_103a).
 *
 * The operations follow the TileInfer.jl "Performance" page:
 *  - section "Fused kernels, FlashAttention and PagedAttention": the KV cache
 *    write, paged flash attention as an online softmax over the pages read in
 *    place through the block table, split-KV for decode, and a combine kernel
 *    kept separate from the split kernel;
 *  - section "INT8 KV cache": an INT8 cache with one scale per cached vector,
 *    keys smoothed by the key norm's weight;
 *  - section "Speculative decoding", "Attention for verify steps": the prefill
 *    kernel runs a block per head over every page.
 *
 * Conventions (all calls):
 *  - Every pointer argument is a DEVICE pointer unless its comment says host.
 *    The caller owns all memory; the library allocates nothing on any call.
 *  - Calls are asynchronous on the given stream (a cudaStream_t passed as
 *    void*; NULL means the legacy default stream).  A status other than
 *    PKV_OK means nothing was launched, except PKV_ERR_CUDA, which reports a
 *    failed launch.
 *  - Arguments are checked on the host before any launch: a NULL pointer
 *    that is required, head_dim != 128, page_size != 16, num_q_heads not a
 *    multiple of num_kv_heads, negative sizes or a short workspace return
 *    PKV_ERR_INVALID.  The CONTENTS of device arrays (block tables, sequence
 *    lengths, offsets) are the caller's contract and are not read on the host.
 *  - bf16 tensors hold IEEE bfloat16; fp32 is IEEE binary32.
 *  - GQA: query head h reads KV head h / (num_q_heads / num_kv_heads).
 *  - lse is the natural-log log-sum-exp of the scaled scores, softmax_scale *
 *    q.k, over the keys a row sees; a row that sees no key gets out = 0 and
 *    lse = -inf.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID = -1,      /* bad argument; nothing launched */
  PKV_ERR_UNSUPPORTED = -2,  /* valid but not provided (e.g. INT8 prefill) */
  PKV_ERR_CUDA = -3,         /* a CUDA call or launch failed */
  PKV_ERR_TIMEOUT = -4       /* a kernel's bounded wait ran out (pkv_poll_device_error) */
} pkv_status;

typedef enum { PKV_BF16 = 0, PKV_INT8 = 1 } pkv_kv_dtype;

/*
 * One paged KV pool (TileInfer.jl "Performance" page: "the pool", read
 * "through the block table").  K and V are separate arrays of
 * [num_pages][num_kv_heads][page_size][head_dim]; one (page, head) slab is
 * contiguous (4 KiB for bf16, 2 KiB for int8).  For PKV_INT8, k_scale and
 * v_scale hold one fp32 scale per cached vector, [num_pages][num_kv_heads]
 * [page_size] ("INT8 KV cache": one scale per cached vector); for PKV_BF16
 * they must be NULL.  k and v must be 16-byte aligned.  Position p of
 * sequence b lives in page block_table[b][p / page_size], slot p % page_size.
 */
typedef struct {
  void* k;
  void* v;
  float* k_scale;
  float* v_scale;
  int32_t num_pages;
  int32_t num_kv_heads;
  int32_t page_size;   /* must be 16 */
  int32_t head_dim;    /* must be 128 */
  int32_t dtype;       /* pkv_kv_dtype */
} pkv_pool;

/*
 * kv_append -- write new K/V vectors into the pool pages named by the block
 * table ("Fused kernels ...": the KV cache write; "INT8 KV cache": one scale
 * per vector).
 *
 *  k_new, v_new  bf16 [num_tokens][num_kv_heads][128]; rows cu_new[b] ..
 *                cu_new[b+1]-1 belong to sequence b.
 *  cu_new        int32 [batch+1], non-decreasing, cu_new[batch] = num_tokens.
 *  block_table   int32 [batch][max_pages] page ids.
 *  seq_lens      int32 [batch] cached positions of each sequence AFTER this
 *                append; new row i of sequence b goes to position
 *                seq_lens[b] - n_b + i, n_b = cu_new[b+1] - cu_new[b].
 *  k_smooth      fp32 [128] per-channel key weight (> 0) or NULL.  INT8
 *                pools only: keys are divided by it before quantisation.
 *                Must be NULL for bf16 pools.
 *
 * bf16 pools: the vectors are copied bit for bit.  INT8 pools: per vector x
 * (fp32; k / w for smoothed keys), scale = max|x| / 127 in fp32, code =
 * round-half-even(x / scale) as an IEEE fp32 quotient, clamped to +-127; an
 * all-zero vector stores scale 0 and codes 0.  Slots not named are left
 * untouched.  num_tokens == 0 launches nothing and returns PKV_OK.
 */
pkv_status pkv_kv_append(const pkv_pool* pool, const void* k_new, const void* v_new,
                         int32_t num_tokens, const int32_t* cu_new, int32_t batch,
                         const int32_t* block_table, int32_t max_pages,
                         const int32_t* seq_lens, const float* k_smooth, void* stream);

/*
 * Split plan of a decode call ("Fused kernels ...": split-KV for decode).
 * Host-only; launches nothing.  max_seq_len (host) bounds every seq_lens[b];
 * dtype is the pool's pkv_kv_dtype (the heuristic plans the two kernels
 * differently: INT8 pages, half the bytes, get longer splits, and the INT8
 * kernel, bound by its work per page, gets a full wave of CTAs); a plan is
 * for its dtype only; num_splits 0 asks for the built-in
 * heuristic (split count chosen from the batch, the heads, the dtype and the
 * device's SM count), > 0 forces that many splits.
 * Outputs (host pointers, each may be NULL): the split count S, the pages per
 * split, the workspace bytes the decode call needs (0 when S == 1), and how
 * many leading bytes of that workspace must be zero before its first use
 * (256 KiB of part counters when S > 1, else 0).  More than 65,536
 * (sequence, KV head) pairs are never split by the heuristic, and a forced
 * num_splits > 1 for them is PKV_ERR_INVALID.
 */
pkv_status pkv_decode_plan(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                           int32_t max_seq_len, int32_t dtype, int32_t num_splits,
                           int32_t* splits_out,
                           int32_t* pages_per_split_out, size_t* workspace_bytes_out,
                           size_t* zero_bytes_out);

/*
 * paged_attn_decode -- one query token per sequence against its cached
 * positions 0 .. seq_lens[b]-1 (the token's own position included): split-KV
 * partials, then a log-sum-exp combine ("Fused kernels ...": online softmax
 * over the pages in place, split-KV for decode, separate combine kernel).  A
 * row whose keys fit one split is finished by that split.
 *
 *  q            bf16 [batch][num_q_heads][128].
 *  block_table  int32 [batch][max_pages]; seq_lens int32 [batch] (device);
 *               max_seq_len (host) >= every seq_lens[b].
 *  k_smooth     INT8 pools: the same fp32 [128] weight given to kv_append,
 *               or NULL if the keys were not smoothed; NULL for bf16.
 *  num_splits   0 = heuristic, > 0 forces (see pkv_decode_plan).
 *  workspace    scratch of at least pkv_decode_plan's bytes for this pool's
 *               dtype and these sizes (256-byte
 *               aligned), may be NULL when that is 0.  Holds the split
 *               partials; its contents are dead after the call (its first
 *               zero_bytes are not used by this call).
 *  out          bf16 [batch][num_q_heads][128]; lse fp32 [batch][num_q_heads]
 *               or NULL.
 */
pkv_status pkv_paged_attn_decode(const pkv_pool* pool, const void* q, int32_t batch,
                                 int32_t num_q_heads, const int32_t* block_table,
                                 int32_t max_pages, const int32_t* seq_lens,
                                 int32_t max_seq_len, float softmax_scale,
                                 const float* k_smooth, int32_t num_splits, void* workspace,
                                 size_t workspace_bytes, void* out, float* lse, void* stream);

/*
 * paged_attn_decode_fused -- the same decode with the combine fused into the
 * split kernel ("Not kept: the attention combine fused into the split-KV
 * kernel", re-measured on GB300; the separate combine above stays the
 * default because it is faster there except on a single cold launch).  Each
 * split stores its partial and counts it with an acquire-release atomic; the
 * split that completes the count of a (sequence, KV head) merges the partials
 * in split order (bit-identical to the separate combine) and resets the
 * count.  No split waits on another.
 *
 * Arguments: as pkv_paged_attn_decode.  The workspace's first zero_bytes
 * (pkv_decode_plan) hold the part counters: they must be zero before the
 * first use; every call that completes leaves them zero again, so a
 * workspace is zeroed once and reused by calls of any shape that fits it
 * (zero it again after PKV_ERR_TIMEOUT).  Calls sharing a workspace must not
 * overlap.
 */
pkv_status pkv_paged_attn_decode_fused(const pkv_pool* pool, const void* q, int32_t batch,
                                       int32_t num_q_heads, const int32_t* block_table,
                                       int32_t max_pages, const int32_t* seq_lens,
                                       int32_t max_seq_len, float softmax_scale,
                                       const float* k_smooth, int32_t num_splits,
                                       void* workspace, size_t workspace_bytes, void* out,
                                       float* lse, void* stream);

/*
 * paged_attn_decode_noalloc -- the same decode as pkv_paged_attn_decode for
 * callers that cannot allocate device memory.  The pages have no counterpart
 * for this call: it exists for users of this library, not for the method.
 *
 * Some callers have no way to obtain the workspace the split partials need:
 * a plain C host program that has no device allocator of its own, a plugin
 * running inside a runtime that owns every byte of device memory and forbids
 * cudaMalloc on its threads (cudaMalloc can synchronise the device and
 * fragments the runtime's pool), or latency-critical code that cannot afford
 * an allocation's implicit synchronisation.  This entry point keeps the
 * partials in a fixed device array that lives in the library itself (16 MiB,
 * 256-byte aligned; every GPU that loads the library holds it until the
 * process exits) and calls no cudaMalloc, cudaFree or other allocating
 * routine.  The caller still passes q, the pool, the tables and out/lse.
 *
 * Arguments: as pkv_paged_attn_decode, without the workspace.  With
 * num_splits == 0 the split heuristic runs first; if its partials would not
 * fit in 16 MiB the split count is lowered until they do (the result differs
 * from pkv_paged_attn_decode only by rounding).  A forced num_splits whose
 * partials need more than 16 MiB (batch * num_q_heads * num_splits * 516 bytes
 * plus alignment and 256 KiB the plan reserves) is rejected with
 * PKV_ERR_INVALID before any launch.
 *
 * The first call on each device looks the array's device address up with
 * cudaGetSymbolAddress (once per device, with that device current); make
 * that first call before any stream capture on the device.  Every call on a
 * device shares the one array and it keeps the last call's contents; nothing
 * in it needs to start at zero (every entry the combine reads is written by
 * the split kernel of the same call).  Calls that overlap on the GPU -- on
 * two streams, or from two host threads without ordering -- race on the
 * array and give wrong results: order them on one stream.
 */
pkv_status pkv_paged_attn_decode_noalloc(const pkv_pool* pool, const void* q, int32_t batch,
                                         int32_t num_q_heads, const int32_t* block_table,
                                         int32_t max_pages, const int32_t* seq_lens,
                                         int32_t max_seq_len, float softmax_scale,
                                         const float* k_smooth, int32_t num_splits, void* out,
                                         float* lse, void* stream);

/*
 * prefill_plan -- the persistent CTA count, workspace size and the size of
 * the workspace's leading part that must be zero before first use, for a
 * prefill call on the current device (one CTA per SM; host only, no GPU
 * work).  Any pointer may be NULL.  Always PKV_OK.
 */
pkv_status pkv_prefill_plan(int32_t* ctas, size_t* workspace_bytes, size_t* zero_bytes);

/*
 * paged_attn_prefill -- causal attention of a chunk of new query rows per
 * sequence against the sequence's cached prefix plus the chunk itself
 * (a block of query rows per head over every page: "Attention for verify
 * steps"; chunked prefill: "What is left to gain").  Tensor-core (tcgen05)
 * QK^T and PV with fp32 accumulation; P is rounded to bf16 for PV.
 *
 *  q         bf16 [total_q][num_q_heads][128]; rows cu_q[b] .. cu_q[b+1]-1
 *            belong to sequence b (all within 0 .. total_q-1).  cu_q int32
 *            [batch+1] (device).  total_q (host) is the row count of q and
 *            out.
 *  seq_lens  int32 [batch] cached positions INCLUDING this chunk (append the
 *            chunk's K/V first).  Row i of sequence b sits at position
 *            seq_lens[b] - q_b + i and sees keys 0 .. that position
 *            (bottom-right causal alignment).
 *  max_q_len (host) >= every q_b.
 *  workspace device scratch of at least pkv_prefill_plan's workspace_bytes,
 *            16-byte aligned, owned by the caller.  Its first zero_bytes
 *            bytes (part counters) must be zero before its first use; every
 *            call that completes leaves them zero again, so a workspace is
 *            zeroed once and reused (zero it again after PKV_ERR_TIMEOUT).
 *            The call runs one persistent CTA per SM.  Each launch either
 *            cuts all (sequence, query-tile pair, head, key block) work into
 *            even shares or gives the CTAs whole units, whichever its
 *            estimate finishes sooner; where a chunk ends in a single
 *            128-row tile and the query heads of a KV head come in pairs, a
 *            unit may hold that tile for two heads.  A unit cut between CTAs
 *            leaves its other parts in the workspace, and the CTA holding its
 *            last blocks merges them (the log-sum-exp rule of "Split-KV
 *            decoding").  PKV_ERR_INVALID if NULL, unaligned or too small.
 *            Calls that share a workspace must not overlap.
 *  num_ctas  persistent CTAs (at most one per SM): 0 = pkv_prefill_plan's
 *            count, every SM; 1 .. that count leaves the other SMs to work
 *            queued on other streams -- a decode step that needs no output
 *            of this call, for one (pkv_overlap_prefill_ctas); larger counts
 *            run as 0.  The workspace is laid out for every SM whatever the
 *            count, so calls with different counts share it.  Negative:
 *            PKV_ERR_INVALID.
 *  out       bf16 [total_q][num_q_heads][128]; lse fp32 [total_q][num_q_heads]
 *            or NULL.
 * bf16 pools only (PKV_ERR_UNSUPPORTED for INT8).
 */
pkv_status pkv_paged_attn_prefill(const pkv_pool* pool, const void* q, int32_t total_q,
                                  const int32_t* cu_q,
                                  int32_t batch, int32_t num_q_heads,
                                  const int32_t* block_table, int32_t max_pages,
                                  const int32_t* seq_lens, int32_t max_q_len,
                                  float softmax_scale, void* workspace, size_t workspace_bytes,
                                  int32_t num_ctas, void* out, float* lse, void* stream);

/*
 * overlap_prefill_ctas -- the num_ctas to give a prefill call that runs on
 * one stream while a decode call runs on another, both after the same
 * append (continuous batching: the prompt chunk and the decode rows of one
 * step).  The prefill is bound by the tensor cores and scales with its SMs;
 * the decode is bound by HBM and needs few SMs to draw most of it, so the
 * two together finish sooner than one after the other.  prefill_flops: the
 * prefill's causal flops (4 * 128 * num_q_heads * keys seen, summed over its
 * rows); decode_bytes: the K/V bytes the decode reads.  The split makes the
 * two finish together by rates measured on GB300: 1.45 PFLOP/s plus 10 us
 * for the prefill alone, 6.5 TB/s for the decode alone, and on few SMs the
 * decode drawing twice its whole-GPU bandwidth per SM; *ctas is in
 * [pkv_prefill_plan's count / 3, that count].  Host only, no
 * GPU work.  PKV_ERR_INVALID for a NULL ctas or a negative or non-finite
 * argument.
 */
pkv_status pkv_overlap_prefill_ctas(double prefill_flops, double decode_bytes, int32_t* ctas);

/*
 * decode_multi_plan -- split plan and workspace size of a multi-token decode
 * (pkv_paged_attn_decode_multi): batch sequences holding total_q query
 * tokens in all, at most max_q_len (1..16) each.  num_splits 0 = heuristic
 * (the single-token plan with ceil(max_q_len * G / 64) CTAs per sequence
 * and KV head), > 0 forces.  workspace_bytes_out: 0 when one split is used.
 * PKV_ERR_UNSUPPORTED for max_q_len > 16.  Host only.
 */
pkv_status pkv_decode_multi_plan(int32_t batch, int32_t total_q, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t max_q_len, int32_t max_seq_len,
                                 int32_t num_splits, int32_t* splits_out,
                                 int32_t* pages_per_split_out, size_t* workspace_bytes_out);

/*
 * paged_attn_decode_multi -- attention for steps of 1..16 query tokens per
 * sequence through split-KV decode ("Attention for verify steps": steps of
 * 2-16 tokens, verify steps of speculative decoding among them, run the
 * split-KV decode kernels rather than the prefill kernel), plus the
 * log-sum-exp combine.  Causal inside the step, bottom-right aligned: token
 * i of the q_b tokens of sequence b (seq_lens[b] positions, these tokens
 * included, appended beforehand) sees positions 0 .. seq_lens[b] - q_b + i.
 *
 *  q          bf16 [total_q][num_q_heads][128], 16-byte aligned; sequence b
 *             owns rows cu_q[b] .. cu_q[b+1] - 1 (cu_q int32 [batch + 1],
 *             non-decreasing, cu_q[0] = 0).
 *  block_table, max_pages, seq_lens, max_seq_len, softmax_scale: as
 *             pkv_paged_attn_decode.  max_q_len: the largest q_b (1..16).
 *  num_splits, workspace: as pkv_decode_multi_plan (256-byte aligned
 *             workspace of its size when splits > 1, else may be NULL).
 *  out        bf16 [total_q][num_q_heads][128]; lse fp32 [total_q][Hq]
 *             (natural log) or NULL.
 * bf16 pools only (PKV_ERR_UNSUPPORTED for INT8 and for max_q_len > 16).
 * A sequence with q_b > max_q_len, seq_lens[b] < q_b, a length past the
 * block table or a page id outside the pool is skipped and flagged for
 * pkv_poll_device_error.
 */
pkv_status pkv_paged_attn_decode_multi(const pkv_pool* pool, const void* q, int32_t total_q,
                                       const int32_t* cu_q, int32_t batch, int32_t num_q_heads,
                                       const int32_t* block_table, int32_t max_pages,
                                       const int32_t* seq_lens, int32_t max_q_len,
                                       int32_t max_seq_len, float softmax_scale,
                                       int32_t num_splits, void* workspace,
                                       size_t workspace_bytes, void* out, float* lse,
                                       void* stream);

/*
 * qkv_norm_rope_append -- the fused attention-input step: from the fused
 * q/k/v projection output, per-head RMSNorm of q and k, RoPE, and the KV
 * cache write, in one kernel ("Fused kernels ...": the attention-input
 * kernel that replaces 3 copies, 2 norms, 2 RoPE and 1 write, bit-identical
 * to that chain).
 *
 *  qkv        bf16 [num_tokens][num_q_heads + 2 Hkv][128]: q heads, then k
 *             heads, then v heads (16-byte aligned).
 *  q_norm_w,  fp32 [128] RMSNorm weights of q and of k, or NULL for no norm
 *  k_norm_w   on that part; eps > 0 typical (1e-6).  n_c = bf16((x_c * r)
 *             * w_c) with fp32 products, r = 1 / sqrt(z) correctly rounded,
 *             z = fp32(ms + eps), ms = the exact mean of x_c^2 rounded once
 *             to fp32 (exact while a head vector's values span at most 2^20
 *             in magnitude), so no summation order enters the result.
 *  rope_cos,  fp32 [max_pos][64] each, or both NULL for no RoPE.  Channel i
 *  rope_sin   pairs with i + 64 at the token's position p: o_i = bf16(n_i
 *             cos[p][i] - n_{i+64} sin[p][i]), o_{i+64} = bf16(n_{i+64}
 *             cos[p][i] + n_i sin[p][i]), fp32, each product and sum
 *             rounded once.
 *  cu_new, block_table, max_pages, seq_lens: as pkv_kv_append; token i of
 *             sequence b sits at position seq_lens[b] - n_b + i (p < max_pos
 *             with RoPE).
 *  q_out      bf16 [num_tokens][num_q_heads][128] (16-byte aligned).
 * The k heads (normed and rotated) and the v heads (copied) go to the new
 * tokens' pool slots.  bf16 pools only (PKV_ERR_UNSUPPORTED for INT8: append
 * q_out's K through pkv_kv_append instead).  A token whose position or page
 * falls outside the caller's arrays is skipped and flagged for
 * pkv_poll_device_error.
 */
pkv_status pkv_qkv_norm_rope_append(const pkv_pool* pool, const void* qkv, int32_t num_tokens,
                                    int32_t num_q_heads, const float* q_norm_w,
                                    const float* k_norm_w, float eps, const float* rope_cos,
                                    const float* rope_sin, int32_t max_pos, const int32_t* cu_new,
                                    int32_t batch, const int32_t* block_table, int32_t max_pages,
                                    const int32_t* seq_lens, void* q_out, void* stream);

/*
 * Synchronises the stream, then reports and clears the device-side error
 * words of the kernels: PKV_ERR_TIMEOUT if a bounded wait ran out (its
 * outputs are garbage), else PKV_ERR_INVALID if a device-side check of the
 * caller's arrays failed (a position past the block table, a page id outside
 * the pool: the offending row was skipped), else PKV_OK.  PKV_ERR_CUDA if
 * the stream itself reports an error.  Host-blocking.
 */
pkv_status pkv_poll_device_error(void* stream);

/*
 * Self-test of the error path of the kernels' bounded waits: one device
 * thread waits, with the bounded wait a prefill CTA uses before it merges a
 * unit cut between CTAs, until the uint32 at `counter` (device memory, the
 * caller's, only read) reaches `target`.  If nothing raises it, the wait
 * gives up after one second, the next pkv_poll_device_error reports
 * PKV_ERR_TIMEOUT, and the context stays usable.  Asynchronous on `stream`;
 * PKV_ERR_INVALID for a NULL counter.
 */
pkv_status pkv_selftest_bounded_wait(const uint32_t* counter, uint32_t target, void* stream);

/* Static text for a status code. */
const char* pkv_status_string(pkv_status status);

/* Number of SMs the split heuristic assumes for the current device (host). */
int32_t pkv_device_sm_count(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
