/*
 * pkv_oracle.c -- plain fp64 CPU oracle for attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the bench's CPU-baseline
 * leg use it.  It shares no code, header, table or helper with the CUDA
 * library; it takes the same raw input arrays and nothing else.
 *
 * What it computes, and where the pages state it (TileInfer.jl "Performance"
 * page, section "Fused kernels, FlashAttention and PagedAttention", and the
 * "INT8 KV cache" section of the same page):
 *
 *  - The reference ("ref") attention path gathers the pool pages named by the
 *    block table into dense K and V and materialises the scores; the paged
 *    flash kernels compute the same softmax attention, only online and in
 *    place.  So the oracle is the plain definition: gather, score, softmax
 *    (two passes: max, then sum), weighted sum of V.  orc_paged_attention.
 *  - Split-KV decode writes one partial per split and a separate combine
 *    kernel merges them (same section, the "Not kept" note on the fused
 *    combine).  orc_paged_attention with num_splits > 0 restates that:
 *    partial softmax per position range plus a log-sum-exp merge.
 *  - The INT8 cache keeps one scale per cached vector, keys smoothed by the
 *    key norm's weight ("INT8 KV cache" section).  orc_quantize_row_int8 and
 *    orc_kv_append_int8 follow the reading: x = float(k) (divided by w when
 *    smoothing), scale = max|x| / 127 in fp32, code = round-half-even of the
 *    fp32 quotient x / scale, clamped to [-127, 127]; an all-zero vector gets
 *    scale 0 and codes 0.
 *  - The KV write copies the new K/V vectors into the pages named by the
 *    block table (same page, list of fused kernels, "the KV cache write").
 *    orc_kv_append_bf16.
 *  - The fused attention-input step (same list: q/k RMSNorm, RoPE and the KV
 *    cache write from the fused q/k/v projection) is restated, with its
 *    readings, above orc_qkv_norm_rope_append.
 *
 * Readings where the pages are silent:
 *  - Causal alignment is bottom-right: query row i of a sequence with q_b new
 *    rows and L_b cached positions (new rows included) sits at absolute
 *    position L_b - q_b + i and sees keys 0 .. L_b - q_b + i.
 *  - GQA grouping is consecutive: query head h uses KV head h / (Hq / Hkv).
 *  - lse is the natural log of sum_j exp(scale * q.k_j).
 *  - An empty visible set gives out = 0 and lse = -inf.
 *
 * Pool layout (one pool each for K and V): [num_pages][Hkv][page_size][D];
 * bf16 entries are raw 16-bit patterns, int8 entries carry an fp32 scale per
 * (page, head, slot) in [num_pages][Hkv][page_size].  Position p of sequence
 * b lives in page block_table[b][p / page_size], slot p % page_size.
 *
 * Arithmetic is fp64 except the quantiser, which the reading fixes to fp32.
 * Build without fast-math and with -ffp-contract=off so both the x86 and the
 * Arm host give the same bits.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORC_BF16 0
#define ORC_INT8 1

typedef struct {
  const void* k;            /* bf16 bits (uint16) or int8 codes */
  const void* v;
  const float* k_scale;     /* int8 only: [num_pages][Hkv][page_size] */
  const float* v_scale;
  const float* k_smooth;    /* int8 only, optional: [D] per-channel key weight */
  int num_pages, num_kv_heads, page_size, head_dim, dtype;
} orc_pool;

static double bf16_bits_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static float bf16_bits_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Index of element c of position p of sequence b, KV head h, in the pool. */
static size_t pool_index(const orc_pool* pl, const int32_t* bt_row, int p, int h, int c) {
  int page = bt_row[p / pl->page_size];
  int slot = p % pl->page_size;
  return (((size_t)page * pl->num_kv_heads + h) * pl->page_size + slot) * pl->head_dim + c;
}

static size_t scale_index(const orc_pool* pl, const int32_t* bt_row, int p, int h) {
  int page = bt_row[p / pl->page_size];
  int slot = p % pl->page_size;
  return ((size_t)page * pl->num_kv_heads + h) * pl->page_size + slot;
}

/* Dequantised K[p][c] of KV head h (fp64). */
static double key_at(const orc_pool* pl, const int32_t* bt_row, int p, int h, int c) {
  size_t i = pool_index(pl, bt_row, p, h, c);
  if (pl->dtype == ORC_BF16) return bf16_bits_to_double(((const uint16_t*)pl->k)[i]);
  double code = (double)((const int8_t*)pl->k)[i];
  double s = (double)pl->k_scale[scale_index(pl, bt_row, p, h)];
  double w = pl->k_smooth ? (double)pl->k_smooth[c] : 1.0;
  return code * s * w;
}

static double value_at(const orc_pool* pl, const int32_t* bt_row, int p, int h, int c) {
  size_t i = pool_index(pl, bt_row, p, h, c);
  if (pl->dtype == ORC_BF16) return bf16_bits_to_double(((const uint16_t*)pl->v)[i]);
  double code = (double)((const int8_t*)pl->v)[i];
  return code * (double)pl->v_scale[scale_index(pl, bt_row, p, h)];
}

/*
 * Softmax attention of one query vector q (fp64, length D) over positions
 * [lo, hi) of one sequence and KV head, two passes: max, then sum.  Writes
 * the normalised output o[D] and returns lse = m + ln(sum exp(s - m)).
 * An empty range gives o = 0 and lse = -inf.
 */
static double attend_range(const orc_pool* pl, const int32_t* bt_row, int h_kv,
                           const double* q, double scale, int lo, int hi,
                           double* s_buf, double* o) {
  const int D = pl->head_dim;
  for (int c = 0; c < D; ++c) o[c] = 0.0;
  if (hi <= lo) return -INFINITY;
  double m = -INFINITY;
  for (int p = lo; p < hi; ++p) {
    double dot = 0.0;
    for (int c = 0; c < D; ++c) dot += q[c] * key_at(pl, bt_row, p, h_kv, c);
    s_buf[p - lo] = scale * dot;
    if (s_buf[p - lo] > m) m = s_buf[p - lo];
  }
  double sum = 0.0;
  for (int p = lo; p < hi; ++p) sum += exp(s_buf[p - lo] - m);
  double lse = m + log(sum);
  for (int p = lo; p < hi; ++p) {
    double w = exp(s_buf[p - lo] - lse);
    for (int c = 0; c < D; ++c) o[c] += w * value_at(pl, bt_row, p, h_kv, c);
  }
  return lse;
}

/* ---------------------------------------------------------------- threads */

typedef struct {
  void (*fn)(void* ctx, long task, double* scratch);
  void* ctx;
  long ntasks;
  long next;            /* shared task counter (gcc atomics) */
  size_t scratch_len;   /* doubles of per-thread scratch */
} task_pool;

static void* worker(void* arg) {
  task_pool* tp = (task_pool*)arg;
  double* scratch = (double*)malloc(tp->scratch_len * sizeof(double));
  if (!scratch) return (void*)1;
  for (;;) {
    long t = __atomic_fetch_add(&tp->next, 1, __ATOMIC_RELAXED);
    if (t >= tp->ntasks) break;
    tp->fn(tp->ctx, t, scratch);
  }
  free(scratch);
  return NULL;
}

static int run_tasks(void (*fn)(void*, long, double*), void* ctx, long ntasks,
                     size_t scratch_len, int nthreads) {
  if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > ntasks) nthreads = (int)(ntasks > 0 ? ntasks : 1);
  task_pool tp = {fn, ctx, ntasks, 0, scratch_len};
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  if (!th) return -1;
  int started = 0, rc = 0;
  for (int i = 0; i < nthreads; ++i) {
    if (pthread_create(&th[i], NULL, worker, &tp) != 0) { rc = -1; break; }
    ++started;
  }
  if (started == 0) rc = (worker(&tp) == NULL) ? 0 : -1;
  for (int i = 0; i < started; ++i) {
    void* r = NULL;
    pthread_join(th[i], &r);
    if (r) rc = -1;
  }
  free(th);
  return rc;
}

/* --------------------------------------------------------- attention rows */

typedef struct {
  const orc_pool* pool;
  const uint16_t* q;        /* bf16 bits [total_q][Hq][D] */
  const int32_t* cu_q;      /* [B+1] */
  int B, Hq;
  const int32_t* block_table;
  int max_pages;
  const int32_t* seq_lens;
  double scale;
  const int32_t* rows;      /* query rows (indices into total_q) to evaluate */
  int num_splits;           /* 0: unsplit; >0: split-KV partials + combine */
  double* out;              /* [nrows][Hq][D] */
  double* lse;              /* [nrows][Hq] */
  int status;
} attn_ctx;

/* Sequence that owns query row r: the b with cu_q[b] <= r < cu_q[b+1]. */
static int owner_sequence(const int32_t* cu_q, int B, int r) {
  for (int b = 0; b < B; ++b)
    if (r >= cu_q[b] && r < cu_q[b + 1]) return b;
  return -1;
}

static void attn_task(void* vctx, long task, double* scratch) {
  attn_ctx* a = (attn_ctx*)vctx;
  const orc_pool* pl = a->pool;
  const int D = pl->head_dim;
  const int G = a->Hq / pl->num_kv_heads;
  long ri = task / a->Hq;
  int hq = (int)(task % a->Hq);
  int r = a->rows[ri];
  int b = owner_sequence(a->cu_q, a->B, r);
  if (b < 0) { a->status = -1; return; }
  int qlen = a->cu_q[b + 1] - a->cu_q[b];
  int L = a->seq_lens[b];
  int pos = L - qlen + (r - a->cu_q[b]);   /* bottom-right causal position */
  int visible = pos + 1;                    /* keys 0..pos */
  if (visible > L) visible = L;
  if (visible < 0) visible = 0;
  const int32_t* bt_row = a->block_table + (size_t)b * a->max_pages;
  int h_kv = hq / G;

  double* qd = scratch;               /* D */
  double* o = scratch + D;            /* D */
  double* opart = scratch + 2 * D;    /* D */
  double* s_buf = scratch + 3 * D;    /* up to L */
  for (int c = 0; c < D; ++c)
    qd[c] = bf16_bits_to_double(a->q[((size_t)r * a->Hq + hq) * D + c]);

  double* out = a->out + ((size_t)ri * a->Hq + hq) * D;
  double lse;
  if (a->num_splits <= 0) {
    lse = attend_range(pl, bt_row, h_kv, qd, a->scale, 0, visible, s_buf, o);
    for (int c = 0; c < D; ++c) out[c] = o[c];
  } else {
    /* Split-KV: split sigma covers positions [sigma*C, min((sigma+1)*C, n)),
     * C = ceil(n / S).  Each split yields a normalised partial and its lse;
     * the combine weighs partial sigma by exp(lse_sigma - lse) with
     * lse = ln sum_sigma exp(lse_sigma).  Empty splits have lse = -inf. */
    int S = a->num_splits;
    int C = (visible + S - 1) / S;
    double* lse_part = (double*)malloc(sizeof(double) * (size_t)S);
    double* o_part = (double*)malloc(sizeof(double) * (size_t)S * D);
    if (!lse_part || !o_part) { free(lse_part); free(o_part); a->status = -1; return; }
    double mx = -INFINITY;
    for (int sgm = 0; sgm < S; ++sgm) {
      int lo = sgm * C, hi = (sgm + 1) * C;
      if (hi > visible) hi = visible;
      lse_part[sgm] = attend_range(pl, bt_row, h_kv, qd, a->scale, lo, hi, s_buf, opart);
      for (int c = 0; c < D; ++c) o_part[(size_t)sgm * D + c] = opart[c];
      if (lse_part[sgm] > mx) mx = lse_part[sgm];
    }
    for (int c = 0; c < D; ++c) out[c] = 0.0;
    if (mx == -INFINITY) {
      lse = -INFINITY;
    } else {
      double sum = 0.0;
      for (int sgm = 0; sgm < S; ++sgm) sum += exp(lse_part[sgm] - mx);
      lse = mx + log(sum);
      for (int sgm = 0; sgm < S; ++sgm) {
        if (lse_part[sgm] == -INFINITY) continue;
        double w = exp(lse_part[sgm] - lse);
        for (int c = 0; c < D; ++c) out[c] += w * o_part[(size_t)sgm * D + c];
      }
    }
    free(lse_part);
    free(o_part);
  }
  a->lse[(size_t)ri * a->Hq + hq] = lse;
}

static int check_pool(const orc_pool* pl, int Hq) {
  if (!pl || !pl->k || !pl->v) return -1;
  if (pl->num_kv_heads <= 0 || Hq <= 0 || Hq % pl->num_kv_heads) return -1;
  if (pl->page_size <= 0 || pl->head_dim <= 0) return -1;
  if (pl->dtype == ORC_INT8 && (!pl->k_scale || !pl->v_scale)) return -1;
  return 0;
}

/*
 * Attention of the listed query rows (all Hq heads each) over the paged
 * cache.  q rows of sequence b are cu_q[b] .. cu_q[b+1]-1; seq_lens[b]
 * counts every cached position of b, the rows' own included.  A decode step
 * is the case cu_q = 0, 1, 2, ..., B.  Returns 0, or -1 on bad arguments.
 */
int orc_paged_attention(const orc_pool* pool, const uint16_t* q, const int32_t* cu_q, int B,
                        int num_q_heads, const int32_t* block_table, int max_pages,
                        const int32_t* seq_lens, double scale, const int32_t* rows,
                        int nrows, int num_splits, double* out, double* lse, int nthreads) {
  if (check_pool(pool, num_q_heads) || !q || !cu_q || !block_table || !seq_lens || !rows ||
      !out || !lse || B <= 0 || nrows < 0)
    return -1;
  int maxL = 0;
  for (int b = 0; b < B; ++b) {
    if (seq_lens[b] < 0 || seq_lens[b] > max_pages * pool->page_size) return -1;
    if (cu_q[b + 1] < cu_q[b]) return -1;   /* rows at negative positions see nothing */
    if (seq_lens[b] > maxL) maxL = seq_lens[b];
  }
  attn_ctx ctx = {pool, q, cu_q, B, num_q_heads, block_table, max_pages, seq_lens, scale,
                  rows, num_splits, out, lse, 0};
  size_t scratch = (size_t)3 * pool->head_dim + (size_t)maxL + 1;
  if (run_tasks(attn_task, &ctx, (long)nrows * num_q_heads, scratch, nthreads)) return -1;
  return ctx.status;
}

/* ------------------------------------------------------------- KV writes */

/*
 * Position of new token i of sequence b: seq_lens[b] - n_b + i, with
 * n_b = cu_new[b+1] - cu_new[b] (seq_lens already count the new tokens).
 * Returns the flat slot index page * page_size + slot, or -1 if out of range.
 */
static long new_token_slot(const int32_t* block_table, int max_pages, int page_size,
                           const int32_t* cu_new, const int32_t* seq_lens, int b, int i) {
  int n = cu_new[b + 1] - cu_new[b];
  int p = seq_lens[b] - n + i;
  if (p < 0 || p >= max_pages * page_size) return -1;
  int page = block_table[(size_t)b * max_pages + p / page_size];
  return (long)page * page_size + p % page_size;
}

/* Copy the bf16 K/V vectors of the new tokens into their pool slots. */
int orc_kv_append_bf16(uint16_t* pool_k, uint16_t* pool_v, int num_pages, int Hkv, int page_size,
                       int D, const uint16_t* k_new, const uint16_t* v_new,
                       const int32_t* cu_new, int B, const int32_t* block_table, int max_pages,
                       const int32_t* seq_lens) {
  for (int b = 0; b < B; ++b) {
    for (int i = 0; i < cu_new[b + 1] - cu_new[b]; ++i) {
      long fs = new_token_slot(block_table, max_pages, page_size, cu_new, seq_lens, b, i);
      if (fs < 0) return -1;
      long page = fs / page_size, slot = fs % page_size;
      if (page >= num_pages) return -1;
      int t = cu_new[b] + i;
      for (int h = 0; h < Hkv; ++h) {
        size_t dst = ((size_t)(page * Hkv + h) * page_size + slot) * D;
        size_t src = ((size_t)t * Hkv + h) * D;
        memcpy(pool_k + dst, k_new + src, sizeof(uint16_t) * (size_t)D);
        memcpy(pool_v + dst, v_new + src, sizeof(uint16_t) * (size_t)D);
      }
    }
  }
  return 0;
}

/*
 * One vector to int8 codes and an fp32 scale, every step in fp32:
 * x_c = float(k_c), divided by w_c when a smoothing weight is given;
 * amax = max_c |x_c|; scale = amax / 127; code_c = nearest-even integer to
 * the fp32 quotient x_c / scale, clamped to [-127, 127].  amax = 0 gives
 * scale 0 and all codes 0.
 */
void orc_quantize_row_int8(const uint16_t* x_bf16, const float* w, int D, int8_t* codes,
                           float* scale_out) {
  float amax = 0.0f;
  for (int c = 0; c < D; ++c) {
    float x = bf16_bits_to_float(x_bf16[c]);
    if (w) x = x / w[c];
    float ax = fabsf(x);
    if (ax > amax) amax = ax;
  }
  float scale = amax / 127.0f;
  *scale_out = scale;
  for (int c = 0; c < D; ++c) {
    if (scale == 0.0f) { codes[c] = 0; continue; }
    float x = bf16_bits_to_float(x_bf16[c]);
    if (w) x = x / w[c];
    float qf = x / scale;
    float r = nearbyintf(qf);   /* default rounding mode: to nearest, ties to even */
    if (r > 127.0f) r = 127.0f;
    if (r < -127.0f) r = -127.0f;
    codes[c] = (int8_t)r;
  }
}

/* Quantise the new K/V vectors (K smoothed by w if given) into the int8 pool. */
int orc_kv_append_int8(int8_t* pool_k, int8_t* pool_v, float* k_scale, float* v_scale,
                       int num_pages, int Hkv, int page_size, int D, const uint16_t* k_new,
                       const uint16_t* v_new, const float* k_smooth, const int32_t* cu_new,
                       int B, const int32_t* block_table, int max_pages,
                       const int32_t* seq_lens) {
  for (int b = 0; b < B; ++b) {
    for (int i = 0; i < cu_new[b + 1] - cu_new[b]; ++i) {
      long fs = new_token_slot(block_table, max_pages, page_size, cu_new, seq_lens, b, i);
      if (fs < 0) return -1;
      long page = fs / page_size, slot = fs % page_size;
      if (page >= num_pages) return -1;
      int t = cu_new[b] + i;
      for (int h = 0; h < Hkv; ++h) {
        size_t row = (size_t)(page * Hkv + h) * page_size + slot;
        size_t src = ((size_t)t * Hkv + h) * D;
        orc_quantize_row_int8(k_new + src, k_smooth, D, pool_k + row * D, &k_scale[row]);
        orc_quantize_row_int8(v_new + src, NULL, D, pool_v + row * D, &v_scale[row]);
      }
    }
  }
  return 0;
}

/* ------------------------------------------------ fused attention inputs */

/*
 * The "attention inputs" fused kernel of the same page's list of fused
 * kernels: from the fused q/k/v projection output, q/k RMSNorm, RoPE and the
 * KV cache write, bit-identical to the chain it replaces (3 copies, 2 norms,
 * 2 RoPE, 1 write).  The pages give no formulas; readings (stated once here
 * and in the build's notes), with the chain taken to be fp32 GPU kernels
 * that store bf16:
 *  - RMSNorm over one head's D channels, the chain's fp32 norm kernel:
 *    ms = fp32(sum_c x_c^2 / D) (the exact sum, rounded once; D a power of
 *    two), z = fp32(ms + eps) with eps an fp32 value, r = fp32(1 / sqrt(z))
 *    correctly rounded (orc_rsqrt_rn), n_c = bf16((x_c * r) * w_c) with
 *    both products in fp32.  Every step is one IEEE fp32 rounding of an
 *    exactly defined value, so the result does not depend on the order in
 *    which a kernel sums the squares.  The sum is exact in fp64 while the
 *    head's values span at most 2^15 in magnitude (53 bits hold the 16-bit
 *    squares and 7 bits of carries).  A NULL weight means that part has no
 *    norm (n = x).
 *  - RoPE by halves (channel i pairs with i + D/2, i < D/2) at the token's
 *    position p, with cos/sin from a caller table [max_pos][D/2], every
 *    product and sum in fp32: o_i = bf16(n_i cos - n_{i+D/2} sin),
 *    o_{i+D/2} = bf16(n_{i+D/2} cos + n_i sin).  A NULL table means no RoPE
 *    (o = n).
 *  - q heads go to q_out [T][Hq][D]; k heads, normed and rotated, and v
 *    heads, copied, go to the pool slots of the new tokens (positions as in
 *    orc_kv_append_bf16).  The projection output is [T][Hq + 2 Hkv][D]: q
 *    heads, then k heads, then v heads.
 * Rounding to bf16 is round to nearest, ties to even, exactly where the
 * chain stores bf16.  (The file is built with -ffp-contract=off, so no
 * product and sum below fuse into one rounding.)
 */

/* v rounded to the nearest bf16 (ties to even), as raw bits. */
static uint16_t bf16_bits_from_double(double v) {
  if (isnan(v)) return 0x7FC0;
  const uint16_t sign = signbit(v) ? 0x8000 : 0;
  const double a = fabs(v);
  if (a == 0.0) return sign;
  int e;
  const double m = frexp(a, &e);                /* a = m 2^e, m in [1/2, 1) */
  /* 8 significant bits for normals (2^-126 <= a), fewer below */
  int bits = 8;
  if (e < -125) bits = 8 - (-125 - e);
  const double r = ldexp(nearbyint(ldexp(m, bits)), e - bits);
  if (r >= 0x1.0p128) return sign | 0x7F80;     /* rounds past the largest finite */
  const float f = (float)r;                     /* exact: r is a bf16 value */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return sign | (uint16_t)(u >> 16);
}

/* Sign of m^2 z - 1 for m = M 2^a (M an integer below 2^26) and z a positive
 * normal float, in exact integer arithmetic. */
static int sq_times_z_vs_one(uint64_t M, int a, float z) {
  int bz;
  const double fz = frexp((double)z, &bz);              /* z = fz 2^bz, fz in [1/2, 1) */
  const uint64_t Z = (uint64_t)ldexp(fz, 24);           /* z = Z 2^(bz - 24), exact */
  const int e = 2 * a + bz - 24;                        /* m^2 z = M^2 Z 2^e */
  const unsigned __int128 P = (unsigned __int128)(M * M) * Z;   /* below 2^76 */
  if (P == 0) return -1;
  if (e >= 0) return (e == 0 && P == 1) ? 0 : 1;
  if (-e >= 127) return -1;
  const unsigned __int128 one = (unsigned __int128)1 << -e;
  return P < one ? -1 : (P > one ? 1 : 0);
}

/* The float nearest to 1 / sqrt(z), ties to even, for a positive normal
 * float z.  Start from the double-precision quotient (within one float step
 * of the answer) and test, exactly, where 1/sqrt(z) lies against the
 * midpoints between the candidate and its neighbours: y > m iff m^2 z < 1. */
float orc_rsqrt_rn(float z) {
  float r = (float)(1.0 / sqrt((double)z));
  for (int it = 0; it < 4; ++it) {
    int er;
    const double fr = frexp((double)r, &er);            /* r = fr 2^er */
    const uint64_t R = (uint64_t)ldexp(fr, 24);         /* r = R 2^(er - 24), R in [2^23, 2^24) */
    const int pow2 = R == (1ull << 23);                 /* the step below r halves */
    /* upper midpoint (R + 1/2) 2^(er - 24); lower (R - 1/2) 2^(er - 24), or
     * (R - 1/4) 2^(er - 24) when r is a power of two */
    const int hi = sq_times_z_vs_one(2 * R + 1, er - 25, z);
    const int lo = pow2 ? sq_times_z_vs_one(4 * R - 1, er - 26, z)
                        : sq_times_z_vs_one(2 * R - 1, er - 25, z);
    if (hi < 0) {                     /* 1/sqrt(z) above the upper midpoint */
      r = nextafterf(r, INFINITY);
      continue;
    }
    if (lo > 0) {                     /* 1/sqrt(z) below the lower midpoint */
      r = nextafterf(r, 0.0f);
      continue;
    }
    if (hi == 0) return (R & 1) ? nextafterf(r, INFINITY) : r;   /* a tie: the even one */
    if (lo == 0) return (R & 1) ? nextafterf(r, 0.0f) : r;
    return r;
  }
  return r;
}

/* RMSNorm (if w) then RoPE (if cos_row) of one head vector of D bf16 values. */
static void norm_rope(const uint16_t* x, int D, const float* w, float eps, const float* cos_row,
                      const float* sin_row, uint16_t* out) {
  uint16_t n[1024];
  if (w) {
    double ss = 0.0;
    for (int c = 0; c < D; ++c) {
      const double v = bf16_bits_to_double(x[c]);
      ss += v * v;
    }
    const float ms = (float)(ss / D);
    const float z = ms + eps;
    const float r = orc_rsqrt_rn(z);
    for (int c = 0; c < D; ++c) {
      const float xr = bf16_bits_to_float(x[c]) * r;
      const float y = xr * w[c];
      n[c] = bf16_bits_from_double((double)y);
    }
  } else {
    memcpy(n, x, sizeof(uint16_t) * (size_t)D);
  }
  if (cos_row) {
    const int half = D / 2;
    for (int i = 0; i < half; ++i) {
      const float a = bf16_bits_to_float(n[i]), b = bf16_bits_to_float(n[i + half]);
      const float c = cos_row[i], s = sin_row[i];
      const float ac = a * c, bs = b * s, bc = b * c, as = a * s;
      const float lo = ac - bs, hi = bc + as;
      out[i] = bf16_bits_from_double((double)lo);
      out[i + half] = bf16_bits_from_double((double)hi);
    }
  } else {
    memcpy(out, n, sizeof(uint16_t) * (size_t)D);
  }
}

int orc_qkv_norm_rope_append(const uint16_t* qkv, int Hq, int Hkv, int D, const float* q_w,
                             const float* k_w, double eps, const float* cos_tab,
                             const float* sin_tab, int max_pos, const int32_t* cu_new, int B,
                             const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                             uint16_t* q_out, uint16_t* pool_k, uint16_t* pool_v, int num_pages,
                             int page_size) {
  if (D <= 0 || D > 1024 || D % 2) return -1;
  const int H = Hq + 2 * Hkv;
  for (int b = 0; b < B; ++b) {
    const int n = cu_new[b + 1] - cu_new[b];
    for (int i = 0; i < n; ++i) {
      const int p = seq_lens[b] - n + i;
      const long fs = new_token_slot(block_table, max_pages, page_size, cu_new, seq_lens, b, i);
      if (fs < 0) return -1;
      if (cos_tab && (p < 0 || p >= max_pos)) return -1;
      const long page = fs / page_size, slot = fs % page_size;
      if (page < 0 || page >= num_pages) return -1;
      const int t = cu_new[b] + i;
      const float* cr = cos_tab ? cos_tab + (size_t)p * (D / 2) : NULL;
      const float* sr = sin_tab ? sin_tab + (size_t)p * (D / 2) : NULL;
      const uint16_t* row = qkv + (size_t)t * H * D;
      for (int h = 0; h < Hq; ++h)
        norm_rope(row + (size_t)h * D, D, q_w, (float)eps, cr, sr, q_out + ((size_t)t * Hq + h) * D);
      for (int h = 0; h < Hkv; ++h) {
        const size_t dst = ((size_t)(page * Hkv + h) * page_size + slot) * D;
        norm_rope(row + (size_t)(Hq + h) * D, D, k_w, (float)eps, cr, sr, pool_k + dst);
        memcpy(pool_v + dst, row + (size_t)(Hq + Hkv + h) * D, sizeof(uint16_t) * (size_t)D);
      }
    }
  }
  return 0;
}

/* Exposed for the pins: v rounded to bf16 bits. */
uint16_t orc_bf16_from_double(double v) { return bf16_bits_from_double(v); }
