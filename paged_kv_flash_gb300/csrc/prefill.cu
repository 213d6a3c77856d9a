// prefill.cu -- causal chunked prefill attention over the paged cache on the
// 5th-generation tensor cores (tcgen05 MMAs, TMEM accumulators, TMA loads).
//
// The method: TileInfer.jl "Performance" page -- paged flash attention runs
// an online softmax over the pages read in place through the block table
// ("Fused kernels, FlashAttention and PagedAttention"); the prefill kernel
// runs a block per head over every page ("Attention for verify steps");
// chunked prefill attends a chunk of new rows to the cached prefix ("What is
// left to gain").  Rows sit bottom-right: row i of a chunk of q rows in a
// sequence of L cached positions is position L - q + i and sees keys 0..it.
//
// One CTA per (query head, 128-row query tile, sequence); 6 warps:
//   warp 0     TMA producer: 128-key K and V blocks, each gathered as eight
//              16-row page boxes (one per page named by the block table) per
//              64-channel half, 128-byte swizzled, 2-stage ring per operand;
//   warp 1     MMA issuer (one thread): S = Q K^T into TMEM (double
//              buffered, 2 x 128 columns), O += P V into TMEM (128 columns);
//   warps 2-5  softmax: thread = query row = TMEM lane; reads S with
//              tcgen05.ld, keeps the running max and sum of its row, rescales
//              O in TMEM only when its max grows by more than 2^8 (exact: the
//              final normalisation uses the same stale max), writes P as bf16
//              into shared memory in the swizzled K-major layout the PV MMA
//              reads, and finally normalises O and writes out and lse.
// Q is loaded once by the softmax warps (rows past the chunk are zero) into
// the same swizzled layout.  V rows at positions >= L in the last block are
// zeroed by the MMA warp before the PV MMA, so stale or poisoned pool slots
// can never reach the accumulator (P is 0 there, but 0 * NaN is NaN).
//
// Every wait is bounded (wall clock, one second); a wait that runs out sets
// the device error word and an abort flag that makes every role leave its
// loop; the MMA warp drains its issued MMAs and the producer its loads
// before TMEM is freed and the CTA exits.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"

namespace {

using namespace pkv;

__device__ uint32_t g_err_prefill;

constexpr int BM = 128;                       // query rows per tile (= TMEM lanes)
constexpr int BN = 128;                       // keys per block (8 pages)
constexpr int NSTAGE = 2;                     // K and V ring depth
constexpr int HALF = 16384;                   // one 128 x 64 bf16 swizzled half-tile
constexpr int TILE = 2 * HALF;                // 128 x 128 bf16
constexpr int NUM_THREADS = 320;              // softmax A: warps 0-3, B: 4-7, TMA 8, MMA 9
constexpr int WARP_TMA = 8, WARP_MMA = 9;
constexpr uint32_t TMEM_COLS = 512;
// TMEM columns: S_A 0..127, S_B 128..255, O_A 256..383, O_B 384..511.  P of a
// tile (bf16 pairs, 64 columns) overwrites the upper half of its S columns.
__host__ __device__ constexpr uint32_t tm_s(int x) { return (uint32_t)x * 128u; }
__host__ __device__ constexpr uint32_t tm_o(int x) { return 256u + (uint32_t)x * 128u; }
__host__ __device__ constexpr uint32_t tm_p(int x) { return (uint32_t)x * 128u + 64u; }

// Shared-memory map (offsets from a 1024-byte aligned base).
constexpr int OFF_Q = 0;                      // Q_A, Q_B
constexpr int OFF_K = OFF_Q + 2 * TILE;
constexpr int OFF_V = OFF_K + NSTAGE * TILE;
constexpr int OFF_BAR = OFF_V + NSTAGE * TILE;
// barriers: q_full, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[A,B],
// p_full[A,B], o_done[A,B], drain
constexpr int BAR_Q = 0, BAR_KF = 1, BAR_KE = 3, BAR_VF = 5, BAR_VE = 7, BAR_SF = 9,
              BAR_PF = 11, BAR_OD = 13, BAR_DR = 15, NUM_BARS = 16;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;   // + alignment slack

// kind::f16 instruction descriptor: D fp32, A and B bf16, M = N = 128.
// bits 4-5 D format, 7-9 A format, 10-12 B format, 15/16 A/B major
// (0 = K-major, 1 = MN-major), 17-22 N >> 3, 24-28 M >> 4.
constexpr uint32_t IDESC_QK =
    (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
constexpr uint32_t IDESC_PV = IDESC_QK | (1u << 16);   // B (= V) is MN-major

// Shared-memory matrix descriptor, 128-byte swizzle: start address >> 4
// (bits 0-13), leading byte offset >> 4 (16-29), stride byte offset >> 4
// (32-45), descriptor version 1 (bit 46), swizzle mode 2 = 128B (61-63).
// K-major tiles: 8-row groups 1024 B apart (SBO); the leading offset is
// unused.  MN-major V tiles: 64-channel halves 16 KiB apart (LBO), 8-key
// groups 1024 B apart (SBO).
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)(HALF >> 4) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

#define PKV_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                  "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define PKV_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
                  "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : PKV_R8(0), PKV_R8(8), PKV_R8(16), PKV_R8(24)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      ::"r"(taddr), PKV_W8(0), PKV_W8(8), PKV_W8(16), PKV_W8(24)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

#define PKV_R16(i) PKV_R8(i), PKV_R8(i + 8)
#define PKV_W16(i) PKV_W8(i), PKV_W8(i + 8)

// 64 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,"
      "%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,"
      "%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
      : PKV_R16(0), PKV_R16(16), PKV_R16(32), PKV_R16(48)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,"
      "%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,"
      "%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};"
      ::"r"(taddr), PKV_W16(0), PKV_W16(16), PKV_W16(32), PKV_W16(48)
      : "memory");
}

// D (TMEM) (+)= A (TMEM, 128 lanes x 16 bf16 in 8 columns) * B (shared).
__device__ __forceinline__ void mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate));
}

// Eight back-to-back MMAs over K = 128 (one 128-column block) in one asm
// block, so the issuing warp spends about three instructions per MMA even
// when the softmax warps keep its scheduler busy.  Descriptor start
// addresses advance by immediates (16-byte units): K-major 128B-swizzled
// tiles step 32 B within a 128-byte row, then jump to the second 64-column
// half 16 KiB on; the MN-major V tile steps 16 keys = 2 KiB.
#define PKV_MMA_SS(acc) \
  "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, " acc ";\n\t"
__device__ __forceinline__ void mma8_qk(uint32_t d_tmem, uint64_t a0, uint64_t b0, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred pf, pt;\n\t.reg .b64 ra, rb;\n\t"
      "setp.ne.b32 pf, 0, 0;\n\tsetp.eq.b32 pt, 0, 0;\n\t"
      "mov.b64 ra, %1;\n\tmov.b64 rb, %2;\n\t" PKV_MMA_SS("pf")
      "add.s64 ra, %1, 2;\n\tadd.s64 rb, %2, 2;\n\t" PKV_MMA_SS("pt")
      "add.s64 ra, %1, 4;\n\tadd.s64 rb, %2, 4;\n\t" PKV_MMA_SS("pt")
      "add.s64 ra, %1, 6;\n\tadd.s64 rb, %2, 6;\n\t" PKV_MMA_SS("pt")
      "add.s64 ra, %1, 1024;\n\tadd.s64 rb, %2, 1024;\n\t" PKV_MMA_SS("pt")
      "add.s64 ra, %1, 1026;\n\tadd.s64 rb, %2, 1026;\n\t" PKV_MMA_SS("pt")
      "add.s64 ra, %1, 1028;\n\tadd.s64 rb, %2, 1028;\n\t" PKV_MMA_SS("pt")
      "add.s64 ra, %1, 1030;\n\tadd.s64 rb, %2, 1030;\n\t" PKV_MMA_SS("pt")
      "}"
      ::"r"(d_tmem), "l"(a0), "l"(b0), "r"(idesc));
}
// P (K-major, shared) x V (MN-major, shared); the first MMA accumulates iff acc0.
__device__ __forceinline__ void mma8_pv_ss(uint32_t d_tmem, uint64_t a0, uint64_t b0,
                                           uint32_t idesc, uint32_t acc0) {
  asm volatile(
      "{\n\t.reg .pred p0, pt;\n\t.reg .b64 ra, rb;\n\t"
      "setp.ne.b32 p0, %4, 0;\n\tsetp.eq.b32 pt, 0, 0;\n\t"
      "mov.b64 ra, %1;\n\tmov.b64 rb, %2;\n\t" PKV_MMA_SS("p0")
      "add.s64 ra, %1, 2;\n\tadd.s64 rb, %2, 128;\n\t" PKV_MMA_SS("pt")
      "add.s64 ra, %1, 4;\n\tadd.s64 rb, %2, 256;\n\t" PKV_MMA_SS("pt")
      "add.s64 ra, %1, 6;\n\tadd.s64 rb, %2, 384;\n\t" PKV_MMA_SS("pt")
      "add.s64 ra, %1, 1024;\n\tadd.s64 rb, %2, 512;\n\t" PKV_MMA_SS("pt")
      "add.s64 ra, %1, 1026;\n\tadd.s64 rb, %2, 640;\n\t" PKV_MMA_SS("pt")
      "add.s64 ra, %1, 1028;\n\tadd.s64 rb, %2, 768;\n\t" PKV_MMA_SS("pt")
      "add.s64 ra, %1, 1030;\n\tadd.s64 rb, %2, 896;\n\t" PKV_MMA_SS("pt")
      "}"
      ::"r"(d_tmem), "l"(a0), "l"(b0), "r"(idesc), "r"(acc0));
}
#define PKV_MMA_TS(acc) \
  "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], rb, %3, " acc ";\n\t"
// P (TMEM, 8 columns per 16 keys) x V (MN-major, shared).
__device__ __forceinline__ void mma8_pv_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b0,
                                           uint32_t idesc, uint32_t acc0) {
  asm volatile(
      "{\n\t.reg .pred p0, pt;\n\t.reg .b32 ta;\n\t.reg .b64 rb;\n\t"
      "setp.ne.b32 p0, %4, 0;\n\tsetp.eq.b32 pt, 0, 0;\n\t"
      "mov.b32 ta, %1;\n\tmov.b64 rb, %2;\n\t" PKV_MMA_TS("p0")
      "add.u32 ta, %1, 8;\n\tadd.s64 rb, %2, 128;\n\t" PKV_MMA_TS("pt")
      "add.u32 ta, %1, 16;\n\tadd.s64 rb, %2, 256;\n\t" PKV_MMA_TS("pt")
      "add.u32 ta, %1, 24;\n\tadd.s64 rb, %2, 384;\n\t" PKV_MMA_TS("pt")
      "add.u32 ta, %1, 32;\n\tadd.s64 rb, %2, 512;\n\t" PKV_MMA_TS("pt")
      "add.u32 ta, %1, 40;\n\tadd.s64 rb, %2, 640;\n\t" PKV_MMA_TS("pt")
      "add.u32 ta, %1, 48;\n\tadd.s64 rb, %2, 768;\n\t" PKV_MMA_TS("pt")
      "add.u32 ta, %1, 56;\n\tadd.s64 rb, %2, 896;\n\t" PKV_MMA_TS("pt")
      "}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b0), "r"(idesc), "r"(acc0));
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// (lo, hi) -> bf16x2 with lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// Bounded wait shared by all roles; the result is uniform across the warp.
// Gives up when another role raised the abort flag or after kWaitLimitNs.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t* abort) {
  bool ok = mbar_try_wait(bar, parity);
  if (!ok) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
      if (mbar_try_wait(bar, parity)) { ok = true; break; }
      if ((it & 63u) == 0) {
        if (*abort) break;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          *abort = 1u;
          atomicOr(&g_err_prefill, kErrTimeout);
          break;
        }
      }
    }
  }
  return __all_sync(0xffffffffu, ok);
}

struct PrefillParams {
  pkv_host::PrefillLaunch a;
  int n_pairs;                  // pairs of 128-row tiles of the longest chunk
};

__global__ void __launch_bounds__(NUM_THREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                   const __grid_constant__ PrefillParams prm) {
  const pkv_host::PrefillLaunch& a = prm.a;
  const int hq = blockIdx.x;
  const int pair = prm.n_pairs - 1 - (int)blockIdx.y;   // heaviest tiles first
  const int b = blockIdx.z;
  const int Hq = a.num_q_heads;
  const int G = Hq / a.num_kv_heads;
  const int hkv = hq / G;

  const int q0 = a.cu_q[b];
  const int q_len = a.cu_q[b + 1] - q0;
  if (q_len > prm.n_pairs * 2 * BM && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
    atomicOr(&g_err_prefill, kErrBadIndex);             // chunk longer than max_q_len
  const int row0 = pair * 2 * BM;                       // first chunk row of tile A
  if (row0 >= q_len) return;                            // no rows in this pair
  const int L = a.seq_lens[b];
  if (L < q_len || L > a.max_pages * kPageSize) {
    if (threadIdx.x == 0) atomicOr(&g_err_prefill, kErrBadIndex);
    return;
  }
  // tile x (0 = A, 1 = B): rows row0 + x*128 .. ; positions L - q_len + row
  auto rows_of = [&](int x) { return max(0, min(BM, q_len - row0 - x * BM)); };
  auto pmin_of = [&](int x) { return L - q_len + row0 + x * BM; };
  auto nblk_of = [&](int x) {
    const int rws = rows_of(x);
    return rws > 0 ? (pmin_of(x) + rws - 1) / BN + 1 : 0;
  };
  const int nblk_a = nblk_of(0), nblk_b = nblk_of(1);
  const int n_blk = max(nblk_a, nblk_b);
  const int npages = (L + kPageSize - 1) / kPageSize;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_s - raw_s);
  auto bar = [&](int i) -> uint32_t { return base_s + OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(base + OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(bar(BAR_Q), 2 * BM);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(bar(BAR_KF + s), 1);
      mbar_init(bar(BAR_KE + s), 1);
      mbar_init(bar(BAR_VF + s), 1);
      mbar_init(bar(BAR_VE + s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(BAR_SF + x), 1);
      mbar_init(bar(BAR_PF + x), BM);
      mbar_init(bar(BAR_OD + x), 1);
    }
    mbar_init(bar(BAR_DR), 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == WARP_MMA) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(tmem_slot)), "r"(TMEM_COLS) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  static_assert(NSTAGE == 2, "the producer tracks two stages");
  int last_k0 = -1, last_k1 = -1, last_v0 = -1, last_v1 = -1;   // last block issued per stage
  if (warp == WARP_TMA) {
    // ------------------------------------------------------ TMA producer
    const int32_t* bt_row = a.block_table + (size_t)b * a.max_pages;
    bool ok = true;
    for (int j = 0; j < n_blk && ok; ++j) {
      const int st = j % NSTAGE;
      const int lp = j * (BN / kPageSize) + (lane & 7);
      int pg = 0;
      if (lane < 8 && lp < npages) {
        pg = __ldg(bt_row + lp);
        if (pg < 0 || pg >= a.num_pages) {
          atomicOr(&g_err_prefill, kErrBadIndex);
          pg = 0;
        }
      }
      // lanes 0..7 hold the block's page ids; lane 0 needs them all
      int rowk[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        rowk[i] = (__shfl_sync(0xffffffffu, pg, i) * a.num_kv_heads + hkv) * kPageSize;
      const int nload = min(BN / kPageSize, npages - j * (BN / kPageSize));
      const uint32_t bytes = (uint32_t)nload * 2u * (kPageSize * 64 * 2);
      if (j >= NSTAGE && !(ok = wait_bar(bar(BAR_KE + st), ((j / NSTAGE) - 1) & 1, abort_flag)))
        break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(BAR_KF + st), bytes);
        const uint32_t dst = base_s + OFF_K + st * TILE;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (i < nload) {
            tma_load_2d(dst + i * 2048, &tk, 0, rowk[i], bar(BAR_KF + st));
            tma_load_2d(dst + HALF + i * 2048, &tk, 64, rowk[i], bar(BAR_KF + st));
          }
        }
      }
      (st == 0 ? last_k0 : last_k1) = j;
      if (j >= NSTAGE && !(ok = wait_bar(bar(BAR_VE + st), ((j / NSTAGE) - 1) & 1, abort_flag)))
        break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(BAR_VF + st), bytes);
        const uint32_t dst = base_s + OFF_V + st * TILE;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (i < nload) {
            tma_load_2d(dst + i * 2048, &tv, 0, rowk[i], bar(BAR_VF + st));
            tma_load_2d(dst + HALF + i * 2048, &tv, 64, rowk[i], bar(BAR_VF + st));
          }
        }
      }
      (st == 0 ? last_v0 : last_v1) = j;
    }
  } else if (warp == WARP_MMA) {
    // ------------------------------------------------------- MMA issuer
    // Iteration j: PV_A(j-1), QK_A(j), PV_B(j-1), QK_B(j).  While softmax A
    // works on S_A(j) the tensor core runs PV_B(j-1) and QK_B(j), and the
    // other way round.  QK_x(j) overwrites S_x, which holds P_x(j-1): it is
    // issued after PV_x(j-1), and MMAs of one thread run in issue order.
    bool ok = wait_bar(bar(BAR_Q), 0, abort_flag);
    for (int j = 0; j <= n_blk && ok; ++j) {
      const bool has_qk = j < n_blk;
      const int st = j % NSTAGE, pst = (j + NSTAGE - 1) % NSTAGE;
      if (has_qk && !(ok = wait_bar(bar(BAR_KF + st), (j / NSTAGE) & 1, abort_flag))) break;
      if (j >= 1) {
        if (!(ok = wait_bar(bar(BAR_VF + pst), ((j - 1) / NSTAGE) & 1, abort_flag))) break;
        const int kbase = (j - 1) * BN;
        if (kbase + BN > L) {
          // zero V rows at positions >= L (both 64-channel halves of each row)
          const int first = L - kbase;
          uint8_t* vt = base + OFF_V + pst * TILE;
          for (int idx = lane; idx < (BN - first) * 16; idx += 32) {
            const int row = first + (idx >> 4), c = idx & 15;
            *reinterpret_cast<uint4*>(vt + (c >> 3) * HALF + row * 128 + (c & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_async_smem();
          __syncwarp();
        }
      }
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int nbx = x == 0 ? nblk_a : nblk_b;
        if (j >= 1 && j - 1 < nbx) {
          if (!(ok = wait_bar(bar(BAR_PF + x), (j - 1) & 1, abort_flag))) break;
          tc_fence_after();
          if (lane == 0) {
            const uint32_t v_s = base_s + OFF_V + pst * TILE;
            mma8_pv_ts(tmem + tm_o(x), tmem + tm_p(x), desc_mnmajor(v_s), IDESC_PV,
                       j > 1 ? 1u : 0u);
            if (j - 1 == nbx - 1) mma_commit(bar(BAR_OD + x));
          }
          __syncwarp();
        }
        if (has_qk && j < nbx) {
          tc_fence_after();
          if (lane == 0) {
            const uint32_t q_s = base_s + OFF_Q + x * TILE, k_s = base_s + OFF_K + st * TILE;
            mma8_qk(tmem + tm_s(x), desc_kmajor(q_s), desc_kmajor(k_s), IDESC_QK);
            mma_commit(bar(BAR_SF + x));
          }
          __syncwarp();
        }
      }
      if (!ok) break;
      if (lane == 0) {
        if (has_qk) mma_commit(bar(BAR_KE + st));
        if (j >= 1) mma_commit(bar(BAR_VE + pst));
      }
      __syncwarp();
    }
    // drain: every MMA issued above completes before TMEM is released
    if (lane == 0) mma_commit(bar(BAR_DR));
    __syncwarp();
    (void)mbar_wait(bar(BAR_DR), 0);
  } else {
    // ---------------------------------------------------------- softmax
    const int x = warp >> 2;                      // tile: 0 = A, 1 = B
    const int quarter = warp & 3;                 // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane;            // row of the tile
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    const int rows = rows_of(x);
    const int pos_min = pmin_of(x);
    const int n_x = x == 0 ? nblk_a : nblk_b;
    const int pos_r = min(pos_min + r, L - 1);    // padding rows clamp to the last key
    const bool row_valid = r < rows;
    const int qrow0 = q0 + row0 + x * BM;         // chunk row of tile row 0

    // Q tile -> swizzled shared memory (rows past the chunk are zero).
    {
      const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(a.q);
      uint8_t* qs = base + OFF_Q + x * TILE;
      for (int it = 0; it < 16; ++it) {
        const int row = quarter * 32 + 2 * it + (lane >> 4);
        const int c = lane & 15;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row < rows)
          v = __ldg(reinterpret_cast<const uint4*>(
                        qg + ((size_t)(qrow0 + row) * Hq + hq) * kHeadDim) + c);
        *reinterpret_cast<uint4*>(qs + (c >> 3) * HALF + row * 128 + (((c & 7) ^ (row & 7)) << 4)) =
            v;
      }
      fence_async_smem();
      mbar_arrive(bar(BAR_Q));
    }

    const float sl2 = a.softmax_scale * kLog2e;
    const float2 sl2x2 = make_float2(sl2, sl2);
    float m_run = -INFINITY, l_run = 0.f;        // running max (scaled, log2 domain), sum
    bool ok = true;
    for (int j = 0; j < n_x; ++j) {
      if (!(ok = wait_bar(bar(BAR_SF + x), j & 1, abort_flag))) break;
      tc_fence_after();
      // The whole S row in one round trip (two 64-column loads, one wait);
      // packed P then overwrites the S registers it came from (c <= 2c) and
      // goes to TMEM columns 64..127 of S_x, which are consumed by then.
      const int kbase = j * BN;
      uint32_t sr[128];
      tmem_ld64(t_lane + tm_s(x), *reinterpret_cast<uint32_t(*)[64]>(&sr[0]));
      tmem_ld64(t_lane + tm_s(x) + 64, *reinterpret_cast<uint32_t(*)[64]>(&sr[64]));
      tmem_wait_ld();
      if (kbase + BN - 1 > pos_min) {             // block crosses the causal edge
        const int lim = pos_r - kbase;
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c > lim) sr[c] = __float_as_uint(-INFINITY);
      }
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < BN; c += 2)
        mx[(c >> 1) & 3] = fmax3(mx[(c >> 1) & 3], __uint_as_float(sr[c]),
                                 __uint_as_float(sr[c + 1]));
      const float m_blk = fmax3(mx[0], mx[1], fmaxf(mx[2], mx[3])) * sl2;
      const float m_new = fmaxf(m_run, m_blk);
      const bool need = m_new > m_run + 8.0f;     // lazy rescale threshold (2^8)
      const float m_use = need ? m_new : m_run;
      const float alpha = need ? fast_exp2(m_run - m_use) : 1.0f;
      const float2 negm = make_float2(-m_use, -m_use);
      float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int c = 0; c < BN / 2; ++c) {
        const float2 t = fma2(make_float2(__uint_as_float(sr[2 * c]),
                                          __uint_as_float(sr[2 * c + 1])), sl2x2, negm);
        const float2 pp = make_float2(fast_exp2(t.x), fast_exp2(t.y));
        sum2[c & 1] = add2(sum2[c & 1], pp);
        sr[c] = pack_bf16x2(pp.x, pp.y);
      }
      tmem_st64(t_lane + tm_p(x), *reinterpret_cast<const uint32_t(*)[64]>(&sr[0]));
      const float2 s2 = add2(sum2[0], sum2[1]);
      l_run = l_run * alpha + (s2.x + s2.y);
      m_run = m_use;

      // O rescale: S_x(j) complete implies PV_x(j-1) complete (one thread
      // issues both, in order), so O_x is stable here.
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll 1
        for (int h = 0; h < 4; ++h) {
          uint32_t o[32];
          tmem_ld32(t_lane + tm_o(x) + 32 * h, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 v = mul2(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), a2);
            o[i] = __float_as_uint(v.x);
            o[i + 1] = __float_as_uint(v.y);
          }
          tmem_st32(t_lane + tm_o(x) + 32 * h, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(BAR_PF + x));
    }

    if (ok && n_x > 0 && wait_bar(bar(BAR_OD + x), 0, abort_flag)) {
      tc_fence_after();
      const float inv = 1.0f / l_run;
      const size_t orow = ((size_t)(qrow0 + r) * Hq + hq) * kHeadDim;
      uint4* og = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + orow);
#pragma unroll 1
      for (int h = 0; h < 4; ++h) {
        uint32_t o[32];
        tmem_ld32(t_lane + tm_o(x) + 32 * h, o);
        tmem_wait_ld();
        if (row_valid) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[8 * k + 0]) * inv, __uint_as_float(o[8 * k + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(o[8 * k + 2]) * inv, __uint_as_float(o[8 * k + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(o[8 * k + 4]) * inv, __uint_as_float(o[8 * k + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(o[8 * k + 6]) * inv, __uint_as_float(o[8 * k + 7]) * inv);
            og[4 * h + k] = v;
          }
        }
      }
      if (row_valid && a.lse)
        a.lse[(size_t)(qrow0 + r) * Hq + hq] = (m_run + fast_log2(l_run)) * kLn2;
    }
  }

  // Every role has left its loop.  After an abort, loads may still be in
  // flight: the producer lets each one land before the CTA can exit.
  __syncthreads();
  if (warp == WARP_TMA && *abort_flag) {
    if (last_k0 >= 0) (void)mbar_wait(bar(BAR_KF + 0), (last_k0 / NSTAGE) & 1);
    if (last_k1 >= 0) (void)mbar_wait(bar(BAR_KF + 1), (last_k1 / NSTAGE) & 1);
    if (last_v0 >= 0) (void)mbar_wait(bar(BAR_VF + 0), (last_v0 / NSTAGE) & 1);
    if (last_v1 >= 0) (void)mbar_wait(bar(BAR_VF + 1), (last_v1 / NSTAGE) & 1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS)
                 : "memory");
  }
}

// cuTensorMapEncodeTiled, fetched through the runtime (no libcuda link).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// The pool as a 2-D bf16 tensor of (num_pages * Hkv * 16) rows of 128
// channels; a box is one page slab (16 rows) by 64 channels, 128B-swizzled.
bool encode_pool_map(CUtensorMap* m, const void* base, int num_pages, int hkv) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)num_pages * hkv * kPageSize};
  cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kPageSize};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace pkv_host {

cudaError_t launch_prefill(const PrefillLaunch& a, cudaStream_t s) {
  if ((long long)a.num_pages * a.num_kv_heads * kPageSize >= (1ll << 31))
    return cudaErrorNotSupported;
  CUtensorMap tk, tv;
  if (!encode_pool_map(&tk, a.k, a.num_pages, a.num_kv_heads) ||
      !encode_pool_map(&tv, a.v, a.num_pages, a.num_kv_heads))
    return cudaErrorInvalidValue;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  PrefillParams prm{a, (a.max_q_len + 2 * BM - 1) / (2 * BM)};
  dim3 grid(a.num_q_heads, prm.n_pairs, a.batch);
  prefill_kernel<<<grid, NUM_THREADS, SMEM_BYTES, s>>>(tk, tv, prm);
  return cudaGetLastError();
}

uint32_t take_prefill_error(cudaStream_t s) {
  uint32_t h = 0, zero = 0;
  if (cudaMemcpyFromSymbolAsync(&h, g_err_prefill, sizeof h, 0, cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return ~0u;
  cudaStreamSynchronize(s);
  if (h) cudaMemcpyToSymbolAsync(g_err_prefill, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s);
  cudaStreamSynchronize(s);
  return h;
}

}  // namespace pkv_host
