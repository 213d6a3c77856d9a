// prefill.cu -- causal chunked prefill attention over the paged cache on the
// 5th-generation tensor cores (tcgen05 MMAs, TMEM accumulators, TMA loads).
//
// The method: TileInfer.jl "Performance" page -- paged flash attention runs
// an online softmax over the pages read in place through the block table
// ("Fused kernels, FlashAttention and PagedAttention"); the prefill kernel
// runs a block of query rows per head over every page ("Attention for verify
// steps"); chunked prefill attends a chunk of new rows to the cached prefix
// ("What is left to gain").  Rows sit bottom-right: row i of a chunk of q
// rows in a sequence of L cached positions is position L - q + i and sees
// keys 0..it.
//
// Persistent kernel, one CTA per SM, 10 warps:
//   warps 0-3  softmax of query tile A, warps 4-7 of tile B (thread = query
//              row = TMEM lane): read S with tcgen05.ld, keep the running
//              max and sum of the row, write P (bf16) back into TMEM over the
//              consumed half of S, rescale O in TMEM only when the max grows
//              by more than 2^8 (exact: the final normalisation uses the same
//              stale max), and finish each unit of work;
//   warp 8     producer and scheduler: walks this CTA's share of the work,
//              publishes one descriptor per segment in a 2-entry shared ring,
//              and loads Q tiles (TMA, per segment) and 128-key K and V blocks
//              (TMA, eight 16-row page boxes per 64-channel half, 128-byte
//              swizzled, 2-stage ring per operand);
//   warp 9     MMA issuer (one thread): S_x = Q_x K^T and O_x += P_x V for the
//              two tiles in ping-pong, so that the tensor core works on one
//              tile while the softmax warps work on the other.
// V rows at positions >= L in the last block are zeroed before the PV MMA,
// so stale or poisoned pool slots never reach the accumulator (P is 0 there,
// but 0 * NaN is NaN).
//
// Work split: see "Work decomposition" below.  A unit of work cut between
// CTAs is finished by the CTA holding its last blocks: every other part is
// written (normalised O, log2-domain lse) to the caller's workspace and
// counted in a per-unit counter there; that CTA waits (bounded) for the
// count, merges the parts with its own by the log-sum-exp rule ("Split-KV
// decoding") and resets the counter to zero for the next call.  The kernel
// has two builds: with the template flag HP, a unit whose second row tile
// is past the chunk may hold the same rows of two query heads instead; the
// host picks the build per launch.
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
// Work is measured in tile-blocks (one 128 x 128 QK^T and PV of one tile).
// A unit also costs kUnitCost0 for starting and finishing it (Q load,
// pipeline fill and drain, epilogue), and each CTA gets at least kMinCost.
constexpr int kUnitCost0 = 4;
constexpr int kMinCost = 2 * kUnitCost0;
// CTAs cut units (split mode) when whole units would finish later than an
// even share plus kSplitGain, the cost of storing and merging cut parts.
// Whole units end no earlier than the largest unit, nor than ceil(units / P)
// units of average cost on the most loaded CTA.
constexpr int kSplitGain = 24;
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
// barriers (pairs are per tile or per ring slot): q_full, q_empty, ld (the
// loads of one phase have landed), xe (the MMAs that read a phase's
// buffers are done), s_full, p_full, o_done, drain, seg_full, seg_empty,
// and per tile for a cut unit: st (the tile's 4 warps have stored their
// part), go (every other part is counted: merge)
constexpr int BAR_QF = 0, BAR_QE = 2, BAR_LD = 4, BAR_XE = 6,
              BAR_SF = 12, BAR_PF = 14, BAR_OD = 16, BAR_DR = 18, BAR_SEGF = 19,
              BAR_SEGE = 21, BAR_ST = 23, BAR_GO = 25, NUM_BARS = 27;
constexpr int NSEG = 2;                       // segment descriptor ring depth
constexpr int OFF_SEG = OFF_BAR + 256;        // after the barriers (27 x 8 bytes)
constexpr int OFF_MISC = OFF_SEG + NSEG * 64;
constexpr int SMEM_BYTES = OFF_MISC + 32 + 1024;   // + alignment slack
static_assert(NUM_BARS * 8 <= 256, "barrier area");
constexpr int SLOT_ROWS = 2 * BM;             // rows of one workspace slot (both tiles)

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

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
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

// The same wait for a single thread (no warp vote).
__device__ __forceinline__ bool wait_bar1(uint32_t bar, uint32_t parity, volatile uint32_t* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        *abort = 1u;
        atomicOr(&g_err_prefill, kErrTimeout);
        return false;
      }
    }
  }
}

// Adds to a counter in global memory after every write this thread has seen
// (including other threads' writes ordered before it by a CTA barrier).
__device__ __forceinline__ void red_release_add(uint32_t* ctr, uint32_t v) {
  asm volatile("fence.acq_rel.gpu;\n\tred.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(ctr), "r"(v)
               : "memory");
}

// Bounded wait (one thread) until a counter in global memory reaches target;
// gpu-scope acquire, so what was written before the count is visible after.
__device__ __forceinline__ bool wait_count(const uint32_t* ctr, uint32_t target,
                                           volatile uint32_t* abort) {
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v >= target) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      *abort = 1u;
      atomicOr(&g_err_prefill, kErrTimeout);
      return false;
    }
    __nanosleep(64);
  }
}

// ------------------------------------------------------------------
// Work decomposition (persistent CTAs, "stream-K" style).
//
// A unit is (sequence b, pair p of 128-row query tiles, query head hq); its
// key blocks j = 0 .. nblk-1 cost one tile-block per tile that needs the
// block (tile A needs blocks 0 .. nblk_a-1, tile B 0 .. nblk_b-1; nblk_b is
// nblk_a or nblk_a + 1, or 0 when the pair's second tile is past the chunk),
// plus kUnitCost0 in front of block 0 for starting and finishing the unit.
// When the second tile is past the chunk (a chunk of at most 128 rows, or
// its odd last tile) and the query heads of a KV head come in pairs (G
// even), the unit instead holds the same rows for heads 2u and 2u + 1, which
// read the same K/V: tile B is the next head, not the next 128 rows, and the
// pair has Hq / 2 units.
// Units are ordered by sequence, pairs from the last (heaviest) down, heads
// innermost (the query heads of a KV head are neighbours, so they share K/V
// through L2).  The total cost W is cut into Pe equal ranges, one per active
// CTA (Pe = the grid, or fewer so that each range holds at least kMinCost);
// a block belongs to the CTA whose range holds the block's starting cost
// position.  A range is at least 2 long and the block starts of a unit are
// at most 2 apart, so the CTAs holding parts of one unit are consecutive,
// cf .. cl; and since kMinCost exceeds the largest gap between block starts
// (kUnitCost0 + 2), every active CTA has work.
//
// Whether units are cut at all follows from W, the largest unit and the
// number of units (kSplitGain above); when they are not, CTAs take whole
// units in a snake order.
//
// Each CTA walks its range backwards (units from its last position down),
// so that for a unit cut between CTAs the part in CTA cl (the unit's last
// blocks) is the last segment cl runs, while the part in any lower CTA k is
// the first segment k runs.  CTA k < cl stores its part (normalised O and
// log2-domain lse) in its workspace slot k and counts it; CTA cl, at the end
// of its walk, waits until the cl - cf other parts are counted (they were
// finished long before, by CTAs that started no later than it), then merges
// them with its own part straight from TMEM and resets the count.  Waiting
// only on lower CTAs, which the hardware starts first, keeps the wait safe
// even if the grid were not resident all at once (it is: one CTA per SM).

struct PairGeom {
  int q0, q_len, L, row0, rows_a, rows_b, pmin_a, nblk_a, nblk_b, nblk;
  int nd;                       // blocks both tiles need (cost 2 each); the rest cost 1
  int hpu;                      // heads per unit: 1 (tile B = next rows), 2 (= next head)
};

__device__ __forceinline__ bool seq_valid(const pkv_host::PrefillLaunch& a, int q0, int q_len,
                                          int L) {
  return q0 >= 0 && q_len >= 0 && q0 <= a.total_q - q_len && L >= q_len &&
         L <= a.max_pages * kPageSize;
}

__device__ __forceinline__ int n_pairs_of(int q_len) { return (q_len + 2 * BM - 1) / (2 * BM); }

// The query heads of a KV head come in pairs (G even): units may pair heads.
__device__ __forceinline__ bool heads_pair(const pkv_host::PrefillLaunch& a) {
  return (a.num_q_heads / a.num_kv_heads) % 2 == 0;
}

__device__ __forceinline__ PairGeom pair_geom(int q0, int q_len, int L, int p, bool hp) {
  PairGeom g;
  g.q0 = q0;
  g.q_len = q_len;
  g.L = L;
  g.row0 = p * 2 * BM;
  g.rows_a = max(0, min(BM, q_len - g.row0));
  g.rows_b = max(0, min(BM, q_len - g.row0 - BM));
  g.hpu = 1;
  if (hp && g.rows_b == 0 && g.rows_a > 0) {     // tile B: the same rows, the next head
    g.hpu = 2;
    g.rows_b = g.rows_a;
  }
  g.pmin_a = L - q_len + g.row0;
  g.nblk_a = g.rows_a > 0 ? (g.pmin_a + g.rows_a - 1) / BN + 1 : 0;
  g.nblk_b = g.rows_b > 0 ? (g.pmin_a + (g.hpu == 2 ? 0 : BM) + g.rows_b - 1) / BN + 1 : 0;
  g.nblk = max(g.nblk_a, g.nblk_b);
  g.nd = min(g.nblk_a, g.nblk_b);
  return g;
}

__device__ __forceinline__ int unit_cost(const PairGeom& g) {
  return kUnitCost0 + g.nblk_a + g.nblk_b;
}
// units of a pair of row tiles: one per head, or per head pair
__device__ __forceinline__ int units_of(const pkv_host::PrefillLaunch& a, const PairGeom& g) {
  return a.num_q_heads / g.hpu;
}
// cost offset of block j within its unit (the unit's fixed cost comes first)
__device__ __forceinline__ int block_off(const PairGeom& g, int j) {
  return kUnitCost0 + (j <= g.nd ? 2 * j : 2 * g.nd + (j - g.nd));
}
// first block whose starting offset is >= off (nblk if none)
__device__ __forceinline__ int first_block_at(const PairGeom& g, long long off) {
  if (off <= kUnitCost0) return 0;
  off -= kUnitCost0;
  const long long j = off <= 2 * g.nd ? (off + 1) / 2 : g.nd + (off - 2 * g.nd);
  return j < g.nblk ? (int)j : g.nblk;
}

// a * b / c for non-negative a * b < 2^63, in 32-bit arithmetic when it fits
__device__ __forceinline__ long long muldiv(long long a, long long b, long long c) {
  const unsigned long long p = (unsigned long long)a * (unsigned long long)b;
  if (p < (1ull << 32) && (unsigned long long)c < (1ull << 32))
    return (long long)((uint32_t)p / (uint32_t)c);
  return (long long)(p / (unsigned long long)c);
}

// Cost of sequence b's units (all heads); umax: the largest unit's cost so
// far; nunits: units so far.
__device__ __forceinline__ long long seq_cost(const pkv_host::PrefillLaunch& a, int b, int& umax,
                                              long long& nunits, bool hp) {
  const int q0 = a.cu_q[b];
  const int q_len = a.cu_q[b + 1] - q0;
  const int L = a.seq_lens[b];
  if (!seq_valid(a, q0, q_len, L)) {
    atomicOr(&g_err_prefill, kErrBadIndex);
    return 0;
  }
  long long c = 0;
  for (int p = 0; p < n_pairs_of(q_len); ++p) {
    const PairGeom g = pair_geom(q0, q_len, L, p, hp);
    const int u = unit_cost(g);
    c += (long long)u * units_of(a, g);
    nunits += units_of(a, g);
    umax = max(umax, u);
  }
  return c;
}

// Position of the work walk: unit (b, pair index pi, unit hq of the pair:
// query head hq, or heads 2 hq and 2 hq + 1 when g.hpu == 2).
struct Cursor {
  int b, pi, hq;
  long long ustart;             // cost position of the unit's first block
  PairGeom g;
  bool end;
};

__device__ __forceinline__ int pair_of(const Cursor& c) { return n_pairs_of(c.g.q_len) - 1 - c.pi; }

// Total cost W, the largest unit's cost and the number of units, by one
// warp (every lane gets all three).
__device__ __forceinline__ long long total_cost(const pkv_host::PrefillLaunch& a, int lane,
                                                int& umax, long long& nunits, bool hp) {
  long long t = 0;
  umax = 0;
  nunits = 0;
  for (int b = lane; b < a.batch; b += 32) t += seq_cost(a, b, umax, nunits, hp);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    t += __shfl_xor_sync(0xffffffffu, t, o);
    umax = max(umax, __shfl_xor_sync(0xffffffffu, umax, o));
    nunits += __shfl_xor_sync(0xffffffffu, nunits, o);
  }
  return t;
}

// The unit before the cursor's unit (end if none).
__device__ __forceinline__ void prev_unit(const pkv_host::PrefillLaunch& a, Cursor& c, bool hp) {
  if (c.hq > 0) {
    --c.hq;
    c.ustart -= unit_cost(c.g);
    return;
  }
  if (c.pi > 0) {
    --c.pi;
    c.g = pair_geom(c.g.q0, c.g.q_len, c.g.L, pair_of(c), hp);
    c.hq = units_of(a, c.g) - 1;
    c.ustart -= unit_cost(c.g);
    return;
  }
  for (int b = c.b - 1; b >= 0; --b) {
    const int q0 = a.cu_q[b], q_len = a.cu_q[b + 1] - q0, L = a.seq_lens[b];
    if (!seq_valid(a, q0, q_len, L) || q_len == 0) continue;
    c.b = b;
    c.pi = n_pairs_of(q_len) - 1;
    c.g = pair_geom(q0, q_len, L, 0, hp);
    c.hq = units_of(a, c.g) - 1;
    c.ustart -= unit_cost(c.g);
    return;
  }
  c.end = true;
}

// Moves the cursor n units forward (end if there are fewer).
__device__ __forceinline__ void skip_units(const pkv_host::PrefillLaunch& a, Cursor& c, int n,
                                           bool hp) {
  while (n > 0 && !c.end) {
    const int left = units_of(a, c.g) - c.hq;     // units left in this pair, this one included
    if (n < left) {
      c.hq += n;
      c.ustart += (long long)n * unit_cost(c.g);
      return;
    }
    n -= left;
    c.ustart += (long long)left * unit_cost(c.g);
    c.hq = 0;
    if (c.pi + 1 < n_pairs_of(c.g.q_len)) {
      ++c.pi;
      c.g = pair_geom(c.g.q0, c.g.q_len, c.g.L, pair_of(c), hp);
      continue;
    }
    int b = c.b + 1;
    for (; b < a.batch; ++b) {
      const int q0 = a.cu_q[b], q_len = a.cu_q[b + 1] - q0, L = a.seq_lens[b];
      if (!seq_valid(a, q0, q_len, L) || q_len == 0) continue;
      c.b = b;
      c.pi = 0;
      c.g = pair_geom(q0, q_len, L, n_pairs_of(q_len) - 1, hp);
      break;
    }
    if (b >= a.batch) c.end = true;
  }
}

// Cursor at the unit whose cost range holds pos (0 <= pos < W), by one warp
// (every lane gets the same cursor).
__device__ __forceinline__ Cursor locate_unit(const pkv_host::PrefillLaunch& a, long long pos,
                                              int lane,
                                              bool hp) {
  Cursor c;
  c.end = true;
  c.b = c.pi = c.hq = 0;
  c.ustart = 0;
  long long base = 0;
  int bf = -1;
  long long sb = 0;
  for (int b0 = 0; b0 < a.batch; b0 += 32) {
    const int b = b0 + lane;
    int um = 0;
    long long nu = 0;
    const long long cst = b < a.batch ? seq_cost(a, b, um, nu, hp) : 0;
    long long incl = cst;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const long long excl = incl - cst;
    const unsigned hit = __ballot_sync(0xffffffffu, b < a.batch && cst > 0 && base + incl > pos);
    if (hit) {
      const int src = __ffs(hit) - 1;
      bf = b0 + src;
      sb = base + __shfl_sync(0xffffffffu, excl, src);
      break;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (bf < 0) return c;
  const int q0 = a.cu_q[bf], q_len = a.cu_q[bf + 1] - q0, L = a.seq_lens[bf];
  long long p0 = sb;
  const int np = n_pairs_of(q_len);
  for (int pi = 0; pi < np; ++pi) {
    const PairGeom g = pair_geom(q0, q_len, L, np - 1 - pi, hp);
    const long long cbp = (long long)unit_cost(g) * units_of(a, g);
    if (pos < p0 + cbp) {
      c.b = bf;
      c.pi = pi;
      c.hq = (int)muldiv(pos - p0, 1, unit_cost(g));
      c.ustart = p0 + (long long)c.hq * unit_cost(g);
      c.g = g;
      c.end = false;
      break;
    }
    p0 += cbp;
  }
  return c;
}

__device__ __forceinline__ long long range_lo(long long W, int Pe, int k) { return muldiv(W, k, Pe); }
// the CTA whose range holds cost position pos
__device__ __forceinline__ int owner_of(long long W, int Pe, long long pos) {
  int k = (int)muldiv(pos, Pe, W);
  while (k + 1 < Pe && range_lo(W, Pe, k + 1) <= pos) ++k;
  return k;
}
__device__ __forceinline__ int active_ctas(long long W, int P) {
  const long long n = W / kMinCost;
  return (int)(n < 1 ? 1 : (n < P ? n : P));
}

// One segment as the producer publishes it to the other roles.
struct SegDesc {
  int qrow0;                    // q row of the unit's tile-A row 0
  int hq, L, pmin_a, rows_a, rows_b, nblk_a, nblk_b;
  int j0, j1;                   // blocks of this segment
  int cf, nown;                 // CTAs holding parts of the unit; nown == 1: all here
  int end;                      // no further segment
  int pmin_b, qrow_b, hq_b;     // tile B: first position, q row, head
};
static_assert(sizeof(SegDesc) == 64, "descriptor slot size");

struct PrefillParams {
  pkv_host::PrefillLaunch a;
  uint32_t* counters;           // [P][2] parts stored, per (first CTA of the unit, tile)
  float* ws_lse;                // [P slots][2 tiles][128] log2-domain lse of a stored part
  float4* ws_o;                 // [P slots][2 tiles][32 channel quads][128 rows] normalised O
};

template <bool HP>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                   const __grid_constant__ CUtensorMap tq, const __grid_constant__ PrefillParams prm) {
  const pkv_host::PrefillLaunch& a = prm.a;
  const int Hq = a.num_q_heads;
  const int G = Hq / a.num_kv_heads;
  const int P = gridDim.x, cta = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_s - raw_s);
  auto bar = [&](int i) -> uint32_t { return base_s + OFF_BAR + 8 * i; };
  SegDesc* seg_ring = reinterpret_cast<SegDesc*>(base + OFF_SEG);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(base + OFF_MISC + 4);

  // The producer warp plans this CTA's walk while the barriers and TMEM are
  // set up.  Split mode: the range is walked backwards, from the unit holding
  // its last position down to the unit holding lo; within a unit, blocks j0
  // .. j1-1 run in order.  Whole-unit mode: CTA c takes units c, 2P-1-c,
  // 2P+c, ... (heaviest first, snaking so that the CTAs that took the
  // heaviest units of one round take the lightest of the next).
  long long W = 0, lo = 0, hi = 0;
  bool split = false, hp = false;           // hp: units pair heads (HP builds only)
  int Pe = P;
  Cursor c;
  c.end = true;
  if (warp == WARP_TMA) {
    // the first sequence's block-table row (a CTA's first block may lie
    // anywhere in it), fetched into L2 while the walk is planned
    for (int e = lane * 32; e < a.max_pages; e += 32 * 32)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(a.block_table + e));
    // whole units' makespan vs the split share (in fp32: the products of
    // large launches would not fit 64 bits, and this is only an estimate;
    // fp64 is slow on this GPU)
    auto cut = [&](long long w, int um, long long n) {
      if (n <= 0) return false;
      const float per = (float)((n + P - 1) / P);
      const float whole = fmaxf((float)um, per * (float)w / (float)n);
      return whole > (float)w / (float)P + (float)kSplitGain;
    };
    int umax = 0;
    long long units = 0;
    if (HP && heads_pair(a)) {
      // Pair heads unless whole units of single heads would already leave
      // CTAs idle (then pairs would halve the CTAs at work).
      W = total_cost(a, lane, umax, units, false);
      hp = cut(W, umax, units) || units > P;
    }
    W = total_cost(a, lane, umax, units, hp);
    split = cut(W, umax, units);
    Pe = split ? active_ctas(W, P) : P;
    if (split && cta < Pe) {
      lo = range_lo(W, Pe, cta);
      hi = range_lo(W, Pe, cta + 1);
    }
    if (split) {
      if (lo < hi) c = locate_unit(a, hi - 1, lane, hp);
    } else if (W > 0) {
      c = locate_unit(a, 0, lane, hp);
      skip_units(a, c, cta, hp);
    }
  }

  if (threadIdx.x == 0) {
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(BAR_QF + x), 1);
      mbar_init(bar(BAR_QE + x), 1);
      mbar_init(bar(BAR_LD + x), 1);
      mbar_init(bar(BAR_XE + x), 1);
      mbar_init(bar(BAR_SF + x), 1);
      mbar_init(bar(BAR_PF + x), BM);
      mbar_init(bar(BAR_OD + x), 1);
      mbar_init(bar(BAR_SEGF + x), 1);
      mbar_init(bar(BAR_SEGE + x), 9);            // 8 softmax warps + the MMA warp
      mbar_init(bar(BAR_ST + x), 4);              // the tile's 4 softmax warps
      mbar_init(bar(BAR_GO + x), 1);
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

  static_assert(NSTAGE == 2, "the producer tracks two ring slots");
  // last armed load phase per ring slot and number of Q loads per tile (for
  // the drain after an abort)
  int last_ph0 = -1, last_ph1 = -1, nq_a = 0, nq_b = 0;
  if (warp == WARP_TMA) {
    // ------------------------------------------------ scheduler + producer
    bool ok = true;
    int ph = 0;                                   // load phases armed so far
    for (int sg = 0;; ++sg) {
      int j0 = 0, j1 = 0, cf = cta, nown = 1;
      if (split) {
        // the next unit (going down) with a block start in [lo, hi)
        while (!c.end) {
          j0 = first_block_at(c.g, lo - c.ustart);
          j1 = first_block_at(c.g, hi - c.ustart);
          if (j0 < j1) break;
          if (c.ustart <= lo) c.end = true;
          else prev_unit(a, c, hp);
        }
        if (!c.end) {
          cf = owner_of(W, Pe, c.ustart + block_off(c.g, 0));
          nown = owner_of(W, Pe, c.ustart + block_off(c.g, c.g.nblk - 1)) - cf + 1;
        }
      } else if (!c.end) {
        j1 = c.g.nblk;
      }
      const bool has = !c.end;
      const int ri = sg % NSEG;
      if (sg >= NSEG && !(ok = wait_bar(bar(BAR_SEGE + ri), ((sg / NSEG) - 1) & 1, abort_flag)))
        break;
      if (lane == 0) {
        SegDesc& d = seg_ring[ri];
        d.end = has ? 0 : 1;
        if (has) {
          d.qrow0 = c.g.q0 + c.g.row0;
          if (HP) {
            d.hq = c.hq * c.g.hpu;                // tile A's head
            // tile B: the next 128 rows, or (head pair) the same rows, next head
            d.pmin_b = c.g.pmin_a + (c.g.hpu == 2 ? 0 : BM);
            d.qrow_b = d.qrow0 + (c.g.hpu == 2 ? 0 : BM);
            d.hq_b = d.hq + (c.g.hpu == 2 ? 1 : 0);
          } else {
            d.hq = c.hq;
          }
          d.L = c.g.L;
          d.pmin_a = c.g.pmin_a;
          d.rows_a = c.g.rows_a;
          d.rows_b = c.g.rows_b;
          d.nblk_a = c.g.nblk_a;
          d.nblk_b = c.g.nblk_b;
          d.j0 = j0;
          d.j1 = j1;
          d.cf = cf;
          d.nown = nown;
        }
        mbar_arrive(bar(BAR_SEGF + ri));          // release: the fields above are visible
      }
      __syncwarp();
      if (!has) break;

      const int hkv = (HP ? c.hq * c.g.hpu : c.hq) / G;   // a head pair shares it
      const int npages = (c.g.L + kPageSize - 1) / kPageSize;
      const int32_t* bt_row = a.block_table + (size_t)c.b * a.max_pages;
      // Page ids of block j, one per lane 0..7 (0 past the sequence's pages).
      auto page_ids = [&](int j) -> int {
        const int lp = j * (BN / kPageSize) + lane;
        return (lane < BN / kPageSize && lp < npages) ? __ldg(bt_row + lp) : 0;
      };
      // Load phases.  Phase j of a segment (j = j0 .. j1) carries V of block
      // j - 1 (if j > j0) and K of block j (if j < j1), in ring slot ph % 2
      // of both the K and the V buffers: MMA iteration j reads exactly these
      // (PV(j - 1), then QK(j)) and frees them with one commit, so the slot
      // is refilled for phase ph + 2 once iteration j's MMAs are done.  One
      // barrier wait and one commit per iteration on the MMA thread, whose
      // every barrier operation stalls the tensor core.  Lane i < 8 loads
      // page i of a block (both 64-channel halves).
      // lane i: page i of blocks j - 1 and j, and of block j + 1 (read one
      // phase ahead, so that its latency overlaps this phase's wait)
      int pg_prev = 0, pg_cur = 0, pg_next = page_ids(j0);
      auto issue_phase = [&](int j) -> bool {
        const bool hv = j > j0, hk = j < j1;
        const int slot = ph & 1;
        pg_prev = pg_cur;
        if (hk) {
          int pg = pg_next;
          if (j + 1 < j1) pg_next = page_ids(j + 1);
          if (pg < 0 || pg >= a.num_pages) {
            atomicOr(&g_err_prefill, kErrBadIndex);
            pg = 0;
          }
          pg_cur = pg;
        }
        const int nk = hk ? min(BN / kPageSize, npages - j * (BN / kPageSize)) : 0;
        const int nv = hv ? min(BN / kPageSize, npages - (j - 1) * (BN / kPageSize)) : 0;
        const uint32_t bytes = (uint32_t)(nk + nv) * 2u * (kPageSize * 64 * 2);
        if (ph >= 2 && !wait_bar(bar(BAR_XE + slot), ((ph >> 1) - 1) & 1, abort_flag))
          return false;
        if (lane == 0) mbar_arrive_expect_tx(bar(BAR_LD + slot), bytes);
        __syncwarp();
        if (lane < nv) {
          const int row = (pg_prev * a.num_kv_heads + hkv) * kPageSize;
          const uint32_t dst = base_s + OFF_V + slot * TILE + lane * 2048;
          tma_load_2d(dst, &tv, 0, row, bar(BAR_LD + slot));
          tma_load_2d(dst + HALF, &tv, 64, row, bar(BAR_LD + slot));
        }
        if (lane < nk) {
          const int row = (pg_cur * a.num_kv_heads + hkv) * kPageSize;
          const uint32_t dst = base_s + OFF_K + slot * TILE + lane * 2048;
          tma_load_2d(dst, &tk, 0, row, bar(BAR_LD + slot));
          tma_load_2d(dst + HALF, &tk, 64, row, bar(BAR_LD + slot));
        }
        (slot == 0 ? last_ph0 : last_ph1) = ph;
        ++ph;
        return true;
      };
      // The segment's Q tiles, each once the previous segment's last QK of
      // that tile has completed.  They go after the segment's first phase
      // (K of its first block), so that they land while the previous
      // segment is still finishing.
      auto issue_q = [&]() -> bool {
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (sg > 0 && !wait_bar(bar(BAR_QE + x), (sg - 1) & 1, abort_flag)) return false;
          const int rows = x == 0 ? c.g.rows_a : c.g.rows_b;
          if (lane == 0) {
            if (rows > 0) {
              // rows past the end of q read as zeros; rows of the next
              // sequence only feed padding rows, whose results are never stored
              // tile B: the next 128 rows of the head, or (head pair) the
              // same rows of the next head
              const int row = c.g.q0 + c.g.row0 + (HP && c.g.hpu == 2 ? 0 : x * BM);
              const int head = HP ? c.hq * c.g.hpu + (c.g.hpu == 2 ? x : 0) : c.hq;
              const uint32_t dst = base_s + OFF_Q + x * TILE;
              mbar_arrive_expect_tx(bar(BAR_QF + x), (uint32_t)TILE);
              tma_load_3d(dst, &tq, 0, head, row, bar(BAR_QF + x));
              tma_load_3d(dst + HALF, &tq, 64, head, row, bar(BAR_QF + x));
            } else {
              mbar_arrive(bar(BAR_QF + x));
            }
          }
          (x == 0 ? nq_a : nq_b) = sg + 1;
        }
        return true;
      };
      // The first segment has nothing in flight: its Q goes out first.
      if (sg == 0 && !(ok = issue_q())) break;
      if (!(ok = issue_phase(j0))) break;
      if (sg > 0 && !(ok = issue_q())) break;
      for (int j = j0 + 1; j <= j1; ++j)
        if (!(ok = issue_phase(j))) break;
      if (!ok) break;
      if (split) {
        if (c.ustart <= lo) c.end = true;         // this unit opens the range: done
        else prev_unit(a, c, hp);
      } else {
        skip_units(a, c, (sg & 1) ? 2 * cta + 1 : 2 * P - 1 - 2 * cta, hp);
      }
    }
  } else if (warp == WARP_MMA) {
    // ------------------------------------------------------- MMA issuer
    // One thread (lane 0) runs this role; the other lanes wait at the end.
    // The tensor core takes MMAs only as fast as this thread issues them, so
    // nothing between two groups of eight may stall it: no warp votes or
    // syncs, and as few barrier waits as the dependencies allow.
    // Per segment, iteration j issues PV_A(j-1), QK_A(j), PV_B(j-1), QK_B(j).
    // While softmax A works on S_A(j) the tensor core runs PV_B(j-1) and
    // QK_B(j), and the other way round.  QK_x(j) overwrites S_x, which holds
    // P_x(j-1): it is issued after PV_x(j-1), and MMAs of one thread run in
    // issue order.  A segment's first QKs only touch S, so they overlap the
    // previous segment's epilogue, which reads O.  K(j) is waited for only
    // after PV_A(j-1) is issued: that PV does not need it and runs while K
    // lands.
    if (lane == 0) {
      bool ok = true;
      int ph = 0, cnt_a = 0, cnt_b = 0;            // load phases consumed, P tiles per tile
      for (int sg = 0;; ++sg) {
        const int ri = sg % NSEG;
        if (!(ok = wait_bar1(bar(BAR_SEGF + ri), (sg / NSEG) & 1, abort_flag))) break;
        const SegDesc& d = seg_ring[ri];
        const int end = d.end;
        const int j0 = d.j0, j1 = d.j1, L = d.L;
        const int je_a = min(j1, d.nblk_a), je_b = min(j1, d.nblk_b);
        if (end) break;
        mbar_arrive(bar(BAR_SEGE + ri));
        if (!(ok = wait_bar1(bar(BAR_QF + 0), sg & 1, abort_flag))) break;
        if (!(ok = wait_bar1(bar(BAR_QF + 1), sg & 1, abort_flag))) break;
        // a tile without QK in this segment releases its Q at once
        if (je_a <= j0) mma_commit(bar(BAR_QE + 0));
        if (je_b <= j0) mma_commit(bar(BAR_QE + 1));
        for (int j = j0; j <= j1 && ok; ++j, ++ph) {
          const bool has_qk = j < j1;
          const int slot = ph & 1;                  // V(j - 1) and K(j) of this phase
          if (!(ok = wait_bar1(bar(BAR_LD + slot), (ph >> 1) & 1, abort_flag))) break;
          if (j > j0) {
            const int kbase = (j - 1) * BN;
            if (kbase + BN > L) {
              // zero V rows at positions >= L (both 64-channel halves of each
              // row; rare: the last block of a sequence)
              const int first_row = L - kbase;
              uint8_t* vt = base + OFF_V + slot * TILE;
              for (int idx = 0; idx < (BN - first_row) * 16; ++idx) {
                const int row = first_row + (idx >> 4), cc = idx & 15;
                *reinterpret_cast<uint4*>(vt + (cc >> 3) * HALF + row * 128 + (cc & 7) * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
              }
              fence_async_smem();
            }
          }
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            const int jex = x == 0 ? je_a : je_b;
            int& cnt = x == 0 ? cnt_a : cnt_b;
            if (j > j0 && j - 1 < jex) {
              if (!(ok = wait_bar1(bar(BAR_PF + x), cnt & 1, abort_flag))) break;
              ++cnt;
              tc_fence_after();
              const uint32_t v_s = base_s + OFF_V + slot * TILE;
              mma8_pv_ts(tmem + tm_o(x), tmem + tm_p(x), desc_mnmajor(v_s), IDESC_PV,
                         j - 1 > j0 ? 1u : 0u);
              if (j == jex) mma_commit(bar(BAR_OD + x));
            }
            if (has_qk && j < jex) {
              tc_fence_after();
              const uint32_t q_s = base_s + OFF_Q + x * TILE, k_s = base_s + OFF_K + slot * TILE;
              mma8_qk(tmem + tm_s(x), desc_kmajor(q_s), desc_kmajor(k_s), IDESC_QK);
              mma_commit(bar(BAR_SF + x));
              if (j == jex - 1) mma_commit(bar(BAR_QE + x));
            }
          }
          if (!ok) break;
          mma_commit(bar(BAR_XE + slot));           // this phase's K and V are read
        }
        if (!ok) break;
      }
      // drain: every MMA issued above completes before TMEM is released
      mma_commit(bar(BAR_DR));
      (void)mbar_wait(bar(BAR_DR), 0);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- softmax
    // Per segment the block loop keeps only what it needs in registers; the
    // rest is read again from the segment's descriptor afterwards (it stays
    // valid until this warp releases it at the end of the segment).
    const int x = warp >> 2;                      // tile: 0 = A, 1 = B
    const int quarter = warp & 3;                 // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane;            // row of the tile
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    const float sl2 = a.softmax_scale * kLog2e;
    const float2 sl2x2 = make_float2(sl2, sl2);
    bool ok = true;
    // phase parities: s_full, o_done, st, go
    constexpr uint32_t PAR_S = 1, PAR_O = 2, PAR_ST = 4, PAR_GO = 8;
    uint32_t par = 0;
    for (int sg = 0;; ++sg) {
      const int ri = sg % NSEG;
      if (!(ok = wait_bar(bar(BAR_SEGF + ri), (sg / NSEG) & 1, abort_flag))) break;
      volatile const SegDesc* d = seg_ring + ri;
      auto release = [&]() {
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_SEGE + ri));
      };
      if (d->end) break;
      if ((x == 0 ? d->rows_a : d->rows_b) == 0) {   // second tile past the chunk: no work
        release();
        continue;
      }
      const int j0 = d->j0;
      const int jend = min(d->j1, x == 0 ? d->nblk_a : d->nblk_b);
      const int pos_min = HP ? (x == 0 ? d->pmin_a : d->pmin_b) : d->pmin_a + x * BM;
      const int pos_r = min(pos_min + r, d->L - 1);   // padding rows clamp to the last key

      // Running max (scaled, log2 domain) and sum.  The max starts finite and
      // far below any score: a row with no unmasked key yet (only when a
      // segment starts past block 0) then gets P = 2^(-inf + 1e30) = 0
      // instead of 2^(-inf + inf) = NaN, and its first real block rescales
      // by 2^(-1e30 - m) = 0.
      float m_run = -1e30f, l_run = 0.f;
      for (int j = j0; j < jend; ++j) {
        if (!(ok = wait_bar(bar(BAR_SF + x), par & PAR_S, abort_flag))) break;
        par ^= PAR_S;
        tc_fence_after();
        // The whole S row in one round trip; packed P then overwrites the S
        // registers it came from (c <= 2c) and goes to TMEM columns 64..127
        // of S_x, which are consumed by then: its first half (keys 0..63) as
        // soon as it is complete, so that the store overlaps the second.
        const int kbase = j * BN;
        uint32_t sr[128];
        tmem_ld64(t_lane + tm_s(x), *reinterpret_cast<uint32_t(*)[64]>(&sr[0]));
        tmem_ld64(t_lane + tm_s(x) + 64, *reinterpret_cast<uint32_t(*)[64]>(&sr[64]));
        tmem_wait_ld();
        if (kbase + BN - 1 > pos_min) {           // block crosses the causal edge
          const int lim = pos_r - kbase;
#pragma unroll
          for (int cc = 0; cc < BN; ++cc)
            if (cc > lim) sr[cc] = __float_as_uint(-INFINITY);
        }
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int cc = 0; cc < BN; cc += 2)
          mx[(cc >> 1) & 3] = fmax3(mx[(cc >> 1) & 3], __uint_as_float(sr[cc]),
                                    __uint_as_float(sr[cc + 1]));
        const float m_blk = fmax3(mx[0], mx[1], fmaxf(mx[2], mx[3])) * sl2;
        const float m_new = fmaxf(m_run, m_blk);
        const bool need = m_new > m_run + 8.0f;   // lazy rescale threshold (2^8)
        const float m_use = need ? m_new : m_run;
        const float alpha = need ? fast_exp2(m_run - m_use) : 1.0f;
        const float2 negm = make_float2(-m_use, -m_use);
        float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int cc = 0; cc < BN / 2; ++cc) {
          const float2 tv2 = fma2(make_float2(__uint_as_float(sr[2 * cc]),
                                              __uint_as_float(sr[2 * cc + 1])), sl2x2, negm);
          const float2 pp = make_float2(fast_exp2(tv2.x), fast_exp2(tv2.y));
          sum2[cc & 1] = add2(sum2[cc & 1], pp);
          sr[cc] = pack_bf16x2(pp.x, pp.y);
          if (cc == BN / 4 - 1)
            tmem_st32(t_lane + tm_p(x), *reinterpret_cast<const uint32_t(*)[32]>(&sr[0]));
        }
        tmem_st32(t_lane + tm_p(x) + 32, *reinterpret_cast<const uint32_t(*)[32]>(&sr[32]));
        const float2 s2 = add2(sum2[0], sum2[1]);
        l_run = l_run * alpha + (s2.x + s2.y);
        m_run = m_use;

        // O rescale: S_x(j) complete implies PV_x(j-1) complete (one thread
        // issues both, in order), so O_x is stable here.
        if (j > j0 && __any_sync(0xffffffffu, need)) {
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
      if (!ok) break;
      const bool own = jend > j0;                 // this segment saw keys of this tile
      if (own) {
        if (!(ok = wait_bar(bar(BAR_OD + x), (par & PAR_O) ? 1u : 0u, abort_flag))) break;
        par ^= PAR_O;
        tc_fence_after();
      }
      // q row of this tile's row 0, and its head
      const int qrow0 = HP ? (x == 0 ? d->qrow0 : d->qrow_b) : d->qrow0 + x * BM;
      const int hq = HP ? (x == 0 ? d->hq : d->hq_b) : d->hq;
      const int nown = d->nown;
      const bool row_valid = r < (x == 0 ? d->rows_a : d->rows_b);
      const float inv = 1.0f / l_run;
      if (nown == 1) {
        // ---- the whole unit ran here: normalise and store
        const size_t orow = ((size_t)(qrow0 + r) * Hq + hq) * kHeadDim;
        uint4* og = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + orow);
        uint32_t o[128];                          // the whole O row in one round trip
        tmem_ld64(t_lane + tm_o(x), *reinterpret_cast<uint32_t(*)[64]>(&o[0]));
        tmem_ld64(t_lane + tm_o(x) + 64, *reinterpret_cast<uint32_t(*)[64]>(&o[64]));
        tmem_wait_ld();
        if (row_valid) {
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[8 * k + 0]) * inv, __uint_as_float(o[8 * k + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(o[8 * k + 2]) * inv, __uint_as_float(o[8 * k + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(o[8 * k + 4]) * inv, __uint_as_float(o[8 * k + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(o[8 * k + 6]) * inv, __uint_as_float(o[8 * k + 7]) * inv);
            og[k] = v;
          }
        }
        if (row_valid && a.lse)
          a.lse[(size_t)(qrow0 + r) * Hq + hq] = (m_run + fast_log2(l_run)) * kLn2;
        release();
        continue;
      }

      // ---- one part of a unit cut between CTAs cf .. cl.  A CTA below cl
      // stores its part in its slot and counts it; CTA cl (this is its last
      // segment) waits for the count, then merges.
      const int cf = d->cf;
      const int cl = cf + nown - 1;
      uint32_t* ctr = prm.counters + 2 * cf + x;
      if (cta != cl) {
        const size_t prow = (size_t)(cta * 2 + x);
        if (own) {
          float4* wo = prm.ws_o + prow * 32 * BM + r;
          uint32_t o[128];                        // the whole O row in one round trip
          tmem_ld64(t_lane + tm_o(x), *reinterpret_cast<uint32_t(*)[64]>(&o[0]));
          tmem_ld64(t_lane + tm_o(x) + 64, *reinterpret_cast<uint32_t(*)[64]>(&o[64]));
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k)
            wo[k * BM] = make_float4(__uint_as_float(o[4 * k]) * inv, __uint_as_float(o[4 * k + 1]) * inv,
                                     __uint_as_float(o[4 * k + 2]) * inv, __uint_as_float(o[4 * k + 3]) * inv);
          prm.ws_lse[prow * BM + r] = m_run + fast_log2(l_run);
        } else {
          prm.ws_lse[prow * BM + r] = -INFINITY;  // no key of this tile in this part
        }
        // the tile's 4 warps have stored: one thread releases the count
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_ST + x));
        if (quarter == 0) {
          if (!(ok = wait_bar(bar(BAR_ST + x), (par & PAR_ST) ? 1u : 0u, abort_flag))) break;
          if (lane == 0) red_release_add(ctr, 1u);
        }
        par ^= PAR_ST;
        release();
        continue;
      }
      // the merging CTA: wait until the cl - cf other parts are counted
      if (quarter == 0 && lane == 0) {
        if (wait_count(ctr, (uint32_t)(nown - 1), abort_flag)) {
          *ctr = 0u;                              // ready for the next call
          mbar_arrive(bar(BAR_GO + x));
        }
      }
      __syncwarp();
      if (!(ok = wait_bar(bar(BAR_GO + x), (par & PAR_GO) ? 1u : 0u, abort_flag))) break;
      par ^= PAR_GO;
      // Parts of CTAs cf .. cl: slot k for k < cl, this CTA's own part from
      // TMEM.  Every part enters as the stored parts do (O / l rounded to
      // fp32, lse = m + log2 l), in CTA order.
      const float lse_own = own ? m_run + fast_log2(l_run) : -INFINITY;
      auto part_lse = [&](int k) -> float {
        if (k == cta) return lse_own;
        return __ldcg(prm.ws_lse + (size_t)(k * 2 + x) * BM + r);
      };
      float M = -INFINITY;
#pragma unroll 4
      for (int k = cf; k < cf + nown; ++k) M = fmaxf(M, part_lse(k));
      // a part without keys of this row has lse -inf (weight 0) and no O
      auto weight = [&](float ls) { return ls == -INFINITY ? 0.f : fast_exp2(ls - M); };
      float sum = 0.f;
#pragma unroll 4
      for (int k = cf; k < cf + nown; ++k) sum += weight(part_lse(k));
      const size_t orow = ((size_t)(qrow0 + r) * Hq + hq) * kHeadDim;
      uint4* og = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + orow);
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {             // 64 channels at a time
        float acc[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) acc[i] = 0.f;
        for (int k = cf; k < cf + nown; ++k) {
          const float f = weight(part_lse(k));
          if (k == cta) {
            if (own) {                            // warp-uniform
              uint32_t o[64];
              tmem_ld64(t_lane + tm_o(x) + 64 * h, o);
              tmem_wait_ld();
              // f == 0: no key of this row in this part (l = 0, O / l = NaN)
              if (f != 0.f) {
#pragma unroll
                for (int i = 0; i < 64; ++i) acc[i] = fmaf(f, __uint_as_float(o[i]) * inv, acc[i]);
              }
            }
          } else {
            const size_t pk = (size_t)(k * 2 + x);
            float4 v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __ldcg(prm.ws_o + (pk * 32 + 16 * h + i) * BM + r);
            if (f != 0.f) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                acc[4 * i + 0] = fmaf(f, v[i].x, acc[4 * i + 0]);
                acc[4 * i + 1] = fmaf(f, v[i].y, acc[4 * i + 1]);
                acc[4 * i + 2] = fmaf(f, v[i].z, acc[4 * i + 2]);
                acc[4 * i + 3] = fmaf(f, v[i].w, acc[4 * i + 3]);
              }
            }
          }
        }
        const float is = sum > 0.f ? 1.0f / sum : 0.f;
        if (row_valid) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            uint4 w;
            w.x = pack_bf16x2(acc[8 * i + 0] * is, acc[8 * i + 1] * is);
            w.y = pack_bf16x2(acc[8 * i + 2] * is, acc[8 * i + 3] * is);
            w.z = pack_bf16x2(acc[8 * i + 4] * is, acc[8 * i + 5] * is);
            w.w = pack_bf16x2(acc[8 * i + 6] * is, acc[8 * i + 7] * is);
            og[8 * h + i] = w;
          }
        }
      }
      if (row_valid && a.lse)
        a.lse[(size_t)(qrow0 + r) * Hq + hq] = sum > 0.f ? (M + fast_log2(sum)) * kLn2 : -INFINITY;
      release();
    }
  }

  // Every role has left its loop.  After an abort, loads may still be in
  // flight: the producer lets each one land before the CTA can exit.
  __syncthreads();
  if (warp == WARP_TMA && *abort_flag) {
    if (last_ph0 >= 0) (void)mbar_wait(bar(BAR_LD + 0), (last_ph0 >> 1) & 1);
    if (last_ph1 >= 0) (void)mbar_wait(bar(BAR_LD + 1), (last_ph1 >> 1) & 1);
    if (nq_a > 0) (void)mbar_wait(bar(BAR_QF + 0), (nq_a - 1) & 1);
    if (nq_b > 0) (void)mbar_wait(bar(BAR_QF + 1), (nq_b - 1) & 1);
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

// q [total_q][Hq][128] as a 3-D bf16 tensor (channel, head, row); a box is
// 64 channels of one head over 128 rows, 128B-swizzled: one half of a query
// tile in the K-major layout the QK MMA reads.  Rows past total_q read as 0.
bool encode_q_map(CUtensorMap* m, const void* q, int total_q, int hq) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)hq, (cuuint64_t)total_q};
  cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)hq * kHeadDim * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)BM};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Self-test of the bounded-wait error path: one thread waits, with the wait
// a merging CTA uses, for a counter that nothing will raise.
__global__ void bounded_wait_selftest_kernel(const uint32_t* ctr, uint32_t target) {
  __shared__ uint32_t abort_flag;
  abort_flag = 0u;
  (void)wait_count(ctr, target, &abort_flag);
}

}  // namespace

namespace pkv_host {

cudaError_t launch_wait_selftest(const uint32_t* counter, uint32_t target, cudaStream_t s) {
  bounded_wait_selftest_kernel<<<1, 1, 0, s>>>(counter, target);
  return cudaGetLastError();
}

bool encode_bf16_pool_map(void* map, const void* base, int num_pages, int hkv) {
  return encode_pool_map(static_cast<CUtensorMap*>(map), base, num_pages, hkv);
}

// An INT8 pool as a 2-D uint8 tensor of (num_pages * Hkv * 16) rows of 128
// bytes; a box is one (page, head) slab of 16 rows, 128B-swizzled (the INT8
// decode kernel reads it).
bool encode_int8_slab_map(void* map, const void* base, int num_pages, int hkv) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)num_pages * hkv * kPageSize};
  cuuint64_t strides[1] = {(cuuint64_t)kHeadDim};
  cuuint32_t box[2] = {(cuuint32_t)kHeadDim, (cuuint32_t)kPageSize};
  cuuint32_t estr[2] = {1, 1};
  return fn(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace pkv_host

namespace {

// Workspace: per-(CTA, tile) part counters, then the parts' lse, then their O.
size_t ws_counter_bytes(int ctas) { return ((size_t)2 * ctas * 4 + 255) / 256 * 256; }
size_t ws_lse_bytes(int ctas) { return (size_t)ctas * SLOT_ROWS * 4; }

}  // namespace

namespace pkv_host {

cudaError_t launch_prefill(const PrefillLaunch& a, cudaStream_t s) {
  if ((long long)a.num_pages * a.num_kv_heads * kPageSize >= (1ll << 31))
    return cudaErrorNotSupported;
  CUtensorMap tk, tv, tq;
  if (!encode_pool_map(&tk, a.k, a.num_pages, a.num_kv_heads) ||
      !encode_pool_map(&tv, a.v, a.num_pages, a.num_kv_heads) ||
      !encode_q_map(&tq, a.q, a.total_q, a.num_q_heads))
    return cudaErrorInvalidValue;
  for (auto fn : {prefill_kernel<false>, prefill_kernel<true>}) {
    cudaError_t e = pkv_host::set_max_dynamic_smem(reinterpret_cast<const void*>(fn), SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  if (a.ctas <= 0 || a.ctas > a.ws_ctas || a.ws_ctas > kMaxPrefillCtas || !a.workspace)
    return cudaErrorInvalidValue;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  const int n = a.ws_ctas;
  PrefillParams prm{a, reinterpret_cast<uint32_t*>(ws),
                    reinterpret_cast<float*>(ws + ws_counter_bytes(n)),
                    reinterpret_cast<float4*>(ws + ws_counter_bytes(n) + ws_lse_bytes(n))};
  // The head-pair build (units of two heads on one row tile) only where a
  // chunk ends in a single row tile: max_q_len tells it exactly for one
  // sequence and is a proxy for a batch; either build is correct for any
  // launch, the other one is a little faster where no unit pairs heads.
  const bool hp = (a.num_q_heads / a.num_kv_heads) % 2 == 0 && a.max_q_len % (2 * BM) != 0 &&
                  a.max_q_len % (2 * BM) <= BM;
  if (hp)
    prefill_kernel<true><<<a.ctas, NUM_THREADS, SMEM_BYTES, s>>>(tk, tv, tq, prm);
  else
    prefill_kernel<false><<<a.ctas, NUM_THREADS, SMEM_BYTES, s>>>(tk, tv, tq, prm);
  return cudaGetLastError();
}

int prefill_ctas(int sms) { return sms < kMaxPrefillCtas ? sms : kMaxPrefillCtas; }

size_t prefill_workspace_bytes(int ctas) {
  return ws_counter_bytes(ctas) + ws_lse_bytes(ctas) + (size_t)ctas * SLOT_ROWS * kHeadDim * 4;
}

size_t prefill_workspace_zero_bytes(int ctas) { return ws_counter_bytes(ctas); }

uint32_t take_prefill_error(cudaStream_t s) { return take_error_word(&g_err_prefill, s); }

}  // namespace pkv_host
