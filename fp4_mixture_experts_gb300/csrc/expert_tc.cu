// Prefill-shaped expert projections on the 5th-generation tensor cores.
//
// A grouped GEMM per expert, swap-AB: the expert's weight rows are the UMMA M
// operand (128 rows per accumulator) and the expert's token rows the N
// operand (up to 192 per tile), so an expert with few rows wastes little of
// the MMA ("low-M utilisation" is a limit the DeepSeek-V4-Flash-on-gfx90a
// paper names).  A work item computes two 128 x N accumulators that share the
// token tile: gate and up rows of W13 (so SwiGLU fuses into the epilogue), or
// two adjacent 128-row blocks of W2.  The kernel is persistent: one CTA per
// SM loops over the items.
//
// Warp roles, per 64-wide K step (one stage of a 2- to 4-deep ring):
//   warp 9      TMA producer of the token tile (up to 192 rows in 64-row
//               boxes, 128-byte swizzle; mostly L2 hits, shared by the CTAs
//               of one expert)
//   warp 10     TMA producer of the packed weights, 2-deep ring of
//               128 rows x 128 bytes (4 K steps) per accumulator, 128-byte
//               swizzle
//   warp 0 and the last warp
//               MMA issuers, one per accumulator: 4 tcgen05.mma.kind::f16
//               (M=128, N=tile, K=16) per K step each, fp32 accumulators in
//               TMEM.  An MMA instruction costs the issuing thread about as
//               long as it runs, and so do its barrier wait and commit; with
//               two issuers one of them is always feeding the tensor pipe
//               while the other synchronises.  Warp 0 also owns TMEM
//               (512 columns: the A ring, then both accumulators).
//   warps 1..8  dequantisers, one thread per weight row: the row's 32 packed
//               bytes per K step come from the TMA ring; E2M1 pairs are decoded by
//               cvt.rn.f16x2.e2m1x2, scaled exactly by a power of two
//               (mul.f16x2) and written to the stage's A slot in TMEM with
//               tcgen05.st (lane = weight row), so that the MMA reads its A
//               operand from tensor memory; then the epilogue (tcgen05.ld,
//               SwiGLU + bf16 rounding of h, or y)
// A stage is full once the token tile has landed and all 8 dequantisers have
// written their A slots (one mbarrier: the producer's expect_tx and 8
// arrivals), and empty once both issuers' MMAs on it have completed (one
// mbarrier, two tcgen05.commit arrivals).
// Weights are dequantised exactly (an E2M1 value times a power of two has
// 2 significant bits), so the MMA multiplies exact products and accumulates
// them in fp32.  Operands are f16: the weight row is scaled by 2^(s - s_ref)
// (exact within 36 binades of the row's largest scale) and each token row
// (x for W13; the f16 copy of h for W2) by a power of two of its own; both
// factors come back in the epilogue.  Every mbarrier wait is bounded; a
// timeout sets the error word and an abort flag that releases the other
// roles.  No warp leaves a loop early (after an abort it stops waiting and
// computes on whatever the buffers hold), so warp-wide instructions always
// see the whole warp.  On the way out every copy a producer issued has
// landed (the token producer adds the arrivals the stopped dequantisers never
// made to its last stages, then waits for them) and every MMA an issuer
// issued has completed, before shared and tensor memory are given back; TMEM
// is always freed.
#include <cuda.h>

#include <algorithm>
#include <cuda_fp16.h>

#include "moe_fp4_internal.cuh"
#include "ptx_sm103.cuh"
#include "tc_helpers.cuh"

namespace moe_fp4 {
namespace {

using namespace tc;

constexpr int kBM = 128;                 // weight rows per accumulator
constexpr int kBK = 64;                  // K elements per stage
constexpr int kBN = kTcTileN;            // token rows per tile (<= 192: TMEM holds 2 accumulators + A)
#ifndef MOE_TC_STAGES
#define MOE_TC_STAGES 4
#endif
constexpr int kStages = MOE_TC_STAGES;   // most ring stages (token tile + A slots); TMEM may allow fewer
constexpr int kDqWarps = 8;
#ifndef MOE_TC_DQ_UNROLL
#define MOE_TC_DQ_UNROLL 4
#endif
constexpr int kDqUnroll = MOE_TC_DQ_UNROLL;     // K steps of the dequantiser loop unrolled together
constexpr int kMmaWarp = 0;                      // TMEM allocator, MMA issuer of accumulator 0
constexpr int kFirstDqWarp = 1;                  // dequantisers 1..8, then the epilogue
constexpr int kBWarp = kFirstDqWarp + kDqWarps;  // token-tile TMA producer
constexpr int kRawWarp = kBWarp + 1;             // packed-weight TMA producer
constexpr int kMma1Warp = kRawWarp + 1;          // MMA issuer of accumulator 1
constexpr int kTcThreads = (kMma1Warp + 1) * 32;
#ifndef MOE_TC_STAGES_RAW
#define MOE_TC_STAGES_RAW 2
#endif
constexpr int kStagesRaw = MOE_TC_STAGES_RAW;    // packed-weight ring depth
constexpr int kRawSteps = 4;                     // K steps per packed-weight stage
constexpr int kRawRowBytes = kRawSteps * kBK / 2; // 128 bytes of each weight row per stage (128-byte swizzle)
// TMEM columns, per tile of n token rows (n_acc = n rounded up to 32):
// accumulator 0 at [0, n_acc), accumulator 1 at [n_acc, 2 n_acc), and the
// A slots in the rest: per (stage, acc) a 128-lane x 32-column slot holding
// 64 K values of each row as f16 pairs.  Narrower tiles leave room for
// more stages (2 at n = 192, 3 at 160, 4 at 128).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kASlotCols = kBK / 2;
static_assert(2 * ((kBN + 31) / 32 * 32) + 2 * 2 * kASlotCols <= kTmemCols, "TMEM columns exceeded at the widest tile");
static_assert(kStages >= 2 && kStages <= 4, "ring of 2 to 4 stages");

#ifndef MOE_TC_FUSED_COMBINE
#define MOE_TC_FUSED_COMBINE 1
#endif
// 1: the pair kernel's W2 epilogue also performs the weighted combine
constexpr bool kFusedCombine = MOE_TC_FUSED_COMBINE != 0;
constexpr int kPairBoxRows = 32;                  // token rows per TMA box of the pair kernel
constexpr int kBBoxRows = 64;                     // token rows per TMA box
constexpr int kBBoxBytes = kBBoxRows * kBK * 2;   // 8 KB
constexpr int kBTileBytes = (kBN + kBBoxRows - 1) / kBBoxRows * kBBoxBytes;  // whole 64-row boxes
constexpr int kRawTileBytes = kBM * kRawRowBytes;  // packed tile of one accumulator's 128 rows
constexpr int kOffB = 0;                                       // [stage]
constexpr int kOffRaw = kOffB + kStages * kBTileBytes;         // [stage][acc]
constexpr int kOffRowscale = kOffRaw + kStagesRaw * 2 * kRawTileBytes;
constexpr int kOffBar = kOffRowscale + 2 * 2 * kBM * 4;  // row scales [item parity][acc][row]
constexpr int kSmemTc = kOffBar + 512 + 1024;  // + barriers, 1 KB alignment slack
static_assert((2 * kStagesRaw + 2 * kStages + 4) * 8 + 8 + 4 * kDqWarps <= 512, "barrier area exceeded");
static_assert(kSmemTc <= 227 * 1024, "shared memory of the tensor-core kernel exceeds 227 KB");
static_assert(kBTileBytes % 1024 == 0, "token slots must stay 1 KB aligned for the 128-byte swizzle");

// Geometry of one work item: token rows [row0, row0 + n) of one expert (n <=
// 192) times two 128-row weight blocks (m-block mb).  TMEM holds the ring of
// A slots first ([0, 64 nS) columns) and the two accumulators after it, each
// n rounded up to 32 columns wide; narrower tiles leave room for more stages.
struct TcItem {
  int row0, n, n_mma, nS, wrow0, mb;
  uint32_t acc_cols, acc0;
};

__device__ __forceinline__ TcItem tc_item(const TcParams& P, int item) {
  TcItem t;
  const int tile = item / P.mblocks;
  t.mb = item % P.mblocks;
  const int4 tl = P.tiles[tile];
  t.row0 = tl.y;
  t.n = tl.z;
  t.n_mma = (t.n + 15) & ~15;
  t.acc_cols = (uint32_t)(t.n_mma + 31) & ~31u;
  t.nS = min(kStages, (int)((kTmemCols - 2 * t.acc_cols) / (2 * kASlotCols)));
  t.acc0 = (uint32_t)t.nS * 2 * kASlotCols;
  t.wrow0 = tl.x * P.rows_per_expert + t.mb * P.block_rows;
  return t;
}

// Persistent: each CTA takes the work items blockIdx.x, blockIdx.x + gridDim.x,
// ... (items are (tile, m-block) pairs, tile-major, so neighbouring CTAs share
// token tiles in L2).  The rings run on across items, so the producers load
// the next item's weights and token rows while the current one is finishing;
// TMEM is allocated once.  Operands are f16: weight rows scaled by
// 2^(s - s_ref(row)) with s_ref = (largest E8M0 of the row) - 13, token rows
// (x for W13, h for W2) by a per-row power of two; both are undone in the
// epilogue (per TMEM lane and column), then SwiGLU and bf16 h (W13) or fp32 y
// (W2).
template <bool W13>
__global__ void __launch_bounds__(kTcThreads, 1)
tc_kernel(const __grid_constant__ CUtensorMap map_b, const __grid_constant__ CUtensorMap map_raw, const TcParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* rowscale = reinterpret_cast<float*>(smem + kOffRowscale);  // [item parity][2][128]
  uint64_t* raw_full = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* raw_empty = raw_full + kStagesRaw;
  uint64_t* full = raw_empty + kStagesRaw;    // [stage]: token tile landed and both A slots written
  uint64_t* empty = full + kStages;           // [stage]: the MMAs of both accumulators on it completed
  uint64_t* acc_full = empty + kStages;       // per item: both accumulators final
  uint64_t* acc_empty = acc_full + 1;         // per item: the epilogue has read the accumulators
  uint64_t* mma_done = acc_empty + 1;         // [2]: every MMA of that issuer completed (on the way out)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* dq_arrived = abort_flag + 1;  // [8]: stages each dequantiser signalled (published on the way out)
  const uint64_t lim = P.wait_ns;

  const int items = P.counts[2] * P.mblocks;
  if ((int)blockIdx.x >= items) return;
  const int nk = P.K / kBK;
  const int nrs = (nk + kRawSteps - 1) / kRawSteps;  // packed-weight stages per item (a last partial one reads zeros)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesRaw; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], kDqWarps);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], kDqWarps + 1);  // the dequantisers and the token producer's expect_tx
      mbar_init(&empty[s], 2);            // one commit per MMA issuer
    }
    mbar_init(acc_full, 2);
    mbar_init(acc_empty, kDqWarps);
    mbar_init(&mma_done[0], 1);
    mbar_init(&mma_done[1], 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncwarp();  // warp 0 reconverges before the warp-wide TMEM allocation
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  // Ring bookkeeping: every role walks the same sequence of (item, K step), so
  // per-slot phase bits (bit s = parity of slot s's next use) agree across roles.

  if (warp == kRawWarp) {
    // ---------------- TMA producer: packed weights ----------------
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();  // weights are read once: keep the token tiles in L2
      uint32_t g = 0;                                // packed-weight stages issued so far
      bool ok = true;
      for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
        const TcItem t = tc_item(P, it);
        for (int rs = 0; rs < nrs; ++rs, ++g) {
          const int s = g % kStagesRaw;
          if (!mbar_wait(&raw_empty[s], ((g / kStagesRaw) & 1) ^ 1u, abort_flag, P.err, kErrWaitTimeout, lim)) {
            ok = false;
            break;
          }
          // (a slot comes back only once every dequantiser read its bytes:
          // one copy per slot in flight)
          mbar_expect_tx(&raw_full[s], 2 * kRawTileBytes);
          uint8_t* raw = smem + kOffRaw + s * 2 * kRawTileBytes;
          tma_load_2d_hint(raw, &map_raw, rs * kRawRowBytes, t.wrow0, &raw_full[s], pol);
          tma_load_2d_hint(raw + kRawTileBytes, &map_raw, rs * kRawRowBytes, t.wrow0 + P.acc1_offset, &raw_full[s], pol);
        }
      }
      // every issued copy has landed before the CTA may exit
      for (uint32_t q = g > kStagesRaw ? g - kStagesRaw : 0; q < g; ++q)
        mbar_wait_drain(&raw_full[q % kStagesRaw], (q / kStagesRaw) & 1, P.err, kErrWaitTimeout, lim);
    }
  } else if (warp == kBWarp) {
    // ---------------- TMA producer: token tiles ----------------
    // A slot comes back (empty) only after the MMAs ran on its previous use,
    // whose copy had landed: at most one copy per slot is ever in flight.
    uint32_t ph = 0;   // bit s: parity of slot s's next use
    int g = 0;         // stages passed (issued, or withheld by the fault injection)
    const bool fault_cta = P.fault != 0 && blockIdx.x == 0;
    if (lane == 0) {
      bool ok = true;
      for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
        const TcItem t = tc_item(P, it);
        const int boxes = (t.n_mma + kBBoxRows - 1) / kBBoxRows;
        for (int ks = 0; ks < nk; ++ks, ++g) {
          const int s = ks % t.nS;
          if (!mbar_wait(&empty[s], ((ph >> s) & 1) ^ 1u, abort_flag, P.err, kErrWaitTimeout, lim)) {
            ok = false;
            break;
          }
          ph ^= 1u << s;
          // fault injection: the first tile of the first CTA never arrives,
          // so the MMA issuers' wait on the stage runs out
          if (fault_cta && g == 0) continue;
          mbar_expect_tx(&full[s], boxes * kBBoxBytes);
          uint8_t* b = smem + kOffB + s * kBTileBytes;
          for (int i = 0; i < boxes; ++i)
            tma_load_2d(b + i * kBBoxBytes, &map_b, ks * kBK, t.row0 + i * kBBoxRows, &full[s]);
        }
      }
    }
    // wait for the dequantisers to stop, then (after an abort) let each copy
    // still in flight complete its stage: add the arrivals of the
    // dequantisers that stopped before it, and wait for the bytes
    __syncwarp();
    asm volatile("bar.sync 3, %0;" ::"r"((kDqWarps + 1) * 32) : "memory");
    if (lane == 0 && *abort_flag) {
      // the last stage of each slot: replay the slot sequence up to g
      int last[kStages];
#pragma unroll
      for (int q = 0; q < kStages; ++q) last[q] = -1;
      int g2 = 0;
      for (int it = blockIdx.x; it < items && g2 < g; it += gridDim.x) {
        const TcItem t = tc_item(P, it);
        for (int ks = 0; ks < nk && g2 < g; ++ks, ++g2) {
          const int s2 = ks % t.nS;
#pragma unroll
          for (int q = 0; q < kStages; ++q)
            if (q == s2) last[q] = g2;
        }
      }
#pragma unroll
      for (int s = 0; s < kStages; ++s) {
        if (last[s] < 0 || (fault_cta && last[s] == 0)) continue;  // no copy (or a withheld one)
        int arrived = 0;
        for (int w = 0; w < kDqWarps; ++w) arrived += dq_arrived[w] > last[s] ? 1 : 0;
        if (arrived < kDqWarps)
          asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(&full[s])),
                       "r"(kDqWarps - arrived) : "memory");
        mbar_wait_drain(&full[s], ((ph >> s) & 1) ^ 1u, P.err, kErrWaitTimeout, lim);
      }
    }
  } else if (warp == kMmaWarp || warp == kMma1Warp) {
    // ---------------- MMA issuers, one per accumulator ----------------
    if (lane == 0) {
      const int acc = warp == kMmaWarp ? 0 : 1;
      uint32_t ph = 0;
      int li = 0;  // items done by this CTA
      bool ok = true;
      for (int it = blockIdx.x; it < items && ok; it += gridDim.x, ++li) {
        const TcItem t = tc_item(P, it);
        // the epilogue of the previous item must have read the accumulators
        if (li > 0 && !mbar_wait(acc_empty, (li - 1) & 1, abort_flag, P.err, kErrWaitTimeout, lim)) break;
        const uint32_t idesc = idesc_f16kind(kBM, t.n_mma, 0u);
        const uint32_t d_tmem = tmem + t.acc0 + acc * t.acc_cols;
        for (int ks = 0; ks < nk; ++ks) {
          const int s = ks % t.nS;
          if (!mbar_wait(&full[s], (ph >> s) & 1, abort_flag, P.err, kErrWaitTimeout, lim)) {
            ok = false;
            break;
          }
          ph ^= 1u << s;
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint32_t b_addr = smem_u32(smem + kOffB + s * kBTileBytes);
          const uint32_t a_tmem = tmem + (s * 2 + acc) * kASlotCols;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_tmem_a(d_tmem, a_tmem + kk * 8, desc_sw128(b_addr + kk * 32), idesc, (ks > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&empty[s]);
        }
        if (!ok) break;
        umma_commit(acc_full);
      }
      // every MMA this thread issued has completed before TMEM can be freed,
      // also on an abort (a commit with nothing outstanding arrives at once)
      umma_commit(&mma_done[acc]);
      mbar_wait_drain(&mma_done[acc], 0, P.err, kErrWaitTimeout, lim);
    }
  } else {
    // ---------------- dequantisers (one weight row each), then the epilogue ----------------
    const int dq = warp - kFirstDqWarp;
    const int acc = dq >> 2;                 // 0: first block (gate), 1: second block (up)
    const int q = warp & 3;                  // TMEM lane quadrant this warp may access
    const int r = q * 32 + lane;             // row within the 128-row block = TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    const int kpr = P.K / 32;                // scale bytes per row
    uint32_t ph = 0;                         // A-slot phase bits
    uint32_t g = 0;                          // packed-weight stages of the items before the one being converted
    int li = 0;
    int gdq = 0;                             // stages this warp signalled full (lane 0's count)
    bool ok = true;                          // this lane's waits have all succeeded
    bool stop = false;                       // all dequantisers stop after this item (uniform)
    // The first steps of the next item are converted before the epilogue of
    // the current one (into A slots below the current accumulators), so that
    // its MMAs can start as soon as the epilogue has read the accumulators.
    // Only the step count and the row's reference scale stay live across the
    // epilogue; the rest of the conversion state is rebuilt after it.
    const uint8_t* srow = nullptr;
    int s_ref = 0;
    const bool vec_scales = (kpr & 15) == 0;  // scale bytes 16 at a time (8 K steps), else 2 per step
    uint4 sg_cur = make_uint4(0, 0, 0, 0), sg_next = make_uint4(0, 0, 0, 0);
    uint32_t sc_next = 0;
    // this thread's scale row of item t: a W2 tile whose second block runs
    // past the expert's d rows (d % 256 == 128) reads a valid row there
    // instead (its results are not written), so that no read leaves the
    // weight and scale tensors
    auto scale_row = [&](const TcItem& t) {
      const bool row_in = t.mb * P.block_rows + acc * P.acc1_offset + r < P.rows_per_expert;
      const int wrow = row_in ? t.wrow0 + acc * P.acc1_offset + r : t.wrow0 + r;
      return P.scales + (size_t)wrow * kpr;
    };
    // reference scale of item t (row scale of item parity `buf`) and the
    // scale-byte registers for step 0
    auto prepare = [&](const TcItem& t, int buf) {
      srow = scale_row(t);
      uint32_t smax = 0;
      auto max4 = [](uint32_t m, uint32_t w4) {
        return max(m, max(max(w4 & 0xFFu, (w4 >> 8) & 0xFFu), max((w4 >> 16) & 0xFFu, w4 >> 24)));
      };
      if (vec_scales) {
        constexpr int kSv = 4;  // 16-byte loads in flight at a time (more would spill registers)
        for (int i0 = 0; i0 < kpr; i0 += 16 * kSv) {
          uint4 sv[kSv];
#pragma unroll
          for (int i = 0; i < kSv; ++i)
            if (i0 + 16 * i < kpr) sv[i] = *reinterpret_cast<const uint4*>(srow + i0 + 16 * i);
#pragma unroll
          for (int i = 0; i < kSv; ++i)
            if (i0 + 16 * i < kpr) smax = max4(max4(max4(max4(smax, sv[i].x), sv[i].y), sv[i].z), sv[i].w);
        }
        sg_next = *reinterpret_cast<const uint4*>(srow);
      } else {
        for (int i = 0; i < kpr; i += 4) smax = max4(smax, *reinterpret_cast<const uint32_t*>(srow + i));
        sc_next = *reinterpret_cast<const uint16_t*>(srow);
      }
      s_ref = (int)smax - 13;
      rowscale[buf * 256 + acc * 128 + r] = pow2f(s_ref - 127);
    };
    // K step ks of item t into the A ring; with active false (a step
    // converted ahead) only the scale-byte registers advance
    auto convert = [&](const TcItem& t, int ks, bool active) {
      {
        const int sa = ks % t.nS;
        const int sub = ks % kRawSteps;
        const uint32_t gs = g + ks / kRawSteps;
        const int rs_slot = gs % kStagesRaw;
        // once a wait has failed (or seen the abort) this lane stops waiting
        // but keeps converting, so that the warp-wide tcgen05 instructions
        // below always see all 32 lanes
        if (active && sub == 0 && ok)
          ok = mbar_wait(&raw_full[rs_slot], (gs / kStagesRaw) & 1, abort_flag, P.err, kErrWaitTimeout, lim);
        // 128-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ (r mod 8),
        // so the 8 rows of a warp's quarter hit 8 different bank groups.  The
        // packed bytes are read as they are converted (one byte per register);
        // the stage is released after its last K step's conversion.
        const uint8_t* raw = smem + kOffRaw + (rs_slot * 2 + acc) * kRawTileBytes + r * kRawRowBytes;
        const uint8_t* raw_lo = raw + (((2 * sub) ^ (r & 7)) << 4);
        const uint8_t* raw_hi = raw + (((2 * sub + 1) ^ (r & 7)) << 4);
        uint32_t sc;
        if (vec_scales) {
          if ((ks & 7) == 0) {
            sg_cur = sg_next;
            if (ks + 8 < nk) sg_next = *reinterpret_cast<const uint4*>(srow + 2 * (ks + 8));
          }
          const uint32_t wsel = ((ks & 7) >> 1) == 0 ? sg_cur.x : ((ks & 7) >> 1) == 1 ? sg_cur.y
                              : ((ks & 7) >> 1) == 2 ? sg_cur.z : sg_cur.w;
          sc = (ks & 1) ? wsel >> 16 : wsel & 0xFFFFu;
        } else {
          sc = sc_next;
          if (ks + 1 < nk) sc_next = *reinterpret_cast<const uint16_t*>(srow + 2 * (ks + 1));
        }
        if (active) {
          if (ok) ok = mbar_wait(&empty[sa], ((ph >> sa) & 1) ^ 1u, abort_flag, P.err, kErrWaitTimeout, lim);
          ph ^= 1u << sa;
          const uint32_t s0 = sc & 0xFFu, s1 = (sc >> 8) & 0xFFu;
          const uint32_t m0 = f16x2_pow2((int)s0 - s_ref), m1 = f16x2_pow2((int)s1 - s_ref);
          uint32_t av[32];  // column j = K elements (2j, 2j+1) of this row
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint32_t b[4];  // 8 codes: K elements 8c .. 8c + 7 of this step
            lds_bytes4((c < 4 ? raw_lo : raw_hi) + 4 * (c & 3), b);
            const uint32_t m = c < 4 ? m0 : m1;
#pragma unroll
            for (int i = 0; i < 4; ++i) av[4 * c + i] = f16x2_mul(e2m1x2_to_f16x2(b[i]), m);
          }
          if (sub == kRawSteps - 1 || ks == nk - 1) {
            __syncwarp();
            if (lane == 0 && ok) mbar_arrive(&raw_empty[rs_slot]);  // the stage's packed bytes have all been read
          }
          tmem_st32(lane_base + (sa * 2 + acc) * kASlotCols, av);
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
          asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
          __syncwarp();
          if (lane == 0 && ok) {
            mbar_arrive(&full[sa]);
            ++gdq;
          }
        }
      }
    };
    int pre = 0;  // K steps of the current item converted ahead
    for (int it = blockIdx.x; it < items && !stop; it += gridDim.x, ++li) {
      const TcItem t = tc_item(P, it);
      if (pre == 0) {
        prepare(t, li & 1);
      } else {
        srow = scale_row(t);  // scale-byte registers back at step 0
        if (vec_scales)
          sg_next = *reinterpret_cast<const uint4*>(srow);
        else
          sc_next = *reinterpret_cast<const uint16_t*>(srow);
      }
#pragma unroll kDqUnroll
      for (int ks = 0; ks < nk; ++ks) convert(t, ks, ks >= pre);
      g += nrs;
      // the next item's first steps, into the slots below both items' accumulators
      pre = 0;
      if (it + (int)gridDim.x < items) {
        const TcItem tn = tc_item(P, it + gridDim.x);
        const int m = min(nk, min(t.nS, tn.nS));
        prepare(tn, (li + 1) & 1);
#pragma unroll 1
        for (int ks = 0; ks < m; ++ks) convert(tn, ks, true);
        pre = m;
      }
      // epilogue: the two warps of a lane quadrant take alternate 32-column
      // chunks; their column scales are fetched before the accumulators are ready
      constexpr int kChunks = (kBN + 63) / 64;
      const int half = dq >> 2;
      float xs_pre[kChunks] = {};
      float wt_pre[kChunks] = {};  // W2 with the combine: routing weight and token of each column
      int tk_pre[kChunks] = {};
      {
#pragma unroll
        for (int i = 0; i < kChunks; ++i) {
          const int col = 32 * (2 * i + half) + lane;
          if (col < t.n) {
            xs_pre[i] = P.x_scale[t.row0 + col];
            if (!W13 && P.out) {
              const int slot = P.sorted_slot[t.row0 + col];
              wt_pre[i] = P.topk_w[slot];
              tk_pre[i] = slot / P.k;
            }
          }
        }
      }
      // the row scales written above must be visible to every epilogue warp
      asm volatile("bar.sync 1, %0;" ::"r"(kDqWarps * 32) : "memory");
      if (__all_sync(0xFFFFFFFFu, ok && mbar_wait(acc_full, li & 1, abort_flag, P.err, kErrWaitTimeout, lim))) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const float rs0 = rowscale[(li & 1) * 256 + r], rs1 = rowscale[(li & 1) * 256 + 128 + r];
#pragma unroll
        for (int ci = 0; ci < kChunks; ++ci) {
          const int c0 = 32 * (2 * ci + half);
          if (c0 >= t.n_mma) break;
          float a0[32], a1[32];
          tmem_ld32x2(lane_base + t.acc0 + c0, lane_base + t.acc0 + t.acc_cols + c0, a0, a1);
          const float xs_l = xs_pre[ci];
          if (W13) {
            const int i = t.mb * kBM + r;
            // two columns per conversion (cvt.rn.bf16x2.f32: one instruction
            // for both roundings, nearest even like the single conversion)
            uint16_t* hp = P.h_out + (size_t)(t.row0 + c0) * P.I + i;
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              const float xs0 = __shfl_sync(0xFFFFFFFFu, xs_l, j), xs1 = __shfl_sync(0xFFFFFFFFu, xs_l, j + 1);
              const __nv_bfloat162 hb = __floats2bfloat162_rn(swiglu(a0[j] * rs0 * xs0, a1[j] * rs1 * xs0),
                                                              swiglu(a0[j + 1] * rs0 * xs1, a1[j + 1] * rs1 * xs1));
              if (c0 + j < t.n) hp[(size_t)j * P.I] = __bfloat16_as_ushort(__low2bfloat16(hb));
              if (c0 + j + 1 < t.n) hp[(size_t)(j + 1) * P.I] = __bfloat16_as_ushort(__high2bfloat16(hb));
            }
          } else {
            // 8-byte stores of two adjacent features: for the token pair (j,
            // j + 1) the even lane of each lane pair takes token j and the odd
            // lane token j + 1, swapping one value with its neighbour (half
            // the store instructions, which bound this epilogue)
            const bool odd = lane & 1;
            const int nrow = t.mb * P.block_rows + (r & ~1);  // the pair's first feature
            const bool second_in = nrow + P.acc1_offset < P.d;  // last block may hold 128 rows
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              const float xs0 = __shfl_sync(0xFFFFFFFFu, xs_l, j), xs1 = __shfl_sync(0xFFFFFFFFu, xs_l, j + 1);
              const float p0 = a0[j] * rs0 * xs0, q0 = a0[j + 1] * rs0 * xs1;
              const float p1 = a1[j] * rs1 * xs0, q1 = a1[j + 1] * rs1 * xs1;
              const float o0 = __shfl_xor_sync(0xFFFFFFFFu, odd ? p0 : q0, 1);
              const float o1 = __shfl_xor_sync(0xFFFFFFFFu, odd ? p1 : q1, 1);
              const int jj = j + (odd ? 1 : 0);
              if (P.out) {
                // the weighted combine: the pair of features of token column jj
                // added into that token's out row
                const float wj = __shfl_sync(0xFFFFFFFFu, wt_pre[ci], jj);
                const int tj = __shfl_sync(0xFFFFFFFFu, tk_pre[ci], jj);
                if (c0 + jj < t.n) {
                  float* orow = P.out + (size_t)tj * P.d + nrow;
                  const float2 v0 = odd ? make_float2(o0, q0) : make_float2(p0, o0);
                  red_add_v2_f32(orow, wj * v0.x, wj * v0.y);
                  if (second_in) {
                    const float2 v1 = odd ? make_float2(o1, q1) : make_float2(p1, o1);
                    red_add_v2_f32(orow + P.acc1_offset, wj * v1.x, wj * v1.y);
                  }
                }
              } else if (c0 + jj < t.n) {
                float* yrow = P.y_out + (size_t)(t.row0 + c0 + jj) * P.d + nrow;
                *reinterpret_cast<float2*>(yrow) = odd ? make_float2(o0, q0) : make_float2(p0, o0);
                if (second_in)
                  *reinterpret_cast<float2*>(yrow + P.acc1_offset) = odd ? make_float2(o1, q1) : make_float2(p1, o1);
              }
            }
          }
        }
        // the accumulators are in registers: the next item's MMAs may overwrite them
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty);
      } else {
        ok = false;
      }
      // every dequantiser is done with this item's accumulators and row scales
      // before any of them writes the next item's A slots (which may cover
      // them); a failure seen by any of them stops all of them together, so
      // that they keep meeting at the same named barriers
      uint32_t st;
      asm volatile(
          "{\n\t.reg .pred pin, pout;\n\tsetp.ne.u32 pin, %1, 0;\n\tbar.red.or.pred pout, 1, %2, pin;\n\t"
          "selp.u32 %0, 1, 0, pout;\n}"
          : "=r"(st)
          : "r"((!ok || *abort_flag) ? 1u : 0u), "r"(kDqWarps * 32)
          : "memory");
      stop = st != 0;
    }
    // how far this warp got, for the token producer's way out
    if (lane == 0) dq_arrived[dq] = gdq;
    asm volatile("bar.arrive 3, %0;" ::"r"((kDqWarps + 1) * 32) : "memory");
  }
  // every warp reconverges first: lanes that skipped a lane-0 role must not
  // arrive at the CTA barrier ahead of their lane 0 (an aligned barrier counts
  // a warp as arrived when any of its lanes gets there), so that TMEM is freed
  // only after all epilogue reads
  __syncwarp();
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

template <bool W13>
cudaError_t launch_tc(const CUtensorMap& b, const CUtensorMap& raw, const TcParams& P, int max_tiles, cudaStream_t st) {
  const cudaError_t oe = ensure_smem_optin(reinterpret_cast<const void*>(tc_kernel<W13>), kSmemTc);
  if (oe != cudaSuccess) return oe;
  // one CTA per SM, each looping over work items; no more CTAs than items
  const long long most = (long long)max_tiles * P.mblocks;
  if (most > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  const int grid = (int)std::min<long long>(most, num_sms());
  if (grid <= 0) return cudaSuccess;
  tc_kernel<W13><<<grid, kTcThreads, kSmemTc, st>>>(b, raw, P);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_w13(const moe_fp4_dims& d, const uint8_t* w13, const uint8_t* w13s, const Workspace& ws,
                          bool pairs, cudaStream_t st) {
  const size_t S = (size_t)d.T * d.k;
  CUtensorMap b, raw;
  if (!make_map_2d(&raw, CU_TENSOR_MAP_DATA_TYPE_UINT8, w13, d.d / 2, (uint64_t)d.E * 2 * d.I, d.d / 2, kRawRowBytes, kBM,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_2d(&b, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, ws.x_perm, d.d, S, (uint64_t)d.d * 2, kBK,
                   pairs ? kPairBoxRows : kBBoxRows, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  TcParams P{};
  P.w = w13;
  P.scales = w13s;
  P.tiles = ws.tc_tiles;
  P.counts = ws.counts;
  P.err = ws.err;
  P.h_out = ws.h;
  P.x_scale = ws.x_scale;
  P.K = d.d;
  P.rows_per_expert = 2 * d.I;
  P.I = d.I;
  P.d = d.d;
  P.wait_ns = wait_limit_ns();
  P.fault = fault_site() == MOE_FP4_FAULT_TC_TOKEN_TILE;
  if (pairs) {
    // a pair covers 256 i-values (128 per CTA); gate rows i, up rows I + i
    P.mblocks = (d.I + 2 * kBM - 1) / (2 * kBM);
    P.block_rows = 2 * kBM;
    P.cta_rows = kBM;
    P.acc_idx_step = 0;
    P.acc_row_off = d.I;
    P.limit = d.I;
    return launch_tc2<true>(b, raw, P, ws.max_tc_tiles, st);
  }
  P.mblocks = d.I / kBM;
  P.block_rows = kBM;
  P.acc1_offset = d.I;
  return launch_tc<true>(b, raw, P, ws.max_tc_tiles, st);
}

bool tc_fused_combine(bool pairs) { return pairs && kFusedCombine; }

cudaError_t launch_tc_w2(const moe_fp4_dims& d, const uint8_t* w2, const uint8_t* w2s, const Workspace& ws,
                         float* out, bool pairs, bool atomic_combine, cudaStream_t st) {
  const size_t S = (size_t)d.T * d.k;
  CUtensorMap b, raw;
  if (!make_map_2d(&raw, CU_TENSOR_MAP_DATA_TYPE_UINT8, w2, d.I / 2, (uint64_t)d.E * d.d, d.I / 2, kRawRowBytes, kBM,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_2d(&b, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, ws.h16, d.I, S, (uint64_t)d.I * 2, kBK,
                   pairs ? kPairBoxRows : kBBoxRows, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  TcParams P{};
  P.w = w2;
  P.scales = w2s;
  P.tiles = ws.tc_tiles;
  P.counts = ws.counts;
  P.err = ws.err;
  P.y_out = ws.y;
  P.x_scale = ws.h_scale;
  P.K = d.I;
  P.rows_per_expert = d.d;
  P.I = d.I;
  P.d = d.d;
  P.wait_ns = wait_limit_ns();
  P.fault = 0;
  if (pairs) {
    // a pair covers 512 output features (256 per CTA, two 128-row accumulators)
    P.mblocks = (d.d + 4 * kBM - 1) / (4 * kBM);
    P.block_rows = 4 * kBM;
    P.cta_rows = 2 * kBM;
    P.acc_idx_step = kBM;
    P.acc_row_off = 0;
    P.limit = d.d;
    if (kFusedCombine) {
      P.out = out;
      P.topk_w = ws.topk_w;
      P.sorted_slot = ws.sorted_slot;
      P.slot_pos = ws.slot_pos;
      P.combine_cnt = ws.combine_cnt;
      P.k = d.k;
    }
    return launch_tc2<false>(b, raw, P, ws.max_tc_tiles, st);
  }
  P.mblocks = (d.d + 2 * kBM - 1) / (2 * kBM);  // d % 256 == 128 leaves a 128-row last block
  P.block_rows = 2 * kBM;
  P.acc1_offset = kBM;
  if (atomic_combine) {
    P.out = out;
    P.topk_w = ws.topk_w;
    P.sorted_slot = ws.sorted_slot;
    P.k = d.k;
  }
  return launch_tc<false>(b, raw, P, ws.max_tc_tiles, st);
}

}  // namespace moe_fp4
