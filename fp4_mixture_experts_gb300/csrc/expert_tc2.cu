// Prefill-shaped expert projections on pairs of SMs (tcgen05 cta_group::2).
//
// The same grouped GEMM as the one-CTA tensor-core kernel (swap-AB: weight
// rows are the UMMA M operand, an expert's token rows the N operand; W13
// computes gate and up accumulators and fuses SwiGLU, W2 two 128-row blocks
// of output features), but each MMA instruction covers two SMs: M = 256, the
// 128 weight rows of each CTA of a cluster pair read from that CTA's tensor
// memory, the N token rows split in halves between the two CTAs' shared
// memory.  The motive: one thread issuing tcgen05.mma spends ~200 cycles per
// instruction whatever N is (measured with A in shared or tensor memory,
// N = 64..256: 203-207 cycles per M=128 instruction), while an M=128, N=144
// MMA keeps the tensor pipe busy for only ~72 cycles, so the one-CTA kernel
// (one issuer per accumulator) is bound by instruction issue; a cta_group::2
// instruction with both operands in shared memory costs ~147 cycles for twice
// the work.  Measured on the prefill workload, the pair kernel is slower all
// the same (W13 1.93 ms against 1.13 ms): with A in tensor memory an M=256
// instruction costs its issuer ~200 cycles again, and the dequantisers'
// tensor-memory stores wait while the pair's MMAs read both SMs' tensor
// memory (0.83 us per stage from slot release to arrival against 0.19 us in
// the one-CTA kernel).  Moving A to shared memory instead would make shared-
// memory bandwidth the bound (~107 KB per stage per CTA).  The kernel is kept
// behind MOE_FP4_FLAG_CTA_PAIRS, tested like the default one.
//
// Per pair (leader = CTA rank 0, follower = rank 1) and work item (a token
// tile of one expert times one m-block: 256 i-values of W13 or 512 output
// features of W2, 128 or 256 of them per CTA):
//   warps 1..8 (both)   dequantisers, one weight row each, writing their
//                       CTA's A slots in TMEM, then the epilogue of their
//                       CTA's accumulators (as in the one-CTA kernel)
//   warp 9 (both)       TMA producer of the CTA's half of the token tile
//   warp 10 (both)      TMA producer of the CTA's packed weights
//   warps 0, 11 leader  MMA issuers, one per accumulator (M = 256 over both
//                       CTAs), commits multicast to both CTAs
//   warp 11 follower    relay: watches the follower's token copies land and
//                       forwards each, in order, to the leader's stage
//                       barrier (so that the follower's producer never waits
//                       on a landing)
// The leader's stage barrier (full) completes with 16 dequantiser arrivals
// (8 remote), the leader producer's expect_tx with its bytes, and the relay;
// the empty, accumulator-ready and MMA-done barriers of both CTAs complete
// by multicast commits; the accumulator-free barrier lives in the leader (16
// epilogue arrivals).
//
// Failure handling: every wait is bounded; the abort flag lives in the
// leader and both CTAs watch it.  No warp leaves a loop early.  On the way
// out every role publishes how far it got, the leader's producer completes
// the stages left open (the arrivals the stopped dequantisers and relay never
// made) and waits for its copies, the relay has seen every follower copy
// land, both CTAs wait for the MMAs, and a cluster barrier precedes freeing
// TMEM.
#include <cooperative_groups.h>
#include <cuda.h>

#include <algorithm>

#include "moe_fp4_internal.cuh"
#include "ptx_sm103.cuh"
#include "tc_helpers.cuh"

namespace moe_fp4 {
namespace {

using namespace tc;
namespace cg = cooperative_groups;

constexpr int kBM = 128;                 // weight rows per accumulator per CTA
constexpr int kBK = 64;                  // K elements per stage
constexpr int kBN = kTcTileN;            // token rows per tile (<= 192)
constexpr int kStages = 4;               // most ring stages (TMEM may allow fewer)
constexpr int kDqWarps = 8;
constexpr int kDqUnroll = 4;
constexpr int kMmaWarp = 0;
constexpr int kFirstDqWarp = 1;
constexpr int kBWarp = kFirstDqWarp + kDqWarps;  // 9
constexpr int kRawWarp = kBWarp + 1;             // 10
constexpr int kMma1Warp = kRawWarp + 1;          // 11 (the follower's relay)
constexpr int kThreads = (kMma1Warp + 1) * 32;
constexpr int kStagesRaw = 2;
constexpr int kRawSteps = 4;
constexpr int kRawRowBytes = kRawSteps * kBK / 2;   // 128
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kASlotCols = kBK / 2;            // 32
constexpr int kBBoxRows = 32;                       // token rows per TMA box
constexpr int kHalfRowsMax = ((kBN / 2 + kBBoxRows - 1) / kBBoxRows) * kBBoxRows;  // 96
constexpr int kBHalfBytes = kHalfRowsMax * kBK * 2;   // 12 KB
constexpr int kBoxBytes = kBBoxRows * kBK * 2;        // 4 KB
constexpr int kRawTileBytes = kBM * kRawRowBytes;     // 16 KB
constexpr int kOffB = 0;
constexpr int kOffRaw = kOffB + kStages * kBHalfBytes;
constexpr int kOffRowscale = kOffRaw + kStagesRaw * 2 * kRawTileBytes;
constexpr int kOffBar = kOffRowscale + 2 * kBM * 4;
constexpr int kNumBars = 2 * kStagesRaw + 3 * kStages + 5;
constexpr int kOffInts = kOffBar + kNumBars * 8;
constexpr int kOffFin = kOffInts + 4 * (4 + 2 * kDqWarps);   // [1 + kBN] finalize list of the W2 combine
constexpr int kSmemTc2 = kOffFin + 4 * (1 + kBN) + 1024;
static_assert(kBHalfBytes % 1024 == 0, "token slots must stay 1 KB aligned for the 128-byte swizzle");
static_assert(kSmemTc2 <= 227 * 1024, "shared memory exceeds 227 KB");
static_assert(2 * ((kBN + 31) / 32 * 32) + 2 * 2 * kASlotCols <= kTmemCols, "TMEM columns exceeded");

__device__ __forceinline__ uint32_t mapa_u32(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// arrive (count times) on the barrier at the same offset in the leader CTA
__device__ __forceinline__ void arrive_leader(uint64_t* bar, uint32_t count = 1) {
  const uint32_t a = mapa_u32(smem_u32(bar), 0);
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(a), "r"(count) : "memory");
}

__device__ __forceinline__ bool try_wait_cl(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// bounded wait on a barrier that other CTAs of the pair arrive on
__device__ __forceinline__ bool wait_cl(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int32_t* err,
                                        uint64_t limit_ns) {
  if (try_wait_cl(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (try_wait_cl(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > limit_ns) break;
  }
  *abort_flag = 1;
  atomicOr(err, kErrWaitTimeout);
  return false;
}

// the same, ignoring the abort flag (on the way out)
__device__ __forceinline__ bool wait_cl_drain(uint64_t* bar, uint32_t parity, int32_t* err, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (global_timer_ns() - t0 <= limit_ns)
    if (try_wait_cl(bar, parity)) return true;
  atomicOr(err, kErrWaitTimeout);
  return false;
}

__device__ __forceinline__ void umma2_tmem_a(uint32_t tmem_d, uint32_t tmem_a, uint64_t b, uint32_t idesc,
                                             uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// commit of this thread's MMAs to the barrier at this offset in both CTAs
__device__ __forceinline__ void commit2_both(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"((uint16_t)3)
      : "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// One work item of a pair: token rows [row0, row0 + n) of one expert times
// m-block mbp.  Each CTA holds half of the (16-padded) token rows: rows
// [rank * half, (rank + 1) * half) of the tile.
struct Item2 {
  int row0, n, n_mma, half, nS, expert, first;
  uint32_t acc_cols, acc0;
};

__device__ __forceinline__ Item2 item2(const TcParams& P, int item, uint32_t rank) {
  Item2 t;
  const int tile = item / P.mblocks;
  const int mbp = item % P.mblocks;
  const int4 tl = P.tiles[tile];
  t.expert = tl.x;
  t.row0 = tl.y;
  t.n = tl.z;
  t.n_mma = (t.n + 15) & ~15;
  t.half = t.n_mma / 2;
  t.acc_cols = (uint32_t)(t.n_mma + 31) & ~31u;
  t.nS = min(kStages, (int)((kTmemCols - 2 * t.acc_cols) / (2 * kASlotCols)));
  t.acc0 = (uint32_t)t.nS * 2 * kASlotCols;
  t.first = mbp * P.block_rows + (int)rank * P.cta_rows;
  return t;
}

// The weighted combine in the W2 epilogue, for this CTA's 256-feature block
// of the item (called by the 8 dequantiser warps once their y rows are
// written and fenced).  A counter per (token, block) counts the slots whose
// y block is written; the CTA that brings a token's count to k sums the k
// rows in slot order, out[t] = sum_j w_tj y[slot_pos[t k + j]], exactly as the
// separate combine kernel would (same fmaf order): deterministic.
__device__ __forceinline__ void combine_block(const TcParams& P, const Item2& t, int dq, int lane, int* fin) {
  const int nblk = (P.d + 255) / 256;
  const int cblk = t.first / 256;
  if (cblk >= nblk) return;  // a block wholly past d (the follower of a last, half pair)
  const int tid = dq * 32 + lane;
  if (tid < t.n) {
    const int tok = P.sorted_slot[t.row0 + tid] / P.k;
    const int old = atomicAdd(&P.combine_cnt[tok * nblk + cblk], 1);
    if (old == P.k - 1) {
      __threadfence();  // every other slot's y block is visible from here on
      fin[1 + atomicAdd(&fin[0], 1)] = tok;
    }
  }
  asm volatile("bar.sync 1, %0;" ::"r"(kDqWarps * 32) : "memory");
  const int nf = fin[0];
  const int col = cblk * 256 + lane * 8;
  for (int i = dq; i < nf; i += kDqWarps) {
    const int tok = fin[1 + i];
    if (col < P.d) {
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
      for (int j = 0; j < P.k; ++j) {
        const float w = P.topk_w[(size_t)tok * P.k + j];
        const float4* yr = reinterpret_cast<const float4*>(P.y_out + (size_t)P.slot_pos[(size_t)tok * P.k + j] * P.d + col);
        const float4 u = __ldcg(yr), v = __ldcg(yr + 1);
        a.x = fmaf(w, u.x, a.x);
        a.y = fmaf(w, u.y, a.y);
        a.z = fmaf(w, u.z, a.z);
        a.w = fmaf(w, u.w, a.w);
        b.x = fmaf(w, v.x, b.x);
        b.y = fmaf(w, v.y, b.y);
        b.z = fmaf(w, v.z, b.z);
        b.w = fmaf(w, v.w, b.w);
      }
      float4* o = reinterpret_cast<float4*>(P.out + (size_t)tok * P.d + col);
      o[0] = a;
      o[1] = b;
    }
  }
  // every warp has read the list before it is reset (the next item's
  // entries come after the next item's barriers)
  asm volatile("bar.sync 1, %0;" ::"r"(kDqWarps * 32) : "memory");
  if (tid == 0) fin[0] = 0;
}

template <bool W13>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
tc2_kernel(const __grid_constant__ CUtensorMap map_b, const __grid_constant__ CUtensorMap map_raw, const TcParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* rowscale = reinterpret_cast<float*>(smem + kOffRowscale);  // [2][128]
  uint64_t* raw_full = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* raw_empty = raw_full + kStagesRaw;
  uint64_t* full = raw_empty + kStagesRaw;   // [stage] leader: A slots of both CTAs written, both halves landed
  uint64_t* bfull = full + kStages;          // [stage] follower: its token half landed (relay's view)
  uint64_t* empty = bfull + kStages;         // [stage] both: the MMAs on the stage completed
  uint64_t* acc_full = empty + kStages;      // both: the item's accumulators are final
  uint64_t* acc_empty = acc_full + 1;        // leader: both CTAs' epilogues read the accumulators
  uint64_t* mma_done = acc_empty + 1;        // [2] both: every MMA of that issuer completed
  uint64_t* stopped = mma_done + 2;          // leader: 16 dequantisers and the relay published their counts
  int* ints = reinterpret_cast<int*>(smem + kOffInts);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ints);
  // ints[1]: abort flag (the leader's is the pair's), ints[2]: relayed count
  // (leader), ints[3]: follower producer's issued count, ints[4..19]:
  // stages signalled by each dequantiser of the pair (leader)
  cg::cluster_group cluster = cg::this_cluster();
  const uint32_t rank = cluster.block_rank();
  volatile int* abort_flag = cluster.map_shared_rank(ints + 1, 0);
  volatile int* relayed_l = cluster.map_shared_rank(ints + 2, 0);
  volatile int* f_issued = reinterpret_cast<volatile int*>(ints + 3);  // >= 0: copies issued; -1 - n: stopped after n
  volatile int* dq_arrived_l = cluster.map_shared_rank(ints + 4, 0);
  int* fin = reinterpret_cast<int*>(smem + kOffFin);  // [0]: entries, [1..]: tokens whose block is complete
  const uint64_t lim = P.wait_ns;

  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int items = P.counts[2] * P.mblocks;
  if (pair >= items) return;  // both CTAs of the pair leave together
  const int nk = P.K / kBK;
  const int nrs = (nk + kRawSteps - 1) / kRawSteps;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesRaw; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], kDqWarps);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 2 * kDqWarps + 2);  // 16 dequantisers, the leader's expect_tx, the relay
      mbar_init(&bfull[s], 1);
      mbar_init(&empty[s], 2);                // one commit per issuer (multicast)
    }
    mbar_init(acc_full, 2);
    mbar_init(acc_empty, 2 * kDqWarps);
    mbar_init(&mma_done[0], 1);
    mbar_init(&mma_done[1], 1);
    mbar_init(stopped, 2 * kDqWarps + 1);
    ints[1] = 0;
    ints[2] = 0;
    ints[3] = 0;
    for (int i = 0; i < 2 * kDqWarps; ++i) ints[4 + i] = 0;
    fin[0] = 0;
    mbar_fence_init();
  }
  __syncwarp();
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers initialised and TMEM allocated
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  if (warp == kRawWarp) {
    // ---------------- TMA producer: this CTA's packed weights ----------------
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      uint32_t g = 0;
      bool ok = true;
      for (int it = pair; it < items && ok; it += npairs) {
        const Item2 t = item2(P, it, rank);
        const int y0 = t.expert * P.rows_per_expert + t.first;
        for (int rs = 0; rs < nrs; ++rs, ++g) {
          const int s = g % kStagesRaw;
          if (!mbar_wait(&raw_empty[s], ((g / kStagesRaw) & 1) ^ 1u, abort_flag, P.err, kErrWaitTimeout, lim) ||
              *abort_flag) {
            ok = false;
            break;
          }
          mbar_expect_tx(&raw_full[s], 2 * kRawTileBytes);
          uint8_t* raw = smem + kOffRaw + s * 2 * kRawTileBytes;
          tma_load_2d_hint(raw, &map_raw, rs * kRawRowBytes, y0, &raw_full[s], pol);
          tma_load_2d_hint(raw + kRawTileBytes, &map_raw, rs * kRawRowBytes, y0 + P.acc_row_off + P.acc_idx_step,
                           &raw_full[s], pol);
        }
      }
      for (uint32_t q = g > kStagesRaw ? g - kStagesRaw : 0; q < g; ++q)
        mbar_wait_drain(&raw_full[q % kStagesRaw], (q / kStagesRaw) & 1, P.err, kErrWaitTimeout, lim);
    }
  } else if (warp == kBWarp) {
    // ---------------- TMA producer: this CTA's half of the token tile ----------------
    int slot_g[kStages];
    uint32_t slot_par = 0, slot_real = 0;
#pragma unroll
    for (int s = 0; s < kStages; ++s) slot_g[s] = -1;
    if (lane == 0) {
      uint32_t ph = 0;
      int g = 0;
      bool withhold = P.fault != 0 && pair == 0 && rank == 0;
      bool ok = true;
      for (int it = pair; it < items && ok; it += npairs) {
        const Item2 t = item2(P, it, rank);
        const int boxes = (t.half + kBBoxRows - 1) / kBBoxRows;
        for (int ks = 0; ks < nk; ++ks, ++g) {
          const int s = ks % t.nS;
          const uint32_t par = (ph >> s) & 1;
          if (!mbar_wait(&empty[s], par ^ 1u, abort_flag, P.err, kErrWaitTimeout, lim) || *abort_flag) {
            ok = false;
            break;
          }
          ph ^= 1u << s;
#pragma unroll
          for (int q = 0; q < kStages; ++q)  // unrolled: the records stay in registers
            if (q == s) slot_g[q] = g;
          slot_par = (slot_par & ~(1u << s)) | (par << s);
          if (withhold) {
            // fault injection: the leader's half of this tile never arrives,
            // so the issuers' wait on the stage runs out
            withhold = false;
            slot_real &= ~(1u << s);
            continue;
          }
          slot_real |= 1u << s;
          uint64_t* bar = rank == 0 ? &full[s] : &bfull[s];
          mbar_expect_tx(bar, boxes * kBoxBytes);
          uint8_t* b = smem + kOffB + s * kBHalfBytes;
          for (int i = 0; i < boxes; ++i)
            tma_load_2d(b + i * kBoxBytes, &map_b, ks * kBK, t.row0 + (int)rank * t.half + i * kBBoxRows, bar);
          if (rank == 1) {
            __threadfence_block();
            *f_issued = g + 1;  // the relay may now wait for this copy
          }
        }
      }
      if (rank == 1) {
        // stopped: -1 - (copies issued), so that the relay knows where to end
        __threadfence_block();
        *f_issued = -1 - g;
      }
    }
    // the leader's producer, after every dequantiser and the relay stopped:
    // let each of its copies still in flight complete its stage, adding the
    // arrivals of those that stopped before it, and wait for the bytes
    __syncwarp();
    if (rank == 0 && lane == 0) {
      wait_cl_drain(stopped, 0, P.err, 4 * lim);
      if (*abort_flag) {
        const int relayed = *relayed_l;
#pragma unroll
        for (int s = 0; s < kStages; ++s) {
          if (slot_g[s] < 0 || !((slot_real >> s) & 1)) continue;
          int missing = relayed > slot_g[s] ? 0 : 1;
          for (int w = 0; w < 2 * kDqWarps; ++w) missing += dq_arrived_l[w] > slot_g[s] ? 0 : 1;
          if (missing > 0) arrive_leader(&full[s], (uint32_t)missing);
          wait_cl_drain(&full[s], (slot_par >> s) & 1, P.err, lim);
        }
      }
    }
  } else if (warp == kMmaWarp || warp == kMma1Warp) {
    if (rank == 0) {
      // ---------------- leader: MMA issuers, one per accumulator ----------------
      if (lane == 0) {
        const int acc = warp == kMmaWarp ? 0 : 1;
        uint32_t ph = 0;
        int li = 0;
        bool ok = true;
        for (int it = pair; it < items && ok; it += npairs, ++li) {
          const Item2 t = item2(P, it, 0);
          if (li > 0 && !wait_cl(acc_empty, (li - 1) & 1, abort_flag, P.err, lim)) break;
          const uint32_t idesc = idesc_f16kind(2 * kBM, t.n_mma, 0u);
          const uint32_t d_tmem = tmem + t.acc0 + acc * t.acc_cols;
          for (int ks = 0; ks < nk; ++ks) {
            const int s = ks % t.nS;
            if (!wait_cl(&full[s], (ph >> s) & 1, abort_flag, P.err, lim)) {
              ok = false;
              break;
            }
            ph ^= 1u << s;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t b_addr = smem_u32(smem + kOffB + s * kBHalfBytes);
            const uint32_t a_tmem = tmem + (s * 2 + acc) * kASlotCols;
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              umma2_tmem_a(d_tmem, a_tmem + kk * 8, desc_sw128(b_addr + kk * 32), idesc, (ks > 0 || kk > 0) ? 1u : 0u);
            commit2_both(&empty[s]);
          }
          if (!ok) break;
          commit2_both(acc_full);
        }
        commit2_both(&mma_done[acc]);
        mbar_wait_drain(&mma_done[acc], 0, P.err, kErrWaitTimeout, lim);
      }
    } else if (warp == kMma1Warp) {
      // ---------------- follower: relay of its token copies ----------------
      if (lane == 0) {
        uint32_t ph = 0;
        int g = 0;
        bool done = false;
        for (int it = pair; it < items && !done; it += npairs) {
          const Item2 t = item2(P, it, 1);
          for (int ks = 0; ks < nk; ++ks, ++g) {
            const int s = ks % t.nS;
            const uint32_t par = (ph >> s) & 1;
            ph ^= 1u << s;
            // wait for the copy of stage g, or for the producer to stop short of it
            const uint64_t t0 = global_timer_ns();
            bool landed = false;
            while (true) {
              if (mbar_try_wait_sleep(&bfull[s], par)) {
                landed = true;
                break;
              }
              const int fi = *f_issued;
              if (fi < 0 && g >= -1 - fi) break;  // stopped before issuing it
              if (global_timer_ns() - t0 > lim) {
                *abort_flag = 1;
                atomicOr(P.err, kErrWaitTimeout);
                break;
              }
            }
            if (!landed) {
              done = true;
              break;
            }
            arrive_leader(&full[s]);
          }
        }
        *relayed_l = g;
        arrive_leader(stopped);
      }
    } else {
      // follower, warp 0: the leader's MMAs read this CTA's TMEM and shared
      // memory until they complete
      if (lane == 0) {
        mbar_wait_drain(&mma_done[0], 0, P.err, kErrWaitTimeout, lim);
        mbar_wait_drain(&mma_done[1], 0, P.err, kErrWaitTimeout, lim);
      }
    }
  } else {
    // ---------------- dequantisers (one weight row each), then the epilogue ----------------
    const int dq = warp - kFirstDqWarp;
    const int acc = dq >> 2;
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    const int kpr = P.K / 32;
    uint32_t ph = 0;
    uint32_t g = 0;
    int li = 0;
    int gdq = 0;
    bool ok = true;
    bool stop = false;
    for (int it = pair; it < items && !stop; it += npairs, ++li) {
      const Item2 t = item2(P, it, rank);
      // this row's index (i for W13, output feature for W2); rows past the
      // end read a valid row instead (their results are not written)
      const int idx = t.first + acc * P.acc_idx_step + r;
      const bool row_in = idx < P.limit;
      const int wrow = t.expert * P.rows_per_expert + acc * P.acc_row_off + (row_in ? idx : 0);
      const uint8_t* srow = P.scales + (size_t)wrow * kpr;
      int s_ref = 0;
      {
        uint32_t smax = 0;
        auto max4 = [](uint32_t m, uint32_t w4) {
          return max(m, max(max(w4 & 0xFFu, (w4 >> 8) & 0xFFu), max((w4 >> 16) & 0xFFu, w4 >> 24)));
        };
        if ((kpr & 15) == 0) {
          constexpr int kSv = 16;
          for (int i0 = 0; i0 < kpr; i0 += 16 * kSv) {
            uint4 sv[kSv];
#pragma unroll
            for (int i = 0; i < kSv; ++i)
              if (i0 + 16 * i < kpr) sv[i] = *reinterpret_cast<const uint4*>(srow + i0 + 16 * i);
#pragma unroll
            for (int i = 0; i < kSv; ++i)
              if (i0 + 16 * i < kpr) smax = max4(max4(max4(max4(smax, sv[i].x), sv[i].y), sv[i].z), sv[i].w);
          }
        } else {
          for (int i = 0; i < kpr; i += 4) smax = max4(smax, *reinterpret_cast<const uint32_t*>(srow + i));
        }
        s_ref = (int)smax - 13;
        rowscale[acc * 128 + r] = pow2f(s_ref - 127);
      }
      const bool vec_scales = (kpr & 15) == 0;
      uint4 sg_cur = make_uint4(0, 0, 0, 0), sg_next = make_uint4(0, 0, 0, 0);
      uint32_t sc_next = 0;
      if (vec_scales) {
        sg_next = *reinterpret_cast<const uint4*>(srow);
      } else {
        sc_next = *reinterpret_cast<const uint16_t*>(srow);
      }
#pragma unroll kDqUnroll
      for (int ks = 0; ks < nk; ++ks) {
        const int sa = ks % t.nS;
        const int sub = ks % kRawSteps;
        const uint32_t gs = g + ks / kRawSteps;
        const int rs_slot = gs % kStagesRaw;
        // once a wait has failed (or seen the abort) this lane stops waiting
        // but keeps converting, so that the warp-wide tcgen05 instructions
        // always see all 32 lanes
        if (sub == 0 && ok)
          ok = mbar_wait(&raw_full[rs_slot], (gs / kStagesRaw) & 1, abort_flag, P.err, kErrWaitTimeout, lim);
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
        if (ok) ok = mbar_wait(&empty[sa], ((ph >> sa) & 1) ^ 1u, abort_flag, P.err, kErrWaitTimeout, lim);
        ph ^= 1u << sa;
        const uint32_t s0 = sc & 0xFFu, s1 = (sc >> 8) & 0xFFu;
        const uint32_t m0 = f16x2_pow2((int)s0 - s_ref), m1 = f16x2_pow2((int)s1 - s_ref);
        uint32_t av[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t b[4];
          lds_bytes4((c < 4 ? raw_lo : raw_hi) + 4 * (c & 3), b);
          const uint32_t m = c < 4 ? m0 : m1;
#pragma unroll
          for (int i = 0; i < 4; ++i) av[4 * c + i] = f16x2_mul(e2m1x2_to_f16x2(b[i]), m);
        }
        if (sub == kRawSteps - 1 || ks == nk - 1) {
          __syncwarp();
          if (lane == 0 && ok) mbar_arrive(&raw_empty[rs_slot]);
        }
        tmem_st32(lane_base + (sa * 2 + acc) * kASlotCols, av);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncwarp();
        if (lane == 0 && ok) {
          arrive_leader(&full[sa]);
          ++gdq;
        }
      }
      g += nrs;
      // epilogue: the two warps of a lane quadrant take alternate 32-column
      // chunks of the tile (all n token rows: the accumulators hold them all)
      constexpr int kChunks = (kBN + 63) / 64;
      const int half = dq >> 2;
      float xs_pre[kChunks] = {};
#pragma unroll
      for (int i = 0; i < kChunks; ++i) {
        const int col = 32 * (2 * i + half) + lane;
        if (col < t.n) xs_pre[i] = P.x_scale[t.row0 + col];
      }
      asm volatile("bar.sync 1, %0;" ::"r"(kDqWarps * 32) : "memory");
      if (__all_sync(0xFFFFFFFFu, ok && mbar_wait(acc_full, li & 1, abort_flag, P.err, kErrWaitTimeout, lim))) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const float rs0 = rowscale[r], rs1 = rowscale[128 + r];
#pragma unroll
        for (int ci = 0; ci < kChunks; ++ci) {
          const int c0 = 32 * (2 * ci + half);
          if (c0 >= t.n_mma) break;
          float a0[32], a1[32];
          tmem_ld32x2(lane_base + t.acc0 + c0, lane_base + t.acc0 + t.acc_cols + c0, a0, a1);
          const float xs_l = xs_pre[ci];
          if (W13) {
            const int i = t.first + r;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float xs = __shfl_sync(0xFFFFFFFFu, xs_l, j);
              if (c0 + j < t.n && i < P.I)
                P.h_out[(size_t)(t.row0 + c0 + j) * P.I + i] =
                    f32_to_bf16_rn(swiglu(a0[j] * rs0 * xs, a1[j] * rs1 * xs));
            }
          } else {
            const int n0 = t.first + r, n1 = t.first + P.acc_idx_step + r;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float xs = __shfl_sync(0xFFFFFFFFu, xs_l, j);
              if (c0 + j < t.n) {
                float* yrow = P.y_out + (size_t)(t.row0 + c0 + j) * P.d;
                if (n0 < P.d) yrow[n0] = a0[j] * rs0 * xs;
                if (n1 < P.d) yrow[n1] = a1[j] * rs1 * xs;
              }
            }
          }
        }
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncwarp();
        if (lane == 0) arrive_leader(acc_empty);
      } else {
        ok = false;
      }
      // the combine reads these y rows from other SMs: publish them first
      if (!W13 && P.out != nullptr) __threadfence();
      uint32_t st;
      asm volatile(
          "{\n\t.reg .pred pin, pout;\n\tsetp.ne.u32 pin, %1, 0;\n\tbar.red.or.pred pout, 1, %2, pin;\n\t"
          "selp.u32 %0, 1, 0, pout;\n}"
          : "=r"(st)
          : "r"((!ok || *abort_flag) ? 1u : 0u), "r"(kDqWarps * 32)
          : "memory");
      stop = st != 0;
      if (!W13 && P.out != nullptr && !stop) combine_block(P, t, dq, lane, fin);
    }
    if (lane == 0) {
      dq_arrived_l[(int)rank * kDqWarps + dq] = gdq;
      arrive_leader(stopped);
    }
  }
  __syncwarp();
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while its peer may still reach into it
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

}  // namespace

template <bool W13>
cudaError_t launch_tc2(const CUtensorMap& b, const CUtensorMap& raw, const TcParams& P, int max_tiles,
                       cudaStream_t st) {
  const cudaError_t oe = ensure_smem_optin(reinterpret_cast<const void*>(tc2_kernel<W13>), kSmemTc2);
  if (oe != cudaSuccess) return oe;
  // one pair per two SMs, each looping over work items; no more pairs than items
  const long long most = (long long)max_tiles * P.mblocks;
  if (most > 0x3FFFFFFFLL) return cudaErrorInvalidValue;
  const int pairs = (int)std::min<long long>(most, num_sms() / 2);
  if (pairs <= 0) return cudaSuccess;
  tc2_kernel<W13><<<2 * pairs, kThreads, kSmemTc2, st>>>(b, raw, P);
  return cudaGetLastError();
}

template cudaError_t launch_tc2<true>(const CUtensorMap&, const CUtensorMap&, const TcParams&, int, cudaStream_t);
template cudaError_t launch_tc2<false>(const CUtensorMap&, const CUtensorMap&, const TcParams&, int, cudaStream_t);

}  // namespace moe_fp4
