// Block-scaled (MX) expert projections on the 5th-generation tensor cores.
//
// The layer with MXFP8 activations (readings of the quantised-activation
// variant: E4M3 elements, one E8M0 scale per 32 K elements; the paper
// quantises its decode activations, "DeepSeek-V4-Flash on AMD gfx90a",
// abstract: INT8 activation quantisation, and the MI250 blog names block-wise
// FP8 as the next gain).  The weights stay MXFP4 and reach the tensor core as
// they are: the TMA reads the packed E2M1 codes into shared memory in the
// padded layout the MMA takes (16 codes in 8 bytes, then 8 bytes of padding:
// tensor-map type 16U4_ALIGN16B), the E8M0 scales of both operands go to
// tensor memory, and tcgen05.mma kind::mxf8f6f4 (E2M1 x E4M3, K = 32 per
// instruction, fp32 accumulation) applies them: no software dequantisation.
//
// Scale factors in tensor memory (measured layout, scale_vec::1X): the scale
// of A row m is read from lane m, column base + m / 32, byte a_sf_id; the
// scale of B column n from lane 32 (m / 32) + n % 32 (the reading row's lane
// quadrant: each quadrant holds its own copy), column base + n / 32, byte
// b_sf_id.  A stage covers K = 128, four MMAs, whose scales are the four
// bytes of one 32-bit column word (a_sf_id = b_sf_id = the MMA's index).
//
// Work items as in the exact kernel: a token tile (<= 192 rows of one
// expert, swap-AB: weights are M, tokens N) times two 128-row weight blocks
// (W13: gate and up, SwiGLU in the epilogue; W2: two blocks of output
// features).  Warp roles: warp 9 the TMA producer (both weight blocks and
// the token tile of a stage, one expect_tx); warps 1..8 the scale writers
// (loaded from the scale arrays, written with tcgen05.st) and then the
// epilogue; warps 0 and 11 the MMA issuers, one per accumulator (warp 0 also
// owns TMEM).  The W13 epilogue writes h (bf16); the MXFP8 quantiser then
// writes h's MXFP8 form for W2 in a separate pass (the epilogue runs while
// the MMAs wait, so work moved out of it is work taken off the MMA's path).
// Waits are bounded; no warp leaves a loop early; on an abort the producer
// completes the stages the stopped scale writers left open and waits for its
// copies, and every MMA completes before TMEM is freed.
#include <cuda.h>

#include <algorithm>

#include "moe_fp4_internal.cuh"
#include "mx_common.cuh"
#include "ptx_sm103.cuh"
#include "tc_helpers.cuh"

namespace moe_fp4 {
namespace {

using namespace tc;

constexpr int kBM = 128;
constexpr int kBKs = 128;                  // K elements per stage (4 MMAs of K = 32)
constexpr int kBN = kTcTileN;              // <= 192 token rows per tile
// Ring depth: 3 stages for W13, 4 for W2 (measured).  The scale writers'
// loads hit L1 only while the rows they touch fit beside the stages: a W13
// scale row is 128 bytes (K = 4096), a W2 row 64; with 4 stages L1 is about
// 24 KB and the W13 rows no longer fit.
#ifndef MOE_MX_STAGES_W13
#define MOE_MX_STAGES_W13 3
#endif
#ifndef MOE_MX_STAGES_W2
#define MOE_MX_STAGES_W2 4
#endif
template <bool W13>
__host__ __device__ constexpr int mx_stages() {
  return W13 ? MOE_MX_STAGES_W13 : MOE_MX_STAGES_W2;
}
constexpr int kMaxStages = MOE_MX_STAGES_W13 > MOE_MX_STAGES_W2 ? MOE_MX_STAGES_W13 : MOE_MX_STAGES_W2;
constexpr int kWriters = 8;                // scale writers, then the epilogue
constexpr int kMmaWarp = 0;
constexpr int kFirstWriter = 1;
constexpr int kProdWarp = kFirstWriter + kWriters;  // 9
constexpr int kMma1Warp = kProdWarp + 2;            // 11 (warp 10 idles)
constexpr int kThreads = (kMma1Warp + 1) * 32;
constexpr int kBoxRows = 64;
constexpr int kATileBytes = kBM * 128;              // 128 rows x 128 bytes (128 padded E2M1 codes)
// transaction bytes of one weight tile: the copy counts the packed bytes it
// reads (64 a row), not the padded footprint it leaves in shared memory, and
// it leaves the padding bytes untouched (the MMA ignores them); measured
constexpr int kATileTxBytes = kBM * 64;
constexpr int kBTileBytes = ((kBN + kBoxRows - 1) / kBoxRows) * kBoxRows * 128;  // E4M3, 128 bytes a row
constexpr int kStageBytes = 2 * kATileBytes + kBTileBytes;
constexpr int kSfColsPerStage = 16;                 // SFA acc0 [0,4), acc1 [4,8), SFB [8, 8 + N/32)
constexpr uint32_t kTmemCols = 512;
constexpr int kOffStages = 0;
template <bool W13>
__host__ __device__ constexpr int mx_off_bar() {
  return kOffStages + mx_stages<W13>() * kStageBytes;
}
template <bool W13>
__host__ __device__ constexpr int mx_smem() {
  return mx_off_bar<W13>() + 256 + 1024;
}
static_assert(kStageBytes % 1024 == 0, "stages must stay 1 KB aligned for the 128-byte swizzle");
static_assert(mx_smem<true>() <= 227 * 1024 && mx_smem<false>() <= 227 * 1024, "shared memory exceeds 227 KB");
static_assert(2 * ((kBN + 31) / 32 * 32) + kMaxStages * kSfColsPerStage <= (int)kTmemCols, "TMEM columns exceeded");
static_assert((kBN + 31) / 32 <= kSfColsPerStage - 8, "B scale columns exceed the stage's share");

struct MxParams {
  const uint8_t* w_scales;    // E8M0 [rows][K/32] of the weights
  const uint8_t* b_scales;    // E8M0 [S][K/32] of the token rows (sorted order)
  const int4* tiles;
  const int32_t* counts;
  int32_t* err;
  uint16_t* h_out;            // W13: h bf16 [S, I]
  float* y_out;               // W2: y [S, d]
  int K;
  int rows_per_expert;        // 2I (W13) or d (W2)
  int mblocks;
  int block_rows;             // 128 (W13) or 256 (W2)
  int acc1_offset;            // I (W13: up rows) or 128 (W2)
  int I, d;
  uint64_t wait_ns;
  int fault;                  // nonzero: the first CTA withholds its first stage (fault-injection test)
};

// Block-scaled MMA: D (+)= A[smem] * B[smem] with the E8M0 scales of the
// given TMEM columns (byte sf of each word)
__device__ __forceinline__ void umma_mx(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                        uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n}" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
      : "memory");
}

// Instruction descriptor of kind::mxf8f6f4: A E2M1 (5), B E4M3 (0), E8M0
// scales, scale bytes sf of both operands.
__device__ __forceinline__ uint32_t idesc_mx(int M, int N, uint32_t sf) {
  return (sf << 4)                        // B scale byte
         | (5u << 7)                      // A format E2M1
         | ((uint32_t)(N >> 3) << 17)     // N
         | (1u << 23)                     // E8M0 scales
         | ((uint32_t)(M >> 4) << 24)     // M
         | (sf << 29);                    // A scale byte
}

__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

struct MxItem {
  int row0, n, n_mma, wrow0, mb, nsfb;
  uint32_t acc_cols;
};

// Every role reads the tile record of its next item one item ahead
// (mx_tile), so that no role waits on that load at an item boundary.
__device__ __forceinline__ int4 mx_tile(const MxParams& P, int item, int items) {
  return item < items ? P.tiles[item / P.mblocks] : make_int4(0, 0, 0, 0);
}

__device__ __forceinline__ MxItem mx_item(const MxParams& P, int item, const int4 tl) {
  MxItem t;
  t.mb = item % P.mblocks;
  t.row0 = tl.y;
  t.n = tl.z;
  t.n_mma = (t.n + 15) & ~15;
  t.acc_cols = (uint32_t)(t.n_mma + 31) & ~31u;
  t.nsfb = (t.n_mma + 31) / 32;
  t.wrow0 = tl.x * P.rows_per_expert + t.mb * P.block_rows;
  return t;
}

// One lane's scale words of one stage (four K blocks, one byte each): its
// weight row's for accumulator `half`, and for B chunks 2c + half its token
// row's (padding rows get 1.0, any finite scale would do).
struct MxScales {
  uint32_t a, b[3];
};

__device__ __forceinline__ MxScales mx_fetch(const MxParams& P, const MxItem& t, int half, int r, int lane, int kpr,
                                             int ks) {
  MxScales v;
  // rows past the expert (a W2 block of 128 features at the end) read a valid row
  const bool row_in = t.mb * P.block_rows + half * P.acc1_offset + r < P.rows_per_expert;
  const uint8_t* sa_row = P.w_scales + (size_t)(row_in ? t.wrow0 + half * P.acc1_offset + r : t.wrow0 + r) * kpr;
  v.a = *reinterpret_cast<const uint32_t*>(sa_row + 4 * ks);
#pragma unroll
  for (int c = 0; c < 3; ++c) {
    const int cb = 2 * c + half;
    const int n = cb * 32 + lane;
    v.b[c] = (cb < t.nsfb && n < t.n)
                 ? *reinterpret_cast<const uint32_t*>(P.b_scales + (size_t)(t.row0 + n) * kpr + 4 * ks)
                 : 0x7F7F7F7Fu;
  }
  return v;
}

template <bool W13>
__global__ void __launch_bounds__(kThreads, 1)
mx_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b, const MxParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int kStages = mx_stages<W13>();
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + mx_off_bar<W13>());  // [stage]: bytes landed, scales written
  uint64_t* empty = full + kStages;                               // [stage]: its MMAs completed
  uint64_t* acc_full = empty + kStages;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* mma_done = acc_empty + 1;                             // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* wr_arrived = abort_flag + 1;                      // [8]: stages each writer signalled
  const uint64_t lim = P.wait_ns;

  const int items = P.counts[2] * P.mblocks;
  if ((int)blockIdx.x >= items) return;
  const int nks = P.K / kBKs;
  const int kpr = P.K / 32;  // scale bytes per row
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], kWriters + 1);  // the writers and the producer's expect_tx
      mbar_init(&empty[s], 2);
    }
    mbar_init(acc_full, 2);
    mbar_init(acc_empty, kWriters);
    mbar_init(&mma_done[0], 1);
    mbar_init(&mma_done[1], 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncwarp();
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  // TMEM: accumulators at [0, 2 acc_cols) (acc_cols <= 192), scale ring from column 384
  const uint32_t sf_base = 2u * ((kBN + 31) / 32 * 32);

  if (warp == kProdWarp) {
    // ---------------- TMA producer: both weight blocks and the token tile ----------------
    uint32_t ph = 0;
    int g = 0;  // stages passed (issued, or withheld by the fault injection)
    const bool fault_cta = P.fault != 0 && blockIdx.x == 0;
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      bool ok = true;
      int4 tl = mx_tile(P, blockIdx.x, items);
      for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
        const MxItem t = mx_item(P, it, tl);
        tl = mx_tile(P, it + gridDim.x, items);
        const int boxes = (t.n_mma + kBoxRows - 1) / kBoxRows;
        for (int ks = 0; ks < nks; ++ks, ++g) {
          const int s = g % kStages;
          if (!mbar_wait(&empty[s], ((ph >> s) & 1) ^ 1u, abort_flag, P.err, kErrWaitTimeout, lim)) {
            ok = false;
            break;
          }
          ph ^= 1u << s;
          // fault injection: the first stage of the first CTA never arrives,
          // so the MMA issuers' wait on it runs out
          if (fault_cta && g == 0) continue;
          uint8_t* st = smem + kOffStages + s * kStageBytes;
          mbar_expect_tx(&full[s], 2 * kATileTxBytes + boxes * kBoxRows * 128);
          tma_load_2d_hint(st, &map_a, ks * kBKs, t.wrow0, &full[s], pol);
          tma_load_2d_hint(st + kATileBytes, &map_a, ks * kBKs, t.wrow0 + P.acc1_offset, &full[s], pol);
          for (int i = 0; i < boxes; ++i)
            tma_load_2d(st + 2 * kATileBytes + i * kBoxRows * 128, &map_b, ks * kBKs, t.row0 + i * kBoxRows, &full[s]);
        }
      }
    }
    // after an abort: complete the stages the stopped writers left open and
    // wait for their bytes (the ring is one sequence: stage g in slot g % 3)
    __syncwarp();
    asm volatile("bar.sync 3, %0;" ::"r"((kWriters + 1) * 32) : "memory");
    if (lane == 0 && *abort_flag) {
      for (int q = g > kStages ? g - kStages : 0; q < g; ++q) {
        if (fault_cta && q == 0) continue;  // withheld: no copy to wait for
        const int s = q % kStages;
        int arrived = 0;
        for (int w = 0; w < kWriters; ++w) arrived += wr_arrived[w] > q ? 1 : 0;
        if (arrived < kWriters)
          asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(&full[s])), "r"(kWriters - arrived)
                       : "memory");
        mbar_wait_drain(&full[s], (q / kStages) & 1, P.err, kErrWaitTimeout, lim);
      }
    }
  } else if (warp == kMmaWarp || warp == kMma1Warp) {
    // ---------------- MMA issuers, one per accumulator ----------------
    if (lane == 0) {
      const int acc = warp == kMmaWarp ? 0 : 1;
      int g = 0, li = 0;
      bool ok = true;
      int4 tl = mx_tile(P, blockIdx.x, items);
      for (int it = blockIdx.x; it < items && ok; it += gridDim.x, ++li) {
        const MxItem t = mx_item(P, it, tl);
        tl = mx_tile(P, it + gridDim.x, items);
        if (li > 0 && !mbar_wait(acc_empty, (li - 1) & 1, abort_flag, P.err, kErrWaitTimeout, lim)) break;
        const uint32_t d_tmem = tmem + acc * t.acc_cols;
        for (int ks = 0; ks < nks; ++ks, ++g) {
          const int s = g % kStages;
          if (!mbar_wait(&full[s], (g / kStages) & 1, abort_flag, P.err, kErrWaitTimeout, lim)) {
            ok = false;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint8_t* st = smem + kOffStages + s * kStageBytes;
          const uint32_t a_addr = smem_u32(st + acc * kATileBytes), b_addr = smem_u32(st + 2 * kATileBytes);
          const uint32_t sf = tmem + sf_base + s * kSfColsPerStage;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_mx(d_tmem, desc_sw128(a_addr + kk * 32), desc_sw128(b_addr + kk * 32), idesc_mx(kBM, t.n_mma, kk),
                    sf + acc * 4, sf + 8, (ks > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&empty[s]);
        }
        if (!ok) break;
        umma_commit(acc_full);
      }
      umma_commit(&mma_done[acc]);
      mbar_wait_drain(&mma_done[acc], 0, P.err, kErrWaitTimeout, lim);
    }
  } else if (warp != kProdWarp + 1) {
    // ---------------- scale writers, then the epilogue ----------------
    const int wr = warp - kFirstWriter;       // 0..7
    const int q = warp & 3;                   // lane quadrant this warp may access
    const int half = wr >> 2;                 // 0: acc0 scales + even B chunks; 1: acc1 + odd
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    const int r = q * 32 + lane;              // weight row (within the block) = TMEM lane
    int g = 0, li = 0, garr = 0;
    bool ok = true, stop = false;
    // The scale words of a stage come from global memory (L2); they are
    // fetched two stages ahead, and the next item's first two stages before
    // the epilogue, so that their latency stays off the pipeline.
    MxItem t = mx_item(P, blockIdx.x, mx_tile(P, blockIdx.x, items));
    MxScales q0 = mx_fetch(P, t, half, r, lane, kpr, 0);
    MxScales q1 = mx_fetch(P, t, half, r, lane, kpr, nks > 1 ? 1 : 0);
    for (int it = blockIdx.x; it < items && !stop; it += gridDim.x, ++li) {
      const int4 tl_next = mx_tile(P, it + gridDim.x, items);
      for (int ks = 0; ks < nks; ++ks, ++g) {
        const int s = g % kStages;
        const MxScales cur = q0;
        q0 = q1;
        if (ks + 2 < nks) q1 = mx_fetch(P, t, half, r, lane, kpr, ks + 2);
        const uint32_t wa = cur.a;
        const uint32_t wb[3] = {cur.b[0], cur.b[1], cur.b[2]};
        if (ok) ok = mbar_wait(&empty[s], ((g / kStages) & 1) ^ 1u, abort_flag, P.err, kErrWaitTimeout, lim);
        const uint32_t sf = lane_base + sf_base + s * kSfColsPerStage;
        tmem_st1(sf + half * 4 + q, wa);     // A scales: column base + quadrant
#pragma unroll
        for (int c = 0; c < 3; ++c)
          if (2 * c + half < t.nsfb) tmem_st1(sf + 8 + 2 * c + half, wb[c]);  // B scales, this quadrant's copy
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncwarp();
        if (lane == 0 && ok) {
          mbar_arrive(&full[s]);
          ++garr;
        }
      }
      // ---------------- epilogue ----------------
      const MxItem tc = t;
      if (it + (int)gridDim.x < items) {
        t = mx_item(P, it + gridDim.x, tl_next);
        q0 = mx_fetch(P, t, half, r, lane, kpr, 0);
        q1 = mx_fetch(P, t, half, r, lane, kpr, nks > 1 ? 1 : 0);
      }
      if (__all_sync(0xFFFFFFFFu, ok && mbar_wait(acc_full, li & 1, abort_flag, P.err, kErrWaitTimeout, lim))) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        constexpr int kChunks = (kBN + 63) / 64;
#pragma unroll
        for (int ci = 0; ci < kChunks; ++ci) {
          const int c0 = 32 * (2 * ci + half);
          if (c0 >= tc.n_mma) break;
          float a0[32], a1[32];
          tmem_ld32x2(lane_base + c0, lane_base + tc.acc_cols + c0, a0, a1);
          if (W13) {
            // all 32 columns are computed (those past the tile's rows too: no
            // side effects), so that the 32 independent chains interleave;
            // only the stores are predicated
            const int i = tc.mb * kBM + r;
            const int nj = min(32, tc.n - c0);
            uint16_t* hp = P.h_out + (size_t)(tc.row0 + c0) * P.I + i;
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              // two columns per conversion (cvt.rn.bf16x2.f32)
              const __nv_bfloat162 hb = __floats2bfloat162_rn(swiglu(a0[j], a1[j]), swiglu(a0[j + 1], a1[j + 1]));
              if (j < nj) hp[(size_t)j * P.I] = __bfloat16_as_ushort(__low2bfloat16(hb));
              if (j + 1 < nj) hp[(size_t)(j + 1) * P.I] = __bfloat16_as_ushort(__high2bfloat16(hb));
            }
          } else {
            // 8-byte stores of two adjacent features: for the token pair (j,
            // j + 1) the even lane of each lane pair takes token j and the odd
            // lane token j + 1, swapping one value with its neighbour
            const bool odd = lane & 1;
            const int nrow = tc.mb * P.block_rows + (r & ~1);  // the pair's first feature
            const bool second_in = nrow + P.acc1_offset < P.d;  // last block may hold 128 rows
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              const float o0 = __shfl_xor_sync(0xFFFFFFFFu, odd ? a0[j] : a0[j + 1], 1);
              const float o1 = __shfl_xor_sync(0xFFFFFFFFu, odd ? a1[j] : a1[j + 1], 1);
              const int jj = j + (odd ? 1 : 0);
              if (c0 + jj < tc.n) {
                float* yrow = P.y_out + (size_t)(tc.row0 + c0 + jj) * P.d + nrow;
                *reinterpret_cast<float2*>(yrow) = odd ? make_float2(o0, a0[j + 1]) : make_float2(a0[j], o0);
                if (second_in)
                  *reinterpret_cast<float2*>(yrow + P.acc1_offset) =
                      odd ? make_float2(o1, a1[j + 1]) : make_float2(a1[j], o1);
              }
            }
          }
        }
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty);
      } else {
        ok = false;
      }
      uint32_t st;
      asm volatile(
          "{\n\t.reg .pred pin, pout;\n\tsetp.ne.u32 pin, %1, 0;\n\tbar.red.or.pred pout, 1, %2, pin;\n\t"
          "selp.u32 %0, 1, 0, pout;\n}"
          : "=r"(st)
          : "r"((!ok || *abort_flag) ? 1u : 0u), "r"(kWriters * 32)
          : "memory");
      stop = st != 0;
    }
    if (lane == 0) wr_arrived[wr] = garr;
    asm volatile("bar.arrive 3, %0;" ::"r"((kWriters + 1) * 32) : "memory");
  }
  __syncwarp();
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

template <bool W13>
cudaError_t launch_mx(const CUtensorMap& a, const CUtensorMap& b, const MxParams& P, int max_tiles, cudaStream_t st) {
  constexpr int kSmemMx = mx_smem<W13>();
  const cudaError_t oe = ensure_smem_optin(reinterpret_cast<const void*>(mx_kernel<W13>), kSmemMx);
  if (oe != cudaSuccess) return oe;
  const long long most = (long long)max_tiles * P.mblocks;
  if (most > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  const int grid = (int)std::min<long long>(most, num_sms());
  if (grid <= 0) return cudaSuccess;
  mx_kernel<W13><<<grid, kThreads, kSmemMx, st>>>(a, b, P);
  return cudaGetLastError();
}

// One warp per sorted row: x[sorted_slot[r] / k] quantised to MXFP8 (codes
// [S, d], scales [S, d/32]), each lane taking 32-element blocks.
__global__ void __launch_bounds__(256)
gather_mx_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ sorted_slot, int S, int k, int d,
                 uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  const int nb = d / 32;
  for (int r = warp; r < S; r += nwarps) {
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)(sorted_slot[r] / k) * d);
    for (int b = lane; b < nb; b += 32) {
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 q = src[4 * b + i];
        w[4 * i] = q.x;
        w[4 * i + 1] = q.y;
        w[4 * i + 2] = q.z;
        w[4 * i + 3] = q.w;
      }
      uint32_t amax = 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) amax = max(amax, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
      const uint32_t sb = mx_scale_byte(amax);
      uint32_t out[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t a = w[2 * i], c = w[2 * i + 1];
        out[i] = sb == 0xFFu ? 0x7F7F7F7Fu
                             : mx_e4m3_code(a & 0xFFFFu, sb) | (mx_e4m3_code(a >> 16, sb) << 8) |
                                   (mx_e4m3_code(c & 0xFFFFu, sb) << 16) | (mx_e4m3_code(c >> 16, sb) << 24);
      }
      uint4* dst = reinterpret_cast<uint4*>(codes + (size_t)r * d + 32 * b);
      dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
      dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
      scales[(size_t)r * nb + b] = (uint8_t)sb;
    }
  }
}

bool map_fp4(CUtensorMap* m, const uint8_t* w, uint64_t K, uint64_t rows) {
  // packed E2M1 codes read as 4-bit elements, written to shared memory padded
  // (16 codes in 8 bytes, then 8 bytes of padding), 128 codes x 128 rows a box
  return make_map_2d(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, w, K, rows, K / 2, 128, kBM,
                     CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

cudaError_t launch_mx_forward(const moe_fp4_dims& d, const uint16_t* x, const uint8_t* w13, const uint8_t* w13s,
                              const uint8_t* w2, const uint8_t* w2s, const Workspace& ws, cudaStream_t st,
                              const std::function<void(int)>& mark) {
  const size_t S = (size_t)d.T * d.k;
  // quantising gather of x into sorted order
  {
    int blocks = (int)std::min<size_t>((S + 7) / 8, (size_t)num_sms() * 16);
    gather_mx_kernel<<<blocks, 256, 0, st>>>(x, ws.sorted_slot, (int)S, d.k, d.d, ws.xq, ws.xq_scales);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (mark) mark(2);
  CUtensorMap a, b;
  // W13: weights [E*2I rows][d], tokens xq [S][d]
  if (!map_fp4(&a, w13, d.d, (uint64_t)d.E * 2 * d.I) ||
      !make_map_2d(&b, CU_TENSOR_MAP_DATA_TYPE_UINT8, ws.xq, d.d, S, d.d, 128, kBoxRows, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  MxParams P{};
  P.w_scales = w13s;
  P.b_scales = ws.xq_scales;
  P.tiles = ws.tc_tiles;
  P.counts = ws.counts;
  P.err = ws.err;
  P.h_out = ws.h;
  P.K = d.d;
  P.rows_per_expert = 2 * d.I;
  P.mblocks = d.I / kBM;
  P.block_rows = kBM;
  P.acc1_offset = d.I;
  P.I = d.I;
  P.d = d.d;
  P.wait_ns = wait_limit_ns();
  P.fault = fault_site() == MOE_FP4_FAULT_TC_TOKEN_TILE;
  cudaError_t e = launch_mx<true>(a, b, P, ws.max_tc_tiles, st);
  if (e != cudaSuccess) return e;
  if (mark) mark(3);
  // h in MXFP8 for W2 (a separate HBM-bound pass: cheaper than quantising
  // inside the W13 epilogue, whose time the MMAs cannot overlap)
  e = launch_mxfp8_quantize(ws.h, (long long)S, d.I, ws.hq, ws.hq_scales, st);
  if (e != cudaSuccess) return e;
  // W2: weights [E*d rows][I], tokens hq [S][I]
  if (!map_fp4(&a, w2, d.I, (uint64_t)d.E * d.d) ||
      !make_map_2d(&b, CU_TENSOR_MAP_DATA_TYPE_UINT8, ws.hq, d.I, S, d.I, 128, kBoxRows, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  MxParams Q{};
  Q.w_scales = w2s;
  Q.b_scales = ws.hq_scales;
  Q.tiles = ws.tc_tiles;
  Q.counts = ws.counts;
  Q.err = ws.err;
  Q.y_out = ws.y;
  Q.K = d.I;
  Q.rows_per_expert = d.d;
  Q.mblocks = (d.d + 2 * kBM - 1) / (2 * kBM);
  Q.block_rows = 2 * kBM;
  Q.acc1_offset = kBM;
  Q.I = d.I;
  Q.d = d.d;
  Q.wait_ns = wait_limit_ns();
  return launch_mx<false>(a, b, Q, ws.max_tc_tiles, st);
}

}  // namespace moe_fp4
