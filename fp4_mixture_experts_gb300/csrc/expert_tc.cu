// Prefill-shaped expert projections on the 5th-generation tensor cores.
//
// A grouped GEMM per expert, swap-AB: the expert's weight rows are the UMMA M
// operand (128 rows per accumulator) and the expert's token rows the N
// operand (up to 128 per tile), so an expert with few rows wastes little of
// the MMA ("low-M utilisation" is a limit the DeepSeek-V4-Flash-on-gfx90a
// paper names).  One CTA computes two 128 x N accumulators that share the
// token tile: gate and up rows of W13 (so SwiGLU fuses into the epilogue), or
// two adjacent 128-row blocks of W2.
//
// Warp roles (192 threads):
//   warp 0      TMA producer: per 64-wide K step, the token tile (bf16, 128-byte
//               swizzle) and the two packed weight tiles (128 rows x 32 bytes)
//   warp 1      TMEM allocator and MMA issuer: 2 x 4 tcgen05.mma.kind::f16
//               (M=128, N=tile, K=16) per K step, fp32 accumulators in TMEM;
//               tcgen05.commit frees the stage
//   warps 2..5  dequantisers: one thread per weight row; E2M1 pairs decoded by
//               cvt.rn.f16x2.e2m1x2, moved to bf16 and scaled exactly by the
//               E8M0 power of two (mul.bf16x2), stored in the UMMA K-major
//               128-byte-swizzled layout; then the epilogue (tcgen05.ld,
//               SwiGLU + bf16 rounding of h, or fp32 y)
// Weights are dequantised exactly (an E2M1 value times a power of two has
// 2 significant bits), so the MMA multiplies the same bf16 products the
// definition does and accumulates them in fp32.  Every mbarrier wait is
// bounded; a timeout sets the error word and an abort flag that releases the
// other roles, and TMEM is always freed.
#include <cuda.h>
#include <cuda_fp16.h>

#include "moe_fp4_internal.cuh"
#include "ptx_sm103.cuh"

namespace moe_fp4 {
namespace {

constexpr int kBM = 128;                 // weight rows per accumulator
constexpr int kBK = 64;                  // K elements per stage
constexpr int kBN = kTcTileN;            // token rows per tile (<= 128)
constexpr int kStagesTc = 3;
constexpr int kNumDequantWarps = 4;
constexpr int kTcThreads = (2 + kNumDequantWarps) * 32;
constexpr uint32_t kTmemCols = 256;      // 2 accumulators x 128 columns

constexpr int kATileBytes = kBM * kBK * 2;        // 16 KB bf16
constexpr int kBTileBytes = kBN * kBK * 2;        // 16 KB bf16
constexpr int kRawTileBytes = kBM * kBK / 2;      // 4 KB packed
constexpr int kOffA = 0;                                       // [stage][acc]
constexpr int kOffB = kOffA + kStagesTc * 2 * kATileBytes;     // [stage]
constexpr int kOffRaw = kOffB + kStagesTc * kBTileBytes;       // [stage][acc]
constexpr int kOffBar = kOffRaw + kStagesTc * 2 * kRawTileBytes;
constexpr int kSmemTc = kOffBar + 256 + 1024;                  // + barriers, slack for 1 KB alignment

struct TcParams {
  const uint8_t* scales;   // E8M0 [rows][K/32]
  const int4* tiles;       // (expert, first sorted row, rows, 0)
  const int32_t* counts;   // counts[2] = number of tiles
  int32_t* err;
  uint16_t* h_out;         // W13: h [S, I]
  float* y_out;            // W2: y [S, d]
  int K;                   // reduction length
  int rows_per_expert;     // rows of the weight tensor per expert (2I or d)
  int mblocks;             // CTAs per token tile along the weight rows
  int block_rows;          // weight rows advanced per m-block (128 W13, 256 W2)
  int acc1_offset;         // row offset of accumulator 1 (I for up rows, 128 for W2)
  int I, d;
};

// UMMA shared-memory descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(16u >> 4) << 16;     // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024u >> 4) << 32;   // stride byte offset
  d |= (uint64_t)1 << 46;              // descriptor version
  d |= (uint64_t)2 << 61;              // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16: bf16 x bf16 -> f32, both K-major.
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
  return (1u << 4)                      // D format f32
         | (1u << 7) | (1u << 10)       // A, B format bf16
         | ((uint32_t)(N >> 3) << 17)   // N
         | ((uint32_t)(M >> 4) << 24);  // M
}

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// E8M0 byte s -> the bf16x2 factor (m, m) that turns the shifted bf16 pattern
// of an E2M1 value (its value times 2^-112) into value * 2^(s-127): m = 2^(s-15)
// for s <= 142; larger s take two factors (2^112, then 2^(s-127)).
__device__ __forceinline__ uint32_t bf16x2_pow2(int e_unbiased) {
  const uint32_t b = (uint32_t)(e_unbiased + 127) << 7;
  return b | (b << 16);
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// 4 packed bytes (8 E2M1 codes, K ascending) -> 8 exact bf16 values scaled by 2^(s-127)
__device__ __forceinline__ uint4 dequant8(uint32_t packed, uint32_t s) {
  uint32_t o[4];
  const bool big = s > 142;
  const uint32_t m1 = big ? bf16x2_pow2(112) : bf16x2_pow2((int)s - 15);
  const uint32_t m2 = bf16x2_pow2((int)s - 127);
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const uint32_t h2 = e2m1x2_to_f16x2((packed >> (8 * b)) & 0xFFu);
    // f16 -> bf16 bit pattern of value * 2^-112 (exponent and mantissa shift, sign kept)
    uint32_t v = ((h2 >> 3) & 0x0FFF0FFFu) | (h2 & 0x80008000u);
    v = bf16x2_mul(v, m1);
    if (big) v = bf16x2_mul(v, m2);
    o[b] = v;
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

template <bool W13>
__global__ void __launch_bounds__(kTcThreads, 1)
tc_kernel(const __grid_constant__ CUtensorMap map_raw, const __grid_constant__ CUtensorMap map_b, const TcParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* a_ready = full + kStagesTc;
  uint64_t* empty = a_ready + kStagesTc;
  uint64_t* acc_full = empty + kStagesTc;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tile = blockIdx.x / P.mblocks, mb = blockIdx.x % P.mblocks;
  if (tile >= P.counts[2]) return;
  const int4 tl = P.tiles[tile];
  const int e = tl.x, row0 = tl.y, n = tl.z;
  const int n_mma = (n + 15) & ~15;
  const int wrow0 = e * P.rows_per_expert + mb * P.block_rows;
  const int nk = P.K / kBK;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesTc; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&a_ready[s], kNumDequantWarps);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      for (int ks = 0; ks < nk; ++ks) {
        const int s = ks % kStagesTc;
        const uint32_t ph = (ks / kStagesTc) & 1;
        if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, P.err, kErrWaitTimeout)) break;
        mbar_expect_tx(&full[s], 2 * kRawTileBytes + kBTileBytes);
        tma_load_2d(smem + kOffRaw + (s * 2 + 0) * kRawTileBytes, &map_raw, ks * (kBK / 2), wrow0, &full[s]);
        tma_load_2d(smem + kOffRaw + (s * 2 + 1) * kRawTileBytes, &map_raw, ks * (kBK / 2), wrow0 + P.acc1_offset,
                    &full[s]);
        tma_load_2d(smem + kOffB + s * kBTileBytes, &map_b, ks * kBK, row0, &full[s]);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(kBM, n_mma);
      bool ok = true;
      for (int ks = 0; ks < nk && ok; ++ks) {
        const int s = ks % kStagesTc;
        const uint32_t ph = (ks / kStagesTc) & 1;
        if (!mbar_wait(&full[s], ph, abort_flag, P.err, kErrWaitTimeout) || !mbar_wait(&a_ready[s], ph, abort_flag, P.err, kErrWaitTimeout)) {
          ok = false;
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t b_addr = smem_u32(smem + kOffB + s * kBTileBytes);
#pragma unroll
        for (int acc = 0; acc < 2; ++acc) {
          const uint32_t a_addr = smem_u32(smem + kOffA + (s * 2 + acc) * kATileBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_bf16(tmem + acc * 128, desc_sw128(a_addr + kk * 32), desc_sw128(b_addr + kk * 32), idesc,
                      (ks > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&empty[s]);
      }
      umma_commit(acc_full);
      // the accumulators must be final before TMEM can be freed, also on an abort
      mbar_wait(acc_full, 0, abort_flag, P.err, kErrWaitTimeout);
    }
  } else {
    // ---------------- dequantisers, then the epilogue ----------------
    const int t = threadIdx.x - 64;       // weight row within the 128-row block
    const int kpr = P.K / 32;             // scale bytes per row
    const uint8_t* srow0 = P.scales + (size_t)(wrow0 + t) * kpr;
    const uint8_t* srow1 = P.scales + (size_t)(wrow0 + P.acc1_offset + t) * kpr;
    const int sw = t & 7;
    bool ok = true;
    for (int ks = 0; ks < nk; ++ks) {
      const int s = ks % kStagesTc;
      const uint32_t ph = (ks / kStagesTc) & 1;
      const uint32_t sc00 = srow0[2 * ks], sc01 = srow0[2 * ks + 1];
      const uint32_t sc10 = srow1[2 * ks], sc11 = srow1[2 * ks + 1];
      if (!mbar_wait(&full[s], ph, abort_flag, P.err, kErrWaitTimeout)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int acc = 0; acc < 2; ++acc) {
        const uint4* raw = reinterpret_cast<const uint4*>(smem + kOffRaw + (s * 2 + acc) * kRawTileBytes + t * 32);
        const uint4 r0 = raw[0], r1 = raw[1];
        const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
        uint8_t* arow = smem + kOffA + (s * 2 + acc) * kATileBytes + (t >> 3) * 1024 + (t & 7) * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t sc = acc == 0 ? (c < 4 ? sc00 : sc01) : (c < 4 ? sc10 : sc11);
          *reinterpret_cast<uint4*>(arow + ((c ^ sw) << 4)) = dequant8(w[c], sc);
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_ready[s]);
    }
    // epilogue: this warp reads TMEM lanes 32*(warp % 4) .. +31
    if (ok && mbar_wait(acc_full, 0, abort_flag, P.err, kErrWaitTimeout)) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int q = warp & 3;
      const int r = q * 32 + lane;  // row within the block
      for (int c0 = 0; c0 < n_mma; c0 += 32) {
        float a0[32], a1[32];
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + c0, a0);
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + 128 + c0, a1);
        if (W13) {
          const int i = mb * kBM + r;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (c0 + j < n) P.h_out[(size_t)(row0 + c0 + j) * P.I + i] = f32_to_bf16_rn(swiglu(a0[j], a1[j]));
        } else {
          const int nrow = mb * P.block_rows + r;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (c0 + j < n) {
              float* yrow = P.y_out + (size_t)(row0 + c0 + j) * P.d;
              yrow[nrow] = a0[j];
              if (nrow + P.acc1_offset < P.d) yrow[nrow + P.acc1_offset] = a1[j];  // last block may hold 128 rows
            }
          }
        }
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

template <bool W13>
cudaError_t launch_tc(const CUtensorMap& raw, const CUtensorMap& b, const TcParams& P, int max_tiles, cudaStream_t st) {
  static bool configured = false;
  if (!configured) {
    cudaFuncSetAttribute(tc_kernel<W13>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTc);
    configured = true;
  }
  const long long grid = (long long)max_tiles * P.mblocks;
  if (grid > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  tc_kernel<W13><<<(unsigned)grid, kTcThreads, kSmemTc, st>>>(raw, b, P);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_w13(const moe_fp4_dims& d, const uint8_t* w13, const uint8_t* w13s, const Workspace& ws,
                          cudaStream_t st) {
  const size_t S = (size_t)d.T * d.k;
  CUtensorMap raw, b;
  if (!make_map_2d(&raw, CU_TENSOR_MAP_DATA_TYPE_UINT8, w13, d.d / 2, (uint64_t)d.E * 2 * d.I, d.d / 2, kBK / 2, kBM,
                   CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map_2d(&b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ws.x_perm, d.d, S, (uint64_t)d.d * 2, kBK, kBN,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  TcParams P{};
  P.scales = w13s;
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
  return launch_tc<true>(raw, b, P, ws.max_tc_tiles, st);
}

cudaError_t launch_tc_w2(const moe_fp4_dims& d, const uint8_t* w2, const uint8_t* w2s, const Workspace& ws,
                         cudaStream_t st) {
  const size_t S = (size_t)d.T * d.k;
  CUtensorMap raw, b;
  if (!make_map_2d(&raw, CU_TENSOR_MAP_DATA_TYPE_UINT8, w2, d.I / 2, (uint64_t)d.E * d.d, d.I / 2, kBK / 2, kBM,
                   CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map_2d(&b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ws.h, d.I, S, (uint64_t)d.I * 2, kBK, kBN,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  TcParams P{};
  P.scales = w2s;
  P.tiles = ws.tc_tiles;
  P.counts = ws.counts;
  P.err = ws.err;
  P.y_out = ws.y;
  P.K = d.I;
  P.rows_per_expert = d.d;
  P.mblocks = (d.d + 2 * kBM - 1) / (2 * kBM);  // d % 256 == 128 leaves a 128-row last block
  P.block_rows = 2 * kBM;
  P.acc1_offset = kBM;
  P.I = d.I;
  P.d = d.d;
  return launch_tc<false>(raw, b, P, ws.max_tc_tiles, st);
}

}  // namespace moe_fp4
