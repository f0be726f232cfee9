// Router projection ahead of top-k: logits[t, e] = sum_K x[t, K] * Wg[e, K].
//
// The step before routing (the gate network of the MoE layer).  The MI250
// correctness blog lets this projection take low-precision inputs with FP32
// accumulation and requires the top-k comparison in FP32 (section 4.1 and
// its table): x and Wg are bf16, every product is exact in fp32, the sums are
// fp32 and the logits fp32.
//
// Warp-level tensor-core MMAs (mma.sync m16n8k16, bf16 in, fp32 out):
// experts are the M rows (16 per tile), tokens the N columns (8 per tile).
// The K order inside each 32-element chunk is permuted identically for both
// operands (the sum does not depend on it, and the products are exact), so
// that each thread loads 16 contiguous bytes of a row per chunk: thread t of
// a quad owns elements 8t .. 8t+7, the first four for the chunk's first
// 16-wide step and the last four for the second.  A CTA splits K among its
// warp groups; the partial sums are added in shared memory in a fixed order,
// so the logits are deterministic.
#include "moe_fp4_internal.cuh"

namespace moe_fp4 {
namespace {

constexpr int kRouterThreads = 256;  // 8 warps

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 ld_row16(const uint16_t* base, size_t row_elems, int row, int nrows, int k) {
  if (row >= nrows) return make_uint4(0, 0, 0, 0);
  return __ldg(reinterpret_cast<const uint4*>(base + (size_t)row * row_elems + k));
}

// CTA tile: (16 MT WM) experts x (8 NT WN) tokens; WM x WN x KS = 8 warps,
// the KS warp groups taking interleaved 32-element K chunks.
template <int MT, int NT, int WM, int WN, int KS>
__global__ void __launch_bounds__(kRouterThreads)
router_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ wg, int T, int E, int d,
              float* __restrict__ logits) {
  static_assert(WM * WN * KS == 8, "8 warps");
  constexpr int TE = 16 * MT * WM, TT = 8 * NT * WN;
  __shared__ float part[KS > 1 ? KS - 1 : 1][TE][TT + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int ks = warp / (WM * WN), wmn = warp % (WM * WN);
  const int wm = wmn % WM, wn = wmn / WM;
  const int e0 = blockIdx.x * TE + wm * 16 * MT;   // this warp's first expert row
  const int n0 = blockIdx.y * TT + wn * 8 * NT;    // this warp's first token
  float acc[MT][NT][4];
#pragma unroll
  for (int i = 0; i < MT; ++i)
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[i][j][0] = acc[i][j][1] = acc[i][j][2] = acc[i][j][3] = 0.f;
  const int nchunks = d / 32;
#pragma unroll 2
  for (int c = ks; c < nchunks; c += KS) {
    const int k = c * 32 + 8 * t;
    uint4 ra[MT][2], rb[NT];
#pragma unroll
    for (int i = 0; i < MT; ++i) {
      ra[i][0] = ld_row16(wg, d, e0 + 16 * i + g, E, k);
      ra[i][1] = ld_row16(wg, d, e0 + 16 * i + g + 8, E, k);
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) rb[j] = ld_row16(x, d, n0 + 8 * j + g, T, k);
#pragma unroll
    for (int i = 0; i < MT; ++i)
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        mma_bf16_16816(acc[i][j], ra[i][0].x, ra[i][1].x, ra[i][0].y, ra[i][1].y, rb[j].x, rb[j].y);
        mma_bf16_16816(acc[i][j], ra[i][0].z, ra[i][1].z, ra[i][0].w, ra[i][1].w, rb[j].z, rb[j].w);
      }
  }
  // accumulator (i, j): c0, c1 = expert row g, tokens 2t, 2t+1; c2, c3 = row g + 8
  const int le0 = wm * 16 * MT, ln0 = wn * 8 * NT;  // offsets inside the CTA tile
  if (KS > 1 && ks > 0) {
#pragma unroll
    for (int i = 0; i < MT; ++i)
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q)
          part[ks - 1][le0 + 16 * i + g + 8 * (q >> 1)][ln0 + 8 * j + 2 * t + (q & 1)] = acc[i][j][q];
  }
  if (KS > 1) __syncthreads();
  if (ks != 0) return;
#pragma unroll
  for (int i = 0; i < MT; ++i)
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int le = le0 + 16 * i + g + 8 * (q >> 1), ln = ln0 + 8 * j + 2 * t + (q & 1);
        float v = acc[i][j][q];
#pragma unroll
        for (int p = 0; p < KS - 1; ++p) v += part[p][le][ln];  // fixed order: group 0, 1, 2, ...
        const int e = blockIdx.x * TE + le, n = blockIdx.y * TT + ln;
        if (e < E && n < T) logits[(size_t)n * E + e] = v;
      }
}

}  // namespace

cudaError_t launch_router(const moe_fp4_dims& d, const uint16_t* x, const uint16_t* wg, float* logits,
                          cudaStream_t st) {
  // small batches: 16 experts x 32 tokens per CTA, K split 8 ways (many CTAs
  // read the gate weights once); large batches: 64 x 64 tiles, K split 2 ways
  // (less L2 traffic per product)
  const long long small_ctas = (long long)((d.E + 15) / 16) * ((d.T + 31) / 32);
  if (small_ctas <= 2LL * num_sms()) {
    dim3 grid((d.E + 15) / 16, (d.T + 31) / 32);
    router_kernel<1, 4, 1, 1, 8><<<grid, kRouterThreads, 0, st>>>(x, wg, d.T, d.E, d.d, logits);
  } else {
    dim3 grid((d.E + 63) / 64, (d.T + 63) / 64);
    if (grid.y > 65535) return cudaErrorInvalidValue;
    router_kernel<2, 4, 2, 2, 2><<<grid, kRouterThreads, 0, st>>>(x, wg, d.T, d.E, d.d, logits);
  }
  return cudaGetLastError();
}

}  // namespace moe_fp4
