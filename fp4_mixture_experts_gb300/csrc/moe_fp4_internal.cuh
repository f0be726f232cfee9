// Internal declarations shared by the CUDA translation units of the FP4
// routed-MoE library: workspace layout, launch helpers and small device
// utilities (MXFP4 decoding, bf16 rounding).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <functional>

#include "../../include/moe_fp4.h"

namespace moe_fp4 {

constexpr int kRouteTokensPerBlock = 32;   // tokens per routing block (8 warps x 4)
constexpr int kRouteThreads = 256;
constexpr int kGemvTokens = 8;             // token rows per streaming-GEMV chunk (the MMA N = 8)
#ifndef MOE_TC_TILE_N
#define MOE_TC_TILE_N 192
#endif
constexpr int kTcTileN = MOE_TC_TILE_N;    // max token rows per tensor-core tile (UMMA N, a multiple of 64)
// An expert whose rows need several tiles takes tiles of at most
// kTcTileMultiN rows on the exact tensor-core path: a tile above 160 rows
// leaves TMEM room for a 2-deep A ring only, and more tiles of <= 160 rows
// (3- or 4-deep) measured faster there (large layer W13 6.40 -> 5.88 ms,
// skewed 0.614 -> 0.543 ms), while one tile per expert stays best up to 192
// rows (prefill).  The block-scaled path keeps its A operand in shared memory
// and uses kTcTileN throughout.
constexpr int kTcTileMultiN = 160;

// Tensor-core tiles of an expert with cnt rows: one tile up to kTcTileN rows,
// else ceil(cnt / multi) tiles (multi <= kTcTileN).
__host__ __device__ inline int tc_tile_count(int cnt, int multi) {
  return cnt <= 0 ? 0 : cnt <= kTcTileN ? 1 : (cnt + multi - 1) / multi;
}

// Device error word values (moe_fp4_check).
constexpr int kErrBadExpertId = 1;
constexpr int kErrWaitTimeout = 2;

// Pointers into the caller's workspace; every region starts on a 256-byte boundary.
struct Workspace {
  int32_t* err;           // [4]    device error words
  int32_t* counts;        // [4]    n_active, n_gemv_chunks, n_tc_tiles, 0
  int32_t* active;        // [E]    experts with >= 1 row, ascending
  int32_t* block_hist;    // [nb*E] per routing block expert counts, then bases
  int32_t* topk_ids;      // [S]
  float* topk_w;          // [S]
  int32_t* offsets;       // [E+1]
  int32_t* sorted_slot;   // [S]
  int32_t* slot_pos;      // [S]
  int4* gemv_chunks;      // [max_gemv_chunks]  (expert, first sorted row, rows, 0)
  int4* tc_tiles;         // [max_tc_tiles]     (expert, first sorted row, rows, 0)
  uint16_t* x_perm;       // [S, d] f16, each row scaled by a power of two (tensor-core path)
  float* x_scale;         // [S]    the inverse of that power of two
  uint16_t* h;            // [S, I] bf16
  uint16_t* h16;          // [S, I] f16 copy of h, each row scaled by a power of two (tensor-core W2);
                          //        shares x_perm's region, which is dead once W13 has run
  float* h_scale;         // [S]    the inverse of that power of two (shares x_scale's region)
  float* y;               // [S, d] fp32 expert outputs in sorted-row order
  int32_t* combine_cnt;   // [T, ceil(d/256)] per (token, 256-feature block): slots whose y is written
                          //        (tensor-core path; zeroed by the token gather of each call)
  // block-scaled (MX) layer only: MXFP8 operands in sorted-row order
  uint8_t* xq;            // [S, d] E4M3 codes of x   (in x_perm's region)
  uint8_t* hq;            // [S, I] E4M3 codes of h   (in x_perm's region, after xq)
  uint8_t* xq_scales;     // [S, d/32] E8M0
  uint8_t* hq_scales;     // [S, I/32] E8M0
  // staging for the host-buffer entry point (only laid out when requested)
  uint16_t* stage_x;      // [T, d]
  float* stage_logits;    // [T, E]
  float* stage_out;       // [T, d]
  size_t total;
  int nb_route;
  int max_gemv_chunks;
  int max_tc_tiles;
};

// Lays the workspace out from `base` (nullptr: sizes only).  Returns false for
// unsupported sizes.  with_staging: host-buffer staging regions; mx: the
// MXFP8 operand regions of the block-scaled layer.
bool layout_workspace(const moe_fp4_dims& d, void* base, bool with_staging, Workspace* ws, bool mx = false);

// TMA tensor map of a 2-D row-major array (inner = contiguous dimension, in
// elements); false if the driver rejects it.
bool make_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);
// SM count of the current device (cached per device).
int num_sms();
// Raises the kernel's dynamic shared memory limit to `bytes` on the current
// device, once per (kernel, device); returns the CUDA error of the attempt.
cudaError_t ensure_smem_optin(const void* kernel, int bytes);
// Fault-injection setting of moe_fp4_set_fault_injection (process-wide) and
// the limit of every pipeline wait (2 s unless a fault test lowers it).
int fault_site();
uint64_t wait_limit_ns();

// ---- launchers (one per kernel family; each returns cudaGetLastError()) ----
// tile_multi: the tile cap of experts with several tiles (kTcTileMultiN for
// the exact tensor-core path, kTcTileN for the block-scaled one)
cudaError_t launch_route(const moe_fp4_dims& d, const float* logits, const Workspace& ws, cudaStream_t st,
                         int tile_multi = kTcTileMultiN);
cudaError_t launch_gather(const moe_fp4_dims& d, const uint16_t* x, const Workspace& ws, cudaStream_t st);
cudaError_t launch_h_f16(const moe_fp4_dims& d, const Workspace& ws, cudaStream_t st);
cudaError_t launch_gemv_w13(const moe_fp4_dims& d, const uint16_t* x, const uint8_t* w13,
                            const uint8_t* w13s, const Workspace& ws, cudaStream_t st);
cudaError_t launch_gemv_w2(const moe_fp4_dims& d, const uint8_t* w2, const uint8_t* w2s,
                           const Workspace& ws, cudaStream_t st);
bool stream_path_supported(const moe_fp4_dims& d);
// zero_out non-null: the kernel zeroes out (T x d fp32) for the W2 kernel's combine
cudaError_t launch_stream_w13(const moe_fp4_dims& d, const uint16_t* x, const uint8_t* w13, const uint8_t* w13s,
                              const Workspace& ws, float* zero_out, cudaStream_t st);
// out non-null: the W2 epilogue adds each slot's weighted row into out (zeroed
// beforehand) instead of writing y for the combine kernel
cudaError_t launch_stream_w2(const moe_fp4_dims& d, const uint8_t* w2, const uint8_t* w2s, const Workspace& ws,
                             float* out, cudaStream_t st);
cudaError_t launch_stream_fused(const moe_fp4_dims& d, const uint16_t* x, const uint8_t* w13, const uint8_t* w13s,
                                const uint8_t* w2, const uint8_t* w2s, const Workspace& ws, float* out,
                                cudaStream_t st);
cudaError_t launch_tc_w13(const moe_fp4_dims& d, const uint8_t* w13, const uint8_t* w13s, const Workspace& ws,
                          bool pairs, cudaStream_t st);
// one-SM kernel: out non-null as for launch_stream_w2; CTA pairs: see tc_fused_combine
cudaError_t launch_tc_w2(const moe_fp4_dims& d, const uint8_t* w2, const uint8_t* w2s, const Workspace& ws,
                         float* out, bool pairs, bool atomic_combine, cudaStream_t st);
cudaError_t launch_combine(const moe_fp4_dims& d, float* out, const Workspace& ws, cudaStream_t st);
// true: the tensor-core W2 kernel writes out itself (the weighted combine in
// its epilogue; the CTA-pair kernel does)
bool tc_fused_combine(bool pairs);
cudaError_t launch_router(const moe_fp4_dims& d, const uint16_t* x, const uint16_t* wg, float* logits,
                          cudaStream_t st);
// MXFP8 of bf16 rows [rows, K] (K a multiple of 32; x and codes 16-byte aligned)
cudaError_t launch_mxfp8_quantize(const uint16_t* x, long long rows, int K, uint8_t* codes, uint8_t* scales,
                                  cudaStream_t st);
// block-scaled layer after routing: quantising gather, W13 (+ SwiGLU, h and
// its MXFP8 form) and W2 on kind::mxf8f6f4 tensor cores; y in ws.y
// `mark` (optional) is called with 2 after the gather and 3 after W13 (stage events)
cudaError_t launch_mx_forward(const moe_fp4_dims& d, const uint16_t* x, const uint8_t* w13, const uint8_t* w13s,
                              const uint8_t* w2, const uint8_t* w2s, const Workspace& ws, cudaStream_t st,
                              const std::function<void(int)>& mark);

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
#ifdef __CUDACC__

// Two E2M1 codes (one byte, low nibble first) -> two exact halves.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n}" : "=r"(r) : "r"(byte));
  return r;
}

// E8M0 byte -> fp32 2^(s-127); 0 maps to the subnormal 2^-127, 0xFF to NaN.
__device__ __forceinline__ float e8m0_to_f32(uint32_t s) {
  uint32_t bits = s == 0 ? 0x00400000u : (s == 255 ? 0x7FC00000u : (s << 23));
  return __uint_as_float(bits);
}

// bf16 bits -> fp32
__device__ __forceinline__ float bf16_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }

// out[i] += v in global memory, no return value (fp32 reduction at L2); the
// order of concurrent additions is not fixed.
__device__ __forceinline__ void red_add_f32(float* p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// The same for two adjacent floats (p 8-byte aligned).
__device__ __forceinline__ void red_add_v2_f32(float* p, float a, float b) {
  asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(p), "f"(a), "f"(b) : "memory");
}

// fp32 -> bf16 bits, round to nearest even (the CUDA intrinsic).
__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// silu(z) * u in fp32 with the fast exponential and division intrinsics (a
// few ulp of fp32, far below the bf16 rounding of h that follows)
__device__ __forceinline__ float swiglu(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }

// Programmatic dependent launch.  A kernel launched by launch_early() may start
// while the previous kernel of the stream is still running: griddep_wait()
// returns once that kernel has completed and its writes are visible (at once
// for a kernel launched the ordinary way), and the early kernel may touch
// nothing that kernel writes before it.  griddep_launch_dependents() lets the
// next early kernel start before this one ends.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_early(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                         Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

#endif

}  // namespace moe_fp4
