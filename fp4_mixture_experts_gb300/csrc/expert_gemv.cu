// Expert projections on CUDA cores (every shape), the token gather and the
// weighted combine.
//
// w13_swiglu_rows: one warp per (gate row i, up row I+i) pair and a chunk of
//   up to 8 token rows of one expert; lanes split K in 32-element MX blocks
//   (16 packed bytes + 1 E8M0 byte), decode E2M1 pairs with the hardware
//   cvt.rn.f16x2.e2m1x2, accumulate in fp32, reduce across the warp and apply
//   SwiGLU; h is rounded to bf16 (the layer's one rounding point).
// w2_rows: the same pattern over W2 rows, fp32 y in sorted-row order.
// combine: out[t] = sum_j w[t, j] * y[slot_pos[t*k + j]] in slot order
//   (deterministic: no atomics, the MI250 blog's section 3.2 / 4.2 rule);
//   launched early (programmatic dependent launch), it waits for the W2
//   kernel before reading y.
#include <cuda_fp16.h>

#include "moe_fp4_internal.cuh"

namespace moe_fp4 {
namespace {

constexpr int kRowsThreads = 256;  // 8 warps, one row (pair) each

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// 16 packed bytes (32 E2M1 codes, K ascending) -> 32 fp32 values (unscaled)
__device__ __forceinline__ void decode32(const uint4 p, float v[32]) {
  const uint32_t w[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t h2 = e2m1x2_to_f16x2((w[q] >> (8 * b)) & 0xFFu);
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
      v[q * 8 + b * 2 + 0] = f.x;
      v[q * 8 + b * 2 + 1] = f.y;
    }
  }
}

// sum_{j<32} v[j] * x[j] with x 32 consecutive bf16 at p (64 bytes, 16-byte aligned)
__device__ __forceinline__ float dot32_bf16(const float v[32], const uint16_t* p) {
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 q = *reinterpret_cast<const uint4*>(p + 8 * c);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      s = fmaf(v[c * 8 + 2 * i + 0], bf16_to_f32(w[i] & 0xFFFFu), s);
      s = fmaf(v[c * 8 + 2 * i + 1], bf16_to_f32(w[i] >> 16), s);
    }
  }
  return s;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__global__ void __launch_bounds__(kRowsThreads)
w13_swiglu_rows_kernel(const uint16_t* __restrict__ x, const uint8_t* __restrict__ w13,
                       const uint8_t* __restrict__ w13s, const int4* __restrict__ chunks,
                       const int32_t* __restrict__ counts, const int32_t* __restrict__ sorted_slot,
                       int k, int d, int I, uint16_t* __restrict__ h) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * (kRowsThreads / 32) + warp;
  if (i >= I) return;
  const int n_chunks = counts[1];
  const int nkb = d / 32;
  for (int c = blockIdx.y; c < n_chunks; c += gridDim.y) {
    const int4 ch = chunks[c];
    const int e = ch.x, row0 = ch.y, mt = ch.z;
    int tok[kGemvTokens];
#pragma unroll
    for (int q = 0; q < kGemvTokens; ++q) tok[q] = q < mt ? sorted_slot[row0 + q] / k : 0;
    const size_t gate_row = (size_t)e * 2 * I + i, up_row = gate_row + I;
    const uint8_t* wg = w13 + gate_row * (d / 2);
    const uint8_t* wu = w13 + up_row * (d / 2);
    const uint8_t* sg = w13s + gate_row * nkb;
    const uint8_t* su = w13s + up_row * nkb;
    float ag[kGemvTokens] = {}, au[kGemvTokens] = {};
    for (int kb = lane; kb < nkb; kb += 32) {
      float vg[32], vu[32];
      decode32(ldg_nc_v4(wg + kb * 16), vg);
      decode32(ldg_nc_v4(wu + kb * 16), vu);
      const float scg = e8m0_to_f32(sg[kb]), scu = e8m0_to_f32(su[kb]);
#pragma unroll
      for (int q = 0; q < kGemvTokens; ++q) {
        if (q < mt) {
          const uint16_t* xr = x + (size_t)tok[q] * d + kb * 32;
          ag[q] = fmaf(scg, dot32_bf16(vg, xr), ag[q]);
          au[q] = fmaf(scu, dot32_bf16(vu, xr), au[q]);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kGemvTokens; ++q) {
      const float g = warp_sum(ag[q]), u = warp_sum(au[q]);
      if (lane == 0 && q < mt) h[(size_t)(row0 + q) * I + i] = f32_to_bf16_rn(swiglu(g, u));
    }
  }
}

__global__ void __launch_bounds__(kRowsThreads)
w2_rows_kernel(const uint16_t* __restrict__ h, const uint8_t* __restrict__ w2,
               const uint8_t* __restrict__ w2s, const int4* __restrict__ chunks,
               const int32_t* __restrict__ counts, int d, int I, float* __restrict__ y) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * (kRowsThreads / 32) + warp;
  if (n >= d) return;
  const int n_chunks = counts[1];
  const int nkb = I / 32;
  for (int c = blockIdx.y; c < n_chunks; c += gridDim.y) {
    const int4 ch = chunks[c];
    const int e = ch.x, row0 = ch.y, mt = ch.z;
    const size_t row = (size_t)e * d + n;
    const uint8_t* wr = w2 + row * (I / 2);
    const uint8_t* sr = w2s + row * nkb;
    float acc[kGemvTokens] = {};
    for (int kb = lane; kb < nkb; kb += 32) {
      float v[32];
      decode32(ldg_nc_v4(wr + kb * 16), v);
      const float sc = e8m0_to_f32(sr[kb]);
#pragma unroll
      for (int q = 0; q < kGemvTokens; ++q)
        if (q < mt) acc[q] = fmaf(sc, dot32_bf16(v, h + (size_t)(row0 + q) * I + kb * 32), acc[q]);
    }
#pragma unroll
    for (int q = 0; q < kGemvTokens; ++q) {
      const float s = warp_sum(acc[q]);
      if (lane == 0 && q < mt) y[(size_t)(row0 + q) * d + n] = s;
    }
  }
}

// x_perm[r] = x[sorted_slot[r] / k] as f16 scaled by 2^shift_r, with
// x_scale[r] = 2^-shift_r; the row's largest magnitude lands in [2^14, 2^15),
// so every bf16 value within 2^31 of it converts exactly.  One warp per row.
// NV > 0: the row is held in registers (NV 16-byte vectors per lane, all
// loads issued before the first use, so a warp keeps NV loads in flight and
// the row is read once); NV = 0: rows too long for that are read twice.
__device__ __forceinline__ uint32_t bf16x2_max_exp(uint32_t e, uint32_t w) {
  return max(e, max((w >> 7) & 0xFFu, (w >> 23) & 0xFFu));
}

__device__ __forceinline__ uint4 bf16x8_to_f16x8(const uint4 q, float f1, float f2) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 h = __floats2half2_rn(bf16_to_f32(w[i] & 0xFFFFu) * f1 * f2, bf16_to_f32(w[i] >> 16) * f1 * f2);
    o[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

template <int NV>
__global__ void __launch_bounds__(256)
gather_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ sorted_slot, int S, int k, int d,
              uint16_t* __restrict__ x_perm, float* __restrict__ x_scale, int32_t* __restrict__ zero, int n_zero) {
  // the W2 kernel's combine counters of this call start at zero
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_zero; i += gridDim.x * blockDim.x) zero[i] = 0;
  // sorted_slot == nullptr: row r of x itself (the f16 copy of h for the tensor-core W2)
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  const int vec = d / 8;
  for (int r = warp; r < S; r += nwarps) {
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)(sorted_slot ? sorted_slot[r] / k : r) * d);
    uint4* dst = reinterpret_cast<uint4*>(x_perm + (size_t)r * d);
    uint32_t emax = 1;
    uint4 q[NV > 0 ? NV : 1];
    if (NV > 0) {
#pragma unroll
      for (int i = 0; i < NV; ++i)
        if (lane + 32 * i < vec) q[i] = src[lane + 32 * i];
#pragma unroll
      for (int i = 0; i < NV; ++i)
        if (lane + 32 * i < vec)
          emax = bf16x2_max_exp(bf16x2_max_exp(bf16x2_max_exp(bf16x2_max_exp(emax, q[i].x), q[i].y), q[i].z), q[i].w);
    } else {
#pragma unroll 4
      for (int v = lane; v < vec; v += 32) {
        const uint4 t = src[v];
        emax = bf16x2_max_exp(bf16x2_max_exp(bf16x2_max_exp(bf16x2_max_exp(emax, t.x), t.y), t.z), t.w);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) emax = max(emax, __shfl_xor_sync(0xFFFFFFFFu, emax, o));
    const int shift = 141 - (int)emax;
    const float f1 = ldexpf(1.0f, shift / 2), f2 = ldexpf(1.0f, shift - shift / 2);
    if (NV > 0) {
#pragma unroll
      for (int i = 0; i < NV; ++i)
        if (lane + 32 * i < vec) dst[lane + 32 * i] = bf16x8_to_f16x8(q[i], f1, f2);
    } else {
#pragma unroll 4
      for (int v = lane; v < vec; v += 32) dst[v] = bf16x8_to_f16x8(src[v], f1, f2);
    }
    if (lane == 0) x_scale[r] = ldexpf(1.0f, -shift);
  }
}

// the row of d elements in registers when it fits 32 vectors a lane (d <= 8192)
cudaError_t launch_gather_rows(const uint16_t* x, const int32_t* sorted_slot, int S, int k, int d, uint16_t* out,
                               float* scale, int32_t* zero, int n_zero, cudaStream_t st) {
  const int nv = (d / 8 + 31) / 32;
  const int per_block = 8;  // rows (warps) per block
  int blocks = (S + per_block - 1) / per_block;
  const int cap = num_sms() * (nv > 16 ? 4 : 8);
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (nv <= 8)
    gather_kernel<8><<<blocks, 256, 0, st>>>(x, sorted_slot, S, k, d, out, scale, zero, n_zero);
  else if (nv <= 16)
    gather_kernel<16><<<blocks, 256, 0, st>>>(x, sorted_slot, S, k, d, out, scale, zero, n_zero);
  else if (nv <= 32)
    gather_kernel<32><<<blocks, 256, 0, st>>>(x, sorted_slot, S, k, d, out, scale, zero, n_zero);
  else
    gather_kernel<0><<<blocks, 256, 0, st>>>(x, sorted_slot, S, k, d, out, scale, zero, n_zero);
  return cudaGetLastError();
}

// out[t] = sum_j w_tj * y[slot_pos(t, j)]; block (t, c) covers columns
// [1024 c, 1024 c + 1024) of token t, one float4 per thread, so that even a
// decode batch of 32 tokens spreads over d / 1024 times as many blocks
__global__ void __launch_bounds__(256)
combine_kernel(const float* __restrict__ y, const float* __restrict__ topk_w,
               const int32_t* __restrict__ slot_pos, int T, int k, int d, float* __restrict__ out) {
  griddep_wait();  // y comes from the W2 kernel (launched early, see launch_combine)
  const int t = blockIdx.x;
  if (t >= T) return;
  const int vec = d / 4;
  for (int v = blockIdx.y * blockDim.x + threadIdx.x; v < vec; v += gridDim.y * blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const float w = topk_w[(size_t)t * k + j];
      const float4 yv = reinterpret_cast<const float4*>(y + (size_t)slot_pos[(size_t)t * k + j] * d)[v];
      acc.x = fmaf(w, yv.x, acc.x);
      acc.y = fmaf(w, yv.y, acc.y);
      acc.z = fmaf(w, yv.z, acc.z);
      acc.w = fmaf(w, yv.w, acc.w);
    }
    reinterpret_cast<float4*>(out + (size_t)t * d)[v] = acc;
  }
}

int grid_chunks(const Workspace& ws) { return ws.max_gemv_chunks < 65535 ? ws.max_gemv_chunks : 65535; }

}  // namespace

cudaError_t launch_gemv_w13(const moe_fp4_dims& d, const uint16_t* x, const uint8_t* w13,
                            const uint8_t* w13s, const Workspace& ws, cudaStream_t st) {
  dim3 grid((d.I + 7) / 8, grid_chunks(ws));
  w13_swiglu_rows_kernel<<<grid, kRowsThreads, 0, st>>>(x, w13, w13s, ws.gemv_chunks, ws.counts,
                                                        ws.sorted_slot, d.k, d.d, d.I, ws.h);
  return cudaGetLastError();
}

cudaError_t launch_gemv_w2(const moe_fp4_dims& d, const uint8_t* w2, const uint8_t* w2s,
                           const Workspace& ws, cudaStream_t st) {
  dim3 grid((d.d + 7) / 8, grid_chunks(ws));
  w2_rows_kernel<<<grid, kRowsThreads, 0, st>>>(ws.h, w2, w2s, ws.gemv_chunks, ws.counts, d.d, d.I, ws.y);
  return cudaGetLastError();
}

cudaError_t launch_gather(const moe_fp4_dims& d, const uint16_t* x, const Workspace& ws, cudaStream_t st) {
  return launch_gather_rows(x, ws.sorted_slot, d.T * d.k, d.k, d.d, ws.x_perm, ws.x_scale, ws.combine_cnt,
                            d.T * ((d.d + 255) / 256), st);
}

cudaError_t launch_h_f16(const moe_fp4_dims& d, const Workspace& ws, cudaStream_t st) {
  return launch_gather_rows(ws.h, nullptr, d.T * d.k, 1, d.I, ws.h16, ws.h_scale, nullptr, 0, st);
}

cudaError_t launch_combine(const moe_fp4_dims& d, float* out, const Workspace& ws, cudaStream_t st) {
  const dim3 grid(d.T, (d.d / 4 + 255) / 256);
  const float* y = ws.y;
  const float* w = ws.topk_w;
  const int32_t* pos = ws.slot_pos;
  // launched early: blocks start as the W2 kernel's CTAs retire, then wait for it
  return launch_early(combine_kernel, grid, dim3(256), 0, st, y, w, pos, d.T, d.k, d.d, out);
}

}  // namespace moe_fp4
