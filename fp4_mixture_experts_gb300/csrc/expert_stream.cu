// Decode-shaped expert projections: a persistent, TMA-fed streaming GEMV.
//
// With few token rows per expert (decode: T*k/E ~ 1) the layer is bound by
// reading the packed expert weights once from HBM; the paper's decode path
// ("packed FP4 weights", "topology-aware kernel geometry") is a weight-
// streaming problem.  Each CTA (one per SM) walks a contiguous range of work
// items, an item being one stage of weight rows for one chunk of up to four
// token rows of one expert:
//   - one producer warp streams the stage's packed rows and E8M0 scales into a
//     4-deep shared-memory ring with 1-D bulk TMA copies (cp.async.bulk,
//     full/empty mbarriers with transaction counts), so ~130 KB of weights per
//     SM are in flight;
//   - the consumer threads split K into 32-element MX blocks (one 16-byte
//     packed chunk and one scale per thread and row).  Each holds its block of
//     the chunk's activations in registers as f16 pairs, scaled by a power of
//     two per (token, block) so that every bf16 value lands exactly in f16
//     range; E2M1 pairs are decoded by cvt.rn.f16x2.e2m1x2 (exact) and
//     multiplied with the mixed-precision fma.rn.f32.f16 (exact f16 x f16
//     products, fp32 accumulation), so no fp32 conversion of the weights is
//     needed; the block sums are scaled once by 2^(s-127) times the
//     activation scale;
//   - partial sums are reduced with a warp butterfly (reduce-scatter) and a
//     small shared-memory pass across the warps of a row group, synchronised
//     by a per-group named barrier; the W13 epilogue applies SwiGLU and rounds
//     h to bf16, the W2 epilogue writes fp32 y.
// Every mbarrier wait is bounded: past the limit the thread records an error
// word; the threads of a row group take the exit decision together (barrier
// with an OR vote), so no barrier is left waiting (moe_fp4_check reports it).
#include <cuda_fp16.h>

#include "moe_fp4_internal.cuh"

namespace moe_fp4 {
namespace {

constexpr int kStages = 4;          // ring depth
constexpr int kPairsW13 = 4;        // (gate, up) row pairs per consumer thread per stage
constexpr int kRowsW2 = 8;          // W2 rows per consumer thread per stage
constexpr int kMaxConsumers = 256;  // K-split threads x row groups
constexpr uint32_t kWaitLimit = 1u << 22;  // try_wait rounds before giving up (~seconds)
constexpr int kRingOffset = 128 + 2 * kMaxConsumers * sizeof(float);  // barriers, reduction buffers

struct StreamParams {
  const uint8_t* w;        // packed weights of all experts
  const uint8_t* ws;       // E8M0 scales
  const uint16_t* act;     // activations: x [T, d] (W13) or h [S, I] (W2), bf16
  const int4* chunks;      // (expert, first sorted row, rows, 0)
  const int32_t* counts;   // counts[1] = number of chunks
  const int32_t* sorted_slot;
  int32_t* err;
  uint16_t* h_out;         // W13: h [S, I]
  float* y_out;            // W2: y [S, d]
  int k, d, I;
  int K;                   // reduction length: d (W13) or I (W2)
  int nkb;                 // K / 32 (consumer threads per row group)
  int rg;                  // row groups
  int rows_per_expert;     // W13: I pairs, W2: d rows
  int rows_per_stage;      // pairs (W13) or rows (W2) per stage = rg * per-thread
  uint32_t stage_bytes;    // bytes of one ring slot
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// bounded wait; false when the limit ran out
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Named barrier `id` over `n_threads` threads that also ORs a predicate, so
// that every thread of the group takes the same exit decision.
__device__ __forceinline__ bool group_sync_or(int id, int n_threads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(n_threads)
      : "memory");
  return r != 0;
}

// Warp reduce-scatter of V = 2^m values: afterwards lane l holds, in v[0],
// the warp sum of value index l >> (5 - m).
template <int V>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[V], int lane) {
  int n = V;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    if (n > 1) {
      const bool upper = lane & off;
#pragma unroll
      for (int i = 0; i < V / 2; ++i) {
        if (i < n / 2) {
          const float send = upper ? v[i] : v[i + n / 2];
          const float keep = upper ? v[i + n / 2] : v[i];
          v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, off);
        }
      }
      n >>= 1;
    } else {
      v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], off);
    }
  }
  return v[0];
}

// 2^e as fp32 for any e the kernel meets (exponent-field build when normal)
__device__ __forceinline__ float pow2f(int e) {
  return (e >= -126 && e <= 127) ? __uint_as_float((uint32_t)(e + 127) << 23) : ldexpf(1.0f, e);
}

// This thread's 32 activations of one token row, as 16 f16 pairs scaled by a
// power of two: value = f16 * 2^xe.  The largest magnitude lands in
// [2^14, 2^15), so every bf16 value of the block within 2^38 of it is exact.
__device__ __forceinline__ void load_x_block(uint32_t (&xh)[16], int& xe, const uint16_t* src) {
  uint32_t w[16];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 q = reinterpret_cast<const uint4*>(src)[c];
    w[4 * c + 0] = q.x;
    w[4 * c + 1] = q.y;
    w[4 * c + 2] = q.z;
    w[4 * c + 3] = q.w;
  }
  uint32_t emax = 1;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    emax = max(emax, (w[i] >> 7) & 0xFFu);
    emax = max(emax, (w[i] >> 23) & 0xFFu);
  }
  const int shift = 141 - (int)emax;  // 2^shift * 2^(emax-127) = 2^14
  const float f1 = pow2f(shift / 2), f2 = pow2f(shift - shift / 2);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float lo = bf16_to_f32(w[i] & 0xFFFFu) * f1 * f2;
    const float hi = bf16_to_f32(w[i] >> 16) * f1 * f2;
    const __half2 h = __floats2half2_rn(lo, hi);
    xh[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  xe = -shift;
}

__device__ __forceinline__ float fma_f16(uint16_t a, uint16_t b, float c) {
  asm("fma.rn.f32.f16 %0, %1, %2, %0;" : "+f"(c) : "h"(a), "h"(b));
  return c;
}

__device__ __forceinline__ void split16(uint32_t v, uint16_t& lo, uint16_t& hi) {
  asm("mov.b32 {%0, %1}, %2;" : "=h"(lo), "=h"(hi) : "r"(v));
}

// One row's 32-element block (16 packed bytes) dotted with MT token rows:
// unscaled sums s[t] = sum_j e2m1_j * xh_t[j] (exact products, fp32 sums).
template <int MT>
__device__ __forceinline__ void block_dot(const uint4 q, const uint32_t (&xh)[kGemvTokens][16], float (&s)[MT]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  float a0[MT], a1[MT];
#pragma unroll
  for (int t = 0; t < MT; ++t) a0[t] = a1[t] = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      uint16_t wl, wh;
      split16(e2m1x2_to_f16x2((w[c] >> (8 * b)) & 0xFFu), wl, wh);
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        uint16_t xl, xh_;
        split16(xh[t][c * 4 + b], xl, xh_);
        a0[t] = fma_f16(wl, xl, a0[t]);
        a1[t] = fma_f16(wh, xh_, a1[t]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < MT; ++t) s[t] = a0[t] + a1[t];
}

// ---------------------------------------------------------------------------
// consumer work of one stage, templated on the chunk's token count
// ---------------------------------------------------------------------------
template <int MT>
__device__ __forceinline__ void w13_stage(const StreamParams& P, const uint8_t* slot, int rgi, int kb, int lane,
                                          const uint32_t (&xh)[kGemvTokens][16], const int (&xe)[kGemvTokens],
                                          float* red_w) {
  constexpr int V = 2 * kPairsW13 * MT;  // (pair, token, gate/up)
  float v[V];
  const int row_bytes = P.K / 2, nkb = P.nkb, rps = P.rows_per_stage;
  const uint8_t* scales = slot + (size_t)2 * rps * row_bytes;
#pragma unroll
  for (int p = 0; p < kPairsW13; ++p) {
    const int pr = rgi * kPairsW13 + p;
#pragma unroll
    for (int gu = 0; gu < 2; ++gu) {
      const int r = gu * rps + pr;
      float s[MT];
      block_dot<MT>(*reinterpret_cast<const uint4*>(slot + (size_t)r * row_bytes + kb * 16), xh, s);
      const int se = (int)scales[r * nkb + kb] - 127;
#pragma unroll
      for (int t = 0; t < MT; ++t) v[(p * MT + t) * 2 + gu] = s[t] * pow2f(se + xe[t]);
    }
  }
  const float r = warp_reduce_scatter<V>(v, lane);
  constexpr int kLanesPerValue = 32 / V;
  if ((lane % kLanesPerValue) == 0) red_w[lane / kLanesPerValue] = r;
}

template <int MT>
__device__ __forceinline__ void w2_stage(const StreamParams& P, const uint8_t* slot, int rgi, int kb, int lane,
                                         const uint32_t (&xh)[kGemvTokens][16], const int (&xe)[kGemvTokens],
                                         float* red_w) {
  constexpr int V = kRowsW2 * MT;  // (row, token)
  float v[V];
  const int row_bytes = P.K / 2, nkb = P.nkb, rps = P.rows_per_stage;
  const uint8_t* scales = slot + (size_t)rps * row_bytes;
#pragma unroll
  for (int p = 0; p < kRowsW2; ++p) {
    const int r = rgi * kRowsW2 + p;
    float s[MT];
    block_dot<MT>(*reinterpret_cast<const uint4*>(slot + (size_t)r * row_bytes + kb * 16), xh, s);
    const int se = (int)scales[r * nkb + kb] - 127;
#pragma unroll
    for (int t = 0; t < MT; ++t) v[p * MT + t] = s[t] * pow2f(se + xe[t]);
  }
  const float r = warp_reduce_scatter<V>(v, lane);
  constexpr int kLanesPerValue = 32 / V;
  if ((lane % kLanesPerValue) == 0) red_w[lane / kLanesPerValue] = r;
}

template <bool W13>
__device__ __forceinline__ void issue_stage(const StreamParams& P, long long u, int spc, uint8_t* dst, uint64_t* bar,
                                            uint64_t pol) {
  const int c = (int)(u / spc), s = (int)(u % spc);
  const int e = P.chunks[c].x;
  const int row_bytes = P.K / 2, nkb = P.nkb, rps = P.rows_per_stage;
  const uint32_t wb = (uint32_t)(rps * row_bytes), sb = (uint32_t)(rps * nkb);
  if (W13) {
    const size_t gate0 = (size_t)e * 2 * P.I + (size_t)s * rps;
    const size_t up0 = gate0 + P.I;
    mbar_expect_tx(bar, 2 * wb + 2 * sb);
    bulk_g2s(dst, P.w + gate0 * row_bytes, wb, bar, pol);
    bulk_g2s(dst + wb, P.w + up0 * row_bytes, wb, bar, pol);
    bulk_g2s(dst + 2 * wb, P.ws + gate0 * nkb, sb, bar, pol);
    bulk_g2s(dst + 2 * wb + sb, P.ws + up0 * nkb, sb, bar, pol);
  } else {
    const size_t r0 = (size_t)e * P.d + (size_t)s * rps;
    mbar_expect_tx(bar, wb + sb);
    bulk_g2s(dst, P.w + r0 * row_bytes, wb, bar, pol);
    bulk_g2s(dst + wb, P.ws + r0 * nkb, sb, bar, pol);
  }
}

// Consumers: rg row groups of nkb threads (K split in 32-element blocks), at
// most 256; one producer warp after them issues the bulk copies.
template <bool W13>
__global__ void __launch_bounds__(kMaxConsumers + 32, 1) stream_kernel(const StreamParams P) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kStages;
  float* red = reinterpret_cast<float*>(smem + 128);  // [2 buffers][consumer warps][32]
  uint8_t* ring = smem + kRingOffset;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_cons = P.rg * P.nkb;
  const int n_cons_warps = n_cons / 32;
  const int n_chunks = P.counts[1];
  const int spc = P.rows_per_expert / P.rows_per_stage;  // stages per chunk
  const long long n_items = (long long)n_chunks * spc;
  const long long u0 = n_items * blockIdx.x / gridDim.x;
  const long long u1 = n_items * (blockIdx.x + 1) / gridDim.x;
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], n_cons_warps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == n_cons_warps) {
    // ---------------- producer warp ----------------
    if (lane == 0) {
      const uint64_t pol = evict_first_policy();
      int slot = 0;
      uint32_t phase = 0, pending = 0, last_phase = 0;
      bool ok = true;
      for (long long u = u0; u < u1; ++u) {
        if (!mbar_wait(&empty[slot], phase ^ 1u)) {
          atomicOr(P.err, kErrWaitTimeout);
          ok = false;
          break;
        }
        issue_stage<W13>(P, u, spc, ring + (size_t)slot * P.stage_bytes, &full[slot], pol);
        pending |= 1u << slot;
        last_phase = (last_phase & ~(1u << slot)) | (phase << slot);
        if (++slot == kStages) {
          slot = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        // let the copies this CTA issued land before it exits (bounded waits)
        for (int i = 0; i < kStages; ++i)
          if (pending & (1u << i)) mbar_wait(&full[i], (last_phase >> i) & 1u);
      }
    }
    return;
  }

  // ---------------- consumer threads ----------------
  const int nkb = P.nkb, rps = P.rows_per_stage;
  const int rgi = tid / nkb, kb = tid % nkb, warp_in_rg = kb / 32;
  const int wpr = nkb / 32;  // warps per row group
  const int lt = kb;         // thread index within the row group
  uint32_t xh[kGemvTokens][16];
  int xe[kGemvTokens];
  int cur = -1, row0 = 0, mt = 0;
  int slot = 0, buf = 0;
  uint32_t phase = 0;
  for (long long u = u0; u < u1; ++u) {
    const int c = (int)(u / spc), s = (int)(u % spc);
    if (c != cur) {
      const int4 ch = P.chunks[c];
      row0 = ch.y;
      mt = ch.z;
#pragma unroll
      for (int t = 0; t < kGemvTokens; ++t) {
        if (t < mt) {
          const int row = W13 ? P.sorted_slot[row0 + t] / P.k : row0 + t;
          load_x_block(xh[t], xe[t], P.act + (size_t)row * P.K + kb * 32);
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) xh[t][j] = 0u;
          xe[t] = 0;
        }
      }
      cur = c;
    }
    const bool ok = mbar_wait(&full[slot], phase);
    const uint8_t* sp = ring + (size_t)slot * P.stage_bytes;
    float* red_w = red + (buf * n_cons_warps + rgi * wpr + warp_in_rg) * 32;
    if (ok) {
      if (W13) {
        switch (mt) {
          case 1: w13_stage<1>(P, sp, rgi, kb, lane, xh, xe, red_w); break;
          case 2: w13_stage<2>(P, sp, rgi, kb, lane, xh, xe, red_w); break;
          default: w13_stage<4>(P, sp, rgi, kb, lane, xh, xe, red_w); break;
        }
      } else {
        switch (mt) {
          case 1: w2_stage<1>(P, sp, rgi, kb, lane, xh, xe, red_w); break;
          case 2: w2_stage<2>(P, sp, rgi, kb, lane, xh, xe, red_w); break;
          default: w2_stage<4>(P, sp, rgi, kb, lane, xh, xe, red_w); break;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    if (++slot == kStages) {
      slot = 0;
      phase ^= 1u;
    }
    if (group_sync_or(1 + rgi, nkb, !ok)) {
      if (lt == 0) atomicOr(P.err, kErrWaitTimeout);
      break;
    }
    // epilogue of this row group; the reduction buffer is double-buffered, so
    // the group's next stage can write the other half meanwhile
    const float* red_g = red + (buf * n_cons_warps + rgi * wpr) * 32;
    const int mtp = mt == 3 ? 4 : mt;  // token count of the template the stage used
    if (W13) {
      const int outs = kPairsW13 * mtp;
      if (lt < outs) {
        const int p = lt / mtp, t = lt % mtp;  // lt = pair * mtp + token
        if (t < mt) {
          float gs = 0.f, us = 0.f;
          for (int w = 0; w < wpr; ++w) {
            gs += red_g[w * 32 + 2 * lt];
            us += red_g[w * 32 + 2 * lt + 1];
          }
          const int i = s * rps + rgi * kPairsW13 + p;
          P.h_out[(size_t)(row0 + t) * P.I + i] = f32_to_bf16_rn(swiglu(gs, us));
        }
      }
    } else {
      const int outs = kRowsW2 * mtp;
      if (lt < outs) {
        const int p = lt / mtp, t = lt % mtp;  // lt = row * mtp + token
        if (t < mt) {
          float ys = 0.f;
          for (int w = 0; w < wpr; ++w) ys += red_g[w * 32 + lt];
          const int n = s * rps + rgi * kRowsW2 + p;
          P.y_out[(size_t)(row0 + t) * P.d + n] = ys;
        }
      }
    }
    buf ^= 1;
  }
}

int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

size_t smem_bytes(const StreamParams& P) { return kRingOffset + (size_t)kStages * P.stage_bytes; }

template <bool W13>
cudaError_t launch_stream(StreamParams P, cudaStream_t st) {
  const size_t smem = smem_bytes(P);
  static bool configured = false;
  if (!configured) {
    cudaFuncSetAttribute(stream_kernel<W13>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    configured = true;
  }
  stream_kernel<W13><<<num_sms(), P.rg * P.nkb + 32, smem, st>>>(P);
  return cudaGetLastError();
}

}  // namespace

bool stream_path_supported(const moe_fp4_dims& d) {
  // K split into 32-element blocks across whole warps, at most 256 threads
  return d.d % 1024 == 0 && d.I % 1024 == 0 && d.d <= 8192 && d.I <= 8192;
}

cudaError_t launch_stream_w13(const moe_fp4_dims& d, const uint16_t* x, const uint8_t* w13, const uint8_t* w13s,
                              const Workspace& ws, cudaStream_t st) {
  StreamParams P{};
  P.w = w13;
  P.ws = w13s;
  P.act = x;
  P.chunks = ws.gemv_chunks;
  P.counts = ws.counts;
  P.sorted_slot = ws.sorted_slot;
  P.err = ws.err;
  P.h_out = ws.h;
  P.k = d.k;
  P.d = d.d;
  P.I = d.I;
  P.K = d.d;
  P.nkb = d.d / 32;
  P.rg = P.nkb >= kMaxConsumers ? 1 : kMaxConsumers / P.nkb;
  P.rows_per_expert = d.I;
  P.rows_per_stage = P.rg * kPairsW13;
  P.stage_bytes = (uint32_t)(2 * P.rows_per_stage * (P.K / 2 + P.nkb));
  return launch_stream<true>(P, st);
}

cudaError_t launch_stream_w2(const moe_fp4_dims& d, const uint8_t* w2, const uint8_t* w2s, const Workspace& ws,
                             cudaStream_t st) {
  StreamParams P{};
  P.w = w2;
  P.ws = w2s;
  P.act = ws.h;
  P.chunks = ws.gemv_chunks;
  P.counts = ws.counts;
  P.sorted_slot = ws.sorted_slot;
  P.err = ws.err;
  P.y_out = ws.y;
  P.k = d.k;
  P.d = d.d;
  P.I = d.I;
  P.K = d.I;
  P.nkb = d.I / 32;
  P.rg = P.nkb >= kMaxConsumers ? 1 : kMaxConsumers / P.nkb;
  P.rows_per_expert = d.d;
  P.rows_per_stage = P.rg * kRowsW2;
  P.stage_bytes = (uint32_t)(P.rows_per_stage * (P.K / 2 + P.nkb));
  return launch_stream<false>(P, st);
}

}  // namespace moe_fp4
