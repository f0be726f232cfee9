// Decode-shaped expert projections: a persistent, TMA-fed streaming GEMV on
// warp-level tensor-core MMAs with register-sourced weights.
//
// With few token rows per expert (decode: T*k/E ~ 1) the layer is bound by
// reading the packed expert weights once from HBM (the paper's decode path:
// packed FP4 weights, dot-product instructions, kernel geometry).  The cost
// to beat is the per-element decode, so it is kept minimal:
//   - one producer warp streams 128-row x 512-K stages (32 KB of packed
//     E2M1 codes, TMA 2-D boxes with the 128-byte swizzle, plus their E8M0
//     scales) into a shared-memory ring guarded by full/empty mbarriers;
//   - 16 consumer warps: each 16-row tile (W13: 8 gate rows and the 8
//     matching up rows, so SwiGLU stays in-thread; W2: 16 output rows) is
//     shared by two warps, each taking half of the stage's MX blocks; for
//     W13 (and W2 writing y) the pair adds its partial sums once per item
//     through shared memory.  A chunk's token rows (up to 8) sit in shared memory as f16 scaled by a
//     power of two per token (every bf16 value within 2^31 of the row maximum
//     is exact, smaller ones round at 2^-39 of it);
//   - per 32-element MX block a thread loads 4 packed bytes of each of its
//     two rows as one 32-bit word (32-bit shared-window addresses, offsets
//     precomputed per thread: the loop spends its ALU issue on little but the
//     conversions); every cvt.rn.f16x2.e2m1x2 result is directly an
//     A-fragment register of mma.sync.m16n8k16 (the K order inside the block
//     is permuted so that each thread's bytes and activations are contiguous,
//     identically for A and B); two MMAs give the block's sums (f16 x f16
//     products are exact, accumulation fp32), which are scaled by 2^(s-127)
//     in fp32 and accumulated, so every E8M0 value is handled exactly;
//   - the W13 epilogue applies SwiGLU and rounds h to bf16 (the W13 kernel
//     also zeroes out while it waits for the routing); the W2 epilogue adds
//     each warp's half-K sums, times the slot's routing weight, into the
//     token's fp32 out row (atomic adds), or writes fp32 y for the slot-order
//     combine pass.
// Waits are bounded; a timeout raises the CTA abort flag, after which every
// warp runs the same loop without waiting (its arithmetic discarded), so all
// barriers are still met and the kernel exits; the producer waits (also
// bounded) for its copies in flight before it leaves.
#include <cuda_fp16.h>

#include "moe_fp4_internal.cuh"
#include "ptx_sm103.cuh"

namespace moe_fp4 {
namespace {

#ifndef MOE_STREAM_KSPLIT
#define MOE_STREAM_KSPLIT 2
#endif
constexpr int kTiles = 8;                        // 16-row tiles per 128-row stage
constexpr int kKSplit = MOE_STREAM_KSPLIT;       // warps sharing a tile, each taking 16/kKSplit blocks per stage
constexpr int kBlkPerWarp = 16 / kKSplit;
constexpr int kConsWarps = kTiles * kKSplit;
constexpr int kThreads = (kConsWarps + 1) * 32;
constexpr int kRedBytes = 2 * kTiles * (kKSplit - 1) * 32 * 16;  // double-buffered partial sums of the split
constexpr int kRowsPerBlock = 128;     // weight rows per item (W13: 64 gate + 64 up)
constexpr int kKStage = 512;           // K elements per stage
constexpr int kStageA = kRowsPerBlock * kKStage / 2;  // 32 KB packed
constexpr int kStageS = kRowsPerBlock * kKStage / 32; // 2 KB scales
constexpr int kStageBytes = kStageA + kStageS;        // 34 KB (multiple of 1024)
constexpr int kMaxTok = kGemvTokens;   // 8 tokens = the MMA N

struct StreamParams {
  const int4* chunks;      // (expert, first sorted row, rows, 0)
  const int32_t* counts;   // counts[1] = number of chunks
  const int32_t* sorted_slot;
  const uint16_t* act;     // activations: x [T, d] (W13) or h [S, I] (W2), bf16
  int32_t* err;
  uint16_t* h_out;         // W13: h [S, I]
  float* y_out;            // W2: y [S, d]
  float* out;              // W2, non-null: out [T, d] += w * y row by row (fp32 atomic adds), no y
  float4* zero;            // W13, non-null: out, zeroed by this kernel before the W2 kernel adds into it
  long long zero_n4;       // its length in float4
  const float* topk_w;     // routing weights by slot (with out)
  int k, d, I;
  int K;                   // reduction length: d (W13) or I (W2)
  int n_rb;                // row blocks per expert
  int stages;              // ring depth
  int x_pitch;             // bytes per token row of the f16 activation buffer
  uint64_t wait_ns;        // limit of every mbarrier wait
  int fault;               // nonzero: CTA 0 withholds its first weight stage (fault-injection test)
  int act_l2;              // nonzero: read the activations through L2 only (written by other SMs in this launch)
};

// Shared-memory loads by 32-bit shared-window address.  Not volatile, so loads
// of later blocks may be scheduled early; the memory clobber keeps them after
// the wait on the stage's full barrier.
//
// 4 consecutive bytes, one per register (zero-extended): the E8M0 scales.
__device__ __forceinline__ void lds_bytes4(uint32_t a, uint32_t (&b)[4]) {
  asm("ld.shared.v4.u8 {%0,%1,%2,%3}, [%4];"
      : "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3])
      : "r"(a)
      : "memory");
}

__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
  uint32_t v;
  asm("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}

__device__ __forceinline__ uint4 lds_u128(uint32_t a) {
  uint4 v;
  asm("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a) : "memory");
  return v;
}

// The 8 E2M1 codes of a 32-bit word as 4 f16x2 registers (byte j -> r[j],
// low nibble -> low half).  The vector move names the word's bytes for the
// conversions, so no shifts or masks are spent on the ALU pipe.
__device__ __forceinline__ void e2m1x8_f16(uint32_t w, uint32_t (&r)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(w));
}

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                          const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

// An E8M0 byte s as the fp32 factor 2^(s-126) = 2 * 2^(s-127): (s + 1) << 23
// is a normal fp32 for every s in [0, 253] (0 needs no special case); the
// factor 2 is taken back in the token scale.  One integer multiply-add.
__device__ __forceinline__ float scale2_of(uint32_t s) { return __uint_as_float(s * (1u << 23) + (1u << 23)); }

// Item geometry.  W13: rows [i0, i0+64) of gate and up; W2: rows [n0, n0+128).
template <bool W13>
__device__ __forceinline__ void issue_stage(const CUtensorMap* map_w, const CUtensorMap* map_s, const StreamParams& P,
                                            int e, int rb, int ks, uint8_t* dst, uint64_t* bar, uint64_t pol) {
  const int xa = ks * (kKStage / 2);   // byte column of the packed codes
  const int xs = ks * (kKStage / 32);  // byte column of the scales
  mbar_expect_tx(bar, kStageBytes);
  if (W13) {
    const int gate = e * 2 * P.I + rb * 64, up = gate + P.I;
    tma_load_2d_hint(dst + 0 * 8192, map_w, xa, gate, bar, pol);
    tma_load_2d_hint(dst + 1 * 8192, map_w, xa + 128, gate, bar, pol);
    tma_load_2d_hint(dst + 2 * 8192, map_w, xa, up, bar, pol);
    tma_load_2d_hint(dst + 3 * 8192, map_w, xa + 128, up, bar, pol);
    tma_load_2d(dst + kStageA, map_s, xs, gate, bar);
    tma_load_2d(dst + kStageA + 1024, map_s, xs, up, bar);
  } else {
    const int r0 = e * P.d + rb * 128;
    tma_load_2d_hint(dst, map_w, xa, r0, bar, pol);
    tma_load_2d_hint(dst + 16384, map_w, xa + 128, r0, bar, pol);
    tma_load_2d(dst + kStageA, map_s, xs, r0, bar);
  }
}

// Shared memory of the streaming kernels (one layout for every phase).
struct StreamSmem {
  uint8_t* ring;           // [stages][kStageBytes]
  uint8_t* xs_buf;         // [8 tokens][x_pitch] f16 activations of the current chunk
  float4* red;             // [2][kKSplit-1][8 tiles][32] partial sums of the K split
  float* tok_scale;        // [8]
  int* tok_row;            // [8] W2 with out: token of each chunk row
  float* tok_w;            // [8] W2 with out: routing weight of each chunk row
  uint64_t* full;          // [stages]
  uint64_t* empty;         // [stages]
  volatile int* abort_flag;
};

__device__ __forceinline__ StreamSmem stream_smem(uint8_t* smem_raw, int stages, int x_pitch) {
  StreamSmem S;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  S.ring = smem;
  S.xs_buf = S.ring + (size_t)stages * kStageBytes;
  S.red = reinterpret_cast<float4*>(S.xs_buf + (size_t)kMaxTok * x_pitch);
  S.tok_scale = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(S.red) + kRedBytes);
  S.tok_row = reinterpret_cast<int*>(S.tok_scale + kMaxTok);
  S.tok_w = reinterpret_cast<float*>(S.tok_row + kMaxTok);
  S.full = reinterpret_cast<uint64_t*>(S.tok_w + kMaxTok);
  S.empty = S.full + stages;
  S.abort_flag = reinterpret_cast<volatile int*>(S.empty + stages);
  return S;
}

__device__ __forceinline__ void stream_init(const StreamSmem& S, int stages) {
  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], kConsWarps);
    }
    *S.abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
}

// The producer's ring state, carried from one phase to the next.
struct ProdRing {
  int slot = 0;
  uint32_t phase = 0;
  uint32_t nxt = 0;    // bit s: parity of the next copy into slot s (its full-barrier phase)
  uint32_t has = 0;    // bit s: slot s received a copy
  bool ok = true;
};

// The consumers' ring state, carried from one phase to the next.
struct ConsRing {
  int slot = 0;
  int rbuf = 0;
  uint32_t phase = 0;
};

// This CTA's share [it0, it1) of the items (chunk, row block) of one projection.
__device__ __forceinline__ void stream_items(const StreamParams& P, long long& it0, long long& it1) {
  const int n_chunks = __ldcg(P.counts + 1);
  const long long n_items = (long long)n_chunks * P.n_rb;
  it0 = n_items * blockIdx.x / gridDim.x;
  it1 = n_items * (blockIdx.x + 1) / gridDim.x;
}

// Producer (one thread): streams the weight stages of this CTA's items.
template <bool W13>
__device__ __forceinline__ void stream_produce(const CUtensorMap* map_w, const CUtensorMap* map_s,
                                               const StreamParams& P, const StreamSmem& S, ProdRing& R) {
  long long it0, it1;
  stream_items(P, it0, it1);
  const int nst = P.K / kKStage;
  const uint64_t pol = l2_evict_first_policy();
  bool withhold = P.fault != 0 && blockIdx.x == 0;
  for (long long it = it0; it < it1 && R.ok; ++it) {
    const int c = (int)(it / P.n_rb), rb = (int)(it % P.n_rb);
    const int e = __ldcg(P.chunks + c).x;
    for (int ks = 0; ks < nst; ++ks) {
      if (!mbar_wait(&S.empty[R.slot], R.phase ^ 1u, S.abort_flag, P.err, kErrWaitTimeout, P.wait_ns) ||
          *S.abort_flag) {
        R.ok = false;
        break;
      }
      // (a slot comes back only once every consumer read its stage, or saw
      // the abort that the check above catches: one copy per slot in flight)
      if (withhold) {
        // fault injection: this stage never arrives, so the consumers' wait
        // on it runs out and the kernel takes its abort path
        withhold = false;
      } else {
        issue_stage<W13>(map_w, map_s, P, e, rb, ks, S.ring + (size_t)R.slot * kStageBytes, &S.full[R.slot], pol);
        R.nxt ^= 1u << R.slot;
        R.has |= 1u << R.slot;
      }
      if (++R.slot == P.stages) {
        R.slot = 0;
        R.phase ^= 1u;
      }
    }
  }
}

// Every copy the producer issued has landed before the CTA may exit.
__device__ __forceinline__ void stream_drain(const StreamParams& P, const StreamSmem& S, const ProdRing& R) {
  for (int q = 0; q < P.stages; ++q)
    if ((R.has >> q) & 1) mbar_wait_drain(&S.full[q], ((R.nxt >> q) & 1) ^ 1u, P.err, kErrWaitTimeout, P.wait_ns);
}

// Consumer warps (16): this CTA's items of one projection.
template <bool W13>
__device__ __forceinline__ void stream_consume(const StreamParams& P, const StreamSmem& S, ConsRing& R) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long it0, it1;
  stream_items(P, it0, it1);
  const int nst = P.K / kKStage;
  uint8_t* const ring = S.ring;
  uint8_t* const xs_buf = S.xs_buf;
  float4* const red = S.red;
  float* const tok_scale = S.tok_scale;
  uint64_t* const full = S.full;
  uint64_t* const empty = S.empty;
  volatile int* const abort_flag = S.abort_flag;
  const int g = lane >> 2, t = lane & 3;
  const int tile = warp % kTiles, kpart = warp / kTiles;  // 16-row tile, share of the stage's blocks
  // rows of this thread inside the stage's 128 rows (A-fragment rows g and g+8)
  const int rowA = W13 ? tile * 8 + g : tile * 16 + g;  // gate row / first W2 row; row B: the
  // matching up row 64 rows on (W13) or the row 8 rows on (W2).  Both rows have the
  // same 128-byte swizzle phase (g), so row B's bytes sit a fixed distance after
  // row A's: the up half of the stage (W13) or 8 rows of 128 bytes (W2).
  constexpr uint32_t kDeltaB = W13 ? 16384 : 8 * 128;
  constexpr uint32_t kDeltaS = W13 ? 64 * 16 : 8 * 16;  // the same for the scale rows
  // packed boxes: K 0..255 and 256..511, each 128 rows (W2) or 2 x 64 rows (W13)
  const int box_stride = W13 ? 8192 : 16384;
  const int ra = W13 ? rowA & 63 : rowA;
  const int baseA = ra * 128 + 4 * t;
  // 32-bit shared addresses; per block of this warp's share, the swizzled offset
  // of this thread's 4 packed bytes of row A inside a stage
  const uint32_t ring_s = smem_u32(ring), xs_s = smem_u32(xs_buf);
  const uint32_t sofA = kStageA + rowA * 16 + kpart * kBlkPerWarp;
  uint32_t offA[kBlkPerWarp];
#pragma unroll
  for (int bi = 0; bi < kBlkPerWarp; ++bi) {
    const int blk = kpart * kBlkPerWarp + bi;
    offA[bi] = baseA + (blk >> 3) * box_stride + (((blk & 7) ^ (ra & 7)) << 4);
  }
  int cur = -1, row0 = 0, mt = 0;
  int& slot = R.slot;
  int& rbuf = R.rbuf;
  uint32_t& phase = R.phase;
  for (long long it = it0; it < it1; ++it) {
    const int c = (int)(it / P.n_rb), rb = (int)(it % P.n_rb);
    if (c != cur) {
      // new token chunk: stage its activations (warp w <- token w) as scaled f16
      asm volatile("bar.sync 1, %0;" ::"r"(kConsWarps * 32) : "memory");
      const int4 ch = P.chunks[c];
      row0 = ch.y;
      mt = ch.z;
      uint8_t* xrow = xs_buf + (size_t)warp * P.x_pitch;
      if (warp >= kMaxTok) {
        // no token row for this warp
      } else if (warp < mt) {
        const int src_row = W13 ? P.sorted_slot[row0 + warp] / P.k : row0 + warp;
        const uint4* src = reinterpret_cast<const uint4*>(P.act + (size_t)src_row * P.K);
        uint32_t emax = 1;
        for (int v = lane; v < P.K / 8; v += 32) {
          const uint4 q = P.act_l2 ? __ldcg(src + v) : src[v];
          const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) emax = max(emax, max((w[i] >> 7) & 0xFFu, (w[i] >> 23) & 0xFFu));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) emax = max(emax, __shfl_xor_sync(0xFFFFFFFFu, emax, o));
        const int shift = 141 - (int)emax;  // the largest magnitude lands in [2^14, 2^15)
        const float f1 = pow2f(shift / 2), f2 = pow2f(shift - shift / 2);
        for (int v = lane; v < P.K / 8; v += 32) {
          const uint4 q = P.act_l2 ? __ldcg(src + v) : src[v];
          const uint32_t w[4] = {q.x, q.y, q.z, q.w};
          uint32_t o[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const __half2 h = __floats2half2_rn(bf16_to_f32(w[i] & 0xFFFFu) * f1 * f2, bf16_to_f32(w[i] >> 16) * f1 * f2);
            o[i] = *reinterpret_cast<const uint32_t*>(&h);
          }
          reinterpret_cast<uint4*>(xrow)[v] = make_uint4(o[0], o[1], o[2], o[3]);
        }
        if (lane == 0) {
          tok_scale[warp] = pow2f(-shift - 1);  // 2^-shift / 2 (scale2_of carries a factor 2)
          if (!W13 && P.out) {
            const int slot = P.sorted_slot[row0 + warp];
            S.tok_row[warp] = slot / P.k;
            S.tok_w[warp] = P.topk_w[slot];
          }
        }
      } else {
        for (int v = lane; v < P.K / 8; v += 32) reinterpret_cast<uint4*>(xrow)[v] = make_uint4(0, 0, 0, 0);
        if (lane == 0) tok_scale[warp] = 0.f;
      }
      asm volatile("bar.sync 1, %0;" ::"r"(kConsWarps * 32) : "memory");
      cur = c;
    }
    // after an abort the waits are skipped but the arithmetic still runs (on
    // whatever the ring holds; nothing is kept), so that the warp-wide
    // mma.sync below always sees all 32 lanes
    const bool run = !*abort_flag;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t xk0 = xs_s + g * P.x_pitch + 16 * t + kpart * kBlkPerWarp * 64;
    for (int ks = 0; ks < nst; ++ks) {
      if (run) mbar_wait(&full[slot], phase, abort_flag, P.err, kErrWaitTimeout, P.wait_ns);
      {
        const uint32_t st = ring_s + slot * kStageBytes;
        // the E8M0 bytes of this warp's blocks [kpart * kBlkPerWarp, +kBlkPerWarp), one per register
        uint32_t sbA[kBlkPerWarp], sbB[kBlkPerWarp];
#pragma unroll
        for (int i = 0; i < kBlkPerWarp / 4; ++i) {
          uint32_t ta[4], tb[4];
          lds_bytes4(st + sofA + 4 * i, ta);
          lds_bytes4(st + sofA + kDeltaS + 4 * i, tb);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            sbA[4 * i + j] = ta[j];
            sbB[4 * i + j] = tb[j];
          }
        }
        const uint32_t xk = xk0 + ks * kKStage * 2;
#pragma unroll
        for (int bi = 0; bi < kBlkPerWarp; ++bi) {
          uint32_t ha[4], hb[4];  // this thread's 8 codes of rows A and B as f16 pairs
          const uint32_t pa = st + offA[bi];
          e2m1x8_f16(lds_u32(pa), ha);
          e2m1x8_f16(lds_u32(pa + kDeltaB), hb);
          const uint4 xf = lds_u128(xk + bi * 64);
          const float zero[4] = {0.f, 0.f, 0.f, 0.f};
          float cb[4];
          uint32_t a[4] = {ha[0], hb[0], ha[1], hb[1]};
          mma_16816(cb, a, xf.x, xf.y, zero);
          a[0] = ha[2];
          a[1] = hb[2];
          a[2] = ha[3];
          a[3] = hb[3];
          mma_16816(cb, a, xf.z, xf.w, cb);
          const float fa = scale2_of(sbA[bi]), fb = scale2_of(sbB[bi]);
          acc[0] = fmaf(cb[0], fa, acc[0]);
          acc[1] = fmaf(cb[1], fa, acc[1]);
          acc[2] = fmaf(cb[2], fb, acc[2]);
          acc[3] = fmaf(cb[3], fb, acc[3]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      if (++slot == P.stages) {
        slot = 0;
        phase ^= 1u;
      }
    }
    // the warps sharing a tile add their partial sums; the exit decision on an
    // abort is taken jointly (barrier with an OR vote) so no barrier is left
    // waiting.  With the combine in the W2 epilogue each warp adds its own
    // partial sums into out (the order of the additions is free), no exchange.
    const bool pair_sum = W13 || !P.out;
    bool aborted = *abort_flag;
    if (kKSplit > 1 && pair_sum) {
      if (kpart > 0)
        red[((rbuf * (kKSplit - 1) + kpart - 1) * kTiles + tile) * 32 + lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      uint32_t any;
      asm volatile(
          "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n}"
          : "=r"(any)
          : "r"((uint32_t)aborted), "r"(2 + tile), "r"(32 * kKSplit)
          : "memory");
      aborted = any != 0;
      if (kpart == 0) {
#pragma unroll
        for (int p = 0; p < kKSplit - 1; ++p) {
          const float4 o = red[((rbuf * (kKSplit - 1) + p) * kTiles + tile) * 32 + lane];
          acc[0] += o.x;
          acc[1] += o.y;
          acc[2] += o.z;
          acc[3] += o.w;
        }
      }
      rbuf ^= 1;
    }
    if (aborted || (pair_sum && kpart > 0)) continue;  // keep meeting the chunk barriers, no output
    // epilogue: acc[0..1] = row A x tokens 2t, 2t+1; acc[2..3] = row B
    const int t0 = 2 * t, t1 = 2 * t + 1;
    const float s0 = tok_scale[t0], s1 = tok_scale[t1];
    if (W13) {
      const int i = rb * 64 + tile * 8 + g;
      if (t0 < mt) P.h_out[(size_t)(row0 + t0) * P.I + i] = f32_to_bf16_rn(swiglu(acc[0] * s0, acc[2] * s0));
      if (t1 < mt) P.h_out[(size_t)(row0 + t1) * P.I + i] = f32_to_bf16_rn(swiglu(acc[1] * s1, acc[3] * s1));
    } else if (P.out) {
      // the weighted combine: each slot's row added into its token's out row
      const int n = rb * 128 + tile * 16 + g;
      if (t0 < mt) {
        float* o = P.out + (size_t)S.tok_row[t0] * P.d + n;
        const float w = S.tok_w[t0];
        red_add_f32(o, w * (acc[0] * s0));
        red_add_f32(o + 8, w * (acc[2] * s0));
      }
      if (t1 < mt) {
        float* o = P.out + (size_t)S.tok_row[t1] * P.d + n;
        const float w = S.tok_w[t1];
        red_add_f32(o, w * (acc[1] * s1));
        red_add_f32(o + 8, w * (acc[3] * s1));
      }
    } else {
      const int n = rb * 128 + tile * 16 + g;
      if (t0 < mt) {
        P.y_out[(size_t)(row0 + t0) * P.d + n] = acc[0] * s0;
        P.y_out[(size_t)(row0 + t0) * P.d + n + 8] = acc[2] * s0;
      }
      if (t1 < mt) {
        P.y_out[(size_t)(row0 + t1) * P.d + n] = acc[1] * s1;
        P.y_out[(size_t)(row0 + t1) * P.d + n + 8] = acc[3] * s1;
      }
    }
  }
}

template <bool W13>
__global__ void __launch_bounds__(kThreads, 1)
stream_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_s,
              const StreamParams P) {
  extern __shared__ uint8_t smem_raw[];
  const StreamSmem S = stream_smem(smem_raw, P.stages, P.x_pitch);
  stream_init(S, P.stages);
  // Both kernels are launched early.  W13 waits here for the routing kernel
  // (the work list); W2 was let start only after every W13 CTA had passed
  // that wait, so the work list is complete, and it reads it through L2
  // (ld.global.cg) so that its producer can stream weights while W13 ends;
  // its consumers wait for W13 (h) below.
  // out is zeroed while the routing kernel still runs (nothing of this call
  // reads or writes it before the W2 kernel, which waits for this one)
  if (W13 && P.zero)
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < P.zero_n4; i += (long long)gridDim.x * blockDim.x)
      P.zero[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (W13) griddep_wait();
  griddep_launch_dependents();
  if ((threadIdx.x >> 5) == kConsWarps) {
    if ((threadIdx.x & 31) == 0) {
      ProdRing R;
      stream_produce<W13>(&map_w, &map_s, P, S, R);
      stream_drain(P, S, R);
    }
    return;
  }
  if (!W13) griddep_wait();  // h comes from the W13 kernel
  ConsRing R;
  stream_consume<W13>(P, S, R);
}

// The decode layer's two projections in one persistent launch: W13 + SwiGLU
// over this CTA's items, a grid-wide arrival counter, then W2.  One weight
// ring serves both phases, so the producer streams W2's first stages while
// the consumers finish W13 (weights do not depend on h).  The counter lives
// in the workspace (zeroed by the routing kernel of the same call); its wait
// is bounded, and on a timeout the consumers skip W2's arithmetic (error bit
// 2).  Launched cooperatively: all CTAs (one per SM) are resident together.
__global__ void __launch_bounds__(kThreads, 1)
stream_fused_kernel(const __grid_constant__ CUtensorMap map_w13, const __grid_constant__ CUtensorMap map_s13,
                    const __grid_constant__ CUtensorMap map_w2, const __grid_constant__ CUtensorMap map_s2,
                    const StreamParams P13, const StreamParams P2, int32_t* arrivals) {
  extern __shared__ uint8_t smem_raw[];
  const StreamSmem S = stream_smem(smem_raw, P13.stages, P13.x_pitch);
  // out is zeroed before the W2 phase adds into it (the grid-wide barrier
  // between the phases orders the two)
  if (P13.zero)
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < P13.zero_n4; i += (long long)gridDim.x * blockDim.x)
      P13.zero[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  stream_init(S, P13.stages);
  griddep_launch_dependents();
  if ((threadIdx.x >> 5) == kConsWarps) {
    if ((threadIdx.x & 31) == 0) {
      ProdRing R;
      stream_produce<true>(&map_w13, &map_s13, P13, S, R);
      stream_produce<false>(&map_w2, &map_s2, P2, S, R);
      stream_drain(P2, S, R);
    }
    return;
  }
  ConsRing R;
  stream_consume<true>(P13, S, R);
  // grid-wide barrier between the phases: every CTA's h is written
  asm volatile("bar.sync 1, %0;" ::"r"(kConsWarps * 32) : "memory");
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(arrivals, 1);
    const uint64_t t0 = global_timer_ns();
    while (true) {
      int seen;
      asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(seen) : "l"(arrivals) : "memory");
      if (seen >= (int)gridDim.x) break;
      if (global_timer_ns() - t0 > P2.wait_ns) {
        *S.abort_flag = 1;
        atomicOr(P2.err, kErrWaitTimeout);
        break;
      }
      __nanosleep(200);
    }
    __threadfence();
  }
  asm volatile("bar.sync 1, %0;" ::"r"(kConsWarps * 32) : "memory");
  stream_consume<false>(P2, S, R);
}

size_t smem_needed(int stages, int x_pitch) {
  return 1024 /* alignment slack */ + (size_t)stages * kStageBytes + (size_t)kMaxTok * x_pitch + kRedBytes +
         3 * kMaxTok * sizeof(float) + 2 * stages * sizeof(uint64_t) + 16;
}

template <bool W13>
cudaError_t launch_stream(const CUtensorMap& mw, const CUtensorMap& ms, StreamParams P, cudaStream_t st) {
  P.x_pitch = P.K * 2 + 64;  // 64-byte skew: conflict-free 16-byte reads across tokens
  P.stages = 4;
  while (P.stages > 2 && smem_needed(P.stages, P.x_pitch) > 227 * 1024) --P.stages;
  const size_t smem = smem_needed(P.stages, P.x_pitch);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  const cudaError_t oe = ensure_smem_optin(reinterpret_cast<const void*>(stream_kernel<W13>), 227 * 1024);
  if (oe != cudaSuccess) return oe;
  return launch_early(stream_kernel<W13>, dim3(num_sms()), dim3(kThreads), smem, st, mw, ms, P);
}

bool maps_w13(const moe_fp4_dims& d, const uint8_t* w13, const uint8_t* w13s, CUtensorMap* mw, CUtensorMap* ms) {
  const uint64_t rows = (uint64_t)d.E * 2 * d.I;
  return make_map_2d(mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, w13, d.d / 2, rows, d.d / 2, 128, 64,
                     CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_map_2d(ms, CU_TENSOR_MAP_DATA_TYPE_UINT8, w13s, d.d / 32, rows, d.d / 32, 16, 64,
                     CU_TENSOR_MAP_SWIZZLE_NONE);
}

bool maps_w2(const moe_fp4_dims& d, const uint8_t* w2, const uint8_t* w2s, CUtensorMap* mw, CUtensorMap* ms) {
  const uint64_t rows = (uint64_t)d.E * d.d;
  return make_map_2d(mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, w2, d.I / 2, rows, d.I / 2, 128, 128,
                     CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_map_2d(ms, CU_TENSOR_MAP_DATA_TYPE_UINT8, w2s, d.I / 32, rows, d.I / 32, 16, 128,
                     CU_TENSOR_MAP_SWIZZLE_NONE);
}

StreamParams params_w13(const moe_fp4_dims& d, const uint16_t* x, const Workspace& ws) {
  StreamParams P{};
  P.chunks = ws.gemv_chunks;
  P.counts = ws.counts;
  P.sorted_slot = ws.sorted_slot;
  P.act = x;
  P.err = ws.err;
  P.h_out = ws.h;
  P.k = d.k;
  P.d = d.d;
  P.I = d.I;
  P.K = d.d;
  P.n_rb = d.I / 64;
  P.wait_ns = wait_limit_ns();
  P.fault = fault_site() == MOE_FP4_FAULT_STREAM_STAGE;
  return P;
}

StreamParams params_w2(const moe_fp4_dims& d, const Workspace& ws, float* out) {
  StreamParams P{};
  P.out = out;
  P.topk_w = ws.topk_w;
  P.chunks = ws.gemv_chunks;
  P.counts = ws.counts;
  P.sorted_slot = ws.sorted_slot;
  P.act = ws.h;
  P.err = ws.err;
  P.y_out = ws.y;
  P.k = d.k;
  P.d = d.d;
  P.I = d.I;
  P.K = d.I;
  P.n_rb = d.d / 128;
  P.wait_ns = wait_limit_ns();
  P.fault = 0;
  return P;
}

}  // namespace

bool stream_path_supported(const moe_fp4_dims& d) {
  // whole 512-K stages, 64-row W13 blocks, 128-row W2 blocks; 8 token rows of
  // K f16 activations must fit shared memory next to the ring
  return d.d % 1024 == 0 && d.I % 1024 == 0 && d.d <= 7168 && d.I <= 7168;
}

cudaError_t launch_stream_w13(const moe_fp4_dims& d, const uint16_t* x, const uint8_t* w13, const uint8_t* w13s,
                              const Workspace& ws, float* zero_out, cudaStream_t st) {
  CUtensorMap mw, ms;
  if (!maps_w13(d, w13, w13s, &mw, &ms)) return cudaErrorInvalidValue;
  StreamParams P = params_w13(d, x, ws);
  P.zero = reinterpret_cast<float4*>(zero_out);
  P.zero_n4 = (long long)d.T * d.d / 4;
  return launch_stream<true>(mw, ms, P, st);
}

cudaError_t launch_stream_w2(const moe_fp4_dims& d, const uint8_t* w2, const uint8_t* w2s, const Workspace& ws,
                             float* out, cudaStream_t st) {
  CUtensorMap mw, ms;
  if (!maps_w2(d, w2, w2s, &mw, &ms)) return cudaErrorInvalidValue;
  return launch_stream<false>(mw, ms, params_w2(d, ws, out), st);
}

cudaError_t launch_stream_fused(const moe_fp4_dims& d, const uint16_t* x, const uint8_t* w13, const uint8_t* w13s,
                                const uint8_t* w2, const uint8_t* w2s, const Workspace& ws, float* out,
                                cudaStream_t st) {
  CUtensorMap mw13, ms13, mw2, ms2;
  if (!maps_w13(d, w13, w13s, &mw13, &ms13) || !maps_w2(d, w2, w2s, &mw2, &ms2)) return cudaErrorInvalidValue;
  StreamParams P13 = params_w13(d, x, ws), P2 = params_w2(d, ws, out);
  P13.zero = reinterpret_cast<float4*>(out);
  P13.zero_n4 = (long long)d.T * d.d / 4;
  // one shared-memory layout for both phases: the wider activation rows
  const int x_pitch = (d.d > d.I ? d.d : d.I) * 2 + 64;
  int stages = 4;
  while (stages > 2 && smem_needed(stages, x_pitch) > 227 * 1024) --stages;
  const size_t smem = smem_needed(stages, x_pitch);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  P13.x_pitch = P2.x_pitch = x_pitch;
  P13.stages = P2.stages = stages;
  P2.act_l2 = 1;  // h is written by the other CTAs of the same launch
  const cudaError_t oe = ensure_smem_optin(reinterpret_cast<const void*>(stream_fused_kernel), 227 * 1024);
  if (oe != cudaSuccess) return oe;
  // the CTAs wait on one another (the arrival counter): a cooperative launch
  // makes them all resident at once, one per SM
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms());
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int32_t* arrivals = ws.counts + 3;
  return cudaLaunchKernelEx(&cfg, stream_fused_kernel, mw13, ms13, mw2, ms2, P13, P2, arrivals);
}

}  // namespace moe_fp4
