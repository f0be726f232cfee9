// Pieces shared by the tensor-core expert kernels (one CTA per tile, and CTA
// pairs): their parameters and inline-PTX wrappers of the 5th-generation
// tensor-core instructions (UMMA descriptors, tcgen05 loads and stores).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ptx_sm103.cuh"

namespace moe_fp4 {
namespace tc {

struct TcParams {
  const uint8_t* w;        // packed E2M1 weights [rows][K/2]
  const uint8_t* scales;   // E8M0 [rows][K/32]
  const int4* tiles;       // (expert, first sorted row, rows, 0)
  const int32_t* counts;   // counts[2] = number of tiles
  int32_t* err;
  uint16_t* h_out;         // W13: h [S, I]
  float* y_out;            // W2: y [S, d]
  const float* x_scale;    // W13: per sorted row, the inverse activation scale
  int K;                   // reduction length
  int rows_per_expert;     // rows of the weight tensor per expert (2I or d)
  int mblocks;             // CTAs per token tile along the weight rows
  int block_rows;          // weight rows advanced per m-block (128 W13, 256 W2)
  int acc1_offset;         // row offset of accumulator 1 (I for up rows, 128 for W2)
  int I, d;
  uint64_t wait_ns;        // limit of every mbarrier wait
  int fault;               // nonzero: the first CTA withholds its first token tile (fault-injection test)
  // CTA pairs only: a pair covers block_rows indices (i for W13, output
  // feature n for W2) per m-block, cta_rows of them per CTA; accumulator a of
  // a CTA holds indices first + a * acc_idx_step + lane, stored in weight row
  // expert * rows_per_expert + a * acc_row_off + index; indices at or beyond
  // limit are not written
  int cta_rows, acc_idx_step, acc_row_off, limit;
  // W2 with the combine in the epilogue (out != nullptr).  CTA pairs: out[t] =
  // sum_j topk_w[t, j] * y[slot_pos[t k + j]] for each 256-feature block,
  // written by the CTA whose item brings the block's last slot (counters).
  // One-SM kernel: each slot's weighted row added into out (zeroed
  // beforehand) with fp32 atomic adds, no y.
  float* out;
  const float* topk_w;
  const int32_t* sorted_slot;
  const int32_t* slot_pos;
  int32_t* combine_cnt;
  int k;
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

// Instruction descriptor of kind::f16 with f32 accumulation, both operands
// K-major; A and B share one type (f16 = 0, bf16 = 1).
__device__ __forceinline__ uint32_t idesc_f16kind(int M, int N, uint32_t ab_type) {
  return (1u << 4)                                // D format f32
         | (ab_type << 7) | (ab_type << 10)       // A, B format
         | ((uint32_t)(N >> 3) << 17)             // N
         | ((uint32_t)(M >> 4) << 24);            // M
}

// D[tmem] (+)= A[tmem] * B[smem]: the A operand is read from tensor memory
__device__ __forceinline__ void umma_tmem_a(uint32_t tmem_d, uint32_t tmem_a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// this thread's TMEM lane, 32 consecutive 32-bit columns from taddr
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// this thread's TMEM lane, 32 columns from each of two addresses, with one
// wait for both loads
__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, uint32_t tb, float (&va)[32], float (&vb)[32]) {
  uint32_t a[32], b[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]),
        "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]),
        "=r"(a[16]), "=r"(a[17]), "=r"(a[18]), "=r"(a[19]), "=r"(a[20]), "=r"(a[21]), "=r"(a[22]), "=r"(a[23]),
        "=r"(a[24]), "=r"(a[25]), "=r"(a[26]), "=r"(a[27]), "=r"(a[28]), "=r"(a[29]), "=r"(a[30]), "=r"(a[31]),
        "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]),
        "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15]),
        "=r"(b[16]), "=r"(b[17]), "=r"(b[18]), "=r"(b[19]), "=r"(b[20]), "=r"(b[21]), "=r"(b[22]), "=r"(b[23]),
        "=r"(b[24]), "=r"(b[25]), "=r"(b[26]), "=r"(b[27]), "=r"(b[28]), "=r"(b[29]), "=r"(b[30]), "=r"(b[31])
      : "r"(ta), "r"(tb)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    va[i] = __uint_as_float(a[i]);
    vb[i] = __uint_as_float(b[i]);
  }
}

// 4 consecutive bytes of shared memory, one per register (zero-extended):
// one load instead of a word load and three shifts on the busy ALU pipe.  Not
// volatile, so it may be scheduled early; the memory clobber keeps it after the
// barrier waits that make the bytes valid.
__device__ __forceinline__ void lds_bytes4(const uint8_t* p, uint32_t (&b)[4]) {
  asm("ld.shared.v4.u8 {%0,%1,%2,%3}, [%4];"
      : "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3])
      : "r"(smem_u32(p))
      : "memory");
}

__device__ __forceinline__ uint32_t f16x2_mul(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// f16x2 (m, m) with m = 2^e for e in [-24, 15]: normal for e >= -14,
// subnormal below; 0 for e < -24
__device__ __forceinline__ uint32_t f16x2_pow2(int e) {
  const uint32_t b = e >= -14 ? (uint32_t)(e + 15) << 10 : (e >= -24 ? 1u << (e + 24) : 0u);
  return b | (b << 16);
}


}  // namespace tc

// the pair kernel's launcher (expert_tc2.cu)
template <bool W13>
cudaError_t launch_tc2(const CUtensorMap& b, const CUtensorMap& raw, const tc::TcParams& P, int max_tiles,
                       cudaStream_t st);

}  // namespace moe_fp4
