// Routing (top-k with a fixed tie-break and softmax over the picked logits)
// and the stable counting sort of the T*k slots by expert.
//
// Top-k follows the MI250 correctness blog (section 4.1 table: fp32
// comparison and a fixed tie-break; section 4.2: ties go to the lower
// expert id, never to memory order).  The sort is the "expert sorting" step
// of the DeepSeek-V4-Flash-on-gfx90a paper's prefill path: a stable
// counting sort, so the permutation is unique and reproducible.
//
// Three kernels:
//   route_hist  one warp per token: k rounds of a warp-wide argmax over the
//               token's E logits (two warp reductions per round: the largest
//               key, then the lowest index holding it), softmax of the k
//               picked, per-block counts
//   sort_scan   one block: per-expert totals, offsets, per-block bases, the
//               list of non-empty experts and the work lists of the expert
//               kernels (so the host never reads a count)
//   scatter     one block per routing block: stable ranks by warp match,
//               writes sorted_slot and its inverse
#include "moe_fp4_internal.cuh"

namespace moe_fp4 {
namespace {

constexpr int kWarps = kRouteThreads / 32;
constexpr int kTokPerWarp = kRouteTokensPerBlock / kWarps;

// Order-preserving map of a finite fp32 to uint32 (-0 folded onto +0).
__device__ __forceinline__ uint32_t ordered_key(float v) {
  uint32_t u = __float_as_uint(v == 0.0f ? 0.0f : v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Top-k of one token's E logits (staged in `row`, shared memory) by (value
// desc, index asc) and the softmax over the k picked, shifted by the slot-0
// logit with the sum in slot order.  Lane j < k returns slot j.
__device__ __forceinline__ void topk_softmax_warp(const float* row, int E, int k, int lane, int& id, float& w) {
  const int nv = (E + 31) >> 5;  // entries per lane: e = lane + 32 i
  uint32_t taken = 0;            // bit i: entry lane + 32 i already picked
  int my_id = 0;
  float my_val = 0.f;
  if (E <= 256) {
    // up to 8 entries per lane, kept in registers as unique 64-bit keys
    // (ordered value, then the inverted index: equal values rank the lower
    // index first); a picked or absent entry is 0
    unsigned long long kk[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      kk[i] = e < E ? ((unsigned long long)ordered_key(row[e]) << 32) | (0xFFFFFFFFu - (uint32_t)e) : 0ull;
    }
    for (int r = 0; r < k; ++r) {
      unsigned long long b = kk[0];
#pragma unroll
      for (int i = 1; i < 8; ++i) b = kk[i] > b ? kk[i] : b;
      const uint32_t hi = (uint32_t)(b >> 32);
      const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, hi);
      const uint32_t l = __reduce_max_sync(0xFFFFFFFFu, hi == m ? (uint32_t)b : 0u);
      const int e_star = (int)(0xFFFFFFFFu - l);
      const int won = (e_star & 31) == lane ? (e_star >> 5) : -1;
#pragma unroll
      for (int i = 0; i < 8; ++i) kk[i] = i == won ? 0ull : kk[i];
      if (lane == r) {
        my_id = e_star;
        my_val = row[e_star];
      }
    }
  } else for (int r = 0; r < k; ++r) {
    // this lane's best remaining entry (the first of equal keys: lowest index)
    uint32_t best = 0;
    int best_e = -1;
    for (int i = 0; i < nv; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u)) {
        const uint32_t key = ordered_key(row[e]);
        if (best_e < 0 || key > best) {
          best = key;
          best_e = e;
        }
      }
    }
    // warp-wide: the largest key, then the lowest index holding it
    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, best_e < 0 ? 0u : best);
    const uint32_t cand = (best_e >= 0 && best == m) ? (uint32_t)best_e : 0xFFFFFFFFu;
    const int e_star = (int)__reduce_min_sync(0xFFFFFFFFu, cand);
    if ((e_star & 31) == lane) taken |= 1u << (e_star >> 5);
    if (lane == r) {
      my_id = e_star;
      my_val = row[e_star];
    }
  }
  const float m = __shfl_sync(0xFFFFFFFFu, my_val, 0);
  const float ex = lane < k ? expf(my_val - m) : 0.f;
  float sum = 0.f;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(0xFFFFFFFFu, ex, j);
  id = my_id;
  w = ex / sum;
}

__global__ void __launch_bounds__(kRouteThreads)
route_hist_kernel(const float* __restrict__ logits, int T, int E, int k,
                  int32_t* __restrict__ topk_ids, float* __restrict__ topk_w,
                  int32_t* __restrict__ block_hist, int32_t* __restrict__ err) {
  extern __shared__ float smem[];
  // the error words start clear on every call (later kernels of the call set them)
  if (blockIdx.x == 0 && threadIdx.x < 4) err[threadIdx.x] = 0;
  float* rows = smem;                                     // [kWarps][E]
  int* hist = reinterpret_cast<int*>(smem + kWarps * E);  // [E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  float* row = rows + warp * E;
  for (int tt = 0; tt < kTokPerWarp; ++tt) {
    const int t = blockIdx.x * kRouteTokensPerBlock + warp * kTokPerWarp + tt;
    if (t >= T) break;
    const float* src = logits + (size_t)t * E;
    for (int e = lane; e < E; e += 32) row[e] = src[e];
    __syncwarp();
    int id;
    float w;
    topk_softmax_warp(row, E, k, lane, id, w);
    if (lane < k) {
      topk_ids[(size_t)t * k + lane] = id;
      topk_w[(size_t)t * k + lane] = w;
      atomicAdd(&hist[id], 1);
    }
    __syncwarp();
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) block_hist[(size_t)blockIdx.x * E + e] = hist[e];
}

// Exclusive scan over the block (blockDim.x <= 1024, a multiple of 32).
__device__ int block_exclusive_scan(int v, int* scratch /* [32] */, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += n;
  }
  __syncthreads();
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int w = lane < nw ? scratch[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(0xFFFFFFFFu, wi, o);
      if (lane >= o) wi += n;
    }
    scratch[lane] = wi - w;  // exclusive prefix of warp totals
    if (lane == 31) scratch[32] = wi;
  }
  __syncthreads();
  const int res = scratch[warp] + incl - v;
  *total = scratch[32];
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(1024)
sort_scan_kernel(int32_t* __restrict__ block_hist, int nb, int E, int32_t* __restrict__ offsets,
                 int32_t* __restrict__ active, int32_t* __restrict__ counts,
                 int4* __restrict__ gemv_chunks, int4* __restrict__ tc_tiles) {
  __shared__ int scratch[33];
  const int e = threadIdx.x;
  const bool ok = e < E;
  int cnt = 0;
  if (ok)
    for (int b = 0; b < nb; ++b) cnt += block_hist[(size_t)b * E + e];
  int total;
  const int off = block_exclusive_scan(ok ? cnt : 0, scratch, &total);
  if (ok) {
    offsets[e] = off;
    int run = off;
    for (int b = 0; b < nb; ++b) {
      const int c = block_hist[(size_t)b * E + e];
      block_hist[(size_t)b * E + e] = run;
      run += c;
    }
  }
  if (e == 0) offsets[E] = total;
  // non-empty experts
  int n_active;
  const int apos = block_exclusive_scan(ok && cnt > 0 ? 1 : 0, scratch, &n_active);
  if (ok && cnt > 0) active[apos] = e;
  // GEMV chunks of up to kGemvTokens rows
  const int nch = ok ? (cnt + kGemvTokens - 1) / kGemvTokens : 0;
  int n_chunks;
  const int cpos = block_exclusive_scan(nch, scratch, &n_chunks);
  for (int c = 0; c < nch; ++c)
    gemv_chunks[cpos + c] = make_int4(e, off + c * kGemvTokens, min(kGemvTokens, cnt - c * kGemvTokens), 0);
  // tensor-core tiles of up to kTcTileN rows
  // tensor-core tiles: ceil(cnt / kTcTileN) tiles of equal size (rounded up to 16)
  const int ntl = ok ? (cnt + kTcTileN - 1) / kTcTileN : 0;
  const int per = ntl ? (((cnt + ntl - 1) / ntl + 15) & ~15) : 0;
  int n_tiles;
  const int tpos = block_exclusive_scan(ntl, scratch, &n_tiles);
  for (int c = 0; c < ntl; ++c) tc_tiles[tpos + c] = make_int4(e, off + c * per, min(per, cnt - c * per), 0);
  if (e == 0) {
    counts[0] = n_active;
    counts[1] = n_chunks;
    counts[2] = n_tiles;
    counts[3] = 0;
  }
}

__global__ void __launch_bounds__(kRouteThreads)
scatter_kernel(const int32_t* __restrict__ topk_ids, const int32_t* __restrict__ block_base, int T,
               int E, int k, int32_t* __restrict__ sorted_slot, int32_t* __restrict__ slot_pos,
               int32_t* __restrict__ err) {
  extern __shared__ int sm[];
  int* running = sm;            // [E]
  int* wcnt = sm + E;           // [kWarps][E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < E; e += blockDim.x) running[e] = block_base[(size_t)blockIdx.x * E + e];
  for (int i = threadIdx.x; i < kWarps * E; i += blockDim.x) wcnt[i] = 0;
  __syncthreads();
  const long f_begin = (long)blockIdx.x * kRouteTokensPerBlock * k;
  const long f_end = min((long)(blockIdx.x + 1) * kRouteTokensPerBlock, (long)T) * k;
  for (long f0 = f_begin; f0 < f_end; f0 += blockDim.x) {
    const long f = f0 + threadIdx.x;
    int e = f < f_end ? topk_ids[f] : -1;
    if (e >= E || e < -1) {  // corrupted id: report and drop
      atomicOr(err, kErrBadExpertId);
      e = -1;
    }
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const bool leader = rank == 0;
    if (e >= 0 && leader) wcnt[warp * E + e] = __popc(peers);
    __syncthreads();
    if (e >= 0) {
      int pos = running[e] + rank;
      for (int w = 0; w < warp; ++w) pos += wcnt[w * E + e];
      sorted_slot[pos] = (int32_t)f;
      slot_pos[f] = pos;
    }
    __syncthreads();
    if (e >= 0 && leader) {
      atomicAdd(&running[e], __popc(peers));
      wcnt[warp * E + e] = 0;
    }
    __syncthreads();
  }
}


// One block does everything when all tokens fit one routing block (T <= 32,
// the decode shape): routing by 32 warps, per-expert totals, offsets and work
// lists, then the stable scatter by a single warp walking the slots in order.
__global__ void __launch_bounds__(1024)
route_small_kernel(const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ topk_ids,
                   float* __restrict__ topk_w, int32_t* __restrict__ offsets, int32_t* __restrict__ active,
                   int32_t* __restrict__ counts, int4* __restrict__ gemv_chunks, int4* __restrict__ tc_tiles,
                   int32_t* __restrict__ sorted_slot, int32_t* __restrict__ slot_pos, int32_t* __restrict__ err) {
  extern __shared__ int smem_small[];
  int* hist = smem_small;                            // [E] counts, then running positions
  int* ids_s = hist + E;                             // [T*k]
  float* rows = reinterpret_cast<float*>(ids_s + kRouteTokensPerBlock * 32);  // [32 warps][E]
  __shared__ int scratch[33];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x < 4) err[threadIdx.x] = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  if (warp < T) {
    float* row = rows + warp * E;
    const float* src = logits + (size_t)warp * E;
    for (int e = lane; e < E; e += 32) row[e] = src[e];
    __syncwarp();
    int id;
    float w;
    topk_softmax_warp(row, E, k, lane, id, w);
    if (lane < k) {
      topk_ids[warp * k + lane] = id;
      topk_w[warp * k + lane] = w;
      ids_s[warp * k + lane] = id;
      atomicAdd(&hist[id], 1);
    }
  }
  __syncthreads();
  const int e = threadIdx.x;
  const bool ok = e < E;
  const int cnt = ok ? hist[e] : 0;
  int total;
  const int off = block_exclusive_scan(cnt, scratch, &total);
  if (ok) offsets[e] = off;
  if (e == 0) offsets[E] = total;
  int n_active;
  const int apos = block_exclusive_scan(ok && cnt > 0 ? 1 : 0, scratch, &n_active);
  if (ok && cnt > 0) active[apos] = e;
  const int nch = ok ? (cnt + kGemvTokens - 1) / kGemvTokens : 0;
  int n_chunks;
  const int cpos = block_exclusive_scan(nch, scratch, &n_chunks);
  for (int c = 0; c < nch; ++c)
    gemv_chunks[cpos + c] = make_int4(e, off + c * kGemvTokens, min(kGemvTokens, cnt - c * kGemvTokens), 0);
  // tensor-core tiles: ceil(cnt / kTcTileN) tiles of equal size (rounded up to 16)
  const int ntl = ok ? (cnt + kTcTileN - 1) / kTcTileN : 0;
  const int per = ntl ? (((cnt + ntl - 1) / ntl + 15) & ~15) : 0;
  int n_tiles;
  const int tpos = block_exclusive_scan(ntl, scratch, &n_tiles);
  for (int c = 0; c < ntl; ++c) tc_tiles[tpos + c] = make_int4(e, off + c * per, min(per, cnt - c * per), 0);
  if (e == 0) {
    counts[0] = n_active;
    counts[1] = n_chunks;
    counts[2] = n_tiles;
    counts[3] = 0;
  }
  if (ok) hist[e] = off;  // running position of each expert
  __syncthreads();
  if (warp == 0) {
    const int S = T * k;
    for (int f0 = 0; f0 < S; f0 += 32) {
      const int f = f0 + lane;
      const int ef = f < S ? ids_s[f] : -1;
      const unsigned peers = __match_any_sync(0xFFFFFFFFu, ef);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      if (ef >= 0) {
        const int pos = hist[ef] + rank;
        sorted_slot[pos] = f;
        slot_pos[f] = pos;
      }
      __syncwarp();
      if (ef >= 0 && rank == 0) hist[ef] += __popc(peers);
      __syncwarp();
    }
  }
}

}  // namespace

cudaError_t launch_route(const moe_fp4_dims& d, const float* logits, const Workspace& ws, cudaStream_t st) {
  const int nb = ws.nb_route;
  if (nb == 1) {
    const size_t smem = (size_t)d.E * sizeof(int) + kRouteTokensPerBlock * 32 * sizeof(int) +
                        (size_t)32 * d.E * sizeof(float);
    static bool configured = false;
    if (!configured) {
      cudaFuncSetAttribute(route_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
      configured = true;
    }
    route_small_kernel<<<1, 1024, smem, st>>>(logits, d.T, d.E, d.k, ws.topk_ids, ws.topk_w, ws.offsets, ws.active,
                                              ws.counts, ws.gemv_chunks, ws.tc_tiles, ws.sorted_slot, ws.slot_pos,
                                              ws.err);
    return cudaGetLastError();
  }
  size_t smem1 = (size_t)(kWarps * d.E) * sizeof(float) + (size_t)d.E * sizeof(int);
  route_hist_kernel<<<nb, kRouteThreads, smem1, st>>>(logits, d.T, d.E, d.k, ws.topk_ids, ws.topk_w,
                                                     ws.block_hist, ws.err);
  sort_scan_kernel<<<1, 1024, 0, st>>>(ws.block_hist, nb, d.E, ws.offsets, ws.active, ws.counts,
                                       ws.gemv_chunks, ws.tc_tiles);
  size_t smem3 = (size_t)(kWarps + 1) * d.E * sizeof(int);
  scatter_kernel<<<nb, kRouteThreads, smem3, st>>>(ws.topk_ids, ws.block_hist, d.T, d.E, d.k,
                                                   ws.sorted_slot, ws.slot_pos, ws.err);
  return cudaGetLastError();
}

}  // namespace moe_fp4
