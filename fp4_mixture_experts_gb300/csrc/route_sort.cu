// Routing (top-k with a fixed tie-break and softmax over the picked logits)
// and the stable counting sort of the T*k slots by expert.
//
// Top-k follows the MI250 correctness blog (section 4.1 table: fp32
// comparison and a fixed tie-break; section 4.2: ties go to the lower
// expert id, never to memory order).  The sort is the "expert sorting" step
// of the DeepSeek-V4-Flash-on-gfx90a paper's prefill path: a stable
// counting sort, so the permutation is unique and reproducible.
//
// Three kernels for any T:
//   route_hist  one warp per token: k rounds of a warp-wide argmax over the
//               token's E logits (two warp reductions per round: the largest
//               key, then the lowest index holding it), softmax of the k
//               picked, per-block counts
//   sort_scan   one block: per-expert totals (several threads per expert,
//               each summing a contiguous range of routing blocks), offsets,
//               per-block bases, the list of non-empty experts and the work
//               lists of the expert kernels (so the host never reads a count)
//   scatter     one block per routing block: stable ranks by warp match,
//               writes sorted_slot and its inverse
// and one for T <= 32 (the decode batch): route_small, a cluster of CTAs on
// separate SMs, one token per warp, with the sort done in CTA 0.
#include <cooperative_groups.h>

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

// Larger key first.
__device__ __forceinline__ void cmpx_desc(unsigned long long& a, unsigned long long& b) {
  const unsigned long long hi = a > b ? a : b, lo = a > b ? b : a;
  a = hi;
  b = lo;
}

// Top-k of one token's E logits (`row`, shared or global memory) by (value
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
    // index first; an absent entry is 0), sorted once in descending order:
    // a round compares the lanes' first keys only and the winning lane
    // drops its first key
    unsigned long long kk[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      kk[i] = e < E ? ((unsigned long long)ordered_key(row[e]) << 32) | (0xFFFFFFFFu - (uint32_t)e) : 0ull;
    }
    // Batcher's odd-even merge sort of 8 keys (19 compare-exchanges)
    cmpx_desc(kk[0], kk[2]); cmpx_desc(kk[1], kk[3]); cmpx_desc(kk[4], kk[6]); cmpx_desc(kk[5], kk[7]);
    cmpx_desc(kk[0], kk[4]); cmpx_desc(kk[1], kk[5]); cmpx_desc(kk[2], kk[6]); cmpx_desc(kk[3], kk[7]);
    cmpx_desc(kk[0], kk[1]); cmpx_desc(kk[2], kk[3]); cmpx_desc(kk[4], kk[5]); cmpx_desc(kk[6], kk[7]);
    cmpx_desc(kk[2], kk[4]); cmpx_desc(kk[3], kk[5]);
    cmpx_desc(kk[1], kk[4]); cmpx_desc(kk[3], kk[6]);
    cmpx_desc(kk[1], kk[2]); cmpx_desc(kk[3], kk[4]); cmpx_desc(kk[5], kk[6]);
    for (int r = 0; r < k; ++r) {
      const uint32_t hi = (uint32_t)(kk[0] >> 32);
      const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, hi);
      const uint32_t l = __reduce_max_sync(0xFFFFFFFFu, hi == m ? (uint32_t)kk[0] : 0u);
      const int e_star = (int)(0xFFFFFFFFu - l);
      const bool won = (e_star & 31) == lane;
#pragma unroll
      for (int i = 0; i < 7; ++i) kk[i] = won ? kk[i + 1] : kk[i];
      kk[7] = won ? 0ull : kk[7];
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
template <typename V>
__device__ V block_exclusive_scan(V v, V* scratch /* [33] */, V* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  V incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const V n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += n;
  }
  __syncthreads();
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    const V w = lane < nw ? scratch[lane] : V(0);
    V wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const V n = __shfl_up_sync(0xFFFFFFFFu, wi, o);
      if (lane >= o) wi += n;
    }
    scratch[lane] = wi - w;  // exclusive prefix of warp totals
    if (lane == 31) scratch[32] = wi;
  }
  __syncthreads();
  const V res = scratch[warp] + incl - v;
  *total = scratch[32];
  __syncthreads();
  return res;
}

// Two 32-bit counters in one 64-bit word (each total stays below 2^31, so
// sums never carry from the low field into the high one).
__device__ __forceinline__ unsigned long long pack2(int lo, int hi) {
  return (unsigned long long)(uint32_t)lo | ((unsigned long long)(uint32_t)hi << 32);
}

// Threads e*G .. e*G+G-1 serve expert e (G a power of two <= 32, G*E <= 1024),
// part p of G summing routing blocks [p*ceil(nb/G), ...) of that expert.
__global__ void __launch_bounds__(1024, 1)
sort_scan_kernel(int32_t* __restrict__ block_hist, int nb, int E, int G, int32_t* __restrict__ offsets,
                 int32_t* __restrict__ active, int32_t* __restrict__ counts,
                 int4* __restrict__ gemv_chunks, int4* __restrict__ tc_tiles, int tile_multi) {
  __shared__ unsigned long long scratch[33];
  const int e = threadIdx.x / G, p = threadIdx.x & (G - 1);
  const bool ok = e < E;
  const int per = (nb + G - 1) / G;
  const int b0 = min(nb, p * per), b1 = min(nb, b0 + per);
  int part = 0;
  if (ok) {
#pragma unroll 8
    for (int b = b0; b < b1; ++b) part += block_hist[(size_t)b * E + e];
  }
  // prefix over the expert's G parts (consecutive lanes of one warp)
  int pin = part;
  for (int o = 1; o < G; o <<= 1) {
    const int n = __shfl_up_sync(0xFFFFFFFFu, pin, o, G);
    if (p >= o) pin += n;
  }
  const int cnt = __shfl_sync(0xFFFFFFFFu, pin, G - 1, G);
  const bool lead = ok && p == 0;
  // offsets and the non-empty-expert positions in one scan, the GEMV chunk
  // and tensor-core tile positions in another
  const int nch = ok ? (cnt + kGemvTokens - 1) / kGemvTokens : 0;
  const int ntl = ok ? tc_tile_count(cnt, tile_multi) : 0;
  unsigned long long tot1, tot2;
  const unsigned long long x1 =
      block_exclusive_scan(lead ? pack2(cnt, cnt > 0 ? 1 : 0) : 0ull, scratch, &tot1);
  const unsigned long long x2 = block_exclusive_scan(lead ? pack2(nch, ntl) : 0ull, scratch, &tot2);
  const unsigned long long y1 = __shfl_sync(0xFFFFFFFFu, x1, 0, G);
  const unsigned long long y2 = __shfl_sync(0xFFFFFFFFu, x2, 0, G);
  const int off = (int)(uint32_t)y1, apos = (int)(y1 >> 32);
  const int cpos = (int)(uint32_t)y2, tpos = (int)(y2 >> 32);
  if (ok) {
    if (p == 0) {
      offsets[e] = off;
      if (cnt > 0) active[apos] = e;
    }
    int run = off + pin - part;  // rows of this expert in the routing blocks before b0
#pragma unroll 8
    for (int b = b0; b < b1; ++b) {
      const int c = block_hist[(size_t)b * E + e];
      block_hist[(size_t)b * E + e] = run;
      run += c;
    }
    // GEMV chunks of up to kGemvTokens rows
    for (int c = p; c < nch; c += G)
      gemv_chunks[cpos + c] = make_int4(e, off + c * kGemvTokens, min(kGemvTokens, cnt - c * kGemvTokens), 0);
    // tensor-core tiles: tc_tile_count tiles of equal size (rounded up to 16)
    const int per_tile = ntl ? (((cnt + ntl - 1) / ntl + 15) & ~15) : 0;
    for (int c = p; c < ntl; c += G)
      tc_tiles[tpos + c] = make_int4(e, off + c * per_tile, min(per_tile, cnt - c * per_tile), 0);
  }
  if (threadIdx.x == 0) {
    offsets[E] = (int)(uint32_t)tot1;
    counts[0] = (int)(tot1 >> 32);
    counts[1] = (int)(uint32_t)tot2;
    counts[2] = (int)(tot2 >> 32);
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


// Routing and sort when all tokens fit one routing block (T <= 32, the decode
// batch): a cluster of kSmallCtas CTAs on separate SMs, one token per warp
// (32 warps of top-k on one SM are issue-bound), each warp also storing its
// token's k expert ids into CTA 0's shared memory.  After the cluster barrier
// CTA 0 alone builds, per expert, the mask of tokens that picked it, then the
// offsets and work lists (one scan of packed counters) and the stable
// scatter: a token picks an expert at most once, so the rank of slot (t, j)
// among its expert's slots in ascending flat index is the number of tokens
// before t in the expert's mask.
constexpr int kSmallCtas = 8;
constexpr int kSmallWarps = kRouteTokensPerBlock / kSmallCtas;  // tokens per CTA
constexpr int kSmallThreads = kSmallWarps * 32;
constexpr int kMaxExperts = 1024;
static_assert(kSmallCtas * kSmallWarps == 32, "a token mask is one 32-bit word");

// Per-expert counters packed in 16-bit fields: rows, non-empty, GEMV chunks,
// tensor-core tiles.  Each total is at most T*k <= 1024 (or E <= 1024), so
// fields never carry into one another.
__device__ __forceinline__ unsigned long long pack4(int cnt, int tile_multi) {
  const unsigned long long nch = (cnt + kGemvTokens - 1) / kGemvTokens;
  const unsigned long long ntl = tc_tile_count(cnt, tile_multi);
  return (unsigned long long)cnt | ((unsigned long long)(cnt > 0) << 16) | (nch << 32) | (ntl << 48);
}

__global__ void __cluster_dims__(kSmallCtas, 1, 1) __launch_bounds__(kSmallThreads)
route_small_kernel(const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ topk_ids,
                   float* __restrict__ topk_w, int32_t* __restrict__ offsets, int32_t* __restrict__ active,
                   int32_t* __restrict__ counts, int4* __restrict__ gemv_chunks, int4* __restrict__ tc_tiles,
                   int32_t* __restrict__ sorted_slot, int32_t* __restrict__ slot_pos, int32_t* __restrict__ err,
                   int tile_multi) {
  __shared__ int ids_s[kRouteTokensPerBlock * 32];  // [T*k] expert of each slot (CTA 0's copy)
  __shared__ uint32_t mask_s[kMaxExperts];          // bit t: token t picked the expert
  __shared__ int off_s[kMaxExperts];
  __shared__ unsigned long long wsum[kSmallWarps];
  griddep_launch_dependents();  // the W13 kernel may start its prologue (it waits for this kernel)
  cooperative_groups::cluster_group cluster = cooperative_groups::this_cluster();
  const int cta = (int)cluster.block_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (cta == 0) {
    if (threadIdx.x < 4) err[threadIdx.x] = 0;
    for (int e = threadIdx.x; e < E; e += kSmallThreads) mask_s[e] = 0;
  }
  const int t = cta * kSmallWarps + warp;
  if (t < T) {
    int id;
    float w;
    topk_softmax_warp(logits + (size_t)t * E, E, k, lane, id, w);
    if (lane < k) {
      topk_ids[t * k + lane] = id;
      topk_w[t * k + lane] = w;
      cluster.map_shared_rank(ids_s, 0)[t * k + lane] = id;
    }
  }
  cluster.sync();
  if (cta != 0) return;
  const int S = T * k;
  for (int f = threadIdx.x; f < S; f += kSmallThreads) atomicOr(&mask_s[ids_s[f]], 1u << (f / k));
  __syncthreads();
  // this thread's experts [e0, e1), in order
  const int ept = (E + kSmallThreads - 1) / kSmallThreads;
  const int e0 = min(E, (int)threadIdx.x * ept), e1 = min(E, e0 + ept);
  unsigned long long mine = 0;
  for (int e = e0; e < e1; ++e) mine += pack4(__popc(mask_s[e]), tile_multi);
  unsigned long long incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  unsigned long long base = incl - mine, total = 0;
#pragma unroll
  for (int w = 0; w < kSmallWarps; ++w) {
    if (w < warp) base += wsum[w];
    total += wsum[w];
  }
  for (int e = e0; e < e1; ++e) {
    const int cnt = __popc(mask_s[e]);
    const int off = (int)(base & 0xFFFF), apos = (int)((base >> 16) & 0xFFFF);
    const int cpos = (int)((base >> 32) & 0xFFFF), tpos = (int)(base >> 48);
    offsets[e] = off;
    off_s[e] = off;
    if (cnt > 0) active[apos] = e;
    const int nch = (cnt + kGemvTokens - 1) / kGemvTokens;
    for (int c = 0; c < nch; ++c)
      gemv_chunks[cpos + c] = make_int4(e, off + c * kGemvTokens, min(kGemvTokens, cnt - c * kGemvTokens), 0);
    // tensor-core tiles: tc_tile_count tiles of equal size (rounded up to 16)
    const int ntl = tc_tile_count(cnt, tile_multi);
    const int per = ntl ? (((cnt + ntl - 1) / ntl + 15) & ~15) : 0;
    for (int c = 0; c < ntl; ++c) tc_tiles[tpos + c] = make_int4(e, off + c * per, min(per, cnt - c * per), 0);
    base += pack4(cnt, tile_multi);
  }
  if (threadIdx.x == 0) {
    offsets[E] = (int)(total & 0xFFFF);
    counts[0] = (int)((total >> 16) & 0xFFFF);
    counts[1] = (int)((total >> 32) & 0xFFFF);
    counts[2] = (int)(total >> 48);
    counts[3] = 0;
  }
  __syncthreads();
  for (int f = threadIdx.x; f < S; f += kSmallThreads) {
    const int e = ids_s[f];
    const int pos = off_s[e] + __popc(mask_s[e] & ((1u << (f / k)) - 1u));
    sorted_slot[pos] = f;
    slot_pos[f] = pos;
  }
}

}  // namespace

cudaError_t launch_route(const moe_fp4_dims& d, const float* logits, const Workspace& ws, cudaStream_t st,
                         int tile_multi) {
  const int nb = ws.nb_route;
  if (tile_multi < 16 || tile_multi > kTcTileN) return cudaErrorInvalidValue;
  if (nb == 1) {
    route_small_kernel<<<kSmallCtas, kSmallThreads, 0, st>>>(logits, d.T, d.E, d.k, ws.topk_ids, ws.topk_w,
                                                           ws.offsets, ws.active, ws.counts, ws.gemv_chunks,
                                                           ws.tc_tiles, ws.sorted_slot, ws.slot_pos, ws.err,
                                                           tile_multi);
    return cudaGetLastError();
  }
  size_t smem1 = (size_t)(kWarps * d.E) * sizeof(float) + (size_t)d.E * sizeof(int);
  route_hist_kernel<<<nb, kRouteThreads, smem1, st>>>(logits, d.T, d.E, d.k, ws.topk_ids, ws.topk_w,
                                                     ws.block_hist, ws.err);
  int G = 1;  // threads per expert in sort_scan
  while (G < 32 && 2 * G * d.E <= 1024) G *= 2;
  sort_scan_kernel<<<1, 1024, 0, st>>>(ws.block_hist, nb, d.E, G, ws.offsets, ws.active, ws.counts,
                                       ws.gemv_chunks, ws.tc_tiles, tile_multi);
  size_t smem3 = (size_t)(kWarps + 1) * d.E * sizeof(int);
  scatter_kernel<<<nb, kRouteThreads, smem3, st>>>(ws.topk_ids, ws.block_hist, d.T, d.E, d.k,
                                                   ws.sorted_slot, ws.slot_pos, ws.err);
  return cudaGetLastError();
}

}  // namespace moe_fp4
