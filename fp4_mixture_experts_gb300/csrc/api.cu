// C-ABI entry points of the FP4 routed-MoE layer: argument checks, the
// workspace layout and the launch sequence.  All compute happens in the
// kernels of the other translation units.
#include <string.h>

#include <functional>

#include "moe_fp4_internal.cuh"

namespace moe_fp4 {

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

bool dims_supported(const moe_fp4_dims& d) {
  if (d.T < 1 || d.E < 1 || d.E > 1024 || d.k < 1 || d.k > 32 || d.k > d.E) return false;
  if (d.d < 128 || d.d > 16384 || d.d % 128 != 0) return false;
  if (d.I < 128 || d.I > 16384 || d.I % 128 != 0) return false;
  const long long S = (long long)d.T * d.k;
  if (S >= (1LL << 31)) return false;
  const long long widest = d.d > d.I ? d.d : d.I;
  if (S * widest >= (1LL << 40)) return false;
  return true;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

// The address of host memory p on the current device, if the device can
// address it (page-locked memory from the CUDA allocator or registered with
// it), else null.
void* device_view(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // unregistered memory may report an error on older drivers: not sticky
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

}  // namespace

bool layout_workspace(const moe_fp4_dims& d, void* base, bool with_staging, Workspace* ws, bool mx) {
  if (!dims_supported(d)) return false;
  memset(ws, 0, sizeof(*ws));
  const size_t S = (size_t)d.T * d.k;
  ws->nb_route = (d.T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock;
  ws->max_gemv_chunks = d.E + (int)((S + kGemvTokens - 1) / kGemvTokens);
  // at most one partial tile per expert beyond S / (smallest tile cap)
  ws->max_tc_tiles = d.E + (int)((S + kTcTileMultiN - 1) / kTcTileMultiN);
  char* p = static_cast<char*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) -> void* {
    void* r = base ? p + off : nullptr;
    off += align_up(bytes);
    return r;
  };
  ws->err = (int32_t*)take(4 * sizeof(int32_t));
  ws->counts = (int32_t*)take(4 * sizeof(int32_t));
  ws->active = (int32_t*)take((size_t)d.E * sizeof(int32_t));
  ws->block_hist = (int32_t*)take((size_t)ws->nb_route * d.E * sizeof(int32_t));
  ws->topk_ids = (int32_t*)take(S * sizeof(int32_t));
  ws->topk_w = (float*)take(S * sizeof(float));
  ws->offsets = (int32_t*)take((size_t)(d.E + 1) * sizeof(int32_t));
  ws->sorted_slot = (int32_t*)take(S * sizeof(int32_t));
  ws->slot_pos = (int32_t*)take(S * sizeof(int32_t));
  ws->gemv_chunks = (int4*)take((size_t)ws->max_gemv_chunks * sizeof(int4));
  ws->tc_tiles = (int4*)take((size_t)ws->max_tc_tiles * sizeof(int4));
  ws->x_perm = (uint16_t*)take(S * (size_t)(d.d > d.I ? d.d : d.I) * sizeof(uint16_t));
  ws->x_scale = (float*)take(S * sizeof(float));
  ws->h16 = ws->x_perm;
  ws->h_scale = ws->x_scale;
  ws->h = (uint16_t*)take(S * d.I * sizeof(uint16_t));
  ws->y = (float*)take(S * d.d * sizeof(float));
  ws->combine_cnt = (int32_t*)take((size_t)d.T * ((d.d + 255) / 256) * sizeof(int32_t));
  if (mx) {
    // S*(d + I) code bytes fit the x_perm region (2 S max(d, I) bytes); the
    // offset S*d keeps hq 128-byte aligned (d is a multiple of 128)
    ws->xq = reinterpret_cast<uint8_t*>(ws->x_perm);
    ws->hq = base ? ws->xq + S * d.d : nullptr;
    ws->xq_scales = (uint8_t*)take(S * (d.d / 32));
    ws->hq_scales = (uint8_t*)take(S * (d.I / 32));
  }
  if (with_staging) {
    ws->stage_x = (uint16_t*)take((size_t)d.T * d.d * sizeof(uint16_t));
    ws->stage_logits = (float*)take((size_t)d.T * d.E * sizeof(float));
    ws->stage_out = (float*)take((size_t)d.T * d.d * sizeof(float));
  }
  ws->total = off;
  return true;
}

namespace {

bool use_gemv_path(const moe_fp4_dims& d, unsigned flags) {
  if (flags & MOE_FP4_FLAG_FORCE_GEMV) return true;
  if (flags & MOE_FP4_FLAG_FORCE_TC) return false;
  if (d.d % 1024 != 0 || d.I % 1024 != 0) return false;
  // expected rows per expert T*k/E; the streaming path wins while it is small
  return (long long)d.T * d.k <= 4LL * d.E;
}

int run_forward(const moe_fp4_dims& d, const void* x, const float* logits, const uint8_t* w13,
                const uint8_t* w13s, const uint8_t* w2, const uint8_t* w2s, float* out,
                int32_t* topk_ids, float* topk_w, int32_t* offsets, int32_t* sorted_slot, void* h,
                unsigned flags, Workspace ws, cudaStream_t st, void* const* events = nullptr) {
  auto mark = [&](int i) {
    if (events) cudaEventRecord(static_cast<cudaEvent_t>(events[i]), st);
  };
  if (topk_ids) ws.topk_ids = topk_ids;
  if (topk_w) ws.topk_w = topk_w;
  if (offsets) ws.offsets = offsets;
  if (sorted_slot) ws.sorted_slot = sorted_slot;
  if (h) ws.h = static_cast<uint16_t*>(h);
  const uint16_t* xb = static_cast<const uint16_t*>(x);
  const bool det = (flags & MOE_FP4_FLAG_DETERMINISTIC) != 0;
  const size_t out_bytes = (size_t)d.T * d.d * sizeof(float);
  const bool gemv = use_gemv_path(d, flags);
  // the combine in the W2 epilogue (atomic adds into out): the streaming
  // kernels and the one-SM tensor-core kernel, unless reproducibility is asked
  const bool stream_combine = !det && gemv && stream_path_supported(d);
  mark(0);
  // on the streaming path the W13 kernel zeroes out while it waits for the routing
  cudaError_t e = launch_route(d, logits, ws, st);
  if (e != cudaSuccess) return MOE_FP4_ERR_CUDA;
  mark(1);
  bool fused_combine = false;
  if (gemv) {
    mark(2);
    if (stream_path_supported(d) && (flags & MOE_FP4_FLAG_PERSISTENT)) {
      // both projections: the W2 stage reads 0
      e = launch_stream_fused(d, xb, w13, w13s, w2, w2s, ws, stream_combine ? out : nullptr, st);
      mark(3);
    } else if (stream_path_supported(d)) {
      e = launch_stream_w13(d, xb, w13, w13s, ws, stream_combine ? out : nullptr, st);
      mark(3);
      if (e == cudaSuccess) e = launch_stream_w2(d, w2, w2s, ws, stream_combine ? out : nullptr, st);
    } else {
      e = launch_gemv_w13(d, xb, w13, w13s, ws, st);
      mark(3);
      if (e == cudaSuccess) e = launch_gemv_w2(d, w2, w2s, ws, st);
    }
  } else {
    e = launch_gather(d, xb, ws, st);
    mark(2);
    const bool pairs = (flags & MOE_FP4_FLAG_CTA_PAIRS) != 0;
    if (e == cudaSuccess) e = launch_tc_w13(d, w13, w13s, ws, pairs, st);
    mark(3);
    const bool tc_combine = !det && !pairs;
    if (e == cudaSuccess) e = launch_h_f16(d, ws, st);  // counted in the W2 stage
    if (e == cudaSuccess && tc_combine) e = cudaMemsetAsync(out, 0, out_bytes, st);
    if (e == cudaSuccess) e = launch_tc_w2(d, w2, w2s, ws, out, pairs, tc_combine, st);
    fused_combine = tc_combine || tc_fused_combine(pairs);
  }
  mark(4);
  if (e == cudaSuccess && !fused_combine && !stream_combine) e = launch_combine(d, out, ws, st);
  mark(5);
  return e == cudaSuccess ? MOE_FP4_OK : MOE_FP4_ERR_CUDA;
}

int check_flags(unsigned flags) {
  const unsigned known = MOE_FP4_FLAG_FORCE_GEMV | MOE_FP4_FLAG_FORCE_TC | MOE_FP4_FLAG_PERSISTENT |
                         MOE_FP4_FLAG_CTA_PAIRS | MOE_FP4_FLAG_DETERMINISTIC;
  if (flags & ~known) return MOE_FP4_ERR_INVALID_ARG;
  if ((flags & MOE_FP4_FLAG_FORCE_GEMV) && (flags & MOE_FP4_FLAG_FORCE_TC)) return MOE_FP4_ERR_INVALID_ARG;
  return MOE_FP4_OK;
}

}  // namespace
}  // namespace moe_fp4

using namespace moe_fp4;

extern "C" {

size_t moe_fp4_workspace_bytes(const moe_fp4_dims* dims) {
  if (!dims) return 0;
  Workspace ws;
  return layout_workspace(*dims, nullptr, false, &ws) ? ws.total : 0;
}

size_t moe_fp4_host_workspace_bytes(const moe_fp4_dims* dims) {
  if (!dims) return 0;
  Workspace ws;
  return layout_workspace(*dims, nullptr, true, &ws) ? ws.total : 0;
}

int moe_fp4_route(const moe_fp4_dims* dims, const float* router_logits, int32_t* topk_ids,
                  float* topk_weights, int32_t* expert_offsets, int32_t* sorted_slot,
                  void* workspace, size_t workspace_bytes, void* cuda_stream) {
  if (!dims || !router_logits || !topk_ids || !topk_weights || !expert_offsets || !sorted_slot || !workspace)
    return MOE_FP4_ERR_INVALID_ARG;
  const moe_fp4_dims d = *dims;
  Workspace ws;
  if (!layout_workspace(d, workspace, false, &ws)) return MOE_FP4_ERR_UNSUPPORTED;
  if (!aligned(workspace, 256) || !aligned(router_logits, 4) || !aligned(topk_ids, 4) ||
      !aligned(topk_weights, 4) || !aligned(expert_offsets, 4) || !aligned(sorted_slot, 4))
    return MOE_FP4_ERR_INVALID_ARG;
  if (workspace_bytes < ws.total) return MOE_FP4_ERR_WORKSPACE;
  ws.topk_ids = topk_ids;
  ws.topk_w = topk_weights;
  ws.offsets = expert_offsets;
  ws.sorted_slot = sorted_slot;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  return launch_route(d, router_logits, ws, st) == cudaSuccess ? MOE_FP4_OK : MOE_FP4_ERR_CUDA;
}

int moe_fp4_forward_profiled(const moe_fp4_dims* dims, const void* x_bf16, const float* router_logits,
                             const uint8_t* w13, const uint8_t* w13_scale, const uint8_t* w2,
                             const uint8_t* w2_scale, float* out, int32_t* topk_ids, float* topk_weights,
                             int32_t* expert_offsets, int32_t* sorted_slot, void* h_bf16, unsigned flags,
                             void* workspace, size_t workspace_bytes, void* cuda_stream,
                             void* const* stage_events) {
  if (!dims || !x_bf16 || !router_logits || !w13 || !w13_scale || !w2 || !w2_scale || !out || !workspace)
    return MOE_FP4_ERR_INVALID_ARG;
  if (check_flags(flags) != MOE_FP4_OK) return MOE_FP4_ERR_INVALID_ARG;
  const moe_fp4_dims d = *dims;
  Workspace ws;
  if (!layout_workspace(d, workspace, false, &ws)) return MOE_FP4_ERR_UNSUPPORTED;
  if (!aligned(workspace, 256) || !aligned(x_bf16, 16) || !aligned(w13, 16) || !aligned(w2, 16) ||
      !aligned(out, 16) || !aligned(router_logits, 4) || !aligned(w13_scale, 16) || !aligned(w2_scale, 16) ||
      (h_bf16 && !aligned(h_bf16, 16)) || (topk_ids && !aligned(topk_ids, 4)) ||
      (topk_weights && !aligned(topk_weights, 4)) || (expert_offsets && !aligned(expert_offsets, 4)) ||
      (sorted_slot && !aligned(sorted_slot, 4)))
    return MOE_FP4_ERR_INVALID_ARG;
  if ((flags & MOE_FP4_FLAG_FORCE_GEMV) && (d.d % 1024 != 0 || d.I % 1024 != 0)) return MOE_FP4_ERR_UNSUPPORTED;
  if (workspace_bytes < ws.total) return MOE_FP4_ERR_WORKSPACE;
  return run_forward(d, x_bf16, router_logits, w13, w13_scale, w2, w2_scale, out, topk_ids, topk_weights,
                     expert_offsets, sorted_slot, h_bf16, flags, ws, static_cast<cudaStream_t>(cuda_stream),
                     stage_events);
}

int moe_fp4_router(const moe_fp4_dims* dims, const void* x_bf16, const void* w_gate_bf16, float* router_logits,
                   void* cuda_stream) {
  if (!dims || !x_bf16 || !w_gate_bf16 || !router_logits) return MOE_FP4_ERR_INVALID_ARG;
  const moe_fp4_dims d = *dims;
  Workspace ws;
  if (!layout_workspace(d, nullptr, false, &ws)) return MOE_FP4_ERR_UNSUPPORTED;
  if (!aligned(x_bf16, 16) || !aligned(w_gate_bf16, 16) || !aligned(router_logits, 4)) return MOE_FP4_ERR_INVALID_ARG;
  return launch_router(d, static_cast<const uint16_t*>(x_bf16), static_cast<const uint16_t*>(w_gate_bf16),
                       router_logits, static_cast<cudaStream_t>(cuda_stream)) == cudaSuccess
             ? MOE_FP4_OK
             : MOE_FP4_ERR_CUDA;
}

int moe_fp4_forward_gated(const moe_fp4_dims* dims, const void* x_bf16, const void* w_gate_bf16,
                          float* router_logits, const uint8_t* w13, const uint8_t* w13_scale, const uint8_t* w2,
                          const uint8_t* w2_scale, float* out, int32_t* topk_ids, float* topk_weights,
                          int32_t* expert_offsets, int32_t* sorted_slot, void* h_bf16, unsigned flags,
                          void* workspace, size_t workspace_bytes, void* cuda_stream) {
  if (!dims || !w_gate_bf16 || !router_logits) return MOE_FP4_ERR_INVALID_ARG;
  // the layer's own checks first (x, weights, out, workspace, flags), so that
  // nothing is enqueued when any argument is bad
  if (!x_bf16 || !w13 || !w13_scale || !w2 || !w2_scale || !out || !workspace) return MOE_FP4_ERR_INVALID_ARG;
  if (check_flags(flags) != MOE_FP4_OK) return MOE_FP4_ERR_INVALID_ARG;
  const moe_fp4_dims d = *dims;
  Workspace ws;
  if (!layout_workspace(d, workspace, false, &ws)) return MOE_FP4_ERR_UNSUPPORTED;
  if (!aligned(w_gate_bf16, 16) || !aligned(router_logits, 4) || !aligned(workspace, 256) || !aligned(x_bf16, 16) ||
      !aligned(w13, 16) || !aligned(w2, 16) || !aligned(out, 16) || !aligned(w13_scale, 16) ||
      !aligned(w2_scale, 16) || (h_bf16 && !aligned(h_bf16, 16)) || (topk_ids && !aligned(topk_ids, 4)) ||
      (topk_weights && !aligned(topk_weights, 4)) || (expert_offsets && !aligned(expert_offsets, 4)) ||
      (sorted_slot && !aligned(sorted_slot, 4)))
    return MOE_FP4_ERR_INVALID_ARG;
  if ((flags & MOE_FP4_FLAG_FORCE_GEMV) && (d.d % 1024 != 0 || d.I % 1024 != 0)) return MOE_FP4_ERR_UNSUPPORTED;
  if (workspace_bytes < ws.total) return MOE_FP4_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  if (launch_router(d, static_cast<const uint16_t*>(x_bf16), static_cast<const uint16_t*>(w_gate_bf16),
                    router_logits, st) != cudaSuccess)
    return MOE_FP4_ERR_CUDA;
  return run_forward(d, x_bf16, router_logits, w13, w13_scale, w2, w2_scale, out, topk_ids, topk_weights,
                     expert_offsets, sorted_slot, h_bf16, flags, ws, st);
}

int moe_fp4_forward(const moe_fp4_dims* dims, const void* x_bf16, const float* router_logits,
                    const uint8_t* w13, const uint8_t* w13_scale, const uint8_t* w2,
                    const uint8_t* w2_scale, float* out, int32_t* topk_ids, float* topk_weights,
                    int32_t* expert_offsets, int32_t* sorted_slot, void* h_bf16, unsigned flags,
                    void* workspace, size_t workspace_bytes, void* cuda_stream) {
  return moe_fp4_forward_profiled(dims, x_bf16, router_logits, w13, w13_scale, w2, w2_scale, out, topk_ids,
                                  topk_weights, expert_offsets, sorted_slot, h_bf16, flags, workspace,
                                  workspace_bytes, cuda_stream, nullptr);
}

int moe_fp4_forward_host(const moe_fp4_dims* dims, const void* x_bf16_host, const float* router_logits_host,
                         const uint8_t* w13, const uint8_t* w13_scale, const uint8_t* w2,
                         const uint8_t* w2_scale, float* out_host, unsigned flags, void* workspace,
                         size_t workspace_bytes, void* cuda_stream) {
  if (!dims || !x_bf16_host || !router_logits_host || !w13 || !w13_scale || !w2 || !w2_scale || !out_host ||
      !workspace)
    return MOE_FP4_ERR_INVALID_ARG;
  if (check_flags(flags) != MOE_FP4_OK) return MOE_FP4_ERR_INVALID_ARG;
  const moe_fp4_dims d = *dims;
  Workspace ws;
  if (!layout_workspace(d, workspace, true, &ws)) return MOE_FP4_ERR_UNSUPPORTED;
  if (!aligned(workspace, 256) || !aligned(w13, 16) || !aligned(w2, 16) || !aligned(w13_scale, 16) ||
      !aligned(w2_scale, 16))
    return MOE_FP4_ERR_INVALID_ARG;
  if ((flags & MOE_FP4_FLAG_FORCE_GEMV) && (d.d % 1024 != 0 || d.I % 1024 != 0)) return MOE_FP4_ERR_UNSUPPORTED;
  if (workspace_bytes < ws.total) return MOE_FP4_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  // Host buffers the device can address (pinned or registered memory) are
  // used in place: the routing kernel reads the logits, the combine writes
  // out, with no copy and no copy-engine round trip.  x, which many CTAs read
  // again, is copied to device staging; so is anything else.
  const float* logits_dev = static_cast<const float*>(device_view(router_logits_host));
  float* out_dev = static_cast<float*>(device_view(out_host));
  if (logits_dev && !aligned(logits_dev, 4)) logits_dev = nullptr;
  if (out_dev && !aligned(out_dev, 16)) out_dev = nullptr;
  // out in host memory is written by the combine pass with plain stores (no
  // atomic adds across the host link)
  if (out_dev) flags |= MOE_FP4_FLAG_DETERMINISTIC;
  const size_t xb = (size_t)d.T * d.d * sizeof(uint16_t), lb = (size_t)d.T * d.E * sizeof(float),
               ob = (size_t)d.T * d.d * sizeof(float);
  if (cudaMemcpyAsync(ws.stage_x, x_bf16_host, xb, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return MOE_FP4_ERR_CUDA;
  if (!logits_dev &&
      cudaMemcpyAsync(ws.stage_logits, router_logits_host, lb, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return MOE_FP4_ERR_CUDA;
  int rc = run_forward(d, ws.stage_x, logits_dev ? logits_dev : ws.stage_logits, w13, w13_scale, w2, w2_scale,
                       out_dev ? out_dev : ws.stage_out, nullptr, nullptr, nullptr, nullptr, nullptr, flags, ws, st);
  if (rc != MOE_FP4_OK) return rc;
  if (!out_dev && cudaMemcpyAsync(out_host, ws.stage_out, ob, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MOE_FP4_ERR_CUDA;
  return cudaStreamSynchronize(st) == cudaSuccess ? MOE_FP4_OK : MOE_FP4_ERR_CUDA;
}

size_t moe_fp4_mx_workspace_bytes(const moe_fp4_dims* dims) {
  if (!dims) return 0;
  Workspace ws;
  return layout_workspace(*dims, nullptr, false, &ws, true) ? ws.total : 0;
}

int moe_fp4_forward_mx(const moe_fp4_dims* dims, const void* x_bf16, const float* router_logits,
                       const uint8_t* w13, const uint8_t* w13_scale, const uint8_t* w2, const uint8_t* w2_scale,
                       float* out, void* h_bf16, uint8_t* h_codes, uint8_t* h_scales, uint8_t* x_codes,
                       uint8_t* x_scales, void* workspace, size_t workspace_bytes, void* cuda_stream,
                       void* const* stage_events) {
  if (!dims || !x_bf16 || !router_logits || !w13 || !w13_scale || !w2 || !w2_scale || !out || !workspace)
    return MOE_FP4_ERR_INVALID_ARG;
  const moe_fp4_dims d = *dims;
  Workspace ws;
  if (!layout_workspace(d, workspace, false, &ws, true)) return MOE_FP4_ERR_UNSUPPORTED;
  // the weights are read by the tensor memory accelerator as 4-bit elements:
  // 32-byte aligned bases
  if (!aligned(workspace, 256) || !aligned(x_bf16, 16) || !aligned(w13, 32) || !aligned(w2, 32) ||
      !aligned(out, 16) || !aligned(router_logits, 4) || !aligned(w13_scale, 16) || !aligned(w2_scale, 16) ||
      (h_bf16 && !aligned(h_bf16, 16)) || (h_codes && !aligned(h_codes, 16)) || (x_codes && !aligned(x_codes, 16)))
    return MOE_FP4_ERR_INVALID_ARG;
  if (workspace_bytes < ws.total) return MOE_FP4_ERR_WORKSPACE;
  if (h_bf16) ws.h = static_cast<uint16_t*>(h_bf16);
  if (h_codes) ws.hq = h_codes;
  if (h_scales) ws.hq_scales = h_scales;
  if (x_codes) ws.xq = x_codes;
  if (x_scales) ws.xq_scales = x_scales;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  auto mark = [&](int i) {
    if (stage_events) cudaEventRecord(static_cast<cudaEvent_t>(stage_events[i]), st);
  };
  mark(0);
  cudaError_t e = launch_route(d, router_logits, ws, st, kTcTileN);
  mark(1);
  if (e == cudaSuccess)
    e = launch_mx_forward(d, static_cast<const uint16_t*>(x_bf16), w13, w13_scale, w2, w2_scale, ws, st,
                          stage_events ? mark : std::function<void(int)>());
  mark(4);
  if (e == cudaSuccess) e = launch_combine(d, out, ws, st);
  mark(5);
  return e == cudaSuccess ? MOE_FP4_OK : MOE_FP4_ERR_CUDA;
}

int moe_fp4_check(void* workspace, void* cuda_stream) {
  if (!workspace) return MOE_FP4_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  int32_t err[4] = {0, 0, 0, 0};
  // the error words are the first region of every workspace layout
  if (cudaMemcpyAsync(err, workspace, sizeof(err), cudaMemcpyDeviceToHost, st) != cudaSuccess) return MOE_FP4_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_FP4_ERR_CUDA;
  if (err[0] != 0) {
    if (cudaMemsetAsync(workspace, 0, sizeof(err), st) != cudaSuccess) return MOE_FP4_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_FP4_ERR_CUDA;
    return MOE_FP4_ERR_DEVICE;
  }
  return MOE_FP4_OK;
}

const char* moe_fp4_status_string(int status) {
  switch (status) {
    case MOE_FP4_OK: return "ok";
    case MOE_FP4_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, bad size or flags)";
    case MOE_FP4_ERR_UNSUPPORTED: return "unsupported sizes";
    case MOE_FP4_ERR_WORKSPACE: return "workspace too small";
    case MOE_FP4_ERR_CUDA: return "CUDA runtime error";
    case MOE_FP4_ERR_DEVICE: return "a kernel reported an error (an out-of-range index or a timed-out wait)";
    default: return "unknown status";
  }
}

}  // extern "C"
