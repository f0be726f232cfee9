// moe_fp4_forward_noalloc: the layer for callers that cannot allocate device
// memory (an allocator-less runtime, a caller that may not call cudaMalloc
// inside its own stream-ordered or captured region, a plugin handed only
// input and output pointers).  Its scratch is a file-scope device array of
// fixed size that every GPU loading this module holds until the process
// exits; the calls share it.
#include <mutex>

#include "moe_fp4_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = MOE_FP4_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The shared scratch.  In host code this name is only a stand-in for the
// device symbol; its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, with that device
// current.  Outside a stream capture it is looked up again on every call, so
// that an address made stale by a device reset (which reloads this module) is
// never used; during a capture, where the lookup might have to load the
// module, the address recorded by the last call outside a capture is used
// (nullptr, hence an error, if there was none).
void* scratch_address(cudaStream_t st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" int moe_fp4_forward_noalloc(const moe_fp4_dims* dims, const void* x_bf16, const float* router_logits,
                                       const uint8_t* w13, const uint8_t* w13_scale, const uint8_t* w2,
                                       const uint8_t* w2_scale, float* out, unsigned flags, void* cuda_stream) {
  if (!dims) return MOE_FP4_ERR_INVALID_ARG;
  const size_t need = moe_fp4_workspace_bytes(dims);
  if (need == 0) return MOE_FP4_ERR_UNSUPPORTED;
  if (need > kNoAllocScratchBytes) return MOE_FP4_ERR_WORKSPACE;
  void* scratch = scratch_address(static_cast<cudaStream_t>(cuda_stream));
  if (!scratch) return MOE_FP4_ERR_CUDA;
  // every region the layer reads is written earlier in the same call (the
  // error words are cleared by the first kernel), so no clearing is needed
  return moe_fp4_forward(dims, x_bf16, router_logits, w13, w13_scale, w2, w2_scale, out, nullptr, nullptr,
                         nullptr, nullptr, nullptr, flags, scratch, kNoAllocScratchBytes, cuda_stream);
}

extern "C" int moe_fp4_noalloc_check(void* cuda_stream) {
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  int32_t err[4] = {0, 0, 0, 0};
  // the error words are the first region of every workspace layout
  if (cudaMemcpyFromSymbolAsync(err, g_noalloc_scratch, sizeof(err), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MOE_FP4_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_FP4_ERR_CUDA;
  if (err[0] != 0) {
    const int32_t zero[4] = {0, 0, 0, 0};
    if (cudaMemcpyToSymbolAsync(g_noalloc_scratch, zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st) != cudaSuccess)
      return MOE_FP4_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_FP4_ERR_CUDA;
    return MOE_FP4_ERR_DEVICE;
  }
  return MOE_FP4_OK;
}
