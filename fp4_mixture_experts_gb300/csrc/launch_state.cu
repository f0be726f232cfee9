// Per-device launch state of the library: the SM count (grid sizes), the
// large-shared-memory opt-in of each kernel (a per-device setting), and the
// process-wide fault-injection setting used by the failure-path tests.  All
// of it is safe to use from several host threads and several devices.
#include <atomic>
#include <mutex>
#include <utility>
#include <vector>

#include "moe_fp4_internal.cuh"
#include "ptx_sm103.cuh"

namespace moe_fp4 {
namespace {

constexpr int kMaxDevices = 64;

std::atomic<int> g_sms[kMaxDevices];  // 0: not looked up yet

std::mutex g_optin_mu;
std::vector<std::pair<const void*, int>> g_optin;  // (kernel, device) pairs already opted in

std::atomic<int> g_fault_site{MOE_FP4_FAULT_NONE};
std::atomic<unsigned long long> g_wait_ns{kWaitLimitNs};

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}

}  // namespace

int num_sms() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return 148;
  int n = g_sms[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    g_sms[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

cudaError_t ensure_smem_optin(const void* kernel, int bytes) {
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_optin_mu);
  for (const auto& e : g_optin)
    if (e.first == kernel && e.second == dev) return cudaSuccess;
  const cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (err != cudaSuccess) return err;
  g_optin.emplace_back(kernel, dev);
  return cudaSuccess;
}

int fault_site() { return g_fault_site.load(std::memory_order_relaxed); }

uint64_t wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

}  // namespace moe_fp4

extern "C" int moe_fp4_set_fault_injection(int site, uint32_t wait_limit_us) {
  using namespace moe_fp4;
  if (site < MOE_FP4_FAULT_NONE || site > MOE_FP4_FAULT_STREAM_STAGE) return MOE_FP4_ERR_INVALID_ARG;
  if (site != MOE_FP4_FAULT_NONE && wait_limit_us == 0) return MOE_FP4_ERR_INVALID_ARG;
  g_wait_ns.store(site == MOE_FP4_FAULT_NONE ? kWaitLimitNs : (unsigned long long)wait_limit_us * 1000ull,
                  std::memory_order_relaxed);
  g_fault_site.store(site, std::memory_order_relaxed);
  return MOE_FP4_OK;
}
