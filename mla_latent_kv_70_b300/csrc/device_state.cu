// Per-device host state of the library: the SM count used by the split planner and the
// opt-in to more than 48 KB of dynamic shared memory, which is an attribute of a kernel in
// each device's context.  Both are looked up once per device, under a lock, so that
// several host threads and several devices can use the library at once.
#include <atomic>
#include <mutex>

#include "common.cuh"

namespace mla {

namespace {

std::mutex g_mu;
std::atomic<int> g_sm_count[kMaxDevices];   // 0: not looked up yet
std::atomic<int> g_fault_kernels{0};
std::atomic<uint64_t> g_fault_wait_ns{kDefaultWaitNs};

}  // namespace

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  return (dev >= 0 && dev < kMaxDevices) ? dev : -1;
}

int device_sm_count() {
  const int dev = current_device();
  if (dev < 0) return 0;
  int n = g_sm_count[dev].load(std::memory_order_acquire);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 0;
  }
  g_sm_count[dev].store(n, std::memory_order_release);
  return n;
}

cudaError_t ensure_dynamic_smem(const void* kernel, int bytes, SmemOptIn& opt) {
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  if (opt.done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> lock(g_mu);
  if (opt.done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) opt.done[dev].store(true, std::memory_order_release);
  return e;
}

WaitConfig wait_config(int kernel_bit) {
  if (g_fault_kernels.load(std::memory_order_acquire) & kernel_bit)
    return WaitConfig{g_fault_wait_ns.load(std::memory_order_relaxed), 1};
  return WaitConfig{kDefaultWaitNs, 0};
}

}  // namespace mla

extern "C" mla_status mla_debug_inject_timeout(int kernels, double wait_ms) {
  if (kernels & ~(mla::kFaultDecode | mla::kFaultAbsorb | mla::kFaultOutProj)) return MLA_ERR_INVALID;
  if (kernels && !(wait_ms > 0.0 && wait_ms <= 2000.0)) return MLA_ERR_INVALID;
  mla::g_fault_wait_ns.store(kernels ? (uint64_t)(wait_ms * 1e6) : mla::kDefaultWaitNs,
                             std::memory_order_relaxed);
  mla::g_fault_kernels.store(kernels, std::memory_order_release);
  return MLA_OK;
}
