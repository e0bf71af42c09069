// Copies out of pinned host memory done by the SMs: each thread reads 16-byte pieces of the
// host buffer through its device-mapped address (the GPU's loads cross PCIe) and writes
// them to device memory.  On hosts whose copy engines move host-to-device data slowly, many
// SMs' outstanding reads move it faster.
#include <algorithm>

#include "common.cuh"

namespace mla {

namespace {

constexpr int64_t kCopyBlocks = 64;

__global__ void __launch_bounds__(256) k_copy_from_host(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                       int64_t n16) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  // Four independent loads in flight per thread before their stores.
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
    dst[i] = a;
    dst[i + stride] = b;
    dst[i + 2 * stride] = c;
    dst[i + 3 * stride] = d;
  }
  for (; i < n16; i += stride) dst[i] = src[i];
}

}  // namespace

cudaError_t launch_copy_from_host(const void* src_dev_alias, void* dst, int64_t bytes, cudaStream_t st) {
  const int64_t n16 = bytes / 16;
  if (n16 == 0) return cudaSuccess;
  // 64 blocks keep 1 MiB of reads in flight, far above PCIe bandwidth x latency, and leave
  // most SMs free for kernels running beside the copy.
  const int64_t blocks = std::min<int64_t>((n16 + 1023) / 1024, kCopyBlocks);
  k_copy_from_host<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const uint4*>(src_dev_alias),
                                                    static_cast<uint4*>(dst), n16);
  return cudaGetLastError();
}

}  // namespace mla
