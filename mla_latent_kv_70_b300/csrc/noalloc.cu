// mla_decode_latent_noalloc: the latent decode for callers that cannot allocate device
// memory.  The split-KV partials live in a fixed array compiled into this library instead
// of a caller-provided workspace; everything else is mla_decode_latent unchanged.
#include <mutex>

#include "common.cuh"

namespace {

// Scratch for the split partials (fp32 o then lse).  Every device that loads libmla.so
// holds this array until the process exits.  Each call writes every partial it later
// reads, so nothing in it has to start at zero.
__device__ __align__(256) static unsigned char g_noalloc_scratch[MLA_NOALLOC_SCRATCH_BYTES];

void* g_scratch_ptr[mla::kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device.  The host-side name of the
// array is only a stand-in, so the address is asked of the runtime, once per device.
cudaError_t scratch_address(void** out) {
  const int dev = mla::current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" mla_status mla_decode_latent_noalloc(
    const mla_bf16* q_cat, const mla_bf16* kv, int64_t kv_seq_stride, const int32_t* seqlens,
    const int32_t* block_table, int max_pages, int page_size, int num_pages, int B, int S, int H,
    int causal, float scale, int num_splits, int max_seqlen, float* o_lat, float* lse,
    int32_t* status_dev, mla_stream stream) {
  // Every host-side check of mla_decode_latent first: a rejected call makes no CUDA call
  // (the scratch address below is what would first touch the device).
  const mla_status bad = mla::check_decode_args(q_cat, kv, kv_seq_stride, seqlens, block_table,
                                                max_pages, page_size, num_pages, B, S, H, scale,
                                                num_splits, max_seqlen, o_lat, lse);
  if (bad != MLA_OK) return bad;
  const size_t need = mla_decode_workspace_bytes(B, S, H, num_splits, max_seqlen);
  if (need > (size_t)MLA_NOALLOC_SCRATCH_BYTES) return MLA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0 && scratch_address(&scratch) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  return mla_decode_latent(q_cat, kv, kv_seq_stride, seqlens, block_table, max_pages, page_size,
                           num_pages, B, S, H, causal, scale, num_splits, max_seqlen, o_lat, lse,
                           scratch, need > 0 ? (size_t)MLA_NOALLOC_SCRATCH_BYTES : 0, status_dev,
                           stream);
}
