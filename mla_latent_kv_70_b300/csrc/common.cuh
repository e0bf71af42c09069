// Shared definitions of libmla's kernels (internal; the public ABI is include/mla.h).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "mla.h"

namespace mla {

constexpr int kDc = MLA_D_C;      // latent width d_c
constexpr int kDr = MLA_D_R;      // decoupled RoPE width d_r
constexpr int kDn = MLA_D_NOPE;   // per-head content query/key width
constexpr int kDv = MLA_D_V;      // per-head value width
constexpr int kRow = MLA_ROW;     // cached row: c^KV | k^R
constexpr int kPage = 64;         // rows per page of a paged cache

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Device-side error flags OR-ed into the caller's status word.
constexpr int32_t kFlagBlockTable = 1 << MLA_ERR_BLOCK_TABLE;
constexpr int32_t kFlagTimeout = 1 << MLA_ERR_TIMEOUT;

__device__ __forceinline__ void raise_flag(int32_t* status, int32_t flag) {
  if (status) atomicOr(status, flag);
}

__device__ __forceinline__ float2 bf2_to_f2(uint32_t w) {
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&w);
  return __bfloat1622float2(v);
}

__device__ __forceinline__ uint32_t f2_to_bf2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Inverse RoPE frequencies theta^(-2i/64), i = 0..31, computed on the host in double and
// carried as two fp32 terms: hi = fp32(f), lo = fp32(f - hi).
struct RopeFreqs {
  float hi[kDr / 2];
  float lo[kDr / 2];
};
RopeFreqs make_rope_freqs(float theta);

// Rotate one interleaved pair by the angle pos * f, reduced to about [-pi, pi] in fp32
// without losing the angle's low bits (fp64 is slow on this GPU): pos * f is carried as
// two terms (the product's exact rounding error from an FMA, plus pos * f_lo), and 2 pi is
// subtracted Cody-Waite style with a two-term 2 pi, whose first step is exact (for
// positions below 2^24 both terms are multiples of 2^-22 below 2^24 units).  The
// reduced angle is within about 1e-6 rad of pos * f mod 2 pi.
__device__ __forceinline__ float2 rope_pair(float x0, float x1, int pos, float f_hi, float f_lo) {
  constexpr float kTwoPiHi = 6.2831854820251465f;      // fp32(2 pi)
  constexpr float kTwoPiLo = -1.7484555314695172e-07f; // 2 pi - kTwoPiHi
  constexpr float kInvTwoPi = 0.15915493667125702f;
  const float p = (float)pos;
  const float a_hi = p * f_hi;
  const float a_lo = fmaf(p, f_lo, fmaf(p, f_hi, -a_hi));
  const float k = rintf(a_hi * kInvTwoPi);
  float r = fmaf(-k, kTwoPiHi, a_hi);
  r = fmaf(-k, kTwoPiLo, r) + a_lo;
  float s, c;
  sincosf(r, &s, &c);
  return make_float2(x0 * c - x1 * s, x0 * s + x1 * c);
}

// Bounded waits.  Every mbarrier wait of the kernels gives up after wait_ns (2 s unless
// the test hook mla_debug_inject_timeout shortened it); a kernel told to withhold one
// completion signal (`fault`) makes one of its own waits run out, to exercise the abort
// path without faulting anything.
enum : int { kFaultDecode = 1, kFaultAbsorb = 2, kFaultOutProj = 4 };
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
struct WaitConfig {
  uint64_t wait_ns;
  int fault;   // 1: withhold the signal, 0: run normally
};
WaitConfig wait_config(int kernel_bit);   // device_state.cu

// ---------------------------------------------------------------------------
// Decode: per-launch parameters shared by the host planner and the kernel.
// ---------------------------------------------------------------------------
struct DecodeParams {
  const __nv_bfloat16* q_cat;  // [B,S,H,576]
  const __nv_bfloat16* kv;     // contiguous rows or page pool
  int64_t kv_seq_stride;       // rows between sequences (contiguous layout)
  const int32_t* seqlens;      // [B]
  const int32_t* block_table;  // [B,max_pages] or null
  int max_pages;
  int num_pages;
  int max_seqlen;              // rows past this bound are never read (seqlens are clamped)
  int B, S, H;
  int causal;
  float scale_log2;            // softmax scale * log2(e)
  int num_splits;
  float* o_out;                // o_lat [B,S,H,512] (1 split) or partials [splits,B,S,H,512]
  float* lse_out;              // lse [B,S,H] or partials [splits,B,S,H]
  int32_t* status;
  uint64_t wait_ns;            // limit of every mbarrier wait
  int fault;                   // 1: the score issuer withholds the completion of tile 0
  const float* kv_scale;       // FP8 cache only: per-row scale of the E4M3 latent values
};

// Rows [t0, t1) of sequence b that split `split` covers for query token s.  Splits are
// chunks of C = ceil(max_seqlen / num_splits) rows (rounded up to the 64-row tile), the
// same for every sequence, so a short sequence uses fewer splits than a long one and
// its trailing splits are empty (t0 >= t1).
__device__ __forceinline__ void split_range(const DecodeParams& p, int T, int s, int split,
                                            int& t0, int& t1) {
  int n_vis = T;
  if (p.causal) n_vis = min(T, max(0, T - p.S + s + 1));
  int chunk = (p.max_seqlen + p.num_splits - 1) / p.num_splits;
  chunk = (chunk + 63) & ~63;
  t0 = min(split * chunk, n_vis);
  t1 = min(t0 + chunk, n_vis);
}

// A 2D TMA tensor map over `rows` rows of `inner` elements (bf16 or fp32), rows
// `row_stride_bytes` apart, copied in boxes of box_inner x box_rows.  Returns false if
// the driver rejects it (alignment, sizes) or the entry point is unavailable.
bool encode_tma_2d(CUtensorMap* map, bool is_bf16, const void* base, uint64_t inner,
                   uint64_t rows, uint64_t row_stride_bytes, uint32_t box_inner,
                   uint32_t box_rows, CUtensorMapSwizzle swizzle);
// A 3D map over [outer][rows][inner] (bf16 or fp32): strides in bytes of a row and of an
// outer slice, boxes of box_inner x box_rows x 1.  Boxes clip at the end of each slice.
bool encode_tma_3d(CUtensorMap* map, bool is_bf16, const void* base, uint64_t inner, uint64_t rows,
                   uint64_t outer, uint64_t row_stride_bytes, uint64_t outer_stride_bytes,
                   uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle);
// The same over bytes (uint8 elements).
bool encode_tma_2d_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                      uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows,
                      CUtensorMapSwizzle swizzle);

// Launch with programmatic stream serialization: the kernel may start while the previous
// kernel on the stream finishes, running its independent prologue (barriers, TMEM,
// weight or cache loads) early; it calls grid_dep_wait() before it touches anything the
// previous kernel writes or reads.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Per-device host state (device_state.cu).  Devices are numbered below kMaxDevices.
constexpr int kMaxDevices = 64;
int current_device();          // the calling thread's current device, -1 if unusable
int device_sm_count();         // SMs of the current device, 0 if unusable
// One kernel's opt-in to `bytes` of dynamic shared memory, made once per device.
struct SmemOptIn {
  std::atomic<bool> done[kMaxDevices];
};
cudaError_t ensure_dynamic_smem(const void* kernel, int bytes, SmemOptIn& opt);

// The host-side argument checks of mla_decode_latent other than the workspace (api.cu);
// they make no CUDA call.
mla_status check_decode_args(const void* q_cat, const void* kv, int64_t kv_seq_stride,
                             const int32_t* seqlens, const int32_t* block_table, int max_pages,
                             int page_size, int num_pages, int B, int S, int H, float scale,
                             int num_splits, int max_seqlen, const float* o_lat, const float* lse);

cudaError_t launch_prefill_attn(const __nv_bfloat16* q_nope, const __nv_bfloat16* q_rope,
                                const __nv_bfloat16* kv, int64_t kv_seq_stride, const __nv_bfloat16* k_exp,
                                const __nv_bfloat16* v_exp, int B, int T_q, int T_kv, int H, float scale,
                                float* o, float* lse, int32_t* status, cudaStream_t st);

// Launchers (defined next to their kernels).
cudaError_t launch_absorb_q(const __nv_bfloat16* q_nope, const __nv_bfloat16* q_rope,
                            const __nv_bfloat16* w_uk, const int32_t* q_pos, const RopeFreqs& f,
                            int M, int H, __nv_bfloat16* q_cat, cudaStream_t st);
cudaError_t launch_out_proj_uv(const float* o_lat, const __nv_bfloat16* w_uv, int M, int H,
                               float* o, cudaStream_t st);
cudaError_t launch_rope_inplace(__nv_bfloat16* x, int64_t row_stride, int64_t rows,
                                int col_offset, const int32_t* pos, const RopeFreqs& f,
                                cudaStream_t st);
cudaError_t launch_combine(const float* o_part, const float* lse_part, int splits, int64_t rows,
                           float* o, float* lse, cudaStream_t st);
cudaError_t launch_decode(DecodeParams p, cudaStream_t st);
// The decode over the FP8 cache (640-byte rows at p.kv, scales at p.kv_scale).
cudaError_t launch_decode_fp8(DecodeParams p, cudaStream_t st);
cudaError_t launch_quantize_fp8(const __nv_bfloat16* rows, int64_t row_stride, int64_t n, uint8_t* out,
                                float* scales, cudaStream_t st);
cudaError_t launch_append_latent_fp8(const __nv_bfloat16* rows, int B, int S, int32_t* seqlens, uint8_t* kv8,
                                     float* kv_scale, int64_t kv_seq_stride, const int32_t* block_table,
                                     int max_pages, int num_pages, int rotate, const RopeFreqs& f,
                                     int32_t* status, cudaStream_t st);
cudaError_t launch_append_latent(const __nv_bfloat16* rows, int B, int S, int32_t* seqlens,
                                 __nv_bfloat16* kv, int64_t kv_seq_stride, const int32_t* block_table,
                                 int max_pages, int num_pages, int rotate, const RopeFreqs& f,
                                 int32_t* status, cudaStream_t st);

}  // namespace mla
