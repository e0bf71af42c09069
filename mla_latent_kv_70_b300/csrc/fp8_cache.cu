// The FP8 form of the latent cache (page "DeepSeek Multi-Head Latent Attention(MLA) 아키텍처
// 해부", section 5, the checklist item on FP8 mixed precision: E4M3 over the 512-wide
// latent space with a per-token scale).
//
// A cached row of 576 bf16 (c^KV then k^R) becomes 640 bytes: the 512 latent values as
// E4M3 codes of c / s (round to nearest even, saturating at +-448), then k^R as it was
// (64 bf16), with the row's scale s in a separate fp32 array.  s is the least power of
// two with max|c| / s <= 448 (exponent clamped to [-126, 15]; an all-zero row takes 1),
// so that c / s and s * E4M3(c / s) are exact in fp32 and bf16; e <= 15 keeps 2^112 * s, the
// multiplier of the decode's widening to bf16, a finite bf16.
#include <cuda_fp8.h>

#include <algorithm>

#include "common.cuh"

namespace mla {

namespace {

constexpr int kFp8Row = 640;   // bytes of one FP8 cache row

// Exponent e of the row scale 2^e: the least e with amax <= 448 * 2^e, from the bits of
// amax (448 = 1.75 * 2^8, so amax = 1.f * 2^E needs e = E - 8 when its fraction exceeds
// 0.75, else e = E - 9).
__device__ __forceinline__ int fp8_scale_exponent(float amax) {
  const uint32_t bits = __float_as_uint(amax);
  if (amax == 0.f) return 0;
  const int ef = (int)(bits >> 23);
  if (ef == 0) return -126;                       // subnormal: 2^-126 already suffices
  const int e = (ef - 127) - 8 + ((bits & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  return min(15, max(-126, e));
}

__device__ __forceinline__ float exp2i(int e) {   // 2^e for e in [-127, 127], exact
  return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);
}

__device__ __forceinline__ uint32_t fp8x2(float a, float b) {   // a -> low byte
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

__global__ void __launch_bounds__(256) k_quantize_fp8(const __nv_bfloat16* __restrict__ rows, int64_t row_stride,
                                                      int64_t n, uint8_t* __restrict__ out,
                                                      float* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < n; r += warps) {
    const __nv_bfloat16* src = rows + r * row_stride;
    // Lane l: latent values [16 l, 16 l + 16).
    const uint4 u0 = reinterpret_cast<const uint4*>(src)[2 * lane];
    const uint4 u1 = reinterpret_cast<const uint4*>(src)[2 * lane + 1];
    const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    float x[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const int e = fp8_scale_exponent(amax);
    const float inv = exp2i(-e);
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      c[i] = fp8x2(x[4 * i] * inv, x[4 * i + 1] * inv) | (fp8x2(x[4 * i + 2] * inv, x[4 * i + 3] * inv) << 16);
    uint8_t* dst = out + r * kFp8Row;
    reinterpret_cast<uint4*>(dst)[lane] = make_uint4(c[0], c[1], c[2], c[3]);
    if (lane < 8)   // k^R: 64 bf16 = 128 bytes, as they are
      reinterpret_cast<uint4*>(dst + kDc)[lane] = reinterpret_cast<const uint4*>(src + kDc)[lane];
    if (lane == 0) scales[r] = exp2i(e);
  }
}

// The step's new rows straight into the FP8 cache: one CTA per sequence, one warp per new
// row (S <= 4).  Row s goes to position seqlens[b] + s: its latent values quantized as by
// k_quantize_fp8, its k^R rotated at that position (as the bf16 append does) and stored
// as bf16, its scale beside it; seqlens[b] advances by S.  A row with no place is skipped
// and flagged.  No early trigger: the decode after it sees the rows and the new seqlens.
__global__ void __launch_bounds__(128) k_append_latent_fp8(const __nv_bfloat16* __restrict__ rows, int S,
                                                           int32_t* __restrict__ seqlens, uint8_t* __restrict__ kv8,
                                                           float* __restrict__ kv_scale, int64_t kv_seq_stride,
                                                           const int32_t* __restrict__ block_table, int max_pages,
                                                           int num_pages, int rotate, RopeFreqs f,
                                                           int32_t* __restrict__ status) {
  const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = seqlens[b];
  __syncthreads();   // every warp has read seqlens[b] before it is advanced
  for (int s = warp; s < S; s += 4) {
    const int t = T + s;
    int64_t dst = -1;
    if (block_table) {
      const int page = (t >= 0 && t / kPage < max_pages) ? block_table[(int64_t)b * max_pages + t / kPage] : -1;
      if (page >= 0 && page < num_pages) dst = (int64_t)page * kPage + t % kPage;
    } else if (t >= 0 && t < kv_seq_stride) {
      dst = (int64_t)b * kv_seq_stride + t;
    }
    if (dst < 0) {
      if (lane == 0) raise_flag(status, kFlagBlockTable);
      continue;
    }
    const __nv_bfloat16* src = rows + ((int64_t)b * S + s) * kRow;
    const uint4 u0 = reinterpret_cast<const uint4*>(src)[2 * lane];
    const uint4 u1 = reinterpret_cast<const uint4*>(src)[2 * lane + 1];
    const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    float x[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const int e = fp8_scale_exponent(amax);
    const float inv = exp2i(-e);
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      c[i] = fp8x2(x[4 * i] * inv, x[4 * i + 1] * inv) | (fp8x2(x[4 * i + 2] * inv, x[4 * i + 3] * inv) << 16);
    uint8_t* row8 = kv8 + dst * kFp8Row;
    reinterpret_cast<uint4*>(row8)[lane] = make_uint4(c[0], c[1], c[2], c[3]);
    if (lane < 8) {   // k^R: 8 pieces of 4 pairs
      uint4 v = reinterpret_cast<const uint4*>(src + kDc)[lane];
      if (rotate) {
        uint32_t r[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int pair = 4 * lane + j;
          const float2 p = bf2_to_f2(r[j]);
          const float2 q = rope_pair(p.x, p.y, t, f.hi[pair], f.lo[pair]);
          r[j] = f2_to_bf2(q.x, q.y);
        }
        v = make_uint4(r[0], r[1], r[2], r[3]);
      }
      reinterpret_cast<uint4*>(row8 + kDc)[lane] = v;
    }
    if (lane == 0) kv_scale[dst] = exp2i(e);
  }
  __syncthreads();
  if (threadIdx.x == 0) seqlens[b] = T + S;
}

}  // namespace

cudaError_t launch_append_latent_fp8(const __nv_bfloat16* rows, int B, int S, int32_t* seqlens, uint8_t* kv8,
                                     float* kv_scale, int64_t kv_seq_stride, const int32_t* block_table,
                                     int max_pages, int num_pages, int rotate, const RopeFreqs& f,
                                     int32_t* status, cudaStream_t st) {
  k_append_latent_fp8<<<B, 128, 0, st>>>(rows, S, seqlens, kv8, kv_scale, kv_seq_stride, block_table, max_pages,
                                         num_pages, rotate, f, status);
  return cudaGetLastError();
}

cudaError_t launch_quantize_fp8(const __nv_bfloat16* rows, int64_t row_stride, int64_t n, uint8_t* out,
                                float* scales, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const int sms = device_sm_count() > 0 ? device_sm_count() : 148;
  const int64_t blocks = std::min<int64_t>((n + 7) / 8, (int64_t)sms * 8);
  k_quantize_fp8<<<(unsigned)blocks, 256, 0, st>>>(rows, row_stride, n, out, scales);
  return cudaGetLastError();
}

}  // namespace mla
