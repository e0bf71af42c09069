// RoPE of the 64-wide rope slice of rows, and the log-sum-exp merge of split partials.
#include <cmath>

#include "common.cuh"
#include "gemm.cuh"
#include "ptx_sm103.cuh"

namespace mla {

RopeFreqs make_rope_freqs(float theta) {
  // Page "Multi-Head Latent Attention (MLA)", section "구현" (_apply_rope): inverse
  // frequencies theta^(-(0, 2, 4, ..)/d_r) for the interleaved pairs.
  RopeFreqs f;
  for (int i = 0; i < kDr / 2; ++i) {
    const double inv = std::pow((double)theta, -2.0 * i / kDr);
    f.hi[i] = (float)inv;
    f.lo[i] = (float)(inv - (double)f.hi[i]);
  }
  return f;
}

namespace {

using namespace ptx;

__global__ void k_rope_inplace(__nv_bfloat16* __restrict__ x, int64_t row_stride, int64_t rows,
                               int col_offset, const int32_t* __restrict__ pos, RopeFreqs f) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows * (kDr / 2)) return;
  const int64_t r = idx / (kDr / 2);
  const int i = (int)(idx % (kDr / 2));
  uint32_t* p = reinterpret_cast<uint32_t*>(x + r * row_stride + col_offset) + i;
  const float2 v = bf2_to_f2(*p);
  const float2 y = rope_pair(v.x, v.y, pos[r], f.hi[i], f.lo[i]);
  *p = f2_to_bf2(y.x, y.y);
}

// The RoPE slice of q_cat rows, q_cat[r, h, 512:576] = RoPE(q_rope[r, h], q_pos[r]) (or a
// copy without positions): one thread per 16-byte piece (4 pairs).
__global__ void k_rope_slice(const __nv_bfloat16* __restrict__ q_rope, const int32_t* __restrict__ q_pos,
                             RopeFreqs f, int M, int H, __nv_bfloat16* __restrict__ q_cat) {
  grid_dep_launch();
  grid_dep_wait();
  constexpr int kPieces = kDr * 2 / 16;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)M * H * kPieces) return;
  const int64_t mh = idx / kPieces;
  const int piece = (int)(idx % kPieces);
  uint4 v = reinterpret_cast<const uint4*>(q_rope + mh * kDr)[piece];
  if (q_pos) {
    const int pos = q_pos[mh / H];
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 x = bf2_to_f2(w[j]);
      const float2 y = rope_pair(x.x, x.y, pos, f.hi[4 * piece + j], f.lo[4 * piece + j]);
      w[j] = f2_to_bf2(y.x, y.y);
    }
    v = make_uint4(w[0], w[1], w[2], w[3]);
  }
  reinterpret_cast<uint4*>(q_cat + mh * kRow + kDc)[piece] = v;
}

// One CTA of 128 threads per output row: weights exp(lse_k - max) are formed once in
// shared memory, then each thread merges one float4 of the 512-wide latent row.
__global__ void __launch_bounds__(128)
k_combine(const float* __restrict__ o_part, const float* __restrict__ lse_part, int splits,
          int64_t rows, float* __restrict__ o, float* __restrict__ lse) {
  grid_dep_launch();
  grid_dep_wait();   // the partials come from the previous kernel
  const int64_t row = blockIdx.x;
  const int tid = threadIdx.x;
  __shared__ float w_s[MLA_MAX_SPLITS];
  __shared__ float red[4];
  const float l = tid < splits ? lse_part[(int64_t)tid * rows + row] : -INFINITY;
  float m = l;
  for (int off = 16; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if ((tid & 31) == 0) red[tid >> 5] = m;
  __syncthreads();
  m = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  __syncthreads();
  const float w = (l == -INFINITY) ? 0.f : expf(l - m);
  float sum = w;
  for (int off = 16; off; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if ((tid & 31) == 0) red[tid >> 5] = sum;
  __syncthreads();
  sum = red[0] + red[1] + red[2] + red[3];
  const bool empty = (m == -INFINITY);
  const float inv = empty ? 0.f : 1.f / sum;
  if (tid < splits) w_s[tid] = w * inv;
  __syncthreads();
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k = 0; k < splits; ++k) {
    const float wk = w_s[k];
    if (wk == 0.f) continue;
    const float4 v = reinterpret_cast<const float4*>(o_part + ((int64_t)k * rows + row) * kDc)[tid];
    acc.x = fmaf(wk, v.x, acc.x);
    acc.y = fmaf(wk, v.y, acc.y);
    acc.z = fmaf(wk, v.z, acc.z);
    acc.w = fmaf(wk, v.w, acc.w);
  }
  reinterpret_cast<float4*>(o + row * kDc)[tid] = acc;
  if (tid == 0) lse[row] = empty ? -INFINITY : m + logf(sum);
}

}  // namespace

cudaError_t launch_rope_inplace(__nv_bfloat16* x, int64_t row_stride, int64_t rows,
                                int col_offset, const int32_t* pos, const RopeFreqs& f,
                                cudaStream_t st) {
  const int64_t n = rows * (kDr / 2);
  if (n == 0) return cudaSuccess;
  const int threads = 256;
  k_rope_inplace<<<(unsigned)((n + threads - 1) / threads), threads, 0, st>>>(
      x, row_stride, rows, col_offset, pos, f);
  return cudaGetLastError();
}

cudaError_t launch_rope_slice(const __nv_bfloat16* q_rope, const int32_t* q_pos, const RopeFreqs& f, int M,
                              int H, __nv_bfloat16* q_cat, cudaStream_t st) {
  const int64_t n = (int64_t)M * H * (kDr * 2 / 16);
  if (n == 0) return cudaSuccess;
  cudaError_t e = launch_pdl(k_rope_slice, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, q_rope, q_pos, f,
                             M, H, q_cat);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_combine(const float* o_part, const float* lse_part, int splits, int64_t rows,
                           float* o, float* lse, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  cudaError_t e = launch_pdl(k_combine, dim3((unsigned)rows), dim3(128), 0, st, o_part, lse_part,
                             splits, rows, o, lse);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mla
