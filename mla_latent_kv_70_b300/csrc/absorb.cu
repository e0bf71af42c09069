// Key absorption: q_cat[m,h,0:512] = q_nope[m,h,:] . W_UK[h]^T, q_cat[m,h,512:576] = RoPE(q_rope).
//
// Page "MLA의 계산: KV를 펼치지 않고 Attention하기", section "Key 투영을 Query 쪽으로 옮기기"
// (Fig. 3): the content query of each head is mapped once into the latent space.
//
// One CTA per (head h, block of 32 query rows).  W_UK[h] (512 x 128 bf16, 128 KB) is
// streamed once per row block; each thread owns two latent columns i and keeps the
// 32-row dot products in registers, reading the query rows from shared memory as
// broadcasts.  The kernel is bound by reading W_UK (16.8 MB for 128 heads).
#include "common.cuh"

namespace mla {

namespace {

constexpr int kRowsPerCta = 32;
constexpr int kThreads = 256;
constexpr int kKChunk = 32;

__global__ void __launch_bounds__(kThreads)
k_absorb_q(const __nv_bfloat16* __restrict__ q_nope, const __nv_bfloat16* __restrict__ q_rope,
           const __nv_bfloat16* __restrict__ w_uk, const int32_t* __restrict__ q_pos,
           RopeFreqs freqs, int M, int H, __nv_bfloat16* __restrict__ q_cat) {
  const int h = blockIdx.x;
  const int m0 = blockIdx.y * kRowsPerCta;
  const int rows = min(kRowsPerCta, M - m0);
  const int tid = threadIdx.x;

  __shared__ __align__(16) float q_s[kRowsPerCta][kDn + 4];

  for (int idx = tid; idx < kRowsPerCta * (kDn / 2); idx += kThreads) {
    const int r = idx / (kDn / 2), k2 = idx % (kDn / 2);
    float2 v = make_float2(0.f, 0.f);
    if (r < rows) {
      const uint32_t w =
          reinterpret_cast<const uint32_t*>(q_nope + ((size_t)(m0 + r) * H + h) * kDn)[k2];
      v = bf2_to_f2(w);
    }
    q_s[r][2 * k2] = v.x;
    q_s[r][2 * k2 + 1] = v.y;
  }
  __syncthreads();

  // Two latent columns per thread: i = tid and i = tid + 256.
  float acc0[kRowsPerCta], acc1[kRowsPerCta];
#pragma unroll
  for (int r = 0; r < kRowsPerCta; ++r) acc0[r] = acc1[r] = 0.f;

  const __nv_bfloat16* w0 = w_uk + ((size_t)h * kDc + tid) * kDn;
  const __nv_bfloat16* w1 = w0 + (size_t)256 * kDn;
  for (int kc = 0; kc < kDn; kc += kKChunk) {
    float wa[kKChunk], wb[kKChunk];
#pragma unroll
    for (int v = 0; v < kKChunk / 8; ++v) {
      const uint4 a = *reinterpret_cast<const uint4*>(w0 + kc + 8 * v);
      const uint4 b = *reinterpret_cast<const uint4*>(w1 + kc + 8 * v);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float2 fa = bf2_to_f2(aw[u]), fb = bf2_to_f2(bw[u]);
        wa[8 * v + 2 * u] = fa.x;
        wa[8 * v + 2 * u + 1] = fa.y;
        wb[8 * v + 2 * u] = fb.x;
        wb[8 * v + 2 * u + 1] = fb.y;
      }
    }
#pragma unroll
    for (int r = 0; r < kRowsPerCta; ++r) {
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int k = 0; k < kKChunk; k += 4) {
        const float4 q = *reinterpret_cast<const float4*>(&q_s[r][kc + k]);
        s0 = fmaf(q.x, wa[k], s0);
        s0 = fmaf(q.y, wa[k + 1], s0);
        s0 = fmaf(q.z, wa[k + 2], s0);
        s0 = fmaf(q.w, wa[k + 3], s0);
        s1 = fmaf(q.x, wb[k], s1);
        s1 = fmaf(q.y, wb[k + 1], s1);
        s1 = fmaf(q.z, wb[k + 2], s1);
        s1 = fmaf(q.w, wb[k + 3], s1);
      }
      acc0[r] += s0;
      acc1[r] += s1;
    }
  }
#pragma unroll
  for (int r = 0; r < kRowsPerCta; ++r) {
    if (r < rows) {
      __nv_bfloat16* out = q_cat + ((size_t)(m0 + r) * H + h) * kRow;
      out[tid] = __float2bfloat16_rn(acc0[r]);
      out[tid + 256] = __float2bfloat16_rn(acc1[r]);
    }
  }

  // The RoPE slice: rotated at the query position, or copied.
  for (int idx = tid; idx < rows * (kDr / 2); idx += kThreads) {
    const int r = idx / (kDr / 2), i = idx % (kDr / 2);
    const size_t mh = (size_t)(m0 + r) * H + h;
    const uint32_t w = reinterpret_cast<const uint32_t*>(q_rope + mh * kDr)[i];
    uint32_t o = w;
    if (q_pos) {
      const float2 x = bf2_to_f2(w);
      const float2 y = rope_pair(x.x, x.y, q_pos[m0 + r], freqs.inv_freq[i]);
      o = f2_to_bf2(y.x, y.y);
    }
    reinterpret_cast<uint32_t*>(q_cat + mh * kRow + kDc)[i] = o;
  }
}

}  // namespace

cudaError_t launch_absorb_q(const __nv_bfloat16* q_nope, const __nv_bfloat16* q_rope,
                            const __nv_bfloat16* w_uk, const int32_t* q_pos, const RopeFreqs& f,
                            int M, int H, __nv_bfloat16* q_cat, cudaStream_t st) {
  dim3 grid(H, (M + kRowsPerCta - 1) / kRowsPerCta);
  k_absorb_q<<<grid, kThreads, 0, st>>>(q_nope, q_rope, w_uk, q_pos, f, M, H, q_cat);
  return cudaGetLastError();
}

}  // namespace mla
