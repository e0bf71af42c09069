// Value up-projection: o[m,h,:] = o_lat[m,h,:] . W_UV[h]   (W_UV[h] is 512 x 128).
//
// Page "MLA의 계산: KV를 펼치지 않고 Attention하기", section "Value 투영을 가중합 뒤로 옮기기"
// (Fig. 4): a (C U^V) = (a C) U^V, so U^V is applied once per head after aggregation.
//
// One CTA per (head h, block of 16 query rows); thread n owns output column n and
// walks the 512 latent rows of W_UV[h] (coalesced across the CTA), with the o_lat
// rows read from shared memory as broadcasts.  fp32 throughout.
#include "common.cuh"

namespace mla {

namespace {

constexpr int kRowsPerCta = 16;

__global__ void __launch_bounds__(kDv)
k_out_proj_uv(const float* __restrict__ o_lat, const __nv_bfloat16* __restrict__ w_uv, int M,
              int H, float* __restrict__ o) {
  const int h = blockIdx.x;
  const int m0 = blockIdx.y * kRowsPerCta;
  const int rows = min(kRowsPerCta, M - m0);
  const int n = threadIdx.x;

  extern __shared__ __align__(16) float lat_s[];  // [kRowsPerCta][512]
  for (int idx = n; idx < kRowsPerCta * (kDc / 4); idx += kDv) {
    const int r = idx / (kDc / 4), c4 = idx % (kDc / 4);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < rows) v = reinterpret_cast<const float4*>(o_lat + ((size_t)(m0 + r) * H + h) * kDc)[c4];
    reinterpret_cast<float4*>(lat_s + r * kDc)[c4] = v;
  }
  __syncthreads();

  float acc[kRowsPerCta];
#pragma unroll
  for (int r = 0; r < kRowsPerCta; ++r) acc[r] = 0.f;
  const __nv_bfloat16* w = w_uv + (size_t)h * kDc * kDv + n;
#pragma unroll 4
  for (int i = 0; i < kDc; ++i) {
    const float wi = __bfloat162float(w[(size_t)i * kDv]);
#pragma unroll
    for (int r = 0; r < kRowsPerCta; ++r) acc[r] = fmaf(lat_s[r * kDc + i], wi, acc[r]);
  }
#pragma unroll
  for (int r = 0; r < kRowsPerCta; ++r)
    if (r < rows) o[((size_t)(m0 + r) * H + h) * kDv + n] = acc[r];
}

}  // namespace

cudaError_t launch_out_proj_uv(const float* o_lat, const __nv_bfloat16* w_uv, int M, int H,
                               float* o, cudaStream_t st) {
  dim3 grid(H, (M + kRowsPerCta - 1) / kRowsPerCta);
  const size_t smem = sizeof(float) * kRowsPerCta * kDc;
  k_out_proj_uv<<<grid, kDv, smem, st>>>(o_lat, w_uv, M, H, o);
  return cudaGetLastError();
}

}  // namespace mla
