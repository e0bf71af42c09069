// Absorbed MLA decode, plain CUDA-core version.
//
// Page "MLA의 계산: KV를 펼치지 않고 Attention하기": section "Content 점수와 위치 점수 합치기"
// (eq. s_j: content dot plus position dot, one scale, one softmax over all readable
// positions, causal mask between query tokens) and section "Value 투영을 가중합 뒤로
// 옮기기" (Fig. 4: the latents are mixed with the weights; U^V is applied later).
//
// One CTA per (query token, block of 16 heads, split).  Tiles of 32 cache rows are
// staged in shared memory; 16 threads share a head: each scores two rows against
// the 576-wide query, then owns 32 of the 512 latent columns of the running output.
// Online softmax in the log2 domain; rows that are past the readable range, or whose
// page id is outside the pool, are zero-filled so they add nothing.
#include "common.cuh"

namespace mla {

namespace {

constexpr int kNT = 32;          // cache rows per tile
constexpr int kHB = 16;          // heads per CTA
constexpr int kThreads = 256;
constexpr int kRowPad = 584;     // bf16 per staged row (1168 B, 16-B multiple)

struct SimtSmem {
  float q[kHB][kRow];
  __align__(16) __nv_bfloat16 kv[kNT][kRowPad];
  float p[kHB][kNT];
};

__device__ __forceinline__ const __nv_bfloat16* row_ptr(const DecodeParams& p, int b, int t,
                                                        bool& ok) {
  ok = true;
  if (p.block_table) {
    const int page = p.block_table[(int64_t)b * p.max_pages + t / kPage];
    if (page < 0 || page >= p.num_pages) {
      ok = false;
      return nullptr;
    }
    return p.kv + ((int64_t)page * kPage + (t % kPage)) * kRow;
  }
  return p.kv + ((int64_t)b * p.kv_seq_stride + t) * kRow;
}

__global__ void __launch_bounds__(kThreads) k_decode_simt(DecodeParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SimtSmem& sm = *reinterpret_cast<SimtSmem*>(smem_raw);
  const int m = blockIdx.x;  // b*S + s
  const int b = m / p.S, s = m % p.S;
  const int h0 = blockIdx.y * kHB;
  const int split = blockIdx.z;
  const int tid = threadIdx.x;
  const int hh = tid >> 4, l16 = tid & 15;

  const int T = min(max(0, p.seqlens[b]), p.max_seqlen);
  int t0, t1;
  split_range(p, T, s, split, t0, t1);

  for (int idx = tid; idx < kHB * (kRow / 2); idx += kThreads) {
    const int r = idx / (kRow / 2), k2 = idx % (kRow / 2);
    const uint32_t w = reinterpret_cast<const uint32_t*>(
        p.q_cat + ((int64_t)m * p.H + h0 + r) * kRow)[k2];
    const float2 f = bf2_to_f2(w);
    sm.q[r][2 * k2] = f.x;
    sm.q[r][2 * k2 + 1] = f.y;
  }

  float m_run = -INFINITY, l_run = 0.f;
  float o[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) o[i] = 0.f;

  for (int ts = t0; ts < t1; ts += kNT) {
    __syncthreads();
    for (int idx = tid; idx < kNT * (kRow / 8); idx += kThreads) {
      const int r = idx / (kRow / 8), c = idx % (kRow / 8);
      const int t = ts + r;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (t < t1) {
        bool ok;
        const __nv_bfloat16* src = row_ptr(p, b, t, ok);
        if (ok)
          v = reinterpret_cast<const uint4*>(src)[c];
        else if (c == 0)
          raise_flag(p.status, kFlagBlockTable);
      }
      *reinterpret_cast<uint4*>(&sm.kv[r][8 * c]) = v;
    }
    __syncthreads();

    // Scores of rows l16 and l16+16 for head hh.
    float acc0 = 0.f, acc1 = 0.f;
    const uint32_t* r0 = reinterpret_cast<const uint32_t*>(&sm.kv[l16][0]);
    const uint32_t* r1 = reinterpret_cast<const uint32_t*>(&sm.kv[l16 + 16][0]);
#pragma unroll 8
    for (int k2 = 0; k2 < kRow / 2; ++k2) {
      const float2 q = *reinterpret_cast<const float2*>(&sm.q[hh][2 * k2]);
      const float2 a = bf2_to_f2(r0[k2]);
      const float2 c = bf2_to_f2(r1[k2]);
      acc0 = fmaf(q.x, a.x, fmaf(q.y, a.y, acc0));
      acc1 = fmaf(q.x, c.x, fmaf(q.y, c.y, acc1));
    }
    const float y0 = (ts + l16 < t1) ? acc0 * p.scale_log2 : -INFINITY;
    const float y1 = (ts + l16 + 16 < t1) ? acc1 * p.scale_log2 : -INFINITY;
    float tmax = fmaxf(y0, y1);
#pragma unroll
    for (int off = 8; off; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
    const float m_new = fmaxf(m_run, tmax);  // finite: the tile holds a readable row
    const float alpha = exp2f(m_run - m_new);
    const float p0 = exp2f(y0 - m_new), p1 = exp2f(y1 - m_new);
    float ps = p0 + p1;
#pragma unroll
    for (int off = 8; off; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    l_run = l_run * alpha + ps;
    m_run = m_new;
    sm.p[hh][l16] = p0;
    sm.p[hh][l16 + 16] = p1;
    __syncwarp();

#pragma unroll
    for (int i = 0; i < 32; ++i) o[i] *= alpha;
    for (int j = 0; j < kNT; ++j) {
      const float pj = sm.p[hh][j];
      const uint32_t* rw = reinterpret_cast<const uint32_t*>(&sm.kv[j][0]);
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const float2 v = bf2_to_f2(rw[l16 + 16 * t]);
        o[2 * t] = fmaf(pj, v.x, o[2 * t]);
        o[2 * t + 1] = fmaf(pj, v.y, o[2 * t + 1]);
      }
    }
  }

  const bool empty = !(l_run > 0.f);
  const float inv = empty ? 0.f : 1.f / l_run;
  const int64_t rows = (int64_t)p.B * p.S * p.H;
  const int64_t row = (int64_t)m * p.H + h0 + hh;
  const int64_t out_row = (p.num_splits > 1) ? (int64_t)split * rows + row : row;
  float* out = p.o_out + out_row * kDc;
#pragma unroll
  for (int t = 0; t < 16; ++t)
    *reinterpret_cast<float2*>(out + 2 * (l16 + 16 * t)) = make_float2(o[2 * t] * inv, o[2 * t + 1] * inv);
  if (l16 == 0) p.lse_out[out_row] = empty ? -INFINITY : (m_run + log2f(l_run)) * kLn2;
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t st) {
  const size_t smem = sizeof(SimtSmem);
  cudaError_t e = cudaFuncSetAttribute(k_decode_simt, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.B * p.S, p.H / kHB, p.num_splits);
  k_decode_simt<<<grid, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
