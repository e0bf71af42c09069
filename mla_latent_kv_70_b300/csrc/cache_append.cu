// Cache append: the latent rows of the tokens being decoded are written into the cache
// before attention reads it.
//
// Page "MLA의 계산: KV를 펼치지 않고 Attention하기", section "계산 재배치의 효과와 한계":
// in a decode step the current token's latent is added to the cache first, and the token
// then attends to every cached position including its own.  Page "DeepSeek Multi-Head
// Latent Attention(MLA) 아키텍처 해부", section 2: the cached k^R already carries RoPE, so
// it is rotated at its position once, here, and never again at read time.
//
// One CTA per sequence: it reads seqlens[b] once, writes the S new rows at positions
// seqlens[b] .. seqlens[b] + S - 1 (c^KV copied, k^R rotated), then advances seqlens[b].
// The kernel does not let the next kernel start early (no programmatic trigger): the
// latent decode that follows reads the cache and seqlens before its own dependency wait.
#include "common.cuh"

namespace mla {

namespace {

constexpr int kAppendThreads = 128;
constexpr int kChunks = kRow * 2 / 16;          // 72 pieces of 16 bytes per row
constexpr int kRopeChunk0 = kDc * 2 / 16;       // pieces 64..71 hold k^R

__global__ void __launch_bounds__(kAppendThreads)
k_append_latent(const __nv_bfloat16* __restrict__ rows, int S, int32_t* __restrict__ seqlens,
                __nv_bfloat16* __restrict__ kv, int64_t kv_seq_stride,
                const int32_t* __restrict__ block_table, int max_pages, int num_pages, int rotate,
                RopeFreqs f, int32_t* __restrict__ status) {
  const int b = blockIdx.x;
  const int T = seqlens[b];
  __shared__ int bad;
  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  for (int idx = threadIdx.x; idx < S * kChunks; idx += kAppendThreads) {
    const int s = idx / kChunks, piece = idx % kChunks;
    const int t = T + s;   // position of the new row
    int64_t dst_row;
    if (block_table) {
      const int page = (t >= 0 && t / kPage < max_pages) ? block_table[(int64_t)b * max_pages + t / kPage] : -1;
      if (page < 0 || page >= num_pages) {
        bad = 1;
        continue;
      }
      dst_row = (int64_t)page * kPage + t % kPage;
    } else {
      if (t < 0 || t >= kv_seq_stride) {
        bad = 1;
        continue;
      }
      dst_row = (int64_t)b * kv_seq_stride + t;
    }
    uint4 v = reinterpret_cast<const uint4*>(rows + ((int64_t)b * S + s) * kRow)[piece];
    if (rotate && piece >= kRopeChunk0) {
      uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int pair = 4 * (piece - kRopeChunk0) + j;
        const float2 x = bf2_to_f2(w[j]);
        const float2 y = rope_pair(x.x, x.y, t, f.hi[pair], f.lo[pair]);
        w[j] = f2_to_bf2(y.x, y.y);
      }
      v = make_uint4(w[0], w[1], w[2], w[3]);
    }
    reinterpret_cast<uint4*>(kv + dst_row * kRow)[piece] = v;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // Rows that had no place were skipped and flagged; the sequence still advances by S so
    // that later steps keep their positions.
    if (bad) raise_flag(status, kFlagBlockTable);
    seqlens[b] = T + S;
  }
}

}  // namespace

cudaError_t launch_append_latent(const __nv_bfloat16* rows, int B, int S, int32_t* seqlens,
                                 __nv_bfloat16* kv, int64_t kv_seq_stride, const int32_t* block_table,
                                 int max_pages, int num_pages, int rotate, const RopeFreqs& f,
                                 int32_t* status, cudaStream_t st) {
  k_append_latent<<<B, kAppendThreads, 0, st>>>(rows, S, seqlens, kv, kv_seq_stride, block_table,
                                                 max_pages, num_pages, rotate, f, status);
  return cudaGetLastError();
}

}  // namespace mla
