// The two per-head projections either side of the latent attention, on the sm_103a
// tensor cores (tcgen05.mma, TMEM accumulators, TMA-staged operands).
//
// Page "MLA의 계산: KV를 펼치지 않고 Attention하기":
//   section "Key 투영을 Query 쪽으로 옮기기" (Fig. 3): q~ = q U^K^T, the content query of
//     each head mapped once into the latent space (k_absorb_q);
//   section "Value 투영을 가중합 뒤로 옮기기" (Fig. 4): (a C) U^V, the value projection
//     applied once per head after the latents are mixed (k_out_proj_uv).
//
// Both are GEMMs batched over heads whose M (the B*S query rows of one head) is small
// (64 for DeepSeek-V3 decode), so both read their 16.8 MB weight tensor once and are
// bound by HBM.  The operands are swapped: the weights are the MMA's M = 128 side and
// the query rows its N side (a multiple of 16), so no MMA row is padding and each CTA
// moves a small share of the bytes; many CTAs per SM keep the loads in flight.  The
// accumulator then holds one weight column per TMEM lane and one query row per column,
// so each warp stores 32 consecutive outputs of a row at a time.  Every mbarrier wait is
// bounded; a CTA whose wait expires writes NaN to its outputs instead of hanging.
#include <cuda.h>

#include "common.cuh"
#include "ptx_sm103.cuh"

namespace mla {

namespace {

using namespace ptx;

__device__ __forceinline__ unsigned char* align1024(unsigned char* p) {
  return reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// TMEM columns to allocate for n fp32 accumulator columns (a power of two, >= 32).
__host__ __device__ constexpr uint32_t tmem_cols(uint32_t n) {
  return n <= 32 ? 32u : n <= 64 ? 64u : n <= 128 ? 128u : 256u;
}

// ---------------------------------------------------------------------------
// Key absorption.  CTA (t, h, row tile):
//   D[128 latent columns x n rows] = W_UK[h, 128 t + (0..127), :] . q_nope[rows, h, :]^T
// A = 128 rows of W_UK[h] (K-major: the 128 d_nope values of a latent column are
// contiguous) and B = the query rows of head h (K-major), each as two 64-wide K boxes
// (128B swizzle); 8 MMAs of K = 16.  n = the rows of the tile rounded up to 16, <= 256.
// TMEM lane l = latent column 128 t + l, column i = query row m0 + i.
// ---------------------------------------------------------------------------
constexpr int kAbsThreads = 128;
constexpr int kAbsTileL = 128;                          // latent columns per CTA (MMA M)
constexpr int kAbsMaxRows = 256;                        // query rows per CTA (MMA N, max)
constexpr uint32_t kAbsABox = kAbsTileL * 128;          // 128 rows x 64 bf16
constexpr uint32_t abs_smem_bytes(int n) { return 2 * kAbsABox + 2u * (uint32_t)n * 128u + 64 + 1024; }

struct AbsorbMaps {
  CUtensorMap q;   // q_nope viewed as [M rows, H*128], box 64 x n rows, 128B swizzle
  CUtensorMap w;   // W_UK viewed as [H*512 rows, 128], box 64 x 128 rows, 128B swizzle
};

__global__ void __launch_bounds__(kAbsThreads)
k_absorb_q(const __grid_constant__ AbsorbMaps maps, const __nv_bfloat16* __restrict__ q_rope,
           const int32_t* __restrict__ q_pos, RopeFreqs freqs, int M, int H, int n,
           __nv_bfloat16* __restrict__ q_cat, WaitConfig wc) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = align1024(smem_raw);
  const uint32_t s0 = smem_addr(smem);
  const uint32_t b_off = 2 * kAbsABox, b_box = (uint32_t)n * 128u;
  const uint32_t bars = s0 + b_off + 2 * b_box;
  const uint32_t bar_full = bars, bar_mma = bars + 16;   // bar_full: [2] K halves (A and B)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + b_off + 2 * b_box + 24);
  const uint64_t wait_ns = wc.wait_ns;

  const int t = blockIdx.x, h = blockIdx.y, m0 = blockIdx.z * n;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t ncols = tmem_cols((uint32_t)n);

  if (tid == 0) {
    mbar_init(bar_full, 1);
    mbar_init(bar_full + 8, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_addr(tmem_slot), ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = *tmem_slot;

  // The weights do not depend on the previous kernel: they are requested before waiting
  // for it (programmatic dependent launch); q_nope (an input) and q_cat after it.
  // (Test hook: with wc.fault the second K half is never requested, so its wait runs out.)
  grid_dep_launch();
  if (tid == 0) {
    prefetch_tmap(&maps.q);
    prefetch_tmap(&maps.w);
    for (int j = 0; j < 2; ++j) {
      mbar_arrive_expect_tx(bar_full + 8u * j, kAbsABox + b_box);
      if (!(wc.fault && j == 1))
        tma_load_2d(s0 + j * kAbsABox, &maps.w, bar_full + 8u * j, 64 * j, h * kDc + kAbsTileL * t);
    }
  }
  grid_dep_wait();
  if (tid == 0) {
    for (int j = 0; j < 2; ++j)
      if (!(wc.fault && j == 1)) tma_load_2d(s0 + b_off + j * b_box, &maps.q, bar_full + 8u * j, h * kDn + 64 * j, m0);
    // On expiry no further MMA is issued; the copies are waited for once more before exit.
    const uint32_t idesc = idesc_bf16(kAbsTileL, n, false, false);
    bool issued = true;
    for (int j = 0; j < 2 && issued; ++j) {
      if (!mbar_wait(bar_full + 8u * j, 0, wait_ns)) {
        issued = false;
        break;
      }
      tc_fence_after();
      const uint64_t ad = smem_desc(s0 + (uint32_t)j * kAbsABox, 16, 1024, kSwizzle128B);
      const uint64_t bd = smem_desc(s0 + b_off + (uint32_t)j * b_box, 16, 1024, kSwizzle128B);
#pragma unroll
      for (int k = 0; k < 4; ++k)   // K = 16 bf16 = 32 B steps inside a swizzle row
        mma_ss(tb, ad + 2u * k, bd + 2u * k, idesc, (j > 0 || k > 0) ? 1u : 0u);
    }
    if (issued) mma_commit(bar_mma);
  }
  __syncwarp();
  const bool ok = !__any_sync(0xffffffffu, !mbar_wait(bar_mma, 0, wait_ns));
  tc_fence_after();

  // Epilogue: warp w holds latent columns c = 128 t + 32 w + lane (its TMEM lane quarter);
  // for each query row the warp writes 32 consecutive bf16 of q~.
  const int c = kAbsTileL * t + 32 * warp + lane;
  const int rows = min(n, M - m0);
#pragma unroll 1
  for (int i0 = 0; i0 < rows; i0 += 32) {
    uint32_t v[32];
    if (ok) {
      tmem_ld32(tb + ((uint32_t)(32 * warp) << 16) + (uint32_t)i0, v);
      tmem_ld_wait();
    }
    const int cnt = min(32, rows - i0);
    __nv_bfloat16* out = q_cat + ((size_t)(m0 + i0) * H + h) * kRow + c;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < cnt) out[(size_t)i * H * kRow] = ok ? __float2bfloat16_rn(__uint_as_float(v[i])) : __float2bfloat16_rn(NAN);
  }

  // The RoPE slice q_cat[..., 512:576]: rotated at the query position, or copied.  The
  // four CTAs of a (head, row tile) share its rows, in 16-byte pieces (8 per row); every
  // thread loads all of its pieces before it stores any, so the copy costs one memory
  // latency rather than one per piece.
  {
    constexpr int kPieces = kDr * 2 / 16;
    constexpr int kShare = kAbsMaxRows * kPieces / 4;
    constexpr int kPerThread = (kShare + kAbsThreads - 1) / kAbsThreads;
    const int total = rows * kPieces;
    const int share = (total + 3) / 4;
    const int begin = t * share, end = min(total, begin + share);
    uint4 v[kPerThread];
#pragma unroll
    for (int u = 0; u < kPerThread; ++u) {
      const int idx = begin + tid + u * kAbsThreads;
      if (idx < end) {
        const size_t mh = (size_t)(m0 + idx / kPieces) * H + h;
        v[u] = reinterpret_cast<const uint4*>(q_rope + mh * kDr)[idx % kPieces];
      }
    }
#pragma unroll
    for (int u = 0; u < kPerThread; ++u) {
      const int idx = begin + tid + u * kAbsThreads;
      if (idx < end) {
        const int rr = idx / kPieces, piece = idx % kPieces;
        const size_t mh = (size_t)(m0 + rr) * H + h;
        uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        if (q_pos) {
          const int pos = q_pos[m0 + rr];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 x = bf2_to_f2(w[j]);
            const float2 y = rope_pair(x.x, x.y, pos, freqs.hi[4 * piece + j], freqs.lo[4 * piece + j]);
            w[j] = f2_to_bf2(y.x, y.y);
          }
        }
        reinterpret_cast<uint4*>(q_cat + mh * kRow + kDc)[piece] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }

  if (!ok && tid == 0) {   // no copy may land, and no MMA may run, after exit
    mbar_wait(bar_full, 0, wait_ns);
    mbar_wait(bar_full + 8, 0, wait_ns);
    mma_commit(bar_mma);    // bar_mma saw no commit: this one tracks every MMA issued
    mbar_wait(bar_mma, 0, wait_ns);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tb, ncols);
  }
}

// ---------------------------------------------------------------------------
// Value up-projection.  A cluster of two CTAs per (head, tile of 64 query rows); CTA r
// takes the K half [256 r, 256 r + 256) of the latent:
//   D_r[128 output columns x 64 rows] = W_UV[h, K half, :]^T . bf16(o_lat[rows, h, K half])^T
// A = that half of W_UV[h] read MN-major (TMA, two 64-column boxes of 256 K-rows), B =
// the o_lat rows of head h rounded to bf16 by the CTA's threads into the 128B-swizzled
// K-major layout (the fp32 loads are all issued before any is used); 16 MMAs of K = 16.
// The two partial sums meet through distributed shared memory: CTA r owns output columns
// [64 r, 64 r + 64) (TMEM lane quarters 2r, 2r+1), sends the other two quarters to the
// peer with st.async (counted on the peer's mbarrier), adds the peer's share of its own
// quarters and writes them, 32 consecutive floats of a row per warp store.  The share
// lands where the peer's A tile was (two CTAs then fit on an SM), so it is sent only
// once the peer says its MMAs are done (a 4-byte st.async "go").
// ---------------------------------------------------------------------------
constexpr int kOutThreads = 256;
constexpr int kOutRows = 64;                             // query rows per cluster (MMA N)
constexpr int kOutKHalf = kDc / 2;
constexpr uint32_t kOutABox = (uint32_t)kOutKHalf * 128; // 256 K-rows x 64 bf16
constexpr uint32_t kOutBBox = (uint32_t)kOutRows * 128;  // 64 rows x 64 bf16
constexpr uint32_t kOutOffB = 2 * kOutABox;
constexpr uint32_t kOutOffRecv = 0;                      // the A tile, once the MMAs are done
constexpr uint32_t kOutRecvBytes = 2 * 2 * 8 * 32 * 16;  // 2 quarters x 2 row halves x 32 lanes x 32 fp32
constexpr uint32_t kOutOffBar = kOutOffB + 4 * kOutBBox;
constexpr uint32_t kOutSmem = kOutOffBar + 64 + 1024;
static_assert(kOutRecvBytes <= 2 * kOutABox, "the peer's share fits in the A tile");
static_assert(2 * (kOutSmem + 1024) <= 233472, "two CTAs per SM");

struct OutMaps {
  CUtensorMap w;   // W_UV viewed as [H*512 rows, 128], box 64 x 256 rows, 128B swizzle
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kOutThreads)
k_out_proj_uv(const __grid_constant__ OutMaps maps, const float* __restrict__ o_lat, int M, int H,
              float* __restrict__ o, WaitConfig wc) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = align1024(smem_raw);
  const uint32_t s0 = smem_addr(smem);
  const uint32_t bar_w = s0 + kOutOffBar, bar_mma = bar_w + 8, bar_recv = bar_w + 16, bar_go = bar_w + 24;
  const uint32_t go_word = bar_w + 32;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOutOffBar + 40);
  const uint64_t wait_ns = wc.wait_ns;

  const uint32_t r = cluster_ctarank();
  const int h = blockIdx.y, m0 = blockIdx.z * kOutRows;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    mbar_init(bar_w, 1);
    mbar_init(bar_mma, 1);
    mbar_init(bar_recv, 1);
    mbar_init(bar_go, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar_recv, kOutRecvBytes);   // armed before the peer can send
    mbar_arrive_expect_tx(bar_go, 4);
  }
  if (warp == 0) {
    tmem_alloc(smem_addr(tmem_slot), 64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = *tmem_slot;

  // W_UV does not depend on the previous kernel: it is requested before waiting for it
  // (programmatic dependent launch); o_lat, which that kernel writes, after.
  // (Test hook: with wc.fault one weight box is never requested, so its wait runs out.)
  grid_dep_launch();
  if (tid == 0) {
    prefetch_tmap(&maps.w);
    mbar_arrive_expect_tx(bar_w, 2 * kOutABox);
    for (int j = 0; j < 2; ++j)
      if (!(wc.fault && j == 1))
        tma_load_2d(s0 + j * kOutABox, &maps.w, bar_w, 64 * j, h * kDc + kOutKHalf * (int)r);
  }
  cluster_sync();   // the peer's barriers exist before any st.async reaches them
  grid_dep_wait();

  // B: thread t converts float4 f = t + 256 u (u < 16) of the 64 x 256 tile: row f / 64,
  // K values 4 (f % 64) .. +3, i.e. a fixed K quad and rows t / 64 + 4 u.
  {
    const int kq = tid & 63, r0 = tid >> 6;
    const float* src = o_lat + ((size_t)(m0 + r0) * H + h) * kDc + kOutKHalf * r + 4 * kq;
    float4 v[16];
#pragma unroll
    for (int u = 0; u < 16; ++u)
      v[u] = (m0 + r0 + 4 * u < M) ? *reinterpret_cast<const float4*>(src + (size_t)4 * u * H * kDc)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
    const int k = 4 * kq;
    const uint32_t box = s0 + kOutOffB + (uint32_t)(k >> 6) * kOutBBox;
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int row = r0 + 4 * u;
      // 128B swizzle: 16-byte chunk j of row `row` sits at chunk j ^ (row & 7).
      const uint32_t addr = box + (uint32_t)row * 128u +
                            (uint32_t)(((((k & 63) >> 3) ^ (row & 7)) << 4) | ((k & 7) << 1));
      const uint32_t lo = f2_to_bf2(v[u].x, v[u].y), hi = f2_to_bf2(v[u].z, v[u].w);
      asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(lo), "r"(hi) : "memory");
    }
  }
  fence_proxy_async_smem();
  __syncthreads();

  if (tid == 0) {
    if (mbar_wait(bar_w, 0, wait_ns)) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(128, kOutRows, true, false);
      const uint64_t ad = smem_desc(s0, kOutABox, 1024, kSwizzle128B);
#pragma unroll
      for (int k = 0; k < kOutKHalf / 16; ++k) {
        const uint64_t bd = smem_desc(s0 + kOutOffB + (uint32_t)(k >> 2) * kOutBBox, 16, 1024, kSwizzle128B);
        mma_ss(tb, ad + 128u * k, bd + 2u * (k & 3), idesc, k > 0 ? 1u : 0u);
      }
      mma_commit(bar_mma);
    }
  }
  __syncwarp();
  const bool ok = !__any_sync(0xffffffffu, !mbar_wait(bar_mma, 0, wait_ns));
  tc_fence_after();
  // Our A tile is no longer read: the peer may send its share into it.
  if (ok && tid == 0) st_async_b32(map_to_rank(go_word, r ^ 1u), 1u, map_to_rank(bar_go, r ^ 1u));

  // Warp w: TMEM lane quarter q = w % 4 (output columns 32 q + lane), rows 32 (w / 4) + i.
  const int q = warp & 3, rh = warp >> 2;
  uint32_t d[32];
  if (ok) {
    tmem_ld32(tb + ((uint32_t)(32 * q) << 16) + 32u * (uint32_t)rh, d);
    tmem_ld_wait();
  }
  const uint32_t slot = (uint32_t)(((q & 1) * 2 + rh) * 8) * 512u + (uint32_t)lane * 16u;
  if ((q >> 1) != (int)r) {
    // Not ours: to the peer's receive buffer, [quarter & 1][row half][chunk][lane][16 B],
    // once the peer's MMAs no longer read it.
    if (ok && !__any_sync(0xffffffffu, !mbar_wait<true>(bar_go, 0, wait_ns))) {
      const uint32_t dst = map_to_rank(s0 + kOutOffRecv + slot, r ^ 1u);
      const uint32_t rbar = map_to_rank(bar_recv, r ^ 1u);
#pragma unroll
      for (int c = 0; c < 8; ++c)
        st_async_v4(dst + (uint32_t)c * 512u, d[4 * c], d[4 * c + 1], d[4 * c + 2], d[4 * c + 3], rbar);
    }
  } else {
    const bool got = !__any_sync(0xffffffffu, !mbar_wait<true>(bar_recv, 0, wait_ns));
    const int m = m0 + 32 * rh;
    float* out = o + ((size_t)m * H + h) * kDv + 32 * q + lane;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      float4 p = make_float4(NAN, NAN, NAN, NAN);
      if (ok && got) {
        p = ld_shared_v4(s0 + kOutOffRecv + slot + (uint32_t)c * 512u);
        p.x += __uint_as_float(d[4 * c]);
        p.y += __uint_as_float(d[4 * c + 1]);
        p.z += __uint_as_float(d[4 * c + 2]);
        p.w += __uint_as_float(d[4 * c + 3]);
      }
      const float vals[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (m + 4 * c + e < M) out[(size_t)(4 * c + e) * H * kDv] = vals[e];
    }
  }

  if (!ok && tid == 0) {   // no copy may land, and no MMA may run, after exit
    mbar_wait(bar_w, 0, wait_ns);
    mma_commit(bar_mma);    // bar_mma saw no commit: this one tracks every MMA issued
    mbar_wait(bar_mma, 0, wait_ns);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tb, 64);
  }
  cluster_sync();   // neither CTA leaves while the other may still write its shared memory
}

}  // namespace

cudaError_t launch_absorb_q(const __nv_bfloat16* q_nope, const __nv_bfloat16* q_rope,
                            const __nv_bfloat16* w_uk, const int32_t* q_pos, const RopeFreqs& f,
                            int M, int H, __nv_bfloat16* q_cat, cudaStream_t st) {
  const int n = M >= kAbsMaxRows ? kAbsMaxRows : (M + 15) & ~15;   // query rows per CTA
  AbsorbMaps maps;
  if (!encode_tma_2d(&maps.q, true, q_nope, (uint64_t)H * kDn, (uint64_t)M, (uint64_t)H * kDn * 2,
                     64, (uint32_t)n, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tma_2d(&maps.w, true, w_uk, kDn, (uint64_t)H * kDc, (uint64_t)kDn * 2, 64, kAbsTileL,
                     CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  static SmemOptIn opt_in;
  cudaError_t e = ensure_dynamic_smem((const void*)k_absorb_q, (int)abs_smem_bytes(kAbsMaxRows), opt_in);
  if (e != cudaSuccess) return e;
  dim3 grid(kDc / kAbsTileL, H, (M + n - 1) / n);
  e = launch_pdl(k_absorb_q, grid, dim3(kAbsThreads), abs_smem_bytes(n), st, maps, q_rope, q_pos, f, M, H,
                 n, q_cat, wait_config(kFaultAbsorb));
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_out_proj_uv(const float* o_lat, const __nv_bfloat16* w_uv, int M, int H,
                               float* o, cudaStream_t st) {
  OutMaps maps;
  if (!encode_tma_2d(&maps.w, true, w_uv, kDv, (uint64_t)H * kDc, (uint64_t)kDv * 2, 64, kOutKHalf,
                     CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  static SmemOptIn opt_in;
  cudaError_t e = ensure_dynamic_smem((const void*)k_out_proj_uv, (int)kOutSmem, opt_in);
  if (e != cudaSuccess) return e;
  dim3 grid(2, H, (M + kOutRows - 1) / kOutRows);
  e = launch_pdl(k_out_proj_uv, grid, dim3(kOutThreads), kOutSmem, st, maps, o_lat, M, H, o,
                 wait_config(kFaultOutProj));
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mla
