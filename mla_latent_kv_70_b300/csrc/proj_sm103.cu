// The two per-head projections either side of the latent attention, on the sm_103a
// tensor cores (tcgen05.mma, TMEM accumulators, TMA-staged operands).
//
// Page "MLA의 계산: KV를 펼치지 않고 Attention하기":
//   section "Key 투영을 Query 쪽으로 옮기기" (Fig. 3): q~ = q U^K^T, the content query of
//     each head mapped once into the latent space (k_absorb_q);
//   section "Value 투영을 가중합 뒤로 옮기기" (Fig. 4): (a C) U^V, the value projection
//     applied once per head after the latents are mixed (k_out_proj_uv).
//
// Both are GEMMs batched over heads with a small M (the B*S query rows of one head) and
// are bound by reading the 16.8 MB weight tensor: one CTA per (head, 128-row block
// [, half of the output columns]) stages its operands in 128B-swizzled shared memory and
// one thread issues the MMAs into TMEM.  Every mbarrier wait is bounded; a CTA whose
// wait expires writes NaN to its output tile instead of hanging.
#include <cuda.h>

#include "common.cuh"
#include "ptx_sm103.cuh"

namespace mla {

namespace {

using namespace ptx;

constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s per wait
constexpr int kTileM = 128;                   // query rows per CTA (MMA M)

__device__ __forceinline__ unsigned char* align1024(unsigned char* p) {
  return reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// ---------------------------------------------------------------------------
// Key absorption.  CTA (n_half, h, m_blk):
//   D[128 rows x 256 latent columns] = q_nope[rows, h, 0:128] . W_UK[h, 256 n_half + (0..255), :]^T
// A (q_nope rows of head h) and B (W_UK[h] rows, i.e. K-major) arrive by TMA as two
// 64-wide K boxes each; 8 MMAs of K = 16 accumulate into 256 TMEM columns.
// ---------------------------------------------------------------------------
constexpr int kAbsThreads = 128;
constexpr uint32_t kAbsABox = kTileM * 128;            // 128 rows x 64 bf16
constexpr uint32_t kAbsBBox = 256 * 128;               // 256 rows x 64 bf16
constexpr uint32_t kAbsOffB = 2 * kAbsABox;
constexpr uint32_t kAbsOffBar = kAbsOffB + 2 * kAbsBBox;
constexpr uint32_t kAbsSmem = kAbsOffBar + 64 + 1024;  // + slack for 1024-B alignment

struct AbsorbMaps {
  CUtensorMap q;   // q_nope viewed as [M rows, H*128], box 64 x 128 rows, 128B swizzle
  CUtensorMap w;   // W_UK viewed as [H*512 rows, 128], box 64 x 256 rows, 128B swizzle
};

__global__ void __launch_bounds__(kAbsThreads, 1)
k_absorb_q(const __grid_constant__ AbsorbMaps maps, const __nv_bfloat16* __restrict__ q_rope,
           const int32_t* __restrict__ q_pos, RopeFreqs freqs, int M, int H,
           __nv_bfloat16* __restrict__ q_cat) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = align1024(smem_raw);
  const uint32_t s0 = smem_addr(smem);
  const uint32_t bar_full = s0 + kAbsOffBar, bar_mma = bar_full + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kAbsOffBar + 16);

  const int nh = blockIdx.x, h = blockIdx.y, m0 = blockIdx.z * kTileM;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    mbar_init(bar_full, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_addr(tmem_slot), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = *tmem_slot;

  if (tid == 0) {
    prefetch_tmap(&maps.q);
    prefetch_tmap(&maps.w);
    mbar_arrive_expect_tx(bar_full, 2 * kAbsABox + 2 * kAbsBBox);
    for (int j = 0; j < 2; ++j) {
      tma_load_2d(s0 + j * kAbsABox, &maps.q, bar_full, h * kDn + 64 * j, m0);
      tma_load_2d(s0 + kAbsOffB + j * kAbsBBox, &maps.w, bar_full, 64 * j, h * kDc + 256 * nh);
    }
    // On expiry no MMA is issued; the copies are waited for once more before exit.
    if (mbar_wait(bar_full, 0, kWaitNs)) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(kTileM, 256, false, false);
#pragma unroll
      for (int k = 0; k < kDn / 16; ++k) {
        const uint32_t off = (uint32_t)(k & 3) * 32u;   // K = 16 bf16 = 32 B inside a swizzle row
        mma_ss(tb, smem_desc(s0 + (uint32_t)(k >> 2) * kAbsABox + off, 16, 1024, kSwizzle128B),
               smem_desc(s0 + kAbsOffB + (uint32_t)(k >> 2) * kAbsBBox + off, 16, 1024, kSwizzle128B),
               idesc, k > 0 ? 1u : 0u);
      }
      mma_commit(bar_mma);
    }
  }
  __syncwarp();
  const bool ok = !__any_sync(0xffffffffu, !mbar_wait(bar_mma, 0, kWaitNs));
  tc_fence_after();

  // Epilogue: TMEM lane r = query row m0 + r; 256 fp32 columns -> bf16 q~.
  const int r = 32 * warp + lane;
  const int m = m0 + r;
  __nv_bfloat16* out = q_cat + ((size_t)m * H + h) * kRow + 256 * nh;
#pragma unroll 1
  for (int c = 0; c < 8; ++c) {
    uint32_t v[32];
    if (ok) {
      tmem_ld32(tb + ((uint32_t)(32 * warp) << 16) + 32u * c, v);
      tmem_ld_wait();
    }
    if (m < M) {
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        pk[j] = ok ? f2_to_bf2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1])) : 0x7FC07FC0u;
      uint4* dst = reinterpret_cast<uint4*>(out + 32 * c);
#pragma unroll
      for (int j = 0; j < 4; ++j) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
    }
  }

  // The RoPE slice q_cat[..., 512:576]: rotated at the query position, or copied.
  if (nh == 0) {
    const int rows = min(kTileM, M - m0);
    for (int idx = tid; idx < rows * (kDr / 2); idx += kAbsThreads) {
      const int rr = idx / (kDr / 2), i = idx % (kDr / 2);
      const size_t mh = (size_t)(m0 + rr) * H + h;
      const uint32_t w = reinterpret_cast<const uint32_t*>(q_rope + mh * kDr)[i];
      uint32_t o = w;
      if (q_pos) {
        const float2 x = bf2_to_f2(w);
        const float2 y = rope_pair(x.x, x.y, q_pos[m0 + rr], freqs.inv_freq[i]);
        o = f2_to_bf2(y.x, y.y);
      }
      reinterpret_cast<uint32_t*>(q_cat + mh * kRow + kDc)[i] = o;
    }
  }

  if (!ok && tid == 0) mbar_wait(bar_full, 0, kWaitNs);   // no copy may land after exit
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tb, 256);
  }
}

// ---------------------------------------------------------------------------
// Value up-projection.  CTA (h, m_blk):
//   D[128 rows x 128] = bf16(o_lat[rows, h, 0:512]) . W_UV[h] (512 x 128, N contiguous)
// W_UV[h] arrives by TMA in 8 chunks of 64 K-rows (two 64-wide N boxes each, read
// MN-major by the MMA).  o_lat is fp32, so the CTA's threads load it, round it to bf16
// and write it in the 128B-swizzled K-major layout, double-buffered by 64-wide K chunks,
// one chunk of global loads ahead of the shared-memory stores.
// ---------------------------------------------------------------------------
constexpr int kOutThreads = 128;
constexpr int kOutChunks = kDc / 64;                   // 8 K chunks of 64
constexpr uint32_t kOutBBox = 64 * 128;                // 64 K-rows x 64 bf16
constexpr uint32_t kOutBChunk = 2 * kOutBBox;          // N = 128
constexpr uint32_t kOutAChunk = kTileM * 128;          // 128 rows x 64 bf16
constexpr uint32_t kOutOffA = kOutChunks * kOutBChunk;
constexpr uint32_t kOutOffBar = kOutOffA + 2 * kOutAChunk;
constexpr uint32_t kOutSmem = kOutOffBar + 128 + 1024;

struct OutMaps {
  CUtensorMap w;   // W_UV viewed as [H*512 rows, 128], box 64 x 64 rows, 128B swizzle
};

__global__ void __launch_bounds__(kOutThreads, 1)
k_out_proj_uv(const __grid_constant__ OutMaps maps, const float* __restrict__ o_lat, int M, int H,
              float* __restrict__ o) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = align1024(smem_raw);
  const uint32_t s0 = smem_addr(smem);
  const uint32_t bars = s0 + kOutOffBar;
  auto bar_b = [&](int c) { return bars + 8u * (uint32_t)c; };          // [8] W chunk landed
  auto bar_a = [&](int i) { return bars + 64u + 8u * (uint32_t)i; };    // [2] A buffer consumed
  const uint32_t bar_done = bars + 80u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOutOffBar + 96);

  const int h = blockIdx.x, m0 = blockIdx.y * kTileM;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int c = 0; c < kOutChunks; ++c) mbar_init(bar_b(c), 1);
    mbar_init(bar_a(0), 1);
    mbar_init(bar_a(1), 1);
    mbar_init(bar_done, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_addr(tmem_slot), 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = *tmem_slot;

  if (tid == 0) {
    prefetch_tmap(&maps.w);
    for (int c = 0; c < kOutChunks; ++c) {
      mbar_arrive_expect_tx(bar_b(c), kOutBChunk);
      for (int j = 0; j < 2; ++j)
        tma_load_2d(s0 + c * kOutBChunk + j * kOutBBox, &maps.w, bar_b(c), 64 * j, h * kDc + 64 * c);
    }
  }

  // Thread (warp, lane) covers rows 2*(4*it + warp) + (lane >> 4), it = 0..15, and the
  // four K values 4*(lane & 15) .. +3 of the current chunk.
  const int sub = lane >> 4, kq = lane & 15;
  float4 ld[16];
  auto load_chunk = [&](int c) {
#pragma unroll
    for (int it = 0; it < 16; ++it) {
      const int r = 2 * (4 * it + warp) + sub;
      const int m = m0 + r;
      ld[it] = m < M ? *reinterpret_cast<const float4*>(o_lat + ((size_t)m * H + h) * kDc + 64 * c + 4 * kq)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  load_chunk(0);
  bool ok = true;
  for (int c = 0; c < kOutChunks; ++c) {
    const int buf = c & 1;
    if (c >= 2 && ok) ok = !__any_sync(0xffffffffu, !mbar_wait(bar_a(buf), (uint32_t)((c - 2) >> 1) & 1u, kWaitNs));
    const uint32_t abase = s0 + kOutOffA + (uint32_t)buf * kOutAChunk;
#pragma unroll
    for (int it = 0; it < 16; ++it) {
      const int r = 2 * (4 * it + warp) + sub;
      // 128B swizzle: 16-byte chunk j of row r sits at chunk j ^ (r & 7).
      const uint32_t addr = abase + (uint32_t)r * 128u + (uint32_t)((((kq >> 1) ^ (r & 7)) << 4) | ((kq & 1) << 3));
      const uint32_t lo = f2_to_bf2(ld[it].x, ld[it].y), hi = f2_to_bf2(ld[it].z, ld[it].w);
      asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(lo), "r"(hi) : "memory");
    }
    if (c + 1 < kOutChunks) load_chunk(c + 1);
    fence_proxy_async_smem();
    ok = __syncthreads_and(ok);   // also tells every thread of an earlier failed wait
    if (tid == 0) {
      if (ok && mbar_wait(bar_b(c), 0, kWaitNs)) {
        tc_fence_after();
        const uint32_t idesc = idesc_bf16(kTileM, kDv, false, true);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ss(tb, smem_desc(abase + 32u * k, 16, 1024, kSwizzle128B),
                 smem_desc(s0 + c * kOutBChunk + 2048u * k, kOutBBox, 1024, kSwizzle128B), idesc,
                 (c > 0 || k > 0) ? 1u : 0u);
        mma_commit(bar_a(buf));
      } else {
        ok = false;
      }
    }
  }
  if (tid == 0 && ok) mma_commit(bar_done);
  ok = __syncthreads_and(ok);
  if (ok) ok = !__any_sync(0xffffffffu, !mbar_wait(bar_done, 0, kWaitNs));
  ok = __syncthreads_and(ok);
  tc_fence_after();

  // Epilogue: TMEM lane r = query row m0 + r, 128 fp32 columns.
  const int r = 32 * warp + lane;
  const int m = m0 + r;
  float* out = o + ((size_t)m * H + h) * kDv;
#pragma unroll 1
  for (int c = 0; c < kDv / 32; ++c) {
    uint32_t v[32];
    if (ok) {
      tmem_ld32(tb + ((uint32_t)(32 * warp) << 16) + 32u * c, v);
      tmem_ld_wait();
    }
    if (m < M) {
      float4* dst = reinterpret_cast<float4*>(out + 32 * c);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        dst[j] = ok ? make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                  __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]))
                    : make_float4(NAN, NAN, NAN, NAN);
    }
  }

  if (!ok && tid == 0)   // no copy may land after exit
    for (int c = 0; c < kOutChunks; ++c) mbar_wait(bar_b(c), 0, kWaitNs);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tb, 128);
  }
}

template <typename K>
cudaError_t set_smem(K kernel, uint32_t bytes, bool& done) {
  if (done) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) done = true;
  return e;
}

}  // namespace

cudaError_t launch_absorb_q(const __nv_bfloat16* q_nope, const __nv_bfloat16* q_rope,
                            const __nv_bfloat16* w_uk, const int32_t* q_pos, const RopeFreqs& f,
                            int M, int H, __nv_bfloat16* q_cat, cudaStream_t st) {
  AbsorbMaps maps;
  if (!encode_tma_2d(&maps.q, true, q_nope, (uint64_t)H * kDn, (uint64_t)M, (uint64_t)H * kDn * 2,
                     64, kTileM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tma_2d(&maps.w, true, w_uk, kDn, (uint64_t)H * kDc, (uint64_t)kDn * 2, 64, 256,
                     CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  static bool attr = false;
  cudaError_t e = set_smem(k_absorb_q, kAbsSmem, attr);
  if (e != cudaSuccess) return e;
  dim3 grid(2, H, (M + kTileM - 1) / kTileM);
  k_absorb_q<<<grid, kAbsThreads, kAbsSmem, st>>>(maps, q_rope, q_pos, f, M, H, q_cat);
  return cudaGetLastError();
}

cudaError_t launch_out_proj_uv(const float* o_lat, const __nv_bfloat16* w_uv, int M, int H,
                               float* o, cudaStream_t st) {
  OutMaps maps;
  if (!encode_tma_2d(&maps.w, true, w_uv, kDv, (uint64_t)H * kDc, (uint64_t)kDv * 2, 64, 64,
                     CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  static bool attr = false;
  cudaError_t e = set_smem(k_out_proj_uv, kOutSmem, attr);
  if (e != cudaSuccess) return e;
  dim3 grid(H, (M + kTileM - 1) / kTileM);
  k_out_proj_uv<<<grid, kOutThreads, kOutSmem, st>>>(maps, o_lat, M, H, o);
  return cudaGetLastError();
}

}  // namespace mla
