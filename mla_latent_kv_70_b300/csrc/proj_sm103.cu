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
  const uint32_t bar_full = s0 + kAbsOffBar, bar_mma = bar_full + 16;   // bar_full: [2] K halves
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kAbsOffBar + 24);

  const int nh = blockIdx.x, h = blockIdx.y, m0 = blockIdx.z * kTileM;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    mbar_init(bar_full, 1);
    mbar_init(bar_full + 8, 1);
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

  // The weights do not depend on the previous kernel: they are requested before waiting
  // for it (programmatic dependent launch); q_cat, which it reads, is written after.
  grid_dep_launch();
  if (tid == 0) {
    prefetch_tmap(&maps.q);
    prefetch_tmap(&maps.w);
    // Two K halves (64 wide each) on their own barriers: the first half's MMAs run
    // while the second half lands.
    for (int j = 0; j < 2; ++j) {
      mbar_arrive_expect_tx(bar_full + 8u * j, kAbsABox + kAbsBBox);
      tma_load_2d(s0 + kAbsOffB + j * kAbsBBox, &maps.w, bar_full + 8u * j, 64 * j, h * kDc + 256 * nh);
    }
  }
  grid_dep_wait();
  if (tid == 0) {
    for (int j = 0; j < 2; ++j)
      tma_load_2d(s0 + j * kAbsABox, &maps.q, bar_full + 8u * j, h * kDn + 64 * j, m0);
    // On expiry no further MMA is issued; the copies are waited for once more before exit.
    const uint32_t idesc = idesc_bf16(kTileM, 256, false, false);
    bool issued = true;
    for (int j = 0; j < 2 && issued; ++j) {
      if (!mbar_wait(bar_full + 8u * j, 0, kWaitNs)) {
        issued = false;
        break;
      }
      tc_fence_after();
      const uint64_t ad = smem_desc(s0 + (uint32_t)j * kAbsABox, 16, 1024, kSwizzle128B);
      const uint64_t bd = smem_desc(s0 + kAbsOffB + (uint32_t)j * kAbsBBox, 16, 1024, kSwizzle128B);
#pragma unroll
      for (int k = 0; k < 4; ++k)   // K = 16 bf16 = 32 B steps inside a swizzle row
        mma_ss(tb, ad + 2u * k, bd + 2u * k, idesc, (j > 0 || k > 0) ? 1u : 0u);
    }
    if (issued) mma_commit(bar_mma);
  }
  __syncwarp();
  const bool ok = !__any_sync(0xffffffffu, !mbar_wait(bar_mma, 0, kWaitNs));
  tc_fence_after();

  // Epilogue: TMEM lane r = query row m0 + r; 256 fp32 columns -> bf16 q~.
  const int r = 32 * warp + lane;
  const int m = m0 + r;
  __nv_bfloat16* out = q_cat + ((size_t)m * H + h) * kRow + 256 * nh;
#pragma unroll 1
  for (int c = 0; c < 8; c += 2) {
    uint32_t v0[32], v1[32];
    if (ok) {   // two loads in flight per wait (~290 cycles each)
      tmem_ld32(tb + ((uint32_t)(32 * warp) << 16) + 32u * c, v0);
      tmem_ld32(tb + ((uint32_t)(32 * warp) << 16) + 32u * (c + 1), v1);
      tmem_ld_wait();
    }
    if (m < M) {
      uint32_t pk[32];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        pk[j] = ok ? f2_to_bf2(__uint_as_float(v0[2 * j]), __uint_as_float(v0[2 * j + 1])) : 0x7FC07FC0u;
        pk[16 + j] = ok ? f2_to_bf2(__uint_as_float(v1[2 * j]), __uint_as_float(v1[2 * j + 1])) : 0x7FC07FC0u;
      }
      uint4* dst = reinterpret_cast<uint4*>(out + 32 * c);
#pragma unroll
      for (int j = 0; j < 8; ++j) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
    }
  }

  // The RoPE slice q_cat[..., 512:576]: rotated at the query position, or copied.  The
  // two CTAs of a head share the rows, in 16-byte pieces (8 per row); every thread loads
  // all of its pieces before it stores any, so the copy costs one memory latency rather
  // than one per piece.
  {
    constexpr int kPieces = kDr * 2 / 16;
    constexpr int kPerThread = (kTileM * kPieces / 2 + kAbsThreads - 1) / kAbsThreads;
    const int rows = min(kTileM, M - m0);
    const int half = (rows * kPieces + 1) / 2;
    const int begin = nh * half, end = min(rows * kPieces, begin + half);
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
            const float2 y = rope_pair(x.x, x.y, pos, freqs.inv_freq[4 * piece + j]);
            w[j] = f2_to_bf2(y.x, y.y);
          }
        }
        reinterpret_cast<uint4*>(q_cat + mh * kRow + kDc)[piece] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }

  if (!ok && tid == 0) {   // no copy may land after exit
    mbar_wait(bar_full, 0, kWaitNs);
    mbar_wait(bar_full + 8, 0, kWaitNs);
  }
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
// All of W_UV[h] (8 chunks of 64 K-rows, two 64-wide N boxes each, read MN-major by the
// MMA) and the fp32 o_lat rows (64-wide K chunks through a 64 KB ring: 2 deep with
// 128-row boxes, 4 deep with 64-row boxes when M <= 64) arrive by TMA.  The CTA's
// threads round each fp32 chunk to bf16 into the 128B-swizzled K-major layout of the A
// operand (double-buffered) while the next chunks land; one thread issues the MMAs.
// With 64-row boxes, A rows 64..127 are never written: the D rows they produce are
// past M and not stored.
// ---------------------------------------------------------------------------
constexpr int kOutThreads = 128;
constexpr int kOutChunks = kDc / 64;                   // 8 K chunks of 64
constexpr uint32_t kOutBBox = 64 * 128;                // 64 K-rows x 64 bf16
constexpr uint32_t kOutBChunk = 2 * kOutBBox;          // N = 128
constexpr uint32_t kOutAChunk = kTileM * 128;          // 128 rows x 64 bf16
constexpr uint32_t kOutA32Chunk = kTileM * 64 * 4;     // 128 rows x 64 fp32
constexpr uint32_t kOutRingBytes = 2 * kOutA32Chunk;   // fp32 ring: 2 x 128 rows or 4 x 64 rows
constexpr int kOutMaxRing = 4;
constexpr uint32_t kOutOffA = kOutChunks * kOutBChunk;
constexpr uint32_t kOutOffA32 = kOutOffA + 2 * kOutAChunk;
constexpr uint32_t kOutOffBar = kOutOffA32 + kOutRingBytes;
constexpr uint32_t kOutSmem = kOutOffBar + 128 + 1024;
static_assert(kOutSmem <= 232448, "shared memory per CTA");

struct OutMaps {
  CUtensorMap w;     // W_UV viewed as [H*512 rows, 128], box 64 x 64 rows, 128B swizzle
  CUtensorMap lat;   // o_lat viewed as [M rows, H*512] fp32, box 64 x 128 rows, no swizzle
};

__global__ void __launch_bounds__(kOutThreads, 1)
k_out_proj_uv(const __grid_constant__ OutMaps maps, int M, int H, int box_rows, float* __restrict__ o) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = align1024(smem_raw);
  const uint32_t s0 = smem_addr(smem);
  const uint32_t bars = s0 + kOutOffBar;
  auto bar_b = [&](int c) { return bars + 8u * (uint32_t)c; };          // [8] W chunk landed
  auto bar_a = [&](int i) { return bars + 64u + 8u * (uint32_t)i; };    // [2] bf16 A buffer consumed
  auto bar_l = [&](int i) { return bars + 80u + 8u * (uint32_t)i; };    // [4] fp32 chunk landed
  const uint32_t bar_done = bars + 112u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOutOffBar + 120);
  const uint32_t a32_bytes = (uint32_t)box_rows * 64u * 4u;
  const int ring = (int)(kOutRingBytes / a32_bytes);   // 2 or 4

  const int h = blockIdx.x, m0 = blockIdx.y * kTileM;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int c = 0; c < kOutChunks; ++c) mbar_init(bar_b(c), 1);
    for (int i = 0; i < 2; ++i) mbar_init(bar_a(i), 1);
    for (int i = 0; i < kOutMaxRing; ++i) mbar_init(bar_l(i), 1);
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

  auto load_lat = [&](int c) {   // fp32 chunk c of the o_lat rows into ring slot c % ring
    const int sl = c % ring;
    mbar_arrive_expect_tx(bar_l(sl), a32_bytes);
    tma_load_2d(s0 + kOutOffA32 + (uint32_t)sl * a32_bytes, &maps.lat, bar_l(sl), h * kDc + 64 * c, m0);
  };
  // W_UV does not depend on the previous kernel: it is requested before waiting for it
  // (programmatic dependent launch); o_lat, which that kernel writes, after.
  grid_dep_launch();
  if (tid == 0) {
    prefetch_tmap(&maps.w);
    prefetch_tmap(&maps.lat);
    for (int c = 0; c < kOutChunks; ++c) {
      mbar_arrive_expect_tx(bar_b(c), kOutBChunk);
      for (int j = 0; j < 2; ++j)
        tma_load_2d(s0 + c * kOutBChunk + j * kOutBBox, &maps.w, bar_b(c), 64 * j, h * kDc + 64 * c);
    }
  }
  grid_dep_wait();
  if (tid == 0)
    for (int c = 0; c < ring; ++c) load_lat(c);

  // Thread (warp, lane) converts rows 2*(4*it + warp) + (lane >> 4), it < box_rows / 8,
  // and the four K values 4*(lane & 15) .. +3 of the current chunk (a half-warp reads one
  // 256-byte fp32 row: no bank conflicts).
  const int sub = lane >> 4, kq = lane & 15;
  const int iters = box_rows / 8;
  bool ok = true;
  for (int c = 0; c < kOutChunks; ++c) {
    const int buf = c & 1, sl = c % ring;
    if (ok) ok = !__any_sync(0xffffffffu, !mbar_wait(bar_l(sl), (uint32_t)(c / ring) & 1u, kWaitNs));
    if (c >= 2 && ok) ok = !__any_sync(0xffffffffu, !mbar_wait(bar_a(buf), (uint32_t)((c - 2) >> 1) & 1u, kWaitNs));
    const uint32_t a32 = s0 + kOutOffA32 + (uint32_t)sl * a32_bytes;
    const uint32_t abase = s0 + kOutOffA + (uint32_t)buf * kOutAChunk;
    if (ok) {
#pragma unroll 4
      for (int it = 0; it < iters; ++it) {
        const int r = 2 * (4 * it + warp) + sub;
        const float4 v = ld_shared_v4(a32 + (uint32_t)r * 256u + (uint32_t)kq * 16u);
        // 128B swizzle: 16-byte chunk j of row r sits at chunk j ^ (r & 7).
        const uint32_t addr = abase + (uint32_t)r * 128u + (uint32_t)((((kq >> 1) ^ (r & 7)) << 4) | ((kq & 1) << 3));
        const uint32_t lo = f2_to_bf2(v.x, v.y), hi = f2_to_bf2(v.z, v.w);
        asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(lo), "r"(hi) : "memory");
      }
    }
    fence_proxy_async_smem();
    ok = __syncthreads_and(ok);   // also tells every thread of an earlier failed wait
    if (tid == 0 && ok) {
      if (c + ring < kOutChunks) load_lat(c + ring);   // fp32 slot `sl` has been converted
      if (mbar_wait(bar_b(c), 0, kWaitNs)) {
        tc_fence_after();
        const uint32_t idesc = idesc_bf16(kTileM, kDv, false, true);
        const uint64_t ad = smem_desc(abase, 16, 1024, kSwizzle128B);
        const uint64_t bd = smem_desc(s0 + c * kOutBChunk, kOutBBox, 1024, kSwizzle128B);
#pragma unroll
        for (int k = 0; k < 4; ++k) mma_ss(tb, ad + 2u * k, bd + 128u * k, idesc, (c > 0 || k > 0) ? 1u : 0u);
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
  for (int c = 0; c < kDv / 32; c += 2) {
    uint32_t v0[32], v1[32];
    if (ok) {
      tmem_ld32(tb + ((uint32_t)(32 * warp) << 16) + 32u * c, v0);
      tmem_ld32(tb + ((uint32_t)(32 * warp) << 16) + 32u * (c + 1), v1);
      tmem_ld_wait();
    }
    if (m < M) {
      float4* d0 = reinterpret_cast<float4*>(out + 32 * c);
      float4* d1 = reinterpret_cast<float4*>(out + 32 * (c + 1));
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        d0[j] = ok ? make_float4(__uint_as_float(v0[4 * j]), __uint_as_float(v0[4 * j + 1]),
                                 __uint_as_float(v0[4 * j + 2]), __uint_as_float(v0[4 * j + 3]))
                   : make_float4(NAN, NAN, NAN, NAN);
        d1[j] = ok ? make_float4(__uint_as_float(v1[4 * j]), __uint_as_float(v1[4 * j + 1]),
                                 __uint_as_float(v1[4 * j + 2]), __uint_as_float(v1[4 * j + 3]))
                   : make_float4(NAN, NAN, NAN, NAN);
      }
    }
  }

  if (tid == 0) {   // no copy may land after exit
    for (int c = 0; c < kOutChunks; ++c) mbar_wait(bar_b(c), 0, kWaitNs);
    for (int c = kOutChunks - ring; c < kOutChunks; ++c) mbar_wait(bar_l(c % ring), (uint32_t)(c / ring) & 1u, kWaitNs);
  }
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
  e = launch_pdl(k_absorb_q, grid, dim3(kAbsThreads), kAbsSmem, st, maps, q_rope, q_pos, f, M, H, q_cat);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_out_proj_uv(const float* o_lat, const __nv_bfloat16* w_uv, int M, int H,
                               float* o, cudaStream_t st) {
  OutMaps maps;
  const int box_rows = M <= 64 ? 64 : kTileM;   // no padding rows in the fp32 ring when M <= 64
  if (!encode_tma_2d(&maps.w, true, w_uv, kDv, (uint64_t)H * kDc, (uint64_t)kDv * 2, 64, 64,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tma_2d(&maps.lat, false, o_lat, (uint64_t)H * kDc, (uint64_t)M, (uint64_t)H * kDc * 4, 64,
                     box_rows, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  static bool attr = false;
  cudaError_t e = set_smem(k_out_proj_uv, kOutSmem, attr);
  if (e != cudaSuccess) return e;
  dim3 grid(H, (M + kTileM - 1) / kTileM);
  e = launch_pdl(k_out_proj_uv, grid, dim3(kOutThreads), kOutSmem, st, maps, M, H, box_rows, o);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mla
