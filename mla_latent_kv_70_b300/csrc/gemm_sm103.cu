// A batched, K-pipelined GEMM on the sm_103a tensor cores, for the pre-fused weights.
//
// Page "MLA의 계산: KV를 펼치지 않고 Attention하기", section "Query·출력 투영과 합치기": the
// projection moved to the query side can be multiplied into the query projection ahead
// of time (U^Q (U^K)^T), and the one moved behind the weighted sum into the output
// projection (U^V W^O, per head, the heads' contributions summed).  Those products, and
// the two products that use them at decode time, are plain GEMMs:
//
//   D[m, n] = sum_k A[m, k] B[n, k]    (per batch z; m < M, n < N, k < K, K % 64 == 0)
//
// A and B come from 2D TMA maps, each stored K-major (k contiguous) or MN-major (m or n
// contiguous), with batch z at a row offset of the map.  A CTA computes one 128 x n_tile
// tile over a range of k (split-K CTAs add their parts with fp32 atomics into a zeroed
// output): one thread streams 64-wide k blocks through a ring of shared-memory stages by
// TMA, one thread issues the MMAs (K = 16 each) into TMEM, and the four warps write the
// tile (TMEM lane = m, so a warp stores 32 consecutive m of one n at a time).  Every wait
// is bounded; a CTA that gives up writes nothing and raises no fault.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "gemm.cuh"
#include "ptx_sm103.cuh"

namespace mla {

namespace {

using namespace ptx;

constexpr int kGemmThreads = 128;
constexpr int kGemmStages = 4;                // the most stages of the k ring
constexpr uint32_t kGemmABytes = 128 * 128;   // 128 m x 64 k, bf16

__device__ __forceinline__ unsigned char* align1024(unsigned char* p) {
  return reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__host__ __device__ constexpr uint32_t tmem_cols_for(uint32_t n) {
  return n <= 32 ? 32u : n <= 64 ? 64u : n <= 128 ? 128u : 256u;
}

__host__ __device__ constexpr uint32_t gemm_b_bytes(int n_tile) { return (uint32_t)n_tile * 128u; }

__host__ __device__ constexpr uint32_t gemm_smem_bytes(int n_tile, int stages) {
  return (uint32_t)stages * (kGemmABytes + gemm_b_bytes(n_tile)) + 128 + 1024;
}

struct GemmMaps {
  CUtensorMap a;   // K-major: box 64 k x 128 m; MN-major: box 64 m x 64 k
  CUtensorMap b;   // K-major: box 64 k x n_tile n; MN-major: box 64 n x 64 k
};

__global__ void __launch_bounds__(kGemmThreads)
k_gemm(const __grid_constant__ GemmMaps maps, GemmShape g, WaitConfig wc) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = align1024(smem_raw);
  const uint32_t s0 = smem_addr(smem);
  const uint32_t b_bytes = gemm_b_bytes(g.n_tile);
  const uint32_t stage_bytes = kGemmABytes + b_bytes;
  const int nst = g.stages;   // stages of the ring (barrier slots exist for kGemmStages)
  const uint32_t bars = s0 + (uint32_t)nst * stage_bytes;
  auto full = [&](int s) { return bars + 8u * (uint32_t)s; };
  auto empty = [&](int s) { return bars + 8u * (uint32_t)(kGemmStages + s); };
  const uint32_t bar_done = bars + 8u * (2 * kGemmStages);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + nst * stage_bytes + 8 * (2 * kGemmStages + 1));
  const uint64_t wait_ns = wc.wait_ns;
  const uint32_t ncols = tmem_cols_for((uint32_t)g.n_tile);

  const int m0 = blockIdx.x * 128, n0 = blockIdx.y * g.n_tile;
  const int z = blockIdx.z / g.k_splits, split = blockIdx.z % g.k_splits;
  const int nkb = g.K / 64;
  const int kb0 = (int)((int64_t)nkb * split / g.k_splits), kb1 = (int)((int64_t)nkb * (split + 1) / g.k_splits);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(bar_done, 1);
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
  grid_dep_launch();
  grid_dep_wait();

  bool ok = true;
  int loaded = 0;
  if (tid == 0) {
    // ---------------- TMA producer ----------------
    prefetch_tmap(&maps.a);
    prefetch_tmap(&maps.b);
    const int ya = z * g.a_batch_rows, yb = z * g.b_batch_rows;
    for (int kb = kb0; kb < kb1; ++kb, ++loaded) {
      const int it = kb - kb0, s = it % nst;
      if (it >= nst && !mbar_wait(empty(s), (uint32_t)(it / nst - 1) & 1u, wait_ns)) {
        ok = false;
        break;
      }
      const uint32_t sa = s0 + (uint32_t)s * stage_bytes, sb = sa + kGemmABytes;
      mbar_arrive_expect_tx(full(s), stage_bytes);
      if (g.a_mn) {
        tma_load_2d(sa, &maps.a, full(s), m0, ya + 64 * kb);
        tma_load_2d(sa + 8192, &maps.a, full(s), m0 + 64, ya + 64 * kb);
      } else {
        tma_load_2d(sa, &maps.a, full(s), 64 * kb, ya + m0);
      }
      if (g.b_mn) {
        for (int j = 0; j < g.n_tile / 64; ++j)
          tma_load_2d(sb + (uint32_t)j * 8192u, &maps.b, full(s), n0 + 64 * j, yb + 64 * kb);
      } else {
        tma_load_2d(sb, &maps.b, full(s), 64 * kb, yb + n0);
      }
    }
  } else if (tid == 32) {
    // ---------------- MMA issuer ----------------
    const uint32_t idesc = idesc_bf16(128, g.n_tile, g.a_mn != 0, g.b_mn != 0);
    for (int kb = kb0; kb < kb1; ++kb) {
      const int it = kb - kb0, s = it % nst;
      if (!mbar_wait(full(s), (uint32_t)(it / nst) & 1u, wait_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sa = s0 + (uint32_t)s * stage_bytes, sb = sa + kGemmABytes;
      const uint64_t ad = g.a_mn ? smem_desc(sa, 8192, 1024, kSwizzle128B) : smem_desc(sa, 16, 1024, kSwizzle128B);
      const uint64_t bd = g.b_mn ? smem_desc(sb, 8192, 1024, kSwizzle128B) : smem_desc(sb, 16, 1024, kSwizzle128B);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        // K = 16: 32 bytes along a K-major row, or 16 rows of 128 bytes when MN-major.
        const uint32_t da = g.a_mn ? 128u * k : 2u * k, db = g.b_mn ? 128u * k : 2u * k;
        mma_ss(tb, ad + da, bd + db, idesc, (it > 0 || k > 0) ? 1u : 0u);
      }
      mma_commit(empty(s));
    }
    mma_commit(bar_done);   // tracks every MMA issued, whether or not the loop finished
  }
  __syncwarp();
  const bool done = !__any_sync(0xffffffffu, !mbar_wait(bar_done, 0, wait_ns));
  ok = __syncthreads_and(ok && done);
  tc_fence_after();

  // Epilogue: warp w holds rows m0 + 32 w + lane; columns are n.  An empty k range (more
  // splits than k blocks) adds nothing.
  const int m = m0 + 32 * warp + lane;
  if (ok && kb1 > kb0) {
#pragma unroll 1
    for (int c0 = 0; c0 < g.n_tile && n0 + c0 < g.N; c0 += 32) {
      uint32_t v[32];
      tmem_ld32(tb + ((uint32_t)(32 * warp) << 16) + (uint32_t)c0, v);
      tmem_ld_wait();
      if (m < g.M) {
        const int64_t base = (int64_t)z * g.ldc_batch + (int64_t)m * g.ldc_m;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int n = n0 + c0 + i;
          if (c0 + i < g.n_tile && n < g.N) {
            const float x = __uint_as_float(v[i]);
            const int64_t off = base + (int64_t)n * g.ldc_n;
            if (g.out_bf16)
              reinterpret_cast<__nv_bfloat16*>(g.c)[off] = __float2bfloat16_rn(x);
            else if (g.k_splits > 1)
              atomicAdd(reinterpret_cast<float*>(g.c) + off, x);
            else
              reinterpret_cast<float*>(g.c)[off] = x;
          }
        }
      }
    }
  }
  if (!ok && g.status && tid == 0) raise_flag(g.status, kFlagTimeout);
  if (tid == 0) {   // no copy may land after exit
    for (int i = max(0, loaded - nst); i < loaded; ++i)
      mbar_wait(full(i % nst), (uint32_t)(i / nst) & 1u, wait_ns);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tb, ncols);
  }
}

// bf16 copy of an fp32 array (n a multiple of 8), round to nearest even.
__global__ void k_f32_to_bf16(const float* __restrict__ x, int64_t n8, __nv_bfloat16* __restrict__ y) {
  grid_dep_launch();
  grid_dep_wait();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(x)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(x)[2 * i + 1];
    reinterpret_cast<uint4*>(y)[i] = make_uint4(f2_to_bf2(a.x, a.y), f2_to_bf2(a.z, a.w), f2_to_bf2(b.x, b.y),
                                                f2_to_bf2(b.z, b.w));
  }
}

}  // namespace

cudaError_t launch_gemm(const GemmOperand& a, const GemmOperand& b, GemmShape g, cudaStream_t st) {
  if (g.K % 64 || g.n_tile % 16 || g.n_tile < 16 || g.n_tile > 256) return cudaErrorInvalidValue;
  if ((b.mn && g.n_tile % 64) || g.k_splits < 1) return cudaErrorInvalidValue;
  if (g.stages == 0) g.stages = kGemmStages;
  if (g.stages < 2 || g.stages > kGemmStages) return cudaErrorInvalidValue;
  GemmMaps maps;
  // A: K-major rows of K (box 64 x 128); MN-major rows of M (box 64 x 64).
  if (!encode_tma_2d(&maps.a, true, a.ptr, a.cols, a.rows, a.row_stride * 2, 64, a.mn ? 64 : 128,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tma_2d(&maps.b, true, b.ptr, b.cols, b.rows, b.row_stride * 2, 64, b.mn ? 64 : (uint32_t)g.n_tile,
                     CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  g.a_mn = a.mn;
  g.b_mn = b.mn;
  static SmemOptIn opt_in;
  cudaError_t e = ensure_dynamic_smem((const void*)k_gemm, (int)gemm_smem_bytes(256, kGemmStages), opt_in);
  if (e != cudaSuccess) return e;
  dim3 grid((g.M + 127) / 128, (g.N + g.n_tile - 1) / g.n_tile, g.batches * g.k_splits);
  e = launch_pdl(k_gemm, grid, dim3(kGemmThreads), gemm_smem_bytes(g.n_tile, g.stages), st, maps, g,
                 wait_config(0));
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_f32_to_bf16(const float* x, int64_t n, __nv_bfloat16* y, cudaStream_t st) {
  if (n % 8) return cudaErrorInvalidValue;
  const int64_t n8 = n / 8;
  const int blocks = (int)std::min<int64_t>((n8 + 255) / 256, 148 * 8);
  if (n8 == 0) return cudaSuccess;
  cudaError_t e = launch_pdl(k_f32_to_bf16, dim3(blocks), dim3(256), 0, st, x, n8, y);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mla
