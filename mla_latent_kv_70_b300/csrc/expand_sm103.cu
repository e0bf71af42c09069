// The per-head keys and values of prefill, built on the sm_103a tensor cores.
//
// Page "Multi-Head Latent Attention (MLA)", section on prefill and decode, and page "MLA의
// 계산: KV를 펼치지 않고 Attention하기", section "계산 재배치의 효과와 한계": prefill keeps the
// order that expands the cache into per-head keys and values,
//
//   K_h[t] = c_t W_UK[h],   V_h[t] = c_t W_UV[h]     (c_t: the 512 latent values of row t),
//
// stored bf16 as [rows][H][128].  One unit of work is 128 consecutive rows and one head:
//
//   D [128 x 256] = C [128 x 512] . [W_UK[h] | W_UV[h]] [512 x 256]
//
// with the row index on the TMEM lanes, so that each thread of the epilogue holds 128
// consecutive output values of one row.  Persistent CTAs (one per SM) take contiguous
// ranges of units ordered (row block, head): the row block C (128 KB, eight 64-wide k
// boxes) stays in shared memory across the heads of that block, and the weights stream
// through a ring of 32-wide k slices (4 boxes of 64 n x 32 k, MN-major, 16 KB).  TMEM holds
// two 256-column fp32 accumulators: the epilogue of one unit runs while the MMAs of the
// next do.  The epilogue rounds to bf16 and stores 64-column chunks by TMA through one
// 16 KB staging slot.  Warp 0 streams by TMA, warp 1 issues the MMAs, warps 2-5 (one TMEM
// lane quarter each) run the epilogue.  Every wait is bounded; on expiry the CTA records
// MLA_ERR_TIMEOUT, drains and exits.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "ptx_sm103.cuh"

namespace mla {

namespace {

using namespace ptx;

constexpr int kXThreads = 192;
constexpr int kXEpiWarp0 = 2;                    // warps 2..5
constexpr int kXSliceK = 32;                     // k per ring slice
constexpr int kXSlices = kDc / kXSliceK;         // 16 per unit
constexpr int kXStages = 5;
constexpr uint32_t kXABox = 128 * 128;           // 128 rows x 64 bf16
constexpr uint32_t kXBBox = kXSliceK * 128;      // 32 k rows x 64 bf16
constexpr uint32_t kXBStage = 4 * kXBBox;        // n = 256
constexpr uint32_t kXOffA = 0;
constexpr uint32_t kXOffB = kXOffA + 8 * kXABox;
constexpr uint32_t kXOffStg = kXOffB + kXStages * kXBStage;
constexpr uint32_t kXStgBytes = 128 * 128;       // 128 rows x 64 bf16
constexpr uint32_t kXOffBars = kXOffStg + kXStgBytes;
constexpr uint32_t kXSmem = kXOffBars + 256 + 1024;
static_assert(kXSmem <= 232448, "shared memory per CTA");
static_assert(kXOffB % 1024 == 0 && kXOffStg % 1024 == 0 && kXBBox % 1024 == 0, "128B-swizzled tiles");

enum XBar {
  kXAFull = 0,                        // row block landed
  kXAFree,                            // MMAs of the row block done
  kXBFull,                            // [5] weight slice landed
  kXBEmpty = kXBFull + kXStages,      // [5] its MMAs done
  kXAccFull = kXBEmpty + kXStages,    // [2] accumulator complete
  kXAccEmpty = kXAccFull + 2,         // [2] accumulator read (128 threads)
  kXDrain = kXAccEmpty + 2,
  kXNumBars
};
static_assert(kXNumBars * 8 + 8 <= 256, "barrier area");

struct ExpandMaps {
  CUtensorMap c;       // cache rows [rows, 576], box 64 x 128 (k < 512 used)
  CUtensorMap w_uk;    // [H*512, 128], box 64 n x 32 k
  CUtensorMap w_uv;
  CUtensorMap k_out;   // [rows, H*128] bf16, box 64 x 128
  CUtensorMap v_out;
};

struct ExpandParams {
  int H;
  int64_t units;       // row blocks x H
  int32_t* status;
};

__global__ void __launch_bounds__(kXThreads, 1)
k_expand_kv(const __grid_constant__ ExpandMaps maps, const ExpandParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s0 = smem_addr(smem);
  auto bar = [&](int i) { return s0 + kXOffBars + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kXOffBars + 8 * kXNumBars);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t u0 = p.units * blockIdx.x / gridDim.x, u1 = p.units * (blockIdx.x + 1) / gridDim.x;

  if (tid == 0) {
    mbar_init(bar(kXAFull), 1);
    mbar_init(bar(kXAFree), 1);
    for (int s = 0; s < kXStages; ++s) {
      mbar_init(bar(kXBFull + s), 1);
      mbar_init(bar(kXBEmpty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kXAccFull + b), 1);
      mbar_init(bar(kXAccEmpty + b), 128);
    }
    mbar_init(bar(kXDrain), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = *tmem_slot;
  grid_dep_launch();
  grid_dep_wait();

  bool ok = true;
  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      prefetch_tmap(&maps.c);
      prefetch_tmap(&maps.w_uk);
      prefetch_tmap(&maps.w_uv);
      int64_t blk = -1;
      int a_loads = 0;
      uint32_t g = 0;   // slices issued
      int64_t rb = u0 / p.H;   // unit u = (row block rb, head h), counted without divisions
      int h = (int)(u0 % p.H);
      for (int64_t u = u0; u < u1 && ok; ++u, ++h) {
        if (h == p.H) {
          h = 0;
          ++rb;
        }
        if (rb != blk) {   // a new row block, once the MMAs of the previous one are done
          if (a_loads > 0 && !mbar_wait(bar(kXAFree), (uint32_t)(a_loads - 1) & 1u, kDefaultWaitNs)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(kXAFull), 8 * kXABox);
          for (int kb = 0; kb < 8; ++kb)
            tma_load_2d(s0 + kXOffA + (uint32_t)kb * kXABox, &maps.c, bar(kXAFull), 64 * kb, (int)(rb * 128));
          blk = rb;
          ++a_loads;
        }
        for (int s = 0; s < kXSlices; ++s, ++g) {
          const uint32_t st = g % kXStages;
          if (g >= (uint32_t)kXStages &&
              !mbar_wait(bar(kXBEmpty + st), (g / kXStages - 1) & 1u, kDefaultWaitNs)) {
            ok = false;
            break;
          }
          const uint32_t sb = s0 + kXOffB + st * kXBStage;
          const int y = h * kDc + kXSliceK * s;
          mbar_arrive_expect_tx(bar(kXBFull + st), kXBStage);
          tma_load_2d(sb, &maps.w_uk, bar(kXBFull + st), 0, y);
          tma_load_2d(sb + kXBBox, &maps.w_uk, bar(kXBFull + st), 64, y);
          tma_load_2d(sb + 2 * kXBBox, &maps.w_uv, bar(kXBFull + st), 0, y);
          tma_load_2d(sb + 3 * kXBBox, &maps.w_uv, bar(kXBFull + st), 64, y);
        }
      }
      // No copy may land after exit.
      for (uint32_t i = g > (uint32_t)kXStages ? g - kXStages : 0u; i < g; ++i)
        mbar_wait(bar(kXBFull + i % kXStages), (i / kXStages) & 1u, kDefaultWaitNs);
      if (a_loads > 0) mbar_wait(bar(kXAFull), (uint32_t)(a_loads - 1) & 1u, kDefaultWaitNs);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, 256, false, true);
      const uint64_t a_desc = smem_desc(s0 + kXOffA, 16, 1024, kSwizzle128B);
      int64_t blk = -1;
      int a_loads = 0;
      uint32_t g = 0;
      int i = 0;   // units of this CTA so far
      int64_t rb = u0 / p.H;
      int h = (int)(u0 % p.H);
      for (int64_t u = u0; u < u1 && ok; ++u, ++i, ++h) {
        if (h == p.H) {
          h = 0;
          ++rb;
        }
        if (rb != blk) {
          if (!mbar_wait(bar(kXAFull), (uint32_t)a_loads & 1u, kDefaultWaitNs)) {
            ok = false;
            break;
          }
          blk = rb;
          ++a_loads;
        }
        const int ab = i & 1;
        if (i >= 2 && !mbar_wait(bar(kXAccEmpty + ab), (uint32_t)((i >> 1) - 1) & 1u, kDefaultWaitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tb + 256u * (uint32_t)ab;
        for (int s = 0; s < kXSlices; ++s, ++g) {
          const uint32_t st = g % kXStages;
          if (!mbar_wait(bar(kXBFull + st), (g / kXStages) & 1u, kDefaultWaitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t b_desc = smem_desc(s0 + kXOffB + st * kXBStage, kXBBox, 1024, kSwizzle128B);
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            // A: box s / 2, 64 bytes per 32-wide half, 32 bytes per K = 16; B: 16 k rows
            // of 128 bytes per K = 16.
            const uint32_t a_off = ((uint32_t)(s >> 1) * kXABox + (uint32_t)(s & 1) * 64u + 32u * kk) >> 4;
            mma_ss(d, a_desc + a_off, b_desc + ((2048u * kk) >> 4), idesc, (s > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(bar(kXBEmpty + st));
        }
        if (!ok) break;
        mma_commit(bar(kXAccFull + ab));
        if (u + 1 < u1 && h + 1 == p.H) mma_commit(bar(kXAFree));   // the next unit starts a row block
      }
      mma_commit(bar(kXDrain));   // tracks every MMA issued
      mbar_wait(bar(kXDrain), 0, kDefaultWaitNs);
    }
  } else {
    // ---------------- epilogue: warps 2-5, TMEM lane quarter warp % 4 ----------------
    const int quarter = warp & 3;
    const int r = 32 * quarter + lane;   // row within the block
    const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
    const bool leader = warp == kXEpiWarp0 && lane == 0;
    const uint32_t stg = s0 + kXOffStg + (uint32_t)r * 128u;
    int i = 0;
    int64_t rb = u0 / p.H;
    int h = (int)(u0 % p.H);
    for (int64_t u = u0; u < u1; ++u, ++i, ++h) {
      if (h == p.H) {
        h = 0;
        ++rb;
      }
      const int ab = i & 1;
      const bool got = !__any_sync(0xffffffffu, !mbar_wait(bar(kXAccFull + ab), (uint32_t)(i >> 1) & 1u,
                                                            kDefaultWaitNs));
      if (!named_bar_and(1, 128, got)) {   // the four warps give up together
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {   // columns [64 c, 64 c + 64): K_h halves, then V_h halves
        uint32_t v[64];
        tmem_ld32(tb + lane_off + 256u * (uint32_t)ab + 64u * (uint32_t)c, *reinterpret_cast<uint32_t(*)[32]>(v));
        tmem_ld32(tb + lane_off + 256u * (uint32_t)ab + 64u * (uint32_t)c + 32u,
                  *reinterpret_cast<uint32_t(*)[32]>(v + 32));
        tmem_ld_wait();
        if (c == 3) {
          tc_fence_before();
          mbar_arrive(bar(kXAccEmpty + ab));
        }
        if (leader) bulk_wait_group_read0();   // the previous chunk has left the slot
        named_bar_sync(1, 128);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          st_shared_u4(stg + (uint32_t)((q ^ (r & 7)) * 16),
                       f2_to_bf2(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
                       f2_to_bf2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                       f2_to_bf2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                       f2_to_bf2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (leader) {
          tma_store_2d(c < 2 ? &maps.k_out : &maps.v_out, h * 128 + 64 * (c & 1), (int)(rb * 128),
                       s0 + kXOffStg);
          bulk_commit_group();
        }
      }
    }
    if (leader) bulk_wait_group_read0();   // the staging outlives its reads; the writes finish with the grid
  }

  if (!ok) raise_flag(p.status, kFlagTimeout);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tb, 512);
  }
}

}  // namespace

cudaError_t launch_expand_kv(const __nv_bfloat16* kv, uint64_t rows, const __nv_bfloat16* w_uk,
                             const __nv_bfloat16* w_uv, int H, __nv_bfloat16* k_exp, __nv_bfloat16* v_exp,
                             int32_t* status, cudaStream_t st) {
  if (rows == 0 || H < 1) return cudaErrorInvalidValue;
  ExpandMaps maps;
  if (!encode_tma_2d(&maps.c, true, kv, kRow, rows, (uint64_t)kRow * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tma_2d(&maps.w_uk, true, w_uk, kDn, (uint64_t)H * kDc, (uint64_t)kDn * 2, 64, kXSliceK,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tma_2d(&maps.w_uv, true, w_uv, kDv, (uint64_t)H * kDc, (uint64_t)kDv * 2, 64, kXSliceK,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tma_2d(&maps.k_out, true, k_exp, (uint64_t)H * kDn, rows, (uint64_t)H * kDn * 2, 64, 128,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tma_2d(&maps.v_out, true, v_exp, (uint64_t)H * kDv, rows, (uint64_t)H * kDv * 2, 64, 128,
                     CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const int64_t units = (int64_t)((rows + 127) / 128) * H;
  const int sms = device_sm_count() > 0 ? device_sm_count() : 148;
  ExpandParams p{H, units, status};
  static SmemOptIn opt_in;
  cudaError_t e = ensure_dynamic_smem((const void*)k_expand_kv, (int)kXSmem, opt_in);
  if (e != cudaSuccess) return e;
  const int grid = (int)std::min<int64_t>(units, sms);
  e = launch_pdl(k_expand_kv, dim3(grid), dim3(kXThreads), kXSmem, st, maps, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mla
