// Prefill and chunked prefill in the expanded order, on the sm_103a tensor cores.
//
// Page "Multi-Head Latent Attention (MLA)", section on prefill and decode: prefill works on
// many query tokens at once and is bound by compute, so it may keep the order that builds
// the per-head keys and values; page "MLA의 계산: KV를 펼치지 않고 Attention하기", section
// "계산 재배치의 효과와 한계": the absorbed order pays d_c-wide dot products per key, which
// pays off only when reading the cache dominates (decode).  Here:
//   K_h = C W_UK[h], V_h = C W_UV[h]  (the batched GEMM of gemm_sm103.cu), then for each
//   head, causal attention of the T_q query tokens (the last T_q of T_kv positions) over
//   [K_h | k^R] with [q_nope | q^R], one scale, and V_h mixed by the weights.
//
// k_prefill_attn: one CTA per (sequence, head, 256 query tokens), as two tiles A and B of
// 128 queries that share every key tile.  Warps 0-3 run the online softmax of tile A and
// warps 4-7 that of tile B, one query row per thread (TMEM lane = row); warp 8 streams the
// key tiles of 64 positions by TMA, [K_h | k^R] (24 KB) into a ring of two stages and V_h
// (16 KB) into a ring of three; warp 9 issues the MMAs, per key tile j:
//   S_A(j), S_B(j) [128 x 64] = Q_t [128 x 192] . K(j)^T   (12 MMAs each, S double-buffered)
//   O_A, O_B [128 x 128]   += P_t(j-1) [128 x 64] . V(j-1)  (4 MMAs each)
// so the tensor core works on one tile's products while the other tile's softmax runs
// (two query tiles in flight hide the softmax; one tile left the tensor core idle while
// its own softmax ran).  The key half of a stage is released as soon as both score
// products are done, the value half once both aggregations are.  The running maximum is
// raised lazily (O is rescaled only when a row's maximum grows by more than 2^8), as in
// the latent decode.  Key tiles past a tile's last query position are neither loaded nor
// multiplied.  Every wait is bounded; on expiry the CTA records MLA_ERR_TIMEOUT, drains
// and exits.
#include <cuda.h>

#include "common.cuh"
#include "ptx_sm103.cuh"

namespace mla {

namespace {

using namespace ptx;

constexpr int kPQ = 128;                  // query rows per tile (TMEM lanes)
constexpr int kPTiles = 2;                // query tiles per CTA
constexpr int kPKeys = 64;                // keys per tile
constexpr int kPKStages = 2;              // [K_h | k^R] ring
constexpr int kPVStages = 3;              // V_h ring
constexpr int kPMmaWarp = 9, kPTmaWarp = 8;
constexpr int kPThreads = 320;
constexpr uint32_t kPBox = 64 * 128;      // 64 rows x 64 bf16
constexpr uint32_t kPQBox = 128 * 128;    // 128 rows x 64 bf16
constexpr uint32_t kPQBytes = 3 * kPQBox; // q_nope (2 boxes) + q^R (1 box)
constexpr uint32_t kPKBytes = 3 * kPBox;  // K_h (2 boxes) + k^R (1 box)
constexpr uint32_t kPVBytes = 2 * kPBox;
constexpr uint32_t kPOffQ = 0;
constexpr uint32_t kPOffK = kPOffQ + kPTiles * kPQBytes;
constexpr uint32_t kPOffV = kPOffK + kPKStages * kPKBytes;
constexpr uint32_t kPOffP = kPOffV + kPVStages * kPVBytes;
constexpr uint32_t kPOffBars = kPOffP + kPTiles * kPQ * 128;
constexpr uint32_t kPSmem = kPOffBars + 256 + 1024;
static_assert(kPSmem <= 232448, "shared memory per CTA");
static_assert(kPOffK % 1024 == 0 && kPOffV % 1024 == 0 && kPOffP % 1024 == 0, "128B-swizzled tiles");

// TMEM: O of tile t at 128 t; S of tile t at 256 + 128 t (two buffers of 64 columns).
constexpr uint32_t kPTmemO = 0, kPTmemS = 256;
constexpr float kPRescale = 8.0f;

enum PBar {
  kPQFullB = 0,
  kPKFullB,                             // [2] key half of a stage landed
  kPKEmptyB = kPKFullB + kPKStages,     // [2] both score products of the stage done
  kPVFullB = kPKEmptyB + kPKStages,     // [3] value half landed
  kPVEmptyB = kPVFullB + kPVStages,     // [3] both aggregations of the stage done
  kPSFullB = kPVEmptyB + kPVStages,     // [tile][2] S buffer ready
  kPSFreeB = kPSFullB + 2 * kPTiles,    // [tile][2] S buffer read (4 warps)
  kPPFullB = kPSFreeB + 2 * kPTiles,    // [tile] P written (128 threads)
  kPPvDoneB = kPPFullB + kPTiles,       // [tile] PV(j) done: P free, O stable
  kPDrainB = kPPvDoneB + kPTiles,
  kPNumBars
};
static_assert(kPNumBars * 8 + 16 <= 256, "barrier area");

struct PrefillMaps {
  CUtensorMap q_nope;   // [B*T_q, H*128], box 64 x 128
  CUtensorMap q_rope;   // [B*T_q, H*64], box 64 x 128
  CUtensorMap k_exp;    // [rows, H*128], box 64 x 64
  CUtensorMap k_rope;   // cache rows [rows, 576], box 64 x 64 (columns 512..575)
  CUtensorMap v_exp;    // [rows, H*128], box 64 x 64
};

struct PrefillParams {
  int B, T_q, T_kv, H;
  int64_t kv_seq_stride;
  float scale_log2;
  float* o;      // [B, T_q, H, 128]
  float* lse;    // [B, T_q, H]
  int32_t* status;
};

__device__ __forceinline__ bool pwarp_wait(uint32_t bar, uint32_t parity) {
  return !__any_sync(0xffffffffu, !mbar_wait(bar, parity, kDefaultWaitNs));
}

// Key tiles that query tile t of the CTA starting at query q0 reads (0 if it holds no query).
__device__ __forceinline__ int tile_keys(const PrefillParams& p, int q0, int t) {
  const int first = q0 + kPQ * t;
  if (first >= p.T_q) return 0;
  const int last_q = min(first + kPQ - 1, p.T_q - 1);
  const int last_pos = min(p.T_kv - 1, p.T_kv - p.T_q + last_q);
  return last_pos < 0 ? 0 : last_pos / kPKeys + 1;
}

__global__ void __launch_bounds__(kPThreads, 1)
k_prefill_attn(const __grid_constant__ PrefillMaps maps, const PrefillParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s0 = smem_addr(smem);
  const uint32_t bars = s0 + kPOffBars;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kPOffBars + 8 * kPNumBars);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q0 = blockIdx.x * (kPTiles * kPQ), h = blockIdx.y, b = blockIdx.z;
  const int offset = p.T_kv - p.T_q;                 // query i sits at position offset + i
  int ntt[kPTiles];
#pragma unroll
  for (int t = 0; t < kPTiles; ++t) ntt[t] = tile_keys(p, q0, t);
  const int nt = max(ntt[0], ntt[1]);                // key tiles the CTA reads
  const int ntiles_q = ntt[1] > 0 ? 2 : 1;           // query tiles holding a query
  const int64_t krow0 = (int64_t)b * p.kv_seq_stride;

  if (tid == 0) {
    mbar_init(bar(kPQFullB), 1);
    for (int i = 0; i < kPKStages; ++i) {
      mbar_init(bar(kPKFullB + i), 1);
      mbar_init(bar(kPKEmptyB + i), 1);
    }
    for (int i = 0; i < kPVStages; ++i) {
      mbar_init(bar(kPVFullB + i), 1);
      mbar_init(bar(kPVEmptyB + i), 1);
    }
    for (int t = 0; t < kPTiles; ++t) {
      for (int i = 0; i < 2; ++i) {
        mbar_init(bar(kPSFullB + 2 * t + i), 1);
        mbar_init(bar(kPSFreeB + 2 * t + i), 4);
      }
      mbar_init(bar(kPPFullB + t), 128);
      mbar_init(bar(kPPvDoneB + t), 1);
    }
    mbar_init(bar(kPDrainB), 1);
    fence_mbar_init();
  }
  if (warp == kPMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = *tmem_slot;
  grid_dep_launch();
  grid_dep_wait();

  bool aborted = false;
  if (warp == kPTmaWarp) {
    // ---------------- TMA producer ----------------
    // Per key tile j: the key half into K stage j % 2 (free once S_A(j-2), S_B(j-2) are
    // done) and the value half into V stage j % 3 (free once PV_A(j-3), PV_B(j-3) are).
    if (lane == 0) {
      prefetch_tmap(&maps.q_nope);
      prefetch_tmap(&maps.k_exp);
      prefetch_tmap(&maps.v_exp);
      mbar_arrive_expect_tx(bar(kPQFullB), (uint32_t)ntiles_q * kPQBytes);
      for (int t = 0; t < ntiles_q; ++t) {
        const int qy = b * p.T_q + q0 + kPQ * t;
        const uint32_t qs = s0 + kPOffQ + (uint32_t)t * kPQBytes;
        tma_load_2d(qs, &maps.q_nope, bar(kPQFullB), h * 128, qy);
        tma_load_2d(qs + kPQBox, &maps.q_nope, bar(kPQFullB), h * 128 + 64, qy);
        tma_load_2d(qs + 2 * kPQBox, &maps.q_rope, bar(kPQFullB), h * 64, qy);
      }
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < nt; ++j) {
        const int ks = j % kPKStages, vs = j % kPVStages;
        const int y = (int)(krow0 + (int64_t)j * kPKeys);
        if (j >= kPKStages &&
            !mbar_wait(bar(kPKEmptyB + ks), (uint32_t)(j / kPKStages - 1) & 1u, kDefaultWaitNs)) {
          aborted = true;
          break;
        }
        const uint32_t kst = s0 + kPOffK + (uint32_t)ks * kPKBytes;
        mbar_arrive_expect_tx(bar(kPKFullB + ks), kPKBytes);
        tma_load_2d(kst, &maps.k_exp, bar(kPKFullB + ks), h * 128, y);
        tma_load_2d(kst + kPBox, &maps.k_exp, bar(kPKFullB + ks), h * 128 + 64, y);
        tma_load_2d(kst + 2 * kPBox, &maps.k_rope, bar(kPKFullB + ks), kDc, y);
        ++k_issued;
        if (j >= kPVStages &&
            !mbar_wait(bar(kPVEmptyB + vs), (uint32_t)(j / kPVStages - 1) & 1u, kDefaultWaitNs)) {
          aborted = true;
          break;
        }
        const uint32_t vst = s0 + kPOffV + (uint32_t)vs * kPVBytes;
        mbar_arrive_expect_tx(bar(kPVFullB + vs), kPVBytes);
        tma_load_2d(vst, &maps.v_exp, bar(kPVFullB + vs), h * 128, y);
        tma_load_2d(vst + kPBox, &maps.v_exp, bar(kPVFullB + vs), h * 128 + 64, y);
        ++v_issued;
      }
      // No copy may land after exit.
      for (int j = max(0, k_issued - kPKStages); j < k_issued; ++j)
        mbar_wait(bar(kPKFullB + j % kPKStages), (uint32_t)(j / kPKStages) & 1u, kDefaultWaitNs);
      for (int j = max(0, v_issued - kPVStages); j < v_issued; ++j)
        mbar_wait(bar(kPVFullB + j % kPVStages), (uint32_t)(j / kPVStages) & 1u, kDefaultWaitNs);
      mbar_wait(bar(kPQFullB), 0, kDefaultWaitNs);
    }
  } else if (warp == kPMmaWarp) {
    // ---------------- MMA issuer ----------------
    // Round j: S_A(j), S_B(j) (each once its tile's softmax has read buffer j & 1 at tile
    // j-2), the key stage released, then PV_A(j-1), PV_B(j-1) (each once that tile's P is
    // written) and the value stage released.  A tile past its last key tile sits out.
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16(128, kPKeys, false, false);
      const uint32_t id_o = idesc_bf16(128, 128, false, true);
      auto pv = [&](int i) {   // O_t += P_t(i) V(i) for the tiles that read key tile i
        if (!mbar_wait(bar(kPVFullB + i % kPVStages), (uint32_t)(i / kPVStages) & 1u, kDefaultWaitNs)) return false;
        const uint64_t vd = smem_desc(s0 + kPOffV + (uint32_t)(i % kPVStages) * kPVBytes, kPBox, 1024, kSwizzle128B);
        for (int t = 0; t < kPTiles; ++t) {
          if (i >= ntt[t]) continue;
          if (!mbar_wait(bar(kPPFullB + t), (uint32_t)i & 1u, kDefaultWaitNs)) return false;
          tc_fence_after();
          const uint64_t pd = smem_desc(s0 + kPOffP + (uint32_t)t * (kPQ * 128), 16, 1024, kSwizzle128B);
#pragma unroll
          for (int k = 0; k < kPKeys / 16; ++k)
            mma_ss(tb + kPTmemO + 128u * t, pd + 2u * k, vd + 128u * k, id_o, (i > 0 || k > 0) ? 1u : 0u);
          mma_commit(bar(kPPvDoneB + t));
        }
        mma_commit(bar(kPVEmptyB + i % kPVStages));
        return true;
      };
      if (!mbar_wait(bar(kPQFullB), 0, kDefaultWaitNs)) aborted = true;
      for (int j = 0; j < nt && !aborted; ++j) {
        const int ks = j % kPKStages;
        if (!mbar_wait(bar(kPKFullB + ks), (uint32_t)(j / kPKStages) & 1u, kDefaultWaitNs)) {
          aborted = true;
          break;
        }
        const uint32_t kst = s0 + kPOffK + (uint32_t)ks * kPKBytes;
        for (int t = 0; t < kPTiles && !aborted; ++t) {
          if (j >= ntt[t]) continue;
          if (j >= 2 && !mbar_wait(bar(kPSFreeB + 2 * t + (j & 1)), (uint32_t)((j - 2) >> 1) & 1u, kDefaultWaitNs)) {
            aborted = true;
            break;
          }
          tc_fence_after();
          const uint32_t d = tb + kPTmemS + 128u * t + 64u * (uint32_t)(j & 1);
          const uint32_t qs = s0 + kPOffQ + (uint32_t)t * kPQBytes;
#pragma unroll
          for (int bx = 0; bx < 3; ++bx) {
            const uint64_t qd = smem_desc(qs + (uint32_t)bx * kPQBox, 16, 1024, kSwizzle128B);
            const uint64_t kd = smem_desc(kst + (uint32_t)bx * kPBox, 16, 1024, kSwizzle128B);
#pragma unroll
            for (int k = 0; k < 4; ++k) mma_ss(d, qd + 2u * k, kd + 2u * k, id_s, (bx > 0 || k > 0) ? 1u : 0u);
          }
          mma_commit(bar(kPSFullB + 2 * t + (j & 1)));
        }
        if (aborted) break;
        mma_commit(bar(kPKEmptyB + ks));
        if (j >= 1 && !pv(j - 1)) {
          aborted = true;
          break;
        }
      }
      if (!aborted && nt > 0 && !pv(nt - 1)) aborted = true;
      mma_commit(bar(kPDrainB));
      mbar_wait(bar(kPDrainB), 0, kDefaultWaitNs);
    }
  } else {
    // ---------------- softmax warps: one query row per thread ----------------
    const int t = warp >> 2;                      // query tile of this warp
    const int r = 32 * (warp & 3) + lane;         // TMEM lane == query row of the tile
    const int qi = q0 + kPQ * t + r;              // query index in the sequence
    const int qpos = offset + qi;                 // its position
    const int my_nt = ntt[t];
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t s_tm = tb + kPTmemS + 128u * t, o_tm = tb + kPTmemO + 128u * t;
    // The rows of a key tile past the sequence end are cleared by the first tile to read it.
    const int clear_tile = (t == 0 || ntt[0] == 0) ? 0 : ntt[0];
    float m_ref = -INFINITY, l = 0.f;
    for (int j = 0; j < my_nt; ++j) {
      if (!pwarp_wait(bar(kPSFullB + 2 * t + (j & 1)), (uint32_t)(j >> 1) & 1u)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      float x[64];
      {
        const uint32_t ts = s_tm + lane_off + 64u * (uint32_t)(j & 1);
        tmem_ld32f<0>(ts, x);
        tmem_ld32f<32>(ts + 32u, x);
        tmem_ld_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kPSFreeB + 2 * t + (j & 1)));
      // Causal mask and the sequence end (rows of later positions may hold anything).
      const int k0 = j * kPKeys;
      const int vis = min(kPKeys, min(qpos, p.T_kv - 1) - k0 + 1);   // readable keys of this row
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < kPKeys; ++c) {
        if (c >= vis) x[c] = -INFINITY;
        mx = fmaxf(mx, x[c]);
      }
      mx *= p.scale_log2;
      const bool grow = mx > m_ref + kPRescale;
      const float m_new = grow ? mx : m_ref;
      if (grow) l *= ex2_approx(m_ref - m_new);   // 0 when m_ref = -inf (l is 0 then)
      const float alpha = grow ? ex2_approx(m_ref - m_new) : 1.f;
      m_ref = m_new;
      const float bias = (m_new == -INFINITY) ? 0.f : -m_new;
      uint32_t pw[32];
      float ps = 0.f;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float a = ex2_approx(fmaf(x[2 * c], p.scale_log2, bias));
        const float e = ex2_approx(fmaf(x[2 * c + 1], p.scale_log2, bias));
        ps += a + e;
        pw[c] = f2_to_bf2(a, e);
      }
      l += ps;
      // This tile's P buffer is free, and its O stable, once its PV(j-1) is done.
      if (j >= 1 && !pwarp_wait(bar(kPPvDoneB + t), (uint32_t)(j - 1) & 1u)) {
        aborted = true;
        break;
      }
      {
        const uint32_t prow = s0 + kPOffP + (uint32_t)t * (kPQ * 128) + (uint32_t)r * 128u;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          st_shared_u4(prow + (uint32_t)((c ^ (r & 7)) << 4), pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
      }
      if (__any_sync(0xffffffffu, grow && j > 0)) {   // rescale this warp's rows of O
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          const uint32_t ta = o_tm + lane_off + 32u * c;
          tmem_ld32(ta, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(ta, o);
        }
        tmem_st_wait();
        tc_fence_before();
      }
      // Rows of the key tile past the sequence end may hold anything (even NaN): clear
      // them in the V tile so that their zero weights add exactly zero.  Tile A clears the
      // key tiles it reads; tile B those past tile A's range (its aggregation of a tile
      // is issued after tile A's).
      const int rows_valid = min(kPKeys, p.T_kv - k0);
      if (rows_valid < kPKeys && j >= clear_tile) {
        if (!pwarp_wait(bar(kPVFullB + j % kPVStages), (uint32_t)(j / kPVStages) & 1u)) {
          aborted = true;
          break;
        }
        const uint32_t vt = s0 + kPOffV + (uint32_t)(j % kPVStages) * kPVBytes;
        for (int idx = tid - 128 * t; idx < (kPKeys - rows_valid) * 16; idx += 128) {
          const int row = rows_valid + idx / 16, c = idx % 16;   // 2 boxes x 8 chunks per row
          st_shared_v4_zero(vt + (uint32_t)(c >> 3) * kPBox + (uint32_t)row * 128u + (uint32_t)(c & 7) * 16u);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(kPPFullB + t));
    }
    // Epilogue: O / l and the LSE of each query row.
    if (!aborted && my_nt > 0 && !pwarp_wait(bar(kPPvDoneB + t), (uint32_t)(my_nt - 1) & 1u)) aborted = true;
    tc_fence_after();
    const bool have = !aborted && l > 0.f;
    const float inv = have ? 1.f / l : 0.f;
    const bool row_ok = qi < p.T_q;
    float* out = p.o + (((int64_t)b * p.T_q + qi) * p.H + h) * 128;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t o[32];
      if (!aborted && my_nt > 0) {
        tmem_ld32(o_tm + lane_off + 32u * c, o);
        tmem_ld_wait();
      }
      if (row_ok) {
#pragma unroll
        for (int v = 0; v < 8; ++v)
          reinterpret_cast<float4*>(out + 32 * c)[v] =
              have ? make_float4(__uint_as_float(o[4 * v]) * inv, __uint_as_float(o[4 * v + 1]) * inv,
                                 __uint_as_float(o[4 * v + 2]) * inv, __uint_as_float(o[4 * v + 3]) * inv)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    if (row_ok) p.lse[((int64_t)b * p.T_q + qi) * p.H + h] = have ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
  }

  if (aborted) raise_flag(p.status, kFlagTimeout);
  tc_fence_before();
  __syncthreads();
  if (warp == kPMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tb, 512);
  }
}

}  // namespace

cudaError_t launch_prefill_attn(const __nv_bfloat16* q_nope, const __nv_bfloat16* q_rope,
                                const __nv_bfloat16* kv, int64_t kv_seq_stride, const __nv_bfloat16* k_exp,
                                const __nv_bfloat16* v_exp, int B, int T_q, int T_kv, int H, float scale,
                                float* o, float* lse, int32_t* status, cudaStream_t st) {
  PrefillMaps maps;
  const uint64_t qrows = (uint64_t)B * T_q, krows = (uint64_t)B * kv_seq_stride;
  if (!encode_tma_2d(&maps.q_nope, true, q_nope, (uint64_t)H * kDn, qrows, (uint64_t)H * kDn * 2, 64, kPQ,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tma_2d(&maps.q_rope, true, q_rope, (uint64_t)H * kDr, qrows, (uint64_t)H * kDr * 2, 64, kPQ,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tma_2d(&maps.k_exp, true, k_exp, (uint64_t)H * kDn, krows, (uint64_t)H * kDn * 2, 64, kPKeys,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tma_2d(&maps.k_rope, true, kv, kRow, krows, (uint64_t)kRow * 2, 64, kPKeys,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tma_2d(&maps.v_exp, true, v_exp, (uint64_t)H * kDv, krows, (uint64_t)H * kDv * 2, 64, kPKeys,
                     CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  PrefillParams p{B, T_q, T_kv, H, kv_seq_stride, scale * kLog2e, o, lse, status};
  static SmemOptIn opt_in;
  cudaError_t e = ensure_dynamic_smem((const void*)k_prefill_attn, (int)kPSmem, opt_in);
  if (e != cudaSuccess) return e;
  dim3 grid((T_q + kPTiles * kPQ - 1) / (kPTiles * kPQ), H, B);
  e = launch_pdl(k_prefill_attn, grid, dim3(kPThreads), kPSmem, st, maps, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mla
