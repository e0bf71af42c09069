// Prefill and chunked prefill in the expanded order, on the sm_103a tensor cores.
//
// Page "Multi-Head Latent Attention (MLA)", section on prefill and decode: prefill works on
// many query tokens at once and is bound by compute, so it may keep the order that builds
// the per-head keys and values; page "MLA의 계산: KV를 펼치지 않고 Attention하기", section
// "계산 재배치의 효과와 한계": the absorbed order pays d_c-wide dot products per key, which
// pays off only when reading the cache dominates (decode).  Here:
//   K_h = C W_UK[h], V_h = C W_UV[h]  (k_expand_kv, expand_sm103.cu), then for each
//   head, causal attention of the T_q query tokens (the last T_q of T_kv positions) over
//   [K_h | k^R] with [q_nope | q^R], one scale, and V_h mixed by the weights.
//
// k_prefill_attn: persistent CTAs (one per SM) walk a fixed list of work items, an item
// being (sequence, head, 128 query tokens) over key tiles of 128 positions.  The items of a
// head go in pairs (query block i with block n-1-i: for a whole prompt their key tile
// counts add up to a constant), the pairs dealt round-robin, so that every CTA carries the
// same work and the CTAs running at one time share heads (their key and value tiles meet
// in L2).  TMEM holds O (128 columns), two score buffers (128 each) and q_nope as the A
// operand of the score products (64 columns of bf16 pairs).  P(j), the A operand of the
// aggregation, is written into the score buffer of S(j) over the columns its thread has
// read, so P is double-buffered with S; shared memory holds the key tiles [K_h | k^R] (48 KB, a ring
// of two), the value tiles V_h (32 KB, a ring of two), q^R and two 16 KB slots.  q_nope
// comes in by TMA through the slots; O goes out by TMA through the slots and the value
// stage of the item's last tile, stored by the value producer.  Per key tile j:
//   S(j) [128 x 128] = q_nope . K_h(j)^T (8 MMAs, A from TMEM) + q^R . k^R(j)^T (4 MMAs)
//   O [128 x 128]   += P(j-1) [128 x 128] . V(j-1)  (8 MMAs, A from TMEM)
// The rings, the score buffers and P run on from one item to the next: the score products
// of the next item start while the softmax warps finish the current one and store its O.
// Both score products and the aggregation read only the key or value tile from shared
// memory (with N = 64 and both operands in shared memory the products were bound by
// their operand reads).  Warps 0-7 run the online softmax, two threads per query row
// (TMEM lane = row; warp w takes key columns [64 (w / 4), 64 (w / 4) + 64)), the pair
// agreeing on the row maximum through shared memory; they also move the next item's
// q_nope from the slots into TMEM during the current item's last tile.  Warps 8 and 10
// stream the key and value tiles by TMA; warp 9 issues the MMAs, S(j+1) running while the
// softmax of tile j does.  The running maximum is raised lazily (O is rescaled only when a row's maximum
// grows by more than 2^8), as in the latent decode.  Key tiles past the last query's
// position are not loaded.  Every wait is bounded; on expiry the CTA records
// MLA_ERR_TIMEOUT, drains and exits.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "ptx_sm103.cuh"

namespace mla {

namespace {

using namespace ptx;

constexpr int kPQ = 128;                  // query rows per item (TMEM lanes)
constexpr int kPKeys = 128;               // keys per tile
constexpr int kPKStages = 2;              // [K_h | k^R] ring
constexpr int kPVStages = 2;              // V_h ring
constexpr int kPSoftWarps = 8;
constexpr int kPTmaWarp = 8, kPMmaWarp = 9, kPVWarp = 10;
constexpr int kPThreads = 352;
constexpr uint32_t kPBox = 128 * 128;     // 128 rows x 64 bf16 (128B swizzle)
constexpr uint32_t kPKBytes = 3 * kPBox;  // K_h (2 boxes) + k^R (1 box)
constexpr uint32_t kPVBytes = 2 * kPBox;
constexpr uint32_t kPOBox = 128 * 128;    // 128 rows x 32 fp32 (128B swizzle)
constexpr uint32_t kPOffK = 0;
constexpr uint32_t kPOffV = kPOffK + kPKStages * kPKBytes;
constexpr uint32_t kPOffQR = kPOffV + kPVStages * kPVBytes;
constexpr uint32_t kPOffOst = kPOffQR + kPBox;     // two O slots
constexpr uint32_t kPOffRed = kPOffOst + 2 * kPOBox;   // [2 halves][128 rows] fp32
constexpr uint32_t kPOffBars = kPOffRed + 2 * 128 * 4;
constexpr uint32_t kPSmem = kPOffBars + 256 + 1024;
constexpr uint32_t kPEpiBar = 5;          // named barrier of the 256 softmax threads
static_assert(kPSmem <= 232448, "shared memory per CTA");
static_assert(kPOffV % 1024 == 0 && kPOffQR % 1024 == 0 && kPOffOst % 1024 == 0, "128B-swizzled tiles");

// TMEM columns.
constexpr uint32_t kPTmemO = 0;      // [0,128)   O, fp32
constexpr uint32_t kPTmemS = 128;    // [128,384) two score buffers of 128 fp32; P(j) in
                                     // buffer j & 1, keys 0-63 in columns [0,32) and keys
                                     // 64-127 in [64,96), bf16 pairs
constexpr uint32_t kPTmemQ = 384;    // [384,448) q_nope, bf16 pairs; [448,512) unused
constexpr float kPRescale = 8.0f;

// Tiles count up across the items of a CTA (g); items count up too (n).
enum PBar {
  kPQFullB = 0,                         // q^R of item n landed
  kPQReadyB,                            // q_nope of item n in TMEM (256 threads)
  kPQrFreeB,                            // score products of item n done: q^R and q_nope free
  kPQnFullB,                            // q_nope of item n landed in the O slots
  kPOStagedB,                           // O of item n staged (256 threads)
  kPOReadB,                             // O of item n stored: its slots and value stage read
  kPKFullB,                             // [2] key tile landed
  kPKEmptyB = kPKFullB + kPKStages,     // [2] score products of the stage done
  kPVFullB = kPKEmptyB + kPKStages,     // [2] value tile landed
  kPVEmptyB = kPVFullB + kPVStages,     // [2] aggregation of the stage done
  kPSFullB = kPVEmptyB + kPVStages,     // [2] S buffer ready
  kPSFreeB = kPSFullB + 2,              // [2] S buffer read (8 warps)
  kPPFullB = kPSFreeB + 2,              // [2] P(g) in TMEM, by g & 1 (256 threads)
  kPPvDoneB = kPPFullB + 2,             // [2] PV(g) done, by g & 1: O stable
  kPDrainB = kPPvDoneB + 2,
  kPNumBars
};
static_assert(kPNumBars * 8 + 16 <= 256, "barrier area");

struct PrefillMaps {
  CUtensorMap q_rope;   // [B*T_q, H*64], box 64 x 128
  CUtensorMap q_nope;   // [B*T_q, H*128], box 64 x 128
  CUtensorMap k_exp;    // [rows, H*128], box 64 x 128
  CUtensorMap k_rope;   // cache rows [rows, 576], box 64 x 128 (columns 512..575)
  CUtensorMap v_exp;    // [rows, H*128], box 64 x 128
  CUtensorMap o;        // fp32 [B][T_q][H*128], box 32 x 128 x 1 (rows past T_q clipped)
};

struct PrefillParams {
  int B, T_q, T_kv, H;
  int64_t kv_seq_stride;
  float scale_log2;
  int n_qb;         // query blocks per (sequence, head)
  int npu;          // pairs of query blocks per (sequence, head): (n_qb + 1) / 2
  int units;        // B * H * npu
  float* o;      // [B, T_q, H, 128]
  float* lse;    // [B, T_q, H]
  int32_t* status;
};

struct PItem {
  int b, h, q0, nt;   // sequence, head, first query, key tiles any of its rows reads
};

// The items of this CTA in order: units blockIdx.x, blockIdx.x + gridDim.x, ...; unit u is
// (sequence, head) u / npu with query blocks n_qb-1-i and then i (i = u % npu, the second
// absent when the two coincide).  (u, k) is the position; returns false past the end.
__device__ __forceinline__ bool pnext(const PrefillParams& p, int& u, int& k, PItem& it) {
  while (u < p.units) {
    const int hs = u / p.npu;
    const int i = u % p.npu;
    const int qb = k == 0 ? p.n_qb - 1 - i : i;
    const bool have = k == 0 || i < p.n_qb - 1 - i;
    if (k == 0) {
      k = 1;
    } else {
      k = 0;
      u += gridDim.x;
    }
    if (have) {
      it.b = hs / p.H;
      it.h = hs % p.H;
      it.q0 = qb * kPQ;
      const int last_pos = min(p.T_kv - 1, p.T_kv - p.T_q + min(it.q0 + kPQ - 1, p.T_q - 1));
      it.nt = last_pos / kPKeys + 1;
      return true;
    }
  }
  return false;
}

__device__ __forceinline__ bool pwarp_wait(uint32_t bar, uint32_t parity) {
  return !__any_sync(0xffffffffu, !mbar_wait(bar, parity, kDefaultWaitNs));
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
  float* red = reinterpret_cast<float*>(smem + kPOffRed);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    mbar_init(bar(kPQFullB), 1);
    mbar_init(bar(kPQReadyB), 32 * kPSoftWarps);
    mbar_init(bar(kPQrFreeB), 1);
    mbar_init(bar(kPQnFullB), 1);
    mbar_init(bar(kPOStagedB), 32 * kPSoftWarps);
    mbar_init(bar(kPOReadB), 1);
    for (int i = 0; i < kPKStages; ++i) {
      mbar_init(bar(kPKFullB + i), 1);
      mbar_init(bar(kPKEmptyB + i), 1);
    }
    for (int i = 0; i < kPVStages; ++i) {
      mbar_init(bar(kPVFullB + i), 1);
      mbar_init(bar(kPVEmptyB + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kPSFullB + i), 1);
      mbar_init(bar(kPSFreeB + i), kPSoftWarps);
    }
    mbar_init(bar(kPPFullB), 32 * kPSoftWarps);
    mbar_init(bar(kPPFullB + 1), 32 * kPSoftWarps);
    mbar_init(bar(kPPvDoneB), 1);
    mbar_init(bar(kPPvDoneB + 1), 1);
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
    // ---------------- TMA producer: q^R and the key tiles ----------------
    // Key tile g into K stage g % 2, free once S(g-2) is done.  q^R of item n replaces that
    // of item n-1 once the last score products of n-1 are done (after the first key tile
    // of n is on its way).  The value tiles have a producer of their own, so that a key
    // tile is never queued behind a value tile waiting for an aggregation.
    if (lane == 0) {
      prefetch_tmap(&maps.q_rope);
      prefetch_tmap(&maps.q_nope);
      prefetch_tmap(&maps.k_exp);
      prefetch_tmap(&maps.k_rope);
      prefetch_tmap(&maps.v_exp);
      prefetch_tmap(&maps.o);
      int u = blockIdx.x;
      int k = 0, n = 0;
      uint32_t g = 0;
      PItem it;
      bool have = pnext(p, u, k, it);
      while (have && !aborted) {
        int u2 = u;
        int k2 = k;
        PItem nx;
        const bool have_nx = pnext(p, u2, k2, nx);
        if (have_nx) tma_prefetch_2d(&maps.q_rope, nx.h * 64, nx.b * p.T_q + nx.q0);
        const int64_t krow0 = (int64_t)it.b * p.kv_seq_stride;
        for (int j = 0; j < it.nt; ++j, ++g) {
          const uint32_t ks = g % kPKStages;
          if (g >= (uint32_t)kPKStages &&
              !mbar_wait(bar(kPKEmptyB + ks), (g / kPKStages - 1) & 1u, kDefaultWaitNs)) {
            aborted = true;
            break;
          }
          const int y = (int)(krow0 + (int64_t)j * kPKeys);
          const uint32_t kst = s0 + kPOffK + ks * kPKBytes;
          mbar_arrive_expect_tx(bar(kPKFullB + ks), kPKBytes);
          tma_load_2d(kst, &maps.k_exp, bar(kPKFullB + ks), it.h * 128, y);
          tma_load_2d(kst + kPBox, &maps.k_exp, bar(kPKFullB + ks), it.h * 128 + 64, y);
          tma_load_2d(kst + 2 * kPBox, &maps.k_rope, bar(kPKFullB + ks), kDc, y);
          if (j == 0) {
            if (n > 0 && !mbar_wait(bar(kPQrFreeB), (uint32_t)(n - 1) & 1u, kDefaultWaitNs)) {
              aborted = true;
              ++g;
              break;
            }
            mbar_arrive_expect_tx(bar(kPQFullB), kPBox);
            tma_load_2d(s0 + kPOffQR, &maps.q_rope, bar(kPQFullB), it.h * 64, it.b * p.T_q + it.q0);
          }
        }
        it = nx;
        have = have_nx;
        u = u2;
        k = k2;
        ++n;
      }
      // No copy may land after exit.
      for (uint32_t i = g > (uint32_t)kPKStages ? g - kPKStages : 0u; i < g; ++i)
        mbar_wait(bar(kPKFullB + i % kPKStages), (i / kPKStages) & 1u, kDefaultWaitNs);
      if (n > 0) mbar_wait(bar(kPQFullB), (uint32_t)(n - 1) & 1u, kDefaultWaitNs);
    }
  } else if (warp == kPVWarp) {
    // ---------------- TMA producer: the value tiles, and O out ----------------
    // Value tile g into V stage g % 2, free once PV(g-2) is done.  The softmax warps stage
    // an item's O in four 32-column boxes: columns 64 hf + [0, 32) in slot hf, columns
    // 64 hf + [32, 64) in half hf of the value stage of the item's last tile.  This thread
    // stores them by TMA before that stage is loaded again (or at the end), waits until
    // the boxes are read, and says so (the slots then take the next q_nope).
    if (lane == 0) {
      int u = blockIdx.x;
      int k = 0;
      uint32_t g = 0;
      PItem it;
      PItem pend_it[4];          // items whose O is staged or about to be, in order
      uint32_t pend_last[4];     // the last tile of each
      int pend_head = 0, pend_n = 0, stored = 0;
      auto store_o = [&]() {
        const PItem t = pend_it[pend_head];
        const uint32_t vst = s0 + kPOffV + (pend_last[pend_head] % kPVStages) * kPVBytes;
        pend_head = (pend_head + 1) & 3;
        --pend_n;
        if (!mbar_wait(bar(kPOStagedB), (uint32_t)stored & 1u, kDefaultWaitNs)) return false;
        tma_store_3d(&maps.o, t.h * 128, t.q0, t.b, s0 + kPOffOst);
        tma_store_3d(&maps.o, t.h * 128 + 32, t.q0, t.b, vst);
        tma_store_3d(&maps.o, t.h * 128 + 64, t.q0, t.b, s0 + kPOffOst + kPOBox);
        tma_store_3d(&maps.o, t.h * 128 + 96, t.q0, t.b, vst + kPOBox);
        bulk_commit_group();
        bulk_wait_group_read0();
        mbar_arrive(bar(kPOReadB));
        ++stored;
        return true;
      };
      while (!aborted && pnext(p, u, k, it)) {
        const int64_t krow0 = (int64_t)it.b * p.kv_seq_stride;
        for (int j = 0; j < it.nt; ++j, ++g) {
          const uint32_t vs = g % kPVStages;
          if (g >= (uint32_t)kPVStages &&
              !mbar_wait(bar(kPVEmptyB + vs), (g / kPVStages - 1) & 1u, kDefaultWaitNs)) {
            aborted = true;
            break;
          }
          if (pend_n > 0 && pend_last[pend_head] + kPVStages == g && !store_o()) {   // the stage holds O
            aborted = true;
            break;
          }
          const int y = (int)(krow0 + (int64_t)j * kPKeys);
          const uint32_t vst = s0 + kPOffV + vs * kPVBytes;
          mbar_arrive_expect_tx(bar(kPVFullB + vs), kPVBytes);
          tma_load_2d(vst, &maps.v_exp, bar(kPVFullB + vs), it.h * 128, y);
          tma_load_2d(vst + kPBox, &maps.v_exp, bar(kPVFullB + vs), it.h * 128 + 64, y);
        }
        if (aborted) break;
        pend_it[(pend_head + pend_n) & 3] = it;
        pend_last[(pend_head + pend_n) & 3] = g - 1;
        ++pend_n;
      }
      while (!aborted && pend_n > 0)
        if (!store_o()) aborted = true;
      bulk_wait_group_read0();   // the staging outlives its reads; the writes finish with the grid
      for (uint32_t i = g > (uint32_t)kPVStages ? g - kPVStages : 0u; i < g; ++i)   // no copy may land after exit
        mbar_wait(bar(kPVFullB + i % kPVStages), (i / kPVStages) & 1u, kDefaultWaitNs);
    }
  } else if (warp == kPMmaWarp) {
    // ---------------- MMA issuer ----------------
    // Tile g: S(g) once the softmax has read buffer g & 1 at tile g-2 (8 MMAs with q_nope
    // from TMEM against the two K_h boxes, 4 with q^R from shared memory against k^R),
    // then PV(g-1) once P(g-1) is in TMEM (8 MMAs, A = P from score buffer (g-1) & 1, B =
    // the value tile read MN-major).  PV(g-1) is thus always issued before S(g+1), which
    // overwrites its P: the MMAs of one thread run in issue order.  The softmax warps may
    // write P(g) before this thread has waited for P(g-1), but not P(g+1) (it needs S(g+1)),
    // so the P barriers go by parity and none runs two phases ahead of its waiter.  The first PV of an item
    // overwrites O: the softmax warps write its P only after reading the previous item's O
    // out of TMEM.  The last PV of an item goes out before the wait for the next item's q^R
    // and q_nope.
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16(128, kPKeys, false, false);
      const uint32_t id_o = idesc_bf16(128, 128, false, true);
      const uint64_t qr_desc = smem_desc(s0 + kPOffQR, 16, 1024, kSwizzle128B);
      auto pv = [&](uint32_t gi, bool first) {   // O (+)= P(gi) V(gi)
        const uint32_t vs = gi % kPVStages;
        if (!mbar_wait(bar(kPPFullB + (gi & 1u)), (gi >> 1) & 1u, kDefaultWaitNs) ||
            !mbar_wait(bar(kPVFullB + vs), (gi / kPVStages) & 1u, kDefaultWaitNs))
          return false;
        tc_fence_after();
        const uint64_t vd = smem_desc(s0 + kPOffV + vs * kPVBytes, kPBox, 1024, kSwizzle128B);
#pragma unroll
        for (int k = 0; k < kPKeys / 16; ++k)
          mma_ts(tb + kPTmemO, tb + kPTmemS + 128u * (gi & 1u) + 8u * k + (k >= 4 ? 32u : 0u), vd + 128u * k, id_o, (!first || k > 0) ? 1u : 0u);
        mma_commit(bar(kPVEmptyB + vs));
        mma_commit(bar(kPPvDoneB + (gi & 1u)));
        return true;
      };
      int u = blockIdx.x;
      int k = 0, n = 0;
      uint32_t g = 0;
      bool pend = false, pend_first = false;   // PV of tile g-1 still to issue
      PItem it;
      while (!aborted && pnext(p, u, k, it)) {
        // The last aggregation of the previous item goes first.
        if (pend && !pv(g - 1, pend_first)) {
          aborted = true;
          break;
        }
        pend = false;
        if (!mbar_wait(bar(kPQFullB), (uint32_t)n & 1u, kDefaultWaitNs) ||
            !mbar_wait(bar(kPQReadyB), (uint32_t)n & 1u, kDefaultWaitNs)) {
          aborted = true;
          break;
        }
        for (int j = 0; j < it.nt; ++j, ++g) {
          const uint32_t ks = g % kPKStages;
          if ((g >= 2 && !mbar_wait(bar(kPSFreeB + (g & 1)), ((g >> 1) - 1) & 1u, kDefaultWaitNs)) ||
              !mbar_wait(bar(kPKFullB + ks), (g / kPKStages) & 1u, kDefaultWaitNs)) {
            aborted = true;
            break;
          }
          tc_fence_after();
          const uint32_t kst = s0 + kPOffK + ks * kPKBytes;
          const uint32_t d = tb + kPTmemS + 128u * (g & 1);
          const uint64_t kd = smem_desc(kst, 16, 1024, kSwizzle128B);
#pragma unroll
          for (int c = 0; c < 8; ++c)   // 16 dims per MMA: 32 bytes along a 128-byte row, box c / 4
            mma_ts(d, tb + kPTmemQ + 8u * c, kd + (((c >> 2) * kPBox + (c & 3) * 32u) >> 4), id_s, c > 0 ? 1u : 0u);
#pragma unroll
          for (int c = 0; c < 4; ++c) mma_ss(d, qr_desc + 2u * c, kd + ((2 * kPBox) >> 4) + 2u * c, id_s, 1u);
          mma_commit(bar(kPSFullB + (g & 1)));
          mma_commit(bar(kPKEmptyB + ks));
          if (j == it.nt - 1) mma_commit(bar(kPQrFreeB));
          if (pend && !pv(g - 1, pend_first)) {
            aborted = true;
            break;
          }
          pend = true;
          pend_first = j == 0;
        }
        ++n;
      }
      if (!aborted && pend && !pv(g - 1, pend_first)) aborted = true;
      mma_commit(bar(kPDrainB));
      mbar_wait(bar(kPDrainB), 0, kDefaultWaitNs);
    }
  } else {
    // ---------------- softmax warps: two threads per query row ----------------
    const int quarter = warp & 3, hf = warp >> 2;
    const int r = 32 * quarter + lane;            // TMEM lane == query row of the tile
    const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
    const uint32_t pair_bar = 1u + (uint32_t)quarter;   // the two warps of this lane quarter
    const int offset = p.T_kv - p.T_q;            // query i sits at position offset + i
    // q_nope goes through the two O slots: the leader (tid 0) loads item t's rows by TMA,
    // box hf into slot hf (row r, 16-byte chunk c at c ^ (r & 7)); every thread then moves
    // its half row into TMEM, the A operand of the score MMAs.
    auto q_issue = [&](const PItem& t) {
      mbar_arrive_expect_tx(bar(kPQnFullB), 2 * kPBox);
      tma_load_2d(s0 + kPOffOst, &maps.q_nope, bar(kPQnFullB), t.h * 128, t.b * p.T_q + t.q0);
      tma_load_2d(s0 + kPOffOst + kPOBox, &maps.q_nope, bar(kPQnFullB), t.h * 128 + 64, t.b * p.T_q + t.q0);
    };
    auto q_move = [&](int item) {
      const bool got = pwarp_wait(bar(kPQnFullB), (uint32_t)item & 1u);
      if (got) {
        const uint32_t src = s0 + kPOffOst + (uint32_t)hf * kPOBox + (uint32_t)r * 128u;
        uint32_t v[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 w = ld_shared_u4(src + (uint32_t)((c ^ (r & 7)) * 16));
          v[4 * c] = w.x;
          v[4 * c + 1] = w.y;
          v[4 * c + 2] = w.z;
          v[4 * c + 3] = w.w;
        }
        tmem_st32(tb + lane_off + kPTmemQ + 32u * (uint32_t)hf, v);
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(bar(kPQReadyB));
      return got;
    };
    int u = blockIdx.x;
    int k = 0, n = 0;
    uint32_t g = 0;
    PItem it;
    bool have = pnext(p, u, k, it);
    bool q_failed = false;
    if (have) {
      if (tid == 0) q_issue(it);
      q_failed = !q_move(0);
      named_bar_sync(kPEpiBar, 32 * kPSoftWarps);   // the slots are read
    }
    while (have) {
      PItem nx;
      bool have_nx;
      {
        int u2 = u, k2 = k;
        have_nx = pnext(p, u2, k2, nx);
      }
      const int qi = it.q0 + r;                   // query index in the sequence
      const int qpos = offset + qi;               // its position
      const bool row_ok = qi < p.T_q;
      // The two threads of a row meet at named barriers, so they leave the loop together:
      // a failed wait is carried to the next meeting, where the pair agrees to give up.
      float m_ref = -INFINITY, l = 0.f;
      bool failed = q_failed;   // a wait of this thread gave up since the last meeting
      q_failed = false;
      for (int j = 0; j < it.nt; ++j, ++g) {
        float x[64];
        // A tile before the last (or at the only one), the next item's q_nope is loaded
        // into the slots, once the previous item's O has left them.
        if (tid == 0 && have_nx && j == max(0, it.nt - 2)) {
          if (n == 0 || mbar_wait(bar(kPOReadB), (uint32_t)(n - 1) & 1u, kDefaultWaitNs))
            q_issue(nx);
          else
            failed = true;
        }
        if (pwarp_wait(bar(kPSFullB + (g & 1)), (g >> 1) & 1u)) {
          tc_fence_after();
          const uint32_t ts = tb + lane_off + kPTmemS + 128u * (g & 1) + 64u * (uint32_t)hf;
          tmem_ld32f<0>(ts, x);
          tmem_ld32f<32>(ts + 32u, x);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kPSFreeB + (g & 1)));
        } else {
          failed = true;
#pragma unroll
          for (int c = 0; c < 64; ++c) x[c] = -INFINITY;
        }
        // Causal mask and the sequence end (rows of later positions may hold anything).
        const int k0 = j * kPKeys + 64 * hf;
        const int vis = min(64, min(qpos, p.T_kv - 1) - k0 + 1);   // readable keys of this half-row
        float t16[16];
        if (vis < 64) {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (c >= vis) x[c] = -INFINITY;
        }
#pragma unroll
        for (int c = 0; c < 16; ++c) t16[c] = fmaxf(fmaxf(x[c], x[c + 16]), fmaxf(x[c + 32], x[c + 48]));
#pragma unroll
        for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
          for (int c = 0; c < w; ++c) t16[c] = fmaxf(t16[c], t16[c + w]);
        // The row maximum of the two halves, through shared memory: write, meet (agreeing
        // to go on), read, meet (the next tile's write stays behind the partner's read).
        red[hf * 128 + r] = t16[0];
        if (!named_bar_and(pair_bar, 64, !failed)) {
          aborted = true;
          ++g;
          break;
        }
        const float mx = fmaxf(t16[0], red[(hf ^ 1) * 128 + r]) * p.scale_log2;
        named_bar_sync(pair_bar, 64);
        const bool grow = mx > m_ref + kPRescale;
        const float m_new = grow ? mx : m_ref;
        if (grow) l *= ex2_approx(m_ref - m_new);   // 0 when m_ref = -inf (l is 0 then)
        const float alpha = grow ? ex2_approx(m_ref - m_new) : 1.f;
        m_ref = m_new;
        const float bias = (m_new == -INFINITY) ? 0.f : -m_new;
        uint32_t pw[32];
        float ps[4] = {0.f, 0.f, 0.f, 0.f};   // four partial sums: short dependency chains
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float a = ex2_approx(fmaf(x[2 * c], p.scale_log2, bias));
          const float e = ex2_approx(fmaf(x[2 * c + 1], p.scale_log2, bias));
          ps[c & 3] += a + e;
          pw[c] = f2_to_bf2(a, e);
        }
        l += (ps[0] + ps[1]) + (ps[2] + ps[3]);
        // P(g) goes over the S(g) columns this thread has read, so it waits for nothing.  O
        // is stable once PV(g-1) is done: a rescale waits for that.  (At tile g the barrier of
        // PV(g-1) is in its phase or one past it: PV(g-3) preceded S(g-1), and PV(g+1) needs
        // P(g+1).)
        const bool resc = __any_sync(0xffffffffu, grow && j > 0);
        if (resc && !pwarp_wait(bar(kPPvDoneB + ((g - 1) & 1u)), ((g - 1) >> 1) & 1u)) {
          failed = true;
          continue;
        }
        tc_fence_after();
        tmem_st32(tb + lane_off + kPTmemS + 128u * (g & 1) + 64u * (uint32_t)hf, pw);
        if (resc) {   // rescale this thread's half of its O row
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            uint32_t o[32];
            const uint32_t ta = tb + lane_off + kPTmemO + 64u * (uint32_t)hf + 32u * c;
            tmem_ld32(ta, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(ta, o);
          }
        }
        tmem_st_wait();
        // Rows of the key tile past the sequence end may hold anything (even NaN): clear
        // them in the value tile so that their zero weights add exactly zero.
        const int rows_valid = min(kPKeys, p.T_kv - j * kPKeys);
        if (rows_valid < kPKeys) {
          if (!pwarp_wait(bar(kPVFullB + g % kPVStages), (g / kPVStages) & 1u)) {
            failed = true;
            continue;
          }
          const uint32_t vt = s0 + kPOffV + (g % kPVStages) * kPVBytes;
          for (int idx = tid; idx < (kPKeys - rows_valid) * 16; idx += 32 * kPSoftWarps) {
            const int row = rows_valid + idx / 16, c = idx % 16;   // 2 boxes x 8 chunks per row
            st_shared_v4_zero(vt + (uint32_t)(c >> 3) * kPBox + (uint32_t)row * 128u + (uint32_t)(c & 7) * 16u);
          }
          fence_proxy_async_smem();
        }
        tc_fence_before();
        mbar_arrive(bar(kPPFullB + (g & 1)));
        // The item's score products are done (S of its last tile was read): the next
        // item's q_nope goes into TMEM.
        if (j == it.nt - 1 && have_nx && !q_move(n + 1)) failed = true;
      }
      // Epilogue: the row sum of both halves, then this thread's half of O / l, and the LSE.
      if (!aborted && !failed && !pwarp_wait(bar(kPPvDoneB + ((g - 1) & 1u)), ((g - 1) >> 1) & 1u)) failed = true;
      tc_fence_after();
      red[hf * 128 + r] = l;
      if (!named_bar_and(pair_bar, 64, !aborted && !failed)) aborted = true;
      const float l_row = l + red[(hf ^ 1) * 128 + r];
      const bool have_l = !aborted && l_row > 0.f;
      const float inv = have_l ? 1.f / l_row : 0.f;
      // O is staged for the value producer to store: this thread's columns 64 hf + 32 c go
      // to slot hf (c = 0) or to half hf of the value stage of the last tile (c = 1), row r,
      // 16-byte chunk v at v ^ (r & 7).  The slots were emptied before this item's last
      // q_nope came in, except after the last item: then the previous item's O must have
      // left them.  The next item's first P (and with it the PV that overwrites O) follows.
      // If any row gave up, O is written directly (zeros for those rows) and the CTA stops.
      if (tid == 0 && !have_nx && n > 0 && !mbar_wait(bar(kPOReadB), (uint32_t)(n - 1) & 1u, kDefaultWaitNs))
        aborted = true;
      const bool all_ok = named_bar_and(kPEpiBar, 32 * kPSoftWarps, !aborted);
      if (all_ok) {
        const uint32_t vst = s0 + kPOffV + ((g - 1) % kPVStages) * kPVBytes;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t o[32];
          tmem_ld32(tb + lane_off + kPTmemO + 64u * (uint32_t)hf + 32u * c, o);
          tmem_ld_wait();
          const uint32_t dst = (c == 0 ? s0 + kPOffOst : vst) + (uint32_t)hf * kPOBox + (uint32_t)r * 128u;
#pragma unroll
          for (int v = 0; v < 8; ++v)
            st_shared_u4(dst + (uint32_t)((v ^ (r & 7)) * 16), __float_as_uint(__uint_as_float(o[4 * v]) * inv),
                         __float_as_uint(__uint_as_float(o[4 * v + 1]) * inv),
                         __float_as_uint(__uint_as_float(o[4 * v + 2]) * inv),
                         __float_as_uint(__uint_as_float(o[4 * v + 3]) * inv));
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(kPOStagedB));
      } else {
        float* out = p.o + (((int64_t)it.b * p.T_q + qi) * p.H + it.h) * 128 + 64 * hf;
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          uint32_t o[32];
          if (!aborted) {
            tmem_ld32(tb + lane_off + kPTmemO + 64u * (uint32_t)hf + 32u * c, o);
            tmem_ld_wait();
          }
          if (row_ok) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
              reinterpret_cast<float4*>(out + 32 * c)[v] =
                  have_l ? make_float4(__uint_as_float(o[4 * v]) * inv, __uint_as_float(o[4 * v + 1]) * inv,
                                       __uint_as_float(o[4 * v + 2]) * inv, __uint_as_float(o[4 * v + 3]) * inv)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
      }
      if (row_ok && hf == 0)
        p.lse[((int64_t)it.b * p.T_q + qi) * p.H + it.h] = have_l ? (m_ref + log2f(l_row)) * kLn2 : -INFINITY;
      if (!all_ok) {
        aborted = true;
        break;
      }
      have = pnext(p, u, k, it);
      ++n;
    }
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
  if (!encode_tma_2d(&maps.q_rope, true, q_rope, (uint64_t)H * kDr, qrows, (uint64_t)H * kDr * 2, 64, kPQ,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tma_2d(&maps.q_nope, true, q_nope, (uint64_t)H * kDn, qrows, (uint64_t)H * kDn * 2, 64, kPQ,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tma_3d(&maps.o, false, o, (uint64_t)H * kDv, (uint64_t)T_q, (uint64_t)B, (uint64_t)H * kDv * 4,
                     (uint64_t)T_q * H * kDv * 4, 32, kPQ, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tma_2d(&maps.k_exp, true, k_exp, (uint64_t)H * kDn, krows, (uint64_t)H * kDn * 2, 64, kPKeys,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tma_2d(&maps.k_rope, true, kv, kRow, krows, (uint64_t)kRow * 2, 64, kPKeys,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tma_2d(&maps.v_exp, true, v_exp, (uint64_t)H * kDv, krows, (uint64_t)H * kDv * 2, 64, kPKeys,
                     CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const int n_qb = (T_q + kPQ - 1) / kPQ;
  const int npu = (n_qb + 1) / 2;
  if ((int64_t)B * H * npu > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const int units = B * H * npu;
  PrefillParams p{B, T_q, T_kv, H, kv_seq_stride, scale * kLog2e, n_qb, npu, units, o, lse, status};
  static SmemOptIn opt_in;
  cudaError_t e = ensure_dynamic_smem((const void*)k_prefill_attn, (int)kPSmem, opt_in);
  if (e != cudaSuccess) return e;
  const int sms = device_sm_count() > 0 ? device_sm_count() : 148;
  const int grid = std::min(units, sms);
  e = launch_pdl(k_prefill_attn, dim3(grid), dim3(kPThreads), kPSmem, st, maps, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mla
