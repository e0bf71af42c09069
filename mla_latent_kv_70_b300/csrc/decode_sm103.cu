// Absorbed MLA decode on the sm_103a tensor cores (tcgen05 + TMEM + TMA), one CTA pair
// per (query token, split).
//
// What it computes -- page "MLA의 계산: KV를 펼치지 않고 Attention하기":
//   section "Content 점수와 위치 점수 합치기" (eq. s_j): s_j = q~ . c_j + q^R . k^R_j, one
//     scale, one softmax over every readable position, causal mask between query tokens;
//   section "Key 투영을 Query 쪽으로 옮기기" (Fig. 3): q~ = q U^K^T is read straight
//     against the latent rows, no per-head key is built;
//   section "Value 투영을 가중합 뒤로 옮기기" (Fig. 4): z = sum_j a_j c_j is accumulated in
//     the latent space; U^V is applied afterwards (mla_out_proj_uv).
//
// How (B300 design).  All 128 heads read the same latent row, so per tile of 64 cache
// rows the work is two dense products: S[128 x 64] = Q[128 x 576] . K^T and
// O[128 x 512] += P[128 x 64] . V[64 x 512].  O alone fills the 512 TMEM columns of one
// SM, so a cluster of two CTAs shares a query token:
//   * CTA r owns latent columns [256r, 256r+256) and rope columns [512+32r, 512+32r+32)
//     of every cache row; its TMA loads only those (each cache byte is read once);
//   * each CTA computes the partial score over its 288 columns into TMEM (A operand =
//     its half of q~, held in TMEM; the rope half of q from shared memory);
//   * the partials are swapped through distributed shared memory as bf16, by 16-byte
//     st.async into the peer's receive buffer, counted (complete_tx) on its mbarrier.
//     No "buffer free" signal travels back: under HBM load a remote release-arrive took
//     ~3900 cycles to land, and the data flow already orders each reuse (a CTA sends
//     tile i+1 only after reading tile i).  bf16 halves the bytes of fp32 partials and
//     adds an error of the same order as storing q~ in bf16 (2^-8 of the partial sum).
//     Each CTA adds its own fp32 partial to the peer's bf16 partial and normalises its
//     half of O with its own softmax sums, so the two halves need not agree bit for bit;
//   * P (bf16) goes to shared memory
//     in the 128B-swizzled K-major layout, and each CTA accumulates its 256 columns of
//     O in TMEM from P and its own V columns (the same shared-memory tile, read MN-major).
// Warp roles per CTA: warp 0 issues TMA, warp 1 issues the score MMAs (QK) and warp 14
// the aggregation MMAs (PV), so that neither waits behind the other; warps 2-5 (one per
// TMEM lane quarter of 32 heads) read the partial scores out of TMEM (freeing the S
// buffer for the next QK at once), swap them with the peer, and leave the full scores
// relative to each row's tile maximum in shared memory (fp16), two warps per quarter
// taking alternate tiles; warps 10-13 (one per quarter) run the online softmax and the
// epilogue.  Exchange and softmax of different tiles overlap.
// Softmax runs in the log2 domain with a lazily raised reference maximum (the running
// output is rescaled only when the maximum grows by more than 2^8).
// Every mbarrier wait is bounded; on expiry the CTA records MLA_ERR_TIMEOUT in the
// status word, drains its own copies and MMAs, frees TMEM and exits.
#include <cuda.h>

#include "common.cuh"
#include "ptx_sm103.cuh"

namespace mla {

namespace {

using namespace ptx;

constexpr int kN = 64;                            // cache rows per tile
constexpr int kStages = 4;
constexpr int kExchWarps = 8;                     // two per TMEM lane quarter (even / odd tiles)
constexpr int kSoftmaxWarps = 4;                  // one per TMEM lane quarter
constexpr int kPvWarp = 2 + kExchWarps + kSoftmaxWarps;   // the warp that issues PV
constexpr int kThreads = 32 * (kPvWarp + 1);
constexpr uint32_t kBoxBytes = kN * 128;          // 64 rows x 64 bf16 (128B swizzle)
constexpr uint32_t kRopeBoxBytes = kN * 64;       // 64 rows x 32 bf16 (64B swizzle)
constexpr uint32_t kStageBytes = 4 * kBoxBytes + kRopeBoxBytes;
constexpr uint32_t kQRopeBytes = 128 * 64;        // 128 heads x 32 bf16
constexpr uint32_t kRecvBytes = 128 * kN * 2;     // peer's bf16 partial scores
constexpr uint32_t kQuarterXBytes = 32 * kN * 2;  // one lane quarter's share: 32 rows x 64 columns
constexpr uint32_t kPBytes = 128 * kN * 2;        // P, bf16, 128 rows x 128 B
constexpr uint32_t kScoreBytes = 128 * kN * 2;    // full scores handed to the softmax, fp16

constexpr uint32_t kOffQRope = kStages * kStageBytes;
constexpr uint32_t kOffRecv = kOffQRope + kQRopeBytes;
constexpr uint32_t kOffP = kOffRecv + 2 * kRecvBytes;
constexpr uint32_t kOffScore = kOffP + kPBytes;
constexpr uint32_t kOffTmax = kOffScore + kScoreBytes;   // [128] tile maxima, log2 units
constexpr uint32_t kOffBars = kOffTmax + 128 * 4;
constexpr uint32_t kOffSlot = kOffBars + 256;
constexpr uint32_t kSmemBytes = kOffSlot + 16 + 1024;   // + slack for 1024-B alignment
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(kOffP % 1024 == 0, "P tiles need 1024-byte alignment (128B swizzle atoms)");

// TMEM columns.
constexpr uint32_t kTmemO = 0;      // [0,256)   O half, fp32
constexpr uint32_t kTmemS = 256;    // [256,384) two score buffers of 64 fp32
constexpr uint32_t kTmemQ = 384;    // [384,512) q~ half: 256 bf16 packed in pairs

constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s per wait
constexpr float kRescaleThreshold = 8.0f;     // log2 units

enum Bar {
  kKvFull = 0,                   // [kStages] TMA -> MMA
  kKvEmpty = kStages,            // [kStages] MMA -> TMA
  // A parity wait must never skip a phase, or it can return on the stale completion of
  // the phase before.  So barriers that the two exchange groups (even / odd tiles) signal
  // or wait for are kept per tile parity: each waiter then sees every phase of its own.
  kSFull = 2 * kStages,          // [2] MMA -> softmax: partial scores in TMEM
  kSFree = 2 * kStages + 2,      // [2] exchange -> QK issuer: S buffer read (4 warps)
  kPFull = 2 * kStages + 4,      // [2] softmax -> PV issuer: P(i) in shared memory (256 threads)
  kPvDone = 2 * kStages + 6,     // [2] PV issuer -> softmax: PV(i) finished (P buffer, O stable)
  kRecvFull = 2 * kStages + 8,   // [2] peer partial landed (expect_tx by one thread here)
  kQFull = 2 * kStages + 10,
  kQReady = 2 * kStages + 11,
  kDrain = 2 * kStages + 12,
  kSReady = 2 * kStages + 17,    // exchange -> softmax: a tile's scores in smem (128 threads)
  kScoreFree = 2 * kStages + 18, // [2] softmax -> exchange: a tile's scores read (4 warps)
  kDrainPv = 2 * kStages + 20,
  kRecvRead = 2 * kStages + 21,  // [2] exchange -> exchange: a tile's peer partial read (4 warps)
  kNumBars = 2 * kStages + 23
};
static_assert(kNumBars * 8 <= 256, "barrier area");

struct Maps {
  CUtensorMap kv_lat;    // cache rows, box 64 cols x 64 rows, 128B swizzle
  CUtensorMap kv_rope;   // cache rows, box 32 cols x 64 rows, 64B swizzle
  CUtensorMap q_rope;    // q_cat rows, box 32 cols x 128 rows, 64B swizzle
};

__device__ __forceinline__ int tile_page(const DecodeParams& p, int b, int t) {
  return p.block_table[(int64_t)b * p.max_pages + t / kPage];
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
  return !__any_sync(0xffffffffu, !mbar_wait(bar, parity, kWaitNs));
}

__device__ __forceinline__ bool warp_wait_cluster(uint32_t bar, uint32_t parity) {
  return !__any_sync(0xffffffffu, !mbar_wait<true>(bar, parity, kWaitNs));
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
k_decode_sm103(const __grid_constant__ Maps maps, const DecodeParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s0 = smem_addr(smem);
  const uint32_t bars = s0 + kOffBars;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffSlot);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;

  // Work unit of this CTA pair.
  const int unit = blockIdx.x >> 1;
  const int m = unit / p.num_splits;          // query token b*S + s
  const int split = unit % p.num_splits;
  const int b = m / p.S, s = m % p.S;
  const int T = min(max(0, p.seqlens[b]), p.max_seqlen);
  int t0, t1;
  split_range(p, T, s, split, t0, t1);
  const int ntiles = t1 > t0 ? (t1 - t0 + kN - 1) / kN : 0;

  const int64_t rows_all = (int64_t)p.B * p.S * p.H;
  grid_dep_launch();
  if (ntiles == 0) {
    grid_dep_wait();   // the outputs below may still be read by the previous kernel
    // Nothing to read (an empty sequence, or a split past its end): both CTAs of the
    // pair leave before any shared set-up.  A split's partial is marked empty by its
    // lse alone (the merge skips it); an unsplit row is written as o_lat = 0, lse = -inf.
    for (int h = tid; h < p.H; h += kThreads) {
      const int64_t qrow = (int64_t)m * p.H + h;
      if (p.num_splits > 1) {
        if (rank == 0) p.lse_out[(int64_t)split * rows_all + qrow] = -INFINITY;
      } else {
        float4* out = reinterpret_cast<float4*>(p.o_out + qrow * kDc + 256 * rank);
        for (int v = 0; v < 64; ++v) out[v] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (rank == 0) p.lse_out[qrow] = -INFINITY;
      }
    }
    return;
  }

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(kKvFull + i), 1);
      mbar_init(bar(kKvEmpty + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kSFull + i), 1);
      mbar_init(bar(kSFree + i), kExchWarps / 2);
      mbar_init(bar(kScoreFree + i), kSoftmaxWarps);
      mbar_init(bar(kRecvRead + i), kExchWarps / 2);
      mbar_init(bar(kPFull + i), 32 * kSoftmaxWarps);
      mbar_init(bar(kPvDone + i), 1);
      mbar_init(bar(kRecvFull + i), 1);
    }
    mbar_init(bar(kQFull), 1);
    mbar_init(bar(kQReady), 32 * kExchWarps);
    mbar_init(bar(kSReady), 32 * kExchWarps / 2);
    mbar_init(bar(kDrain), 1);
    mbar_init(bar(kDrainPv), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers exist before any remote arrive
  const uint32_t tb = *tmem_slot;

  bool aborted = false;
  // Programmatic dependent launch: the TMA warp requests the first cache tiles (which no
  // earlier kernel writes) before waiting for the previous kernel; every other thread
  // waits here, before reading q_cat or writing outputs.
  if (warp != 0) grid_dep_wait();

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0 && ntiles > 0) {
      prefetch_tmap(&maps.kv_lat);
      prefetch_tmap(&maps.kv_rope);
      prefetch_tmap(&maps.q_rope);
      // Row coordinate of tile i in the tensor maps (a page past the pool for a bad
      // block-table entry: the copy then fills zeros and the tile is masked).
      auto tile_row = [&](int i, bool flag) -> int {
        const int t = t0 + i * kN;
        if (p.block_table) {
          const int page = tile_page(p, b, t);
          if (page < 0 || page >= p.num_pages) {
            if (flag) raise_flag(p.status, kFlagBlockTable);
            return p.num_pages * kPage;
          }
          return page * kPage;
        }
        return (int)((int64_t)b * p.kv_seq_stride + t);
      };
      int issued = 0;
      for (int i = 0; i < ntiles; ++i) {
        const int st = i % kStages;
        const uint32_t ph = (uint32_t)(i / kStages) & 1u;
        if (!mbar_wait(bar(kKvEmpty + st), ph ^ 1u, kWaitNs)) {
          aborted = true;
          break;
        }
        const int y = tile_row(i, true);
        const uint32_t stage = s0 + (uint32_t)st * kStageBytes;
        mbar_arrive_expect_tx(bar(kKvFull + st), kStageBytes);
        for (int j = 0; j < 4; ++j)
          tma_load_2d(stage + j * kBoxBytes, &maps.kv_lat, bar(kKvFull + st), 256 * (int)rank + 64 * j, y);
        tma_load_2d(stage + 4 * kBoxBytes, &maps.kv_rope, bar(kKvFull + st), kDc + 32 * (int)rank, y);
        ++issued;
        if (i == min(kStages, ntiles) - 1) {
          // The ring is full: now wait for the previous kernel, then fetch q^R from q_cat.
          grid_dep_wait();
          mbar_arrive_expect_tx(bar(kQFull), kQRopeBytes);
          tma_load_2d(s0 + kOffQRope, &maps.q_rope, bar(kQFull), kDc + 32 * (int)rank, m * p.H);
        }
      }
      // No copy may still be landing when the CTA exits.
      for (int i = max(0, issued - kStages); i < issued; ++i)
        mbar_wait(bar(kKvFull + i % kStages), (uint32_t)(i / kStages) & 1u, kWaitNs);
      if (!mbar_wait(bar(kQFull), 0, kWaitNs)) aborted = true;
    }
  } else if (warp == 1) {
    // ---------------- QK issuer ----------------
    // QK(i): partial scores of tile i into S buffer i & 1, once the tile has landed and
    // the softmax has read S buffer i & 1 (tile i-2).  Steps 0-15: latent half (A = q~
    // half from TMEM, B = cache rows, K-major, 128B swizzle); steps 16-17: rope half
    // (A = q^R half from smem, B = k^R half, 64B swizzle).  Shared-memory descriptors are
    // built once per tile: the 14-bit start field holds (address >> 4), so stepping
    // through a tile adds a compile-time constant to the 64-bit descriptor.
    if (lane == 0 && ntiles > 0) {
      const uint32_t id_qk = idesc_bf16(128, kN, false, false);
      const uint64_t qrope_desc = smem_desc(s0 + kOffQRope, 16, 512, kSwizzle64B);
      if (!mbar_wait(bar(kQFull), 0, kWaitNs) || !mbar_wait(bar(kQReady), 0, kWaitNs)) aborted = true;
      for (int i = 0; i < ntiles && !aborted; ++i) {
        if ((i >= 2 && !mbar_wait(bar(kSFree + (i & 1)), (uint32_t)((i - 2) >> 1) & 1u, kWaitNs)) ||
            !mbar_wait(bar(kKvFull + i % kStages), (uint32_t)(i / kStages) & 1u, kWaitNs)) {
          aborted = true;
          break;
        }
        tc_fence_after();
        const uint32_t stage = s0 + (uint32_t)(i % kStages) * kStageBytes;
        const uint32_t d = tb + kTmemS + 64u * (uint32_t)(i & 1);
        const uint64_t kv = smem_desc(stage, 16, 1024, kSwizzle128B);
        const uint64_t kr = smem_desc(stage + 4 * kBoxBytes, 16, 512, kSwizzle64B);
#pragma unroll
        for (int k = 0; k < 16; ++k)
          mma_ts(d, tb + kTmemQ + 8u * k, kv + (((k >> 2) * kBoxBytes + (k & 3) * 32u) >> 4), id_qk, k > 0);
#pragma unroll
        for (int k = 0; k < 2; ++k) mma_ss(d, qrope_desc + 2u * k, kr + 2u * k, id_qk, 1);
        mma_commit(bar(kSFull + (i & 1)));
      }
      mma_commit(bar(kDrain));
      mbar_wait(bar(kDrain), 0, kWaitNs);
    }
  } else if (warp == kPvWarp) {
    // ---------------- PV issuer ----------------
    // PV(i): O half += P(i) . V(i) once P(i) is in shared memory, then release the
    // stage and the P buffer.  A separate issuing warp lets a PV enter the tensor pipe
    // while a QK chain (18 dependent MMAs) is still being issued.  A = P (smem, K-major),
    // B = the staged tile read MN-major (N = 256 latent columns over four 64-column
    // boxes, K = 16 rows per step).
    if (lane == 0 && ntiles > 0) {
      const uint32_t id_pv = idesc_bf16(128, 256, false, true);
      for (int i = 0; i < ntiles; ++i) {
        const int buf = i & 1;
        if (!mbar_wait(bar(kPFull + buf), (uint32_t)(i >> 1) & 1u, kWaitNs)) {
          aborted = true;
          break;
        }
        tc_fence_after();
        const uint64_t pd = smem_desc(s0 + kOffP, 16, 1024, kSwizzle128B);
        const uint64_t vd = smem_desc(s0 + (uint32_t)(i % kStages) * kStageBytes, 8192, 1024, kSwizzle128B);
#pragma unroll
        for (int k = 0; k < kN / 16; ++k)
          mma_ss(tb + kTmemO, pd + 2u * k, vd + 128u * k, id_pv, (i > 0 || k > 0) ? 1u : 0u);
        mma_commit(bar(kKvEmpty + i % kStages));
        mma_commit(bar(kPvDone + buf));
      }
      mma_commit(bar(kDrainPv));
      mbar_wait(bar(kDrainPv), 0, kWaitNs);
    }
  } else if (warp < 2 + kExchWarps) {
    // ---------------- exchange (warps 2..9) ----------------
    // Warp w covers TMEM lane quarter q = w % 4 and the tiles i with i % 2 == e,
    // e = (w - 2) / 4 (S buffer e, receive buffer e): two warps per quarter, so that one
    // waits for the peer's partial of its tile while the other sends the next.  Per
    // tile: own fp32 partial scores (64 columns of 32 heads) out of TMEM, a bf16 copy to
    // the peer, the peer's bf16 partial in, the row maximum, and the scores relative to
    // it (fp16) into shared memory for the softmax warps.
    const int quarter = warp & 3;
    const int e = (warp - 2) >> 2;
    const int h = 32 * quarter + lane;               // head row == TMEM lane
    const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
    const bool head_ok = h < p.H;
    const int64_t qrow = (int64_t)m * p.H + h;
    const uint32_t xoff = (uint32_t)quarter * kQuarterXBytes + (uint32_t)lane * 16u;
    const uint32_t recv_local = s0 + kOffRecv;
    const uint32_t recv_peer = map_to_rank(recv_local, peer);
    const uint32_t recv_bar_peer = map_to_rank(bar(kRecvFull), peer);
    if (ntiles > 0) {
      // Half (e) of this head's 256 q~ columns into TMEM (A operand of the score MMA,
      // bf16 pairs packed in 32-bit columns).
      const uint4* src = reinterpret_cast<const uint4*>(p.q_cat + qrow * kRow + 256 * rank + 128 * e);
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t r[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 w = head_ok ? src[c * 8 + v] : make_uint4(0u, 0u, 0u, 0u);
          r[4 * v] = w.x;
          r[4 * v + 1] = w.y;
          r[4 * v + 2] = w.z;
          r[4 * v + 3] = w.w;
        }
        tmem_st32(tb + lane_off + kTmemQ + 64u * e + 32u * c, r);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(kQReady));
      if (h == 0 && e < ntiles) mbar_arrive_expect_tx(bar(kRecvFull + e), kRecvBytes);
    }
    for (int i = e; i < ntiles && !aborted; i += 2) {
      const int buf = e;
      const uint32_t ph = (uint32_t)(i >> 1) & 1u;
      const uint32_t ts = tb + lane_off + kTmemS + 64u * buf;
      if (!warp_wait(bar(kSFull + buf), ph)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      // Own fp32 partial scores; the S buffer is free for QK(i+2) once they are read.
      float x[64];
      tmem_ld32f<0>(ts, x);
      tmem_ld32f<32>(ts + 32u, x);   // both requested before one wait (~290 cycles each)
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kSFree + buf));
      // To the peer: [4 quarters][8 chunks][32 rows][16 B], chunk k = columns 8k..8k+7.
      // Receive buffer `buf` is reused two tiles later without a remote handshake: tile
      // i goes out only after the warps of tile i-1 here have read its peer partial
      // (kRecvRead), and the peer follows the same rule, so it sends tile i+2 only after
      // it has received tile i+1 from us, i.e. after we have read tile i.
      if (i >= 1 && !warp_wait(bar(kRecvRead + ((i - 1) & 1)), (uint32_t)((i - 1) >> 1) & 1u)) {
        aborted = true;
        break;
      }
      {
        const uint32_t dst = recv_peer + (uint32_t)buf * kRecvBytes + xoff;
        const uint32_t rb = recv_bar_peer + 8u * (uint32_t)buf;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          st_async_v4(dst + (uint32_t)c * 512u, f2_to_bf2(x[8 * c], x[8 * c + 1]),
                      f2_to_bf2(x[8 * c + 2], x[8 * c + 3]), f2_to_bf2(x[8 * c + 4], x[8 * c + 5]),
                      f2_to_bf2(x[8 * c + 6], x[8 * c + 7]), rb);
      }
      if (!warp_wait_cluster(bar(kRecvFull + buf), ph)) {
        aborted = true;
        break;
      }
      // Re-arm for tile i+2: the peer sends it only after our warps have read tile i.
      if (h == 0 && i + 2 < ntiles) mbar_arrive_expect_tx(bar(kRecvFull + buf), kRecvBytes);
      {
        const uint32_t rl = recv_local + (uint32_t)buf * kRecvBytes + xoff;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 w = ld_shared_u4(rl + (uint32_t)c * 512u);
          const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            x[8 * c + 2 * u] += __uint_as_float(ww[u] << 16);
            x[8 * c + 2 * u + 1] += __uint_as_float(ww[u] & 0xffff0000u);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kRecvRead + buf));
      // Readable rows of this tile, the row maximum over them (log2 units), and the
      // scores relative to it.  The softmax takes exp2 of these, so they are stored as
      // fp16: its error near 0, where the weights are largest, is under 2^-11 of the
      // value (far below the bf16 rounding of P), and -inf marks an unreadable row.
      const int t = t0 + i * kN;
      int valid = min(kN, t1 - t);
      if (p.block_table) {
        const int page = tile_page(p, b, t);
        if (page < 0 || page >= p.num_pages) valid = 0;
      }
      if (valid < kN) {
#pragma unroll
        for (int j = 0; j < kN; ++j)
          if (j >= valid) x[j] = -INFINITY;
      }
      float mx;
      {
        float t16[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) t16[j] = fmaxf(fmaxf(x[j], x[j + 16]), fmaxf(x[j + 32], x[j + 48]));
#pragma unroll
        for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
          for (int j = 0; j < w; ++j) t16[j] = fmaxf(t16[j], t16[j + w]);
        mx = t16[0] * p.scale_log2;
      }
      const float negmx = (mx == -INFINITY) ? 0.f : -mx;
      if (i >= 1 && !warp_wait(bar(kScoreFree + ((i - 1) & 1)), (uint32_t)((i - 1) >> 1) & 1u)) {
        aborted = true;
        break;
      }
      {
        const uint32_t row = s0 + kOffScore + (uint32_t)h * 128u;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t w[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            __half2 v = __floats2half2_rn(fmaf(x[8 * c + 2 * u], p.scale_log2, negmx),
                                          fmaf(x[8 * c + 2 * u + 1], p.scale_log2, negmx));
            w[u] = *reinterpret_cast<uint32_t*>(&v);
          }
          // Chunk c of row h at chunk c ^ (h & 7): conflict-free for row-per-lane access.
          st_shared_u4(row + (uint32_t)((c ^ (h & 7)) << 4), w[0], w[1], w[2], w[3]);
        }
        reinterpret_cast<float*>(smem + kOffTmax)[h] = mx;
      }
      mbar_arrive(bar(kSReady));
    }
  } else {
    // ---------------- softmax / epilogue (warps 10..13) ----------------
    // Warp w covers heads 32q..32q+31, q = w % 4 (its TMEM lane quarter, for O), and all
    // 64 columns of each tile, from the scores and row maxima the exchange warps leave in
    // shared memory.
    const int quarter = warp & 3;
    const int h = 32 * quarter + lane;
    const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
    const bool head_ok = h < p.H;
    const int64_t qrow = (int64_t)m * p.H + h;
    float m_ref = -INFINITY, l = 0.f;

    for (int i = 0; i < ntiles && !aborted; ++i) {
      const int buf = i & 1;
      if (!warp_wait(bar(kSReady), (uint32_t)i & 1u)) {
        aborted = true;
        break;
      }
      // Readable rows of this tile (for clearing the V rows past them below).
      const int t = t0 + i * kN;
      int valid = min(kN, t1 - t);
      if (p.block_table) {
        const int page = tile_page(p, b, t);
        if (page < 0 || page >= p.num_pages) valid = 0;
      }
      // The 64 scores of this row, relative to the tile maximum mx (log2 units).
      uint32_t xh[32];   // fp16 pairs
      const float mx = reinterpret_cast<const float*>(smem + kOffTmax)[h];
      {
        const uint32_t row = s0 + kOffScore + (uint32_t)h * 128u;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 w = ld_shared_u4(row + (uint32_t)((c ^ (h & 7)) << 4));
          xh[4 * c] = w.x;
          xh[4 * c + 1] = w.y;
          xh[4 * c + 2] = w.z;
          xh[4 * c + 3] = w.w;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kScoreFree + buf));
      // Lazy maximum: move the reference only when the tile exceeds it by > 2^8.
      const bool grow = mx > m_ref + kRescaleThreshold;
      const float m_new = grow ? mx : m_ref;
      const float alpha = grow ? ex2_approx(m_ref - m_new) : 1.f;   // 0 when m_ref = -inf
      l *= alpha;
      m_ref = m_new;
      // The P buffer is free, and O stable, once PV(i-1) is done.
      if (i >= 1 && !warp_wait(bar(kPvDone + ((i - 1) & 1)), (uint32_t)((i - 1) >> 1) & 1u)) {
        aborted = true;
        break;
      }
      // p = 2^(x + mx - m_ref); a tile with no readable row (mx = -inf) gives p = 0.
      const float neg = (mx == -INFINITY) ? -INFINITY : mx - m_ref;
      const uint32_t prow = s0 + kOffP + (uint32_t)h * 128u;
      float ps = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&xh[4 * c + u]));
          const float a = ex2_approx(f.x + neg);
          const float d = ex2_approx(f.y + neg);
          ps += a + d;
          w[u] = f2_to_bf2(a, d);
        }
        // 128B swizzle: 16-byte chunk c of row h sits at chunk c ^ (h & 7).
        st_shared_u4(prow + (uint32_t)((c ^ (h & 7)) << 4), w[0], w[1], w[2], w[3]);
      }
      l += ps;

      // Rescale this warp's rows of O (PV(i-1) has landed); xh is no longer live here.
      if (__any_sync(0xffffffffu, grow && i > 0)) {
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t r[32];
          const uint32_t ta = tb + lane_off + kTmemO + 32u * c;
          tmem_ld32(ta, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
          tmem_st32(ta, r);
        }
        tmem_st_wait();
        tc_fence_before();
      }

      // Rows past the readable range may hold anything (even NaN): clear them in the
      // V columns of the staged tile so that 0-weighted rows add exactly 0.
      if (valid < kN) {
        const uint32_t stage = s0 + (uint32_t)(i % kStages) * kStageBytes;
        const int nrow = kN - valid;
        for (int idx = tid - 32 * (2 + kExchWarps); idx < nrow * 32; idx += 32 * kSoftmaxWarps) {
          const int row = valid + idx / 32, c = idx % 32;   // 4 boxes x 8 chunks per row
          st_shared_v4_zero(stage + (uint32_t)(c >> 3) * kBoxBytes + (uint32_t)row * 128u +
                            (uint32_t)(c & 7) * 16u);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(kPFull + buf));
    }

    // Epilogue: this warp's rows of the O half, divided by the row sum.
    const int64_t orow = (p.num_splits > 1) ? (int64_t)split * rows_all + qrow : qrow;
    float* out = p.o_out + orow * kDc + 256 * rank;
    const bool have = ntiles > 0 && l > 0.f;
    if (ntiles > 0 && !aborted) {
      const int last = ntiles - 1;
      if (!warp_wait(bar(kPvDone + (last & 1)), (uint32_t)(last >> 1) & 1u)) aborted = true;
    }
    tc_fence_after();
    const float inv = have ? 1.f / l : 0.f;
    if (ntiles > 0 && !aborted) {
#pragma unroll 1
      for (int c = 0; c < 8; c += 2) {
        uint32_t r0[32], r1[32];
        tmem_ld32(tb + lane_off + kTmemO + 32u * c, r0);
        tmem_ld32(tb + lane_off + kTmemO + 32u * (c + 1), r1);
        tmem_ld_wait();
        if (head_ok) {
          // A row that saw no readable position (l == 0) is written as exact zeros.
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            reinterpret_cast<float4*>(out + 32 * c)[v] =
                have ? make_float4(__uint_as_float(r0[4 * v]) * inv, __uint_as_float(r0[4 * v + 1]) * inv,
                                   __uint_as_float(r0[4 * v + 2]) * inv, __uint_as_float(r0[4 * v + 3]) * inv)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
            reinterpret_cast<float4*>(out + 32 * (c + 1))[v] =
                have ? make_float4(__uint_as_float(r1[4 * v]) * inv, __uint_as_float(r1[4 * v + 1]) * inv,
                                   __uint_as_float(r1[4 * v + 2]) * inv, __uint_as_float(r1[4 * v + 3]) * inv)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
      }
    } else if (head_ok) {
      for (int v = 0; v < 64; ++v) reinterpret_cast<float4*>(out)[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (head_ok && rank == 0)
      p.lse_out[orow] = have ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
  }

  if (aborted) raise_flag(p.status, kFlagTimeout);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tb, 512);
  }
  cluster_sync();  // neither CTA leaves while the other may still touch its shared memory
}

bool encode_rows(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_cols,
                 uint32_t box_rows, CUtensorMapSwizzle sw) {
  return encode_tma_2d(map, true, base, kRow, rows, (uint64_t)kRow * 2, box_cols, box_rows, sw);
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t st) {
  Maps maps;
  const uint64_t kv_rows = p.block_table ? (uint64_t)p.num_pages * kPage
                                         : (uint64_t)p.B * (uint64_t)p.kv_seq_stride;
  const uint64_t q_rows = (uint64_t)p.B * p.S * p.H;
  if (kv_rows == 0 || kv_rows > 0x7FFFFFFFull) return cudaErrorInvalidValue;
  if (!encode_rows(&maps.kv_lat, p.kv, kv_rows, 64, kN, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_rows(&maps.kv_rope, p.kv, kv_rows, 32, kN, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !encode_rows(&maps.q_rope, p.q_cat, q_rows, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(k_decode_sm103, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const int units = p.B * p.S * p.num_splits;
  cudaError_t e = launch_pdl(k_decode_sm103, dim3(2 * units), dim3(kThreads), kSmemBytes, st, maps, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mla
