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
//   * the partials are swapped through distributed shared memory as fp16 (saturating at
//     +-65504), by 16-byte st.async into the peer's receive buffer (two, by tile parity),
//     counted (complete_tx) on its mbarrier.  A buffer is reused for tile i+2 once the
//     peer has read tile i out of it; the peer says so with a 4-byte st.async counted on
//     our "free" barrier (about 500 cycles under HBM load, where a remote
//     mbarrier.arrive.release took ~3900).  fp16 halves the bytes of fp32 partials and
//     rounds a partial by at most 2^-11 of its magnitude (bf16 would round by 2^-8).
//     Each CTA adds its own fp32 partial to the peer's fp16 partial and normalises its
//     half of O with its own softmax sums, so the two halves need not agree bit for bit;
//   * P (bf16) goes to shared memory in the 128B-swizzled K-major layout, and each CTA
//     accumulates its 256 columns of O in TMEM from P and its own V columns.
// Shared memory holds the score operands in a short ring (3 latent tiles, 2 rope tiles),
// released as soon as a tile's score MMAs are done.  The aggregation reads the same latent
// columns a second time, a few tiles later, into a ring of its own (2 tiles): that read is
// served by L2, and the score ring no longer stays occupied through exchange, softmax
// and aggregation (HBM bytes in flight, not tile compute, set the pace of a decode).
// Warp roles per CTA: warp 0 issues the score-ring TMA, warp 1 the score MMAs (QK), warp
// 14 the V re-reads and the aggregation MMAs (PV); warps 2-13 form three groups of four
// (one warp per TMEM lane quarter of 32 heads), group g taking the tiles i with i % 3 == g
// from partial scores to P: read the partial out of TMEM (freeing the S buffer at once),
// swap it with the peer, add, row maximum, reference maximum (handed from the group of the
// previous tile), exp2, P into shared memory.
// Softmax runs in the log2 domain with a lazily raised reference maximum (the running
// output is rescaled only when the maximum grows by more than 2^8); each group keeps its
// own share of the row sum, merged in the epilogue.
// Every mbarrier wait is bounded; on expiry the CTA records MLA_ERR_TIMEOUT in the
// status word, drains its own copies and MMAs, frees TMEM and exits.
#include <cuda.h>

#include "common.cuh"
#include "ptx_sm103.cuh"

namespace mla {

namespace {

using namespace ptx;

constexpr int kN = 64;                            // cache rows per tile
constexpr int kQkStages = 3;                      // latent tiles in flight for the score MMAs
constexpr int kRopeStages = 2;                    // rope tiles (their two MMAs close each chain)
constexpr int kVStages = 2;                       // latent tiles re-read for the aggregation MMAs
constexpr int kGroups = 3;                        // score-to-P groups: tile i goes to group i % 3
constexpr int kGroupWarps = 4;                    // one warp per TMEM lane quarter
constexpr int kPvWarp = 2 + kGroups * kGroupWarps;   // the warp that issues PV
constexpr int kThreads = 32 * (kPvWarp + 1);
constexpr int kGroupThreads = 32 * kGroupWarps;
constexpr uint32_t kBoxBytes = kN * 128;          // 64 rows x 64 bf16 (128B swizzle)
constexpr uint32_t kLatBytes = 4 * kBoxBytes;     // 64 rows x this CTA's 256 latent columns
constexpr uint32_t kRopeBoxBytes = kN * 64;       // 64 rows x 32 bf16 (64B swizzle)
constexpr uint32_t kQRopeBytes = 128 * 64;        // 128 heads x 32 bf16
constexpr uint32_t kRecvBytes = 128 * kN * 2;     // peer's fp16 partial scores
constexpr uint32_t kQuarterXBytes = 32 * kN * 2;  // one lane quarter's share: 32 rows x 64 columns
constexpr uint32_t kPBytes = 128 * kN * 2;        // P, bf16, 128 rows x 128 B

constexpr uint32_t kOffQk = 0;
constexpr uint32_t kOffRope = kOffQk + kQkStages * kLatBytes;
constexpr uint32_t kOffV = kOffRope + kRopeStages * kRopeBoxBytes;
constexpr uint32_t kOffQRope = kOffV + kVStages * kLatBytes;
constexpr uint32_t kOffRecv = kOffQRope + kQRopeBytes;
constexpr uint32_t kOffP = kOffRecv + 2 * kRecvBytes;
constexpr uint32_t kOffMref = kOffP + kPBytes;    // [128] reference maximum per head, log2 units
constexpr uint32_t kOffBars = kOffMref + 128 * 4;
constexpr uint32_t kOffSlot = kOffBars + 512;
constexpr uint32_t kOffSig = kOffSlot + 16;       // [4] landing words of the peer's "buffer free" signals
constexpr uint32_t kOffScale8 = (kOffSig + 16 + 127) & ~127u;   // FP8: [2 staging buffers][64 rows] fp32 row scales
constexpr uint32_t kSmemBytes = kOffScale8 + 2 * 64 * 4 + 1024;   // + slack for 1024-B alignment
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(kOffScale8 % 128 == 0, "TMA destination alignment");
static_assert(kOffV % 1024 == 0 && kOffP % 1024 == 0, "128B-swizzled tiles need 1024-byte alignment");
static_assert(kOffRope % 512 == 0 && kOffQRope % 512 == 0, "64B-swizzled tiles need 512-byte alignment");
static_assert(kGroups * kGroupThreads * 4 <= 2 * kRecvBytes, "row sums reuse the receive buffers");

// FP8 cache: a ring of kSlots8 bf16 tiles serves both products; a tile's E4M3 bytes (64
// rows x this CTA's 256 latent columns) land by TMA in staging buffer i % 2, from which
// the group that owns the tile (i % 3) widens them into slot i % 4.  Four slots let that
// group widen tile i right after finishing tile i-3 (PV(i-4), which held the slot, is
// done by then).  The staging buffers are shared by the groups, so before waiting for
// tile i's bytes the group waits for tile i-2 to be widened: the buffer's previous phase
// has then completed, and its parity wait cannot take the phase of tile i-2.
constexpr int kSlots8 = 4;
constexpr int kStages8 = 2;
constexpr uint32_t kLat8Bytes = kN * 256;          // 64 rows x 256 E4M3 bytes
constexpr uint32_t kOffStage8 = kOffQk + kSlots8 * kLatBytes;
constexpr uint32_t kOffRope8 = kOffQk + 5 * kLatBytes;   // q^R stays where the bf16 layout has it
constexpr int kRow8 = 640;                         // bytes of an FP8 cache row
static_assert(kOffStage8 + kStages8 * kLat8Bytes <= kOffRope8, "FP8 staging below the rope ring");
static_assert(kOffRope8 + kRopeStages * kRopeBoxBytes == kOffQRope, "the FP8 layout keeps q^R in place");
static_assert(kOffRope8 % 512 == 0 && kOffStage8 % 1024 == 0, "alignment");

// TMEM columns.
constexpr uint32_t kTmemO = 0;      // [0,256)   O half, fp32
constexpr uint32_t kTmemS = 256;    // [256,384) two score buffers of 64 fp32
constexpr uint32_t kTmemQ = 384;    // [384,512) q~ half: 256 bf16 packed in pairs

constexpr float kRescaleThreshold = 8.0f;     // log2 units

enum Bar {
  kQkFull = 0,                        // [kQkStages] TMA -> QK issuer: latent tile landed
  kRopeFull = kQkFull + kQkStages,    // [kRopeStages] TMA -> QK issuer: rope tile landed
  kVFull = kRopeFull + kRopeStages,   // [kVStages] re-read latent tile landed
  kVEmpty = kVFull + kVStages,        // [kVStages] PV done -> PV issuer
  // Barriers that a group waits for are kept per group (tile % 3): a parity wait must never
  // skip a phase, or it can return on the stale completion of the phase before, so every
  // waiter of a barrier must see each of its phases.
  kSFull = kVEmpty + kVStages,        // [3] QK(i) done -> group, and -> TMA (its slots are free)
  kSFree = kSFull + kGroups,          // [3] group -> QK issuer: S buffer read (4 warps)
  kRecvFull = kSFree + kGroups,       // [3] peer partial landed (expect_tx by one thread here)
  kRecvFree = kRecvFull + kGroups,    // [2] peer -> here: it has read our tile in its buffer i & 1
  kFreeSeen = kRecvFree + 2,          // [3] group -> next group: past its kRecvFree wait (4 warps)
  kSigSent = kFreeSeen + kGroups,     // [3] group -> next group: its "free" signal is out (4 warps)
  kMref = kSigSent + kGroups,        // [3] group -> next group: reference maximum (128 threads)
  kPvDone = kMref + kGroups,          // [3] PV issuer -> next group: P buffer free, O stable
  kPFull = kPvDone + kGroups,         // group -> PV issuer: P(i) in shared memory (128 threads)
  kQFull,
  kQReady,
  kDrain,
  kDrainPv,
  kVGo,                               // PV issuer -> TMA: the first V tiles are requested
  // FP8 cache only:
  kStageLoaded,                         // [kStages8] a tile's E4M3 bytes landed (TMA)
  kStageFree = kStageLoaded + kStages8, // [kStages8] the converting group has read them (4 warps)
  kSlotFull = kStageFree + kStages8,    // [kSlots8] bf16 tile in its slot (128 threads)
  kSlotEmpty = kSlotFull + kSlots8,     // [kSlots8] PV of the slot's tile done
  kNumBars = kSlotEmpty + kSlots8
};
static_assert(kNumBars * 8 <= 512, "barrier area");

struct Maps {
  CUtensorMap kv_lat;    // cache rows, box 64 cols x 64 rows, 128B swizzle; FP8: bytes, box 256 x 64
  CUtensorMap kv_rope;   // cache rows, box 32 cols x 64 rows, 64B swizzle (FP8: rows as 320 bf16)
  CUtensorMap q_rope;    // q_cat rows, box 32 cols x 128 rows, 64B swizzle
  CUtensorMap q_lat;     // q_cat rows, box 64 cols x 128 rows, 128B swizzle (bf16 cache: q~ staged)
  CUtensorMap o_store;   // output rows (o_lat or split partials) fp32, box 32 cols x H rows, 128B swizzle
  CUtensorMap kv_scale;  // FP8: the row scales as one line of fp32, box 64
};

// Epilogue staging: chunk c (32 output columns of the 128 head rows, 128 B per row,
// 128B-swizzled) at c * 16 KB, over the score and V rings, which are idle by then.
constexpr uint32_t kOffStage = 0;
constexpr uint32_t kStageChunk = 128 * 128;
static_assert(kOffStage + 8 * kStageChunk <= kOffQRope, "staging stays clear of q^R and the exchange buffers");

// bf16 cache: this CTA's 256 q~ columns of the 128 head rows land by TMA in the V ring
// (four 64-column boxes, 128B-swizzled), which takes its first tile only after groups 0
// and 1 have moved them into TMEM.
constexpr uint32_t kQLatBox = 128 * 128;
static_assert(4 * kQLatBox == kVStages * kLatBytes, "q~ fills the V ring");

__device__ __forceinline__ int tile_page(const DecodeParams& p, int b, int t) {
  return p.block_table[(int64_t)b * p.max_pages + t / kPage];
}

// Row coordinate of the tile starting at position t in the tensor maps (a page past the pool
// for a bad block-table entry: the copy then fills zeros and the tile is masked).
__device__ __forceinline__ int tile_row(const DecodeParams& p, int b, int t, bool flag) {
  if (p.block_table) {
    const int page = tile_page(p, b, t);
    if (page < 0 || page >= p.num_pages) {
      if (flag) raise_flag(p.status, kFlagBlockTable);
      return p.num_pages * kPage;
    }
    return page * kPage;
  }
  return (int)((int64_t)b * p.kv_seq_stride + t);
}

// Four E4M3 values (bytes of w, lowest first) to four bf16 (lo: the first two), times
// the bf16x2 multiplier mul2.  The hardware conversion to f16 is exact (every E4M3 value
// is an f16 normal or zero); moving the f16 exponent and mantissa bits down by 3 puts
// them in bf16 positions, which reads as the value times 2^-112; the multiplication by
// 2^112 * scale then gives scale * value, exactly when the scale is a power of two.
__device__ __forceinline__ void e4m3x4_to_bf16(uint32_t w, uint32_t mul2, uint32_t& lo, uint32_t& hi) {
  uint32_t h0, h1;
  asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n cvt.rn.f16x2.e4m3x2 %0, a;\n cvt.rn.f16x2.e4m3x2 %1, b;\n}"
      : "=r"(h0), "=r"(h1)
      : "r"(w));
  const uint32_t r0 = ((h0 & 0x7FFF7FFFu) >> 3) | (h0 & 0x80008000u);
  const uint32_t r1 = ((h1 & 0x7FFF7FFFu) >> 3) | (h1 & 0x80008000u);
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(lo) : "r"(r0), "r"(mul2));
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(hi) : "r"(r1), "r"(mul2));
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  return !__any_sync(0xffffffffu, !mbar_wait(bar, parity, limit_ns));
}

__device__ __forceinline__ bool warp_wait_cluster(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  return !__any_sync(0xffffffffu, !mbar_wait<true>(bar, parity, limit_ns));
}

// kTestHook: the instance launched only while the test hook mla_debug_inject_timeout is
// on, whose wait limit comes from the launch and whose score issuer may withhold a
// completion; the ordinary instance keeps the 2 s limit a compile-time constant.
// kFp8: the cache is in the FP8 form (E4M3 latent bytes, bf16 k^R, a scale per row).
template <bool kTestHook, bool kFp8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
k_decode_sm103(const __grid_constant__ Maps maps, const DecodeParams p) {
  const uint64_t wait_ns = kTestHook ? p.wait_ns : kDefaultWaitNs;
  constexpr uint32_t kRopeAt = kFp8 ? kOffRope8 : kOffRope;      // rope ring
  constexpr int kRopeX = kFp8 ? 256 : kDc;                        // first k^R column in the rope map
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
    for (int i = 0; i < kQkStages; ++i) mbar_init(bar(kQkFull + i), 1);
    for (int i = 0; i < kRopeStages; ++i) mbar_init(bar(kRopeFull + i), 1);
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(bar(kVFull + i), 1);
      mbar_init(bar(kVEmpty + i), 1);
    }
    for (int g = 0; g < kGroups; ++g) {
      mbar_init(bar(kSFull + g), 1);
      mbar_init(bar(kSFree + g), kGroupWarps);
      mbar_init(bar(kRecvFull + g), 1);
      mbar_init(bar(kFreeSeen + g), kGroupWarps);
      mbar_init(bar(kSigSent + g), kGroupWarps);
      mbar_init(bar(kMref + g), kGroupThreads);
      mbar_init(bar(kPvDone + g), 1);
    }
    mbar_init(bar(kPFull), kGroupThreads);
    mbar_init(bar(kQFull), 1);
    mbar_init(bar(kQReady), 2 * kGroupThreads);
    mbar_init(bar(kDrain), 1);
    mbar_init(bar(kDrainPv), 1);
    mbar_init(bar(kVGo), 1);
    mbar_init(bar(kRecvFree + 0), 1);
    mbar_init(bar(kRecvFree + 1), 1);
    if (kFp8) {
      for (int i = 0; i < kStages8; ++i) {
        mbar_init(bar(kStageLoaded + i), 1);
        mbar_init(bar(kStageFree + i), kGroupWarps);
      }
      for (int i = 0; i < kSlots8; ++i) {
        mbar_init(bar(kSlotFull + i), kGroupThreads);
        mbar_init(bar(kSlotEmpty + i), 1);
      }
    }
    fence_mbar_init();
    // The first waits on kRecvFree are for tiles 2 and 3 (the peer has read tiles 0, 1).
    if (ntiles > 2) mbar_arrive_expect_tx(bar(kRecvFree + 0), 4 * kGroupWarps);
    if (ntiles > 3) mbar_arrive_expect_tx(bar(kRecvFree + 1), 4 * kGroupWarps);
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
    // ---------------- TMA producer: score operands, straight from HBM ----------------
    // Tile i: its 256 latent columns into QK slot i % 3 (free once QK(i-3) is done) and its
    // 32 rope columns into rope slot i % 2 (free once QK(i-2) is done).  "QK(j) done" is the commit the score groups wait for (kSFull):
    // the TMA thread waits for each of its phases in order, and the next phase of that
    // barrier needs a tile that is requested only after the wait.
    if (kFp8 && lane == 0) {
      // FP8 cache: tile i's E4M3 bytes into staging buffer i % 2, free once tile i-2 has
      // been read out of it, and its k^R into rope slot i % 2 as for the bf16 cache.
      prefetch_tmap(&maps.kv_lat);
      prefetch_tmap(&maps.kv_rope);
      prefetch_tmap(&maps.q_rope);
      prefetch_tmap(&maps.kv_scale);
      int issued = 0, rope_issued = 0;
      bool q_issued = false;
      auto load_q = [&]() {
        grid_dep_wait();
        mbar_arrive_expect_tx(bar(kQFull), kQRopeBytes);
        tma_load_2d(s0 + kOffQRope, &maps.q_rope, bar(kQFull), kDc + 32 * (int)rank, m * p.H);
        q_issued = true;
      };
      for (int i = 0; i < ntiles; ++i) {
        const int ss = i % kStages8, rs = i % kRopeStages;
        const int y = tile_row(p, b, t0 + i * kN, true);
        if (i >= 1 && !q_issued) load_q();
        if (i >= kStages8 && !mbar_wait(bar(kStageFree + ss), (uint32_t)(i / kStages8 - 1) & 1u, wait_ns)) {
          aborted = true;
          break;
        }
        mbar_arrive_expect_tx(bar(kStageLoaded + ss), kLat8Bytes + kN * 4);
        tma_load_2d(s0 + kOffStage8 + (uint32_t)ss * kLat8Bytes, &maps.kv_lat, bar(kStageLoaded + ss),
                    256 * (int)rank, y);
        tma_load_2d(s0 + kOffScale8 + (uint32_t)ss * (kN * 4), &maps.kv_scale, bar(kStageLoaded + ss), y, 0);
        ++issued;
        if (i >= kRopeStages &&
            !mbar_wait(bar(kSFull + (i - kRopeStages) % kGroups), (uint32_t)((i - kRopeStages) / kGroups) & 1u, wait_ns)) {
          aborted = true;
          break;
        }
        mbar_arrive_expect_tx(bar(kRopeFull + rs), kRopeBoxBytes);
        tma_load_2d(s0 + kRopeAt + (uint32_t)rs * kRopeBoxBytes, &maps.kv_rope, bar(kRopeFull + rs),
                    kRopeX + 32 * (int)rank, y);
        ++rope_issued;
      }
      if (!q_issued && !aborted) load_q();
      // No copy may still be landing when the CTA exits.
      for (int i = max(0, issued - kStages8); i < issued; ++i)
        mbar_wait(bar(kStageLoaded + i % kStages8), (uint32_t)(i / kStages8) & 1u, wait_ns);
      for (int i = max(0, rope_issued - kRopeStages); i < rope_issued; ++i)
        mbar_wait(bar(kRopeFull + i % kRopeStages), (uint32_t)(i / kRopeStages) & 1u, wait_ns);
      if (q_issued && !mbar_wait(bar(kQFull), 0, wait_ns)) aborted = true;
    }
    if (!kFp8 && lane == 0) {
      prefetch_tmap(&maps.kv_lat);
      prefetch_tmap(&maps.kv_rope);
      prefetch_tmap(&maps.q_rope);
      prefetch_tmap(&maps.q_lat);
      int issued = 0, rope_issued = 0;
      bool q_issued = false;
      // q^R and q~ come from q_cat, which the previous kernel writes: they are requested
      // after the first tiles (which no kernel writes), and before the first wait that
      // needs QK(0).  q~ goes to the V ring (groups 0 and 1 move it into TMEM).
      auto load_q = [&]() {
        grid_dep_wait();
        mbar_arrive_expect_tx(bar(kQFull), kQRopeBytes + 4 * kQLatBox);
        tma_load_2d(s0 + kOffQRope, &maps.q_rope, bar(kQFull), kDc + 32 * (int)rank, m * p.H);
        for (int j = 0; j < 4; ++j)
          tma_load_2d(s0 + kOffV + (uint32_t)j * kQLatBox, &maps.q_lat, bar(kQFull), 256 * (int)rank + 64 * j,
                      m * p.H);
        q_issued = true;
      };
      auto qk_done = [&](int j) {
        return mbar_wait(bar(kSFull + j % kGroups), (uint32_t)(j / kGroups) & 1u, wait_ns);
      };
      for (int i = 0; i < ntiles; ++i) {
        const int qs = i % kQkStages, rs = i % kRopeStages;
        const int y = tile_row(p, b, t0 + i * kN, true);
        // Start-up order: tile 0, then q^R, then the other tiles, so that the first score
        // MMAs are not queued behind the whole start-up burst of every CTA.  Tile 3 reuses
        // the slot of tile 0, whose landing the aggregation issuer waits for (phase 0)
        // before it requests the first V tiles: it is requested only once those requests
        // are out (kVGo), so that wait cannot meet a later phase.
        if (i >= 1 && !q_issued) load_q();
        if (i == kQkStages && !mbar_wait(bar(kVGo), 0, wait_ns)) {
          aborted = true;
          break;
        }
        if (i >= kQkStages && !qk_done(i - kQkStages)) {
          aborted = true;
          break;
        }
        mbar_arrive_expect_tx(bar(kQkFull + qs), kLatBytes);
        for (int j = 0; j < 4; ++j)
          tma_load_2d(s0 + kOffQk + (uint32_t)qs * kLatBytes + j * kBoxBytes, &maps.kv_lat, bar(kQkFull + qs),
                      256 * (int)rank + 64 * j, y);
        ++issued;
        if (i >= kRopeStages && !qk_done(i - kRopeStages)) {
          aborted = true;
          break;
        }
        mbar_arrive_expect_tx(bar(kRopeFull + rs), kRopeBoxBytes);
        tma_load_2d(s0 + kOffRope + (uint32_t)rs * kRopeBoxBytes, &maps.kv_rope, bar(kRopeFull + rs),
                    kDc + 32 * (int)rank, y);
        ++rope_issued;
      }
      if (!q_issued && !aborted) load_q();
      // No copy may still be landing when the CTA exits.
      for (int i = max(0, issued - kQkStages); i < issued; ++i)
        mbar_wait(bar(kQkFull + i % kQkStages), (uint32_t)(i / kQkStages) & 1u, wait_ns);
      for (int i = max(0, rope_issued - kRopeStages); i < rope_issued; ++i)
        mbar_wait(bar(kRopeFull + i % kRopeStages), (uint32_t)(i / kRopeStages) & 1u, wait_ns);
      if (q_issued && !mbar_wait(bar(kQFull), 0, wait_ns)) aborted = true;
    }
  } else if (warp == 1) {
    // ---------------- QK issuer ----------------
    // QK(i): partial scores of tile i into S buffer i & 1, once group (i-2) % 3 has read
    // that buffer: 16 latent MMAs (A = q~ half from TMEM, B = cache rows, K-major, 128B
    // swizzle), then two rope MMAs (A = q^R half from smem, B = k^R half, 64B swizzle; the
    // rope tile is requested last, so it is awaited only here), and one commit.  Every
    // instruction of this thread queues behind the tcgen05 and shared-memory traffic of the
    // other warps, so the loop keeps to few waits and one commit (waits placed between the
    // MMAs of a chain slowed the issue down).  Shared-memory descriptors hold (address >> 4)
    // in their 14-bit start field, so stepping through a tile adds a compile-time constant
    // to the 64-bit descriptor.
    if (lane == 0) {
      const uint32_t id_qk = idesc_bf16(128, kN, false, false);
      const uint64_t qrope_desc = smem_desc(s0 + kOffQRope, 16, 512, kSwizzle64B);
      if (!mbar_wait(bar(kQFull), 0, wait_ns) || !mbar_wait(bar(kQReady), 0, wait_ns)) aborted = true;
      for (int i = 0; i < ntiles && !aborted; ++i) {
        // The latent tile: slot i % 3 of the score ring, or (FP8) of the widened ring.
        const int qs = kFp8 ? i % kSlots8 : i % kQkStages, rs = i % kRopeStages;
        const uint32_t full_bar = kFp8 ? bar(kSlotFull + qs) : bar(kQkFull + qs);
        const uint32_t full_ph = (uint32_t)(i / (kFp8 ? kSlots8 : kQkStages)) & 1u;
        const uint32_t d = tb + kTmemS + 64u * (uint32_t)(i & 1);
        if ((i >= 2 && !mbar_wait(bar(kSFree + (i - 2) % kGroups), (uint32_t)((i - 2) / kGroups) & 1u, wait_ns)) ||
            !mbar_wait(full_bar, full_ph, wait_ns)) {
          aborted = true;
          break;
        }
        tc_fence_after();
        const uint64_t kv = smem_desc(s0 + kOffQk + (uint32_t)qs * kLatBytes, 16, 1024, kSwizzle128B);
        const uint64_t kr = smem_desc(s0 + kRopeAt + (uint32_t)rs * kRopeBoxBytes, 16, 512, kSwizzle64B);
#pragma unroll
        for (int k = 0; k < 16; ++k)
          mma_ts(d, tb + kTmemQ + 8u * k, kv + (((k >> 2) * kBoxBytes + (k & 3) * 32u) >> 4), id_qk, k > 0 ? 1u : 0u);
        if (!mbar_wait(bar(kRopeFull + rs), (uint32_t)(i / kRopeStages) & 1u, wait_ns)) {
          aborted = true;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 2; ++k) mma_ss(d, qrope_desc + 2u * k, kr + 2u * k, id_qk, 1u);
        if (!(kTestHook && p.fault && i == 0)) mma_commit(bar(kSFull + i % kGroups));   // test hook: withheld
      }
      mma_commit(bar(kDrain));
      mbar_wait(bar(kDrain), 0, wait_ns);
    }
  } else if (warp == kPvWarp) {
    // ---------------- PV issuer (and the V re-reads) ----------------
    // The aggregation reads the same 256 latent columns of tile i again, into V slot i % 2,
    // a few tiles after the score ring fetched them (so from L2).  A stage of the score
    // ring is thus held only through the score MMAs, not through exchange and softmax.
    // V(i+1) is requested as soon as PV(i-1) has released its slot.  PV(i): O half +=
    // P(i) . V(i), A = P (smem, K-major), B = the V tile read MN-major (N = 256 latent
    // columns over four 64-column boxes, K = 16 rows per step).
    if (kFp8 && lane == 0) {
      // FP8 cache: PV(i) reads the widened tile in slot i % 4 (still in place: the slot is
      // refilled only after this PV) and releases the slot.
      const uint32_t id_pv = idesc_bf16(128, 256, false, true);
      for (int i = 0; i < ntiles && !aborted; ++i) {
        const int ss = i % kSlots8;
        if (!mbar_wait(bar(kPFull), (uint32_t)i & 1u, wait_ns)) {
          aborted = true;
          break;
        }
        tc_fence_after();
        const uint64_t pd = smem_desc(s0 + kOffP, 16, 1024, kSwizzle128B);
        const uint64_t vd = smem_desc(s0 + kOffQk + (uint32_t)ss * kLatBytes, 8192, 1024, kSwizzle128B);
#pragma unroll
        for (int k = 0; k < kN / 16; ++k)
          mma_ss(tb + kTmemO, pd + 2u * k, vd + 128u * k, id_pv, (i > 0 || k > 0) ? 1u : 0u);
        mma_commit(bar(kSlotEmpty + ss));
        mma_commit(bar(kPvDone + i % kGroups));
      }
      mma_commit(bar(kDrainPv));
      mbar_wait(bar(kDrainPv), 0, wait_ns);
    }
    if (!kFp8 && lane == 0) {
      const uint32_t id_pv = idesc_bf16(128, 256, false, true);
      auto load_v = [&](int i) {
        const int vs = i % kVStages;
        const int y = tile_row(p, b, t0 + i * kN, false);
        mbar_arrive_expect_tx(bar(kVFull + vs), kLatBytes);
        for (int j = 0; j < 4; ++j)
          tma_load_2d(s0 + kOffV + (uint32_t)vs * kLatBytes + j * kBoxBytes, &maps.kv_lat, bar(kVFull + vs),
                      256 * (int)rank + 64 * j, y);
      };
      int v_issued = 0;
      // The V ring holds q~ until groups 0 and 1 have moved it into TMEM.  The first V tiles
      // re-read latent rows that the score ring requested first: asked for once those have
      // landed, they are L2 hits rather than part of the start-up burst from HBM.
      if (!mbar_wait(bar(kQReady), 0, wait_ns)) aborted = true;
      for (; !aborted && v_issued < min(kVStages, ntiles); ++v_issued) {
        if (!mbar_wait(bar(kQkFull + v_issued), 0u, wait_ns)) break;
        load_v(v_issued);
      }
      mbar_arrive(bar(kVGo));
      if (v_issued < min(kVStages, ntiles)) aborted = true;
      for (int i = 0; i < ntiles && !aborted; ++i) {
        const int vs = i % kVStages;
        if (i + 1 < ntiles && i + 1 >= kVStages) {
          if (!mbar_wait(bar(kVEmpty + (i + 1) % kVStages), (uint32_t)((i + 1) / kVStages - 1) & 1u, wait_ns)) {
            aborted = true;
            break;
          }
          load_v(i + 1);
          ++v_issued;
        }
        if (!mbar_wait(bar(kPFull), (uint32_t)i & 1u, wait_ns) ||
            !mbar_wait(bar(kVFull + vs), (uint32_t)(i / kVStages) & 1u, wait_ns)) {
          aborted = true;
          break;
        }
        tc_fence_after();
        const uint64_t pd = smem_desc(s0 + kOffP, 16, 1024, kSwizzle128B);
        const uint64_t vd = smem_desc(s0 + kOffV + (uint32_t)vs * kLatBytes, 8192, 1024, kSwizzle128B);
#pragma unroll
        for (int k = 0; k < kN / 16; ++k)
          mma_ss(tb + kTmemO, pd + 2u * k, vd + 128u * k, id_pv, (i > 0 || k > 0) ? 1u : 0u);
        mma_commit(bar(kVEmpty + vs));
        mma_commit(bar(kPvDone + i % kGroups));
      }
      mma_commit(bar(kDrainPv));
      mbar_wait(bar(kDrainPv), 0, wait_ns);
      for (int i = max(0, v_issued - kVStages); i < v_issued; ++i)
        mbar_wait(bar(kVFull + i % kVStages), (uint32_t)(i / kVStages) & 1u, wait_ns);
    }
  } else {
    // ---------------- score-to-P groups (warps 2..13) ----------------
    // Group g = (w - 2) / 4 takes the tiles i with i % 3 == g; its warp w covers TMEM lane
    // quarter w % 4 (heads 32q..32q+31, one head per lane).  Per tile: own fp32 partial
    // scores out of TMEM, an fp16 copy to the peer, the peer's fp16 partial in, the row
    // maximum, the reference maximum (handed on from the group of tile i-1), P = 2^(s -
    // m_ref) into shared memory, and the running output rescaled when m_ref moves.  Each
    // group keeps its own share of the row sum; the shares are merged at the end.
    const int g = (warp - 2) / kGroupWarps;
    const int quarter = warp & 3;
    const int h = 32 * quarter + lane;               // head row == TMEM lane
    const int gtid = tid - 32 * (2 + g * kGroupWarps);
    const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
    const bool head_ok = h < p.H;
    const int64_t qrow = (int64_t)m * p.H + h;
    const uint32_t xoff = (uint32_t)quarter * kQuarterXBytes + (uint32_t)lane * 16u;
    const uint32_t recv_local = s0 + kOffRecv;
    const uint32_t recv_peer = map_to_rank(recv_local, peer);
    const uint32_t recv_bar_peer = map_to_rank(bar(kRecvFull + g), peer);
    const uint32_t free_bar_peer = map_to_rank(bar(kRecvFree), peer);
    const uint32_t sig_peer = map_to_rank(s0 + kOffSig + 4u * (uint32_t)quarter, peer);
    float* mref_sh = reinterpret_cast<float*>(smem + kOffMref);
    if (g < 2) {
      // Half g of this head's 256 q~ columns into TMEM (A operand of the score MMA,
      // bf16 pairs packed in 32-bit columns): from the boxes 2g and 2g+1 staged in the V
      // ring (row h, 16-byte chunk v at v ^ (h & 7)), or (FP8 cache) from q_cat itself.
      bool got = true;
      if (!kFp8) got = warp_wait(bar(kQFull), 0, wait_ns);
      if (got) {
        const uint4* src = reinterpret_cast<const uint4*>(p.q_cat + qrow * kRow + 256 * rank + 128 * g);
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          uint32_t r[32];
          const uint32_t box = s0 + kOffV + (uint32_t)(2 * g + c) * kQLatBox + (uint32_t)h * 128u;
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const uint4 w = !kFp8 ? ld_shared_u4(box + (uint32_t)((v ^ (h & 7)) << 4))
                                  : head_ok ? src[c * 8 + v] : make_uint4(0u, 0u, 0u, 0u);
            r[4 * v] = w.x;
            r[4 * v + 1] = w.y;
            r[4 * v + 2] = w.z;
            r[4 * v + 3] = w.w;
          }
          tmem_st32(tb + lane_off + kTmemQ + 64u * g + 32u * c, r);
        }
        tmem_st_wait();
      } else {
        aborted = true;
      }
      tc_fence_before();
      mbar_arrive(bar(kQReady));
    }
    if (h == 0 && g < ntiles) mbar_arrive_expect_tx(bar(kRecvFull + g), kRecvBytes);

    // FP8 cache: the group widens its own tiles (i % 3 == g) from staging into their slots,
    // tile g before its first tile and tile i+3 once it has finished tile i, each row
    // times its scale (landed with the bytes); rows past the readable range are written as
    // zeros (so their zero weights add exactly 0 in PV).
    auto tile_valid = [&](int j) {
      const int t = t0 + j * kN;
      int v = min(kN, t1 - t);
      if (p.block_table) {
        const int page = tile_page(p, b, t);
        if (page < 0 || page >= p.num_pages) v = 0;
      }
      return v;
    };
    auto convert = [&](int j) -> bool {
      const int ss = j % kSlots8, gs = j % kStages8;
      const uint32_t slot = s0 + kOffQk + (uint32_t)ss * kLatBytes;
      // Tile j-2 is widened (so staging buffer j % 2 is in the phase of tile j), tile j's
      // E4M3 bytes and scales have landed, and the slot is free (PV(j-4) is done: the group
      // waited for it before finishing tile j-3, so that wait returns at once).
      if ((j >= 2 && !warp_wait(bar(kSlotFull + (j - 2) % kSlots8), (uint32_t)((j - 2) / kSlots8) & 1u, wait_ns)) ||
          !warp_wait(bar(kStageLoaded + gs), (uint32_t)(j / kStages8) & 1u, wait_ns) ||
          (j >= kSlots8 && !warp_wait(bar(kSlotEmpty + ss), (uint32_t)(j / kSlots8 - 1) & 1u, wait_ns)))
        return false;
      // Eight passes over the tile's 64 rows x 16 chunks (16 E4M3 bytes each).  In pass
      // pp, the eight threads of a shared-memory wavefront take four chunks of an even row
      // and the four chunks of the other parity of quarter of the odd row after it: their
      // staging reads hit eight different bank groups, and so do their bf16 stores (the
      // 128B swizzle puts the even row's chunks in even and the odd row's in odd groups).
      const uint32_t stage = s0 + kOffStage8 + (uint32_t)gs * kLat8Bytes;
      const float* scl = reinterpret_cast<const float*>(smem + kOffScale8 + gs * (kN * 4));
      const int valid = tile_valid(j);
      const int sub = (gtid >> 2) & 1, l4 = gtid & 3;
      uint4 w[8];
      int rowv[8], qv[8];
#pragma unroll
      for (int pp = 0; pp < 8; ++pp) {
        const int k = pp * 16 + (gtid >> 3);             // task: row pair k / 4, quarter k % 4
        rowv[pp] = 2 * (k >> 2) + sub;
        qv[pp] = (k & 3) ^ sub;
        w[pp] = ld_shared_u4(stage + (uint32_t)rowv[pp] * 256u + (uint32_t)(16 * (4 * qv[pp] + l4)));
      }
      float sc[8];
#pragma unroll
      for (int pp = 0; pp < 8; ++pp) sc[pp] = scl[rowv[pp]];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kStageFree + gs));   // the staging buffer may be refilled
#pragma unroll
      for (int pp = 0; pp < 8; ++pp) {
        const int r = rowv[pp];
        const float mul = sc[pp] * 0x1p112f;
        const uint32_t mul2 = f2_to_bf2(mul, mul);
        const uint32_t ww[4] = {w[pp].x, w[pp].y, w[pp].z, w[pp].w};
        uint32_t o[8];
#pragma unroll
        for (int u = 0; u < 4; ++u) e4m3x4_to_bf16(ww[u], mul2, o[2 * u], o[2 * u + 1]);
        // Columns 16 (4 q + l4) .. +15: box q, 16-byte chunks 2 l4 and 2 l4 + 1 of the row.
        const uint32_t rowp = slot + (uint32_t)qv[pp] * kBoxBytes + (uint32_t)r * 128u;
        const uint32_t j0 = (uint32_t)(2 * l4), sw = (uint32_t)(r & 7);
        if (r < valid) {   // 128B swizzle: chunk c of row r sits at chunk c ^ (r & 7)
          st_shared_u4(rowp + ((j0 ^ sw) << 4), o[0], o[1], o[2], o[3]);
          st_shared_u4(rowp + (((j0 + 1) ^ sw) << 4), o[4], o[5], o[6], o[7]);
        } else {
          st_shared_v4_zero(rowp + ((j0 ^ sw) << 4));
          st_shared_v4_zero(rowp + (((j0 + 1) ^ sw) << 4));
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(kSlotFull + ss));
      return true;
    };
    if (kFp8 && g < ntiles && !convert(g)) aborted = true;

    float m_g = -INFINITY, l_g = 0.f;   // this group's share of the row sum, relative to m_g
    for (int i = g; i < ntiles && !aborted; i += kGroups) {
      const uint32_t ph = (uint32_t)(i / kGroups) & 1u;
      const uint32_t sb = (uint32_t)(i & 1);          // S buffer and receive buffer
      if (!warp_wait(bar(kSFull + g), ph, wait_ns)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      // Own fp32 partial scores; the S buffer is free for QK(i+2) once they are read.
      float x[64];
      {
        const uint32_t ts = tb + lane_off + kTmemS + 64u * sb;
        tmem_ld32f<0>(ts, x);
        tmem_ld32f<32>(ts + 32u, x);   // both requested before one wait
        tmem_ld_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kSFree + g));
      // To the peer: [4 quarters][8 chunks][32 rows][16 B], chunk k = columns 8k..8k+7, into
      // its receive buffer i & 1, once the peer has read tile i-2 out of it: each of its 4
      // warps then sends a 4-byte st.async counted on our kRecvFree[i & 1] (a remote
      // mbarrier arrive is far slower under load).  The groups pass this wait in tile order
      // (kFreeSeen), so each phase of kRecvFree[i & 1] is awaited after the one before it.
      if (i >= 1 && !warp_wait(bar(kFreeSeen + (i - 1) % kGroups), (uint32_t)((i - 1) / kGroups) & 1u, wait_ns)) {
        aborted = true;
        break;
      }
      if (i >= 2) {
        if (!warp_wait_cluster(bar(kRecvFree + sb), (uint32_t)((i - 2) >> 1) & 1u, wait_ns)) {
          aborted = true;
          break;
        }
        // Re-arm for the wait of tile i+2 (the peer's read of tile i).
        if (h == 0 && i + 2 < ntiles) mbar_arrive_expect_tx(bar(kRecvFree + sb), 4 * kGroupWarps);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kFreeSeen + g));
      {
        const uint32_t dst = recv_peer + sb * kRecvBytes + xoff;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          st_async_v4(dst + (uint32_t)c * 512u, f2_to_h2_sat(x[8 * c], x[8 * c + 1]),
                      f2_to_h2_sat(x[8 * c + 2], x[8 * c + 3]), f2_to_h2_sat(x[8 * c + 4], x[8 * c + 5]),
                      f2_to_h2_sat(x[8 * c + 6], x[8 * c + 7]), recv_bar_peer);
      }
      if (!warp_wait_cluster(bar(kRecvFull + g), ph, wait_ns)) {
        aborted = true;
        break;
      }
      // Re-arm for tile i+3 (its bytes can only come after the phase of tile i completed:
      // the peer sends tile i+3 after our "free" signal for tile i+1).
      if (h == 0 && i + kGroups < ntiles) mbar_arrive_expect_tx(bar(kRecvFull + g), kRecvBytes);
      {
        const uint32_t rl = recv_local + sb * kRecvBytes + xoff;
        uint4 w[8];
        uint32_t sig = 0;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          w[c] = ld_shared_u4(rl + (uint32_t)c * 512u);
          sig ^= w[c].x;
        }
        // Every lane's loads have returned (sig depends on them) before lane 0 tells the
        // peer that buffer i & 1 may be overwritten (by tile i+2, if there is one).  The
        // signals go out in tile order (kSigSent): the peer sends tile i+3, which lands on
        // kRecvFull of this group, only after our signal for tile i+1, hence after this
        // group's phase of tile i has completed and been read.
        asm volatile("" ::"r"(sig));
        if (i >= 1 && !warp_wait(bar(kSigSent + (i - 1) % kGroups), (uint32_t)((i - 1) / kGroups) & 1u, wait_ns)) {
          aborted = true;
          break;
        }
        if (lane == 0) {
          if (i + 2 < ntiles) st_async_b32(sig_peer, sig, free_bar_peer + 8u * sb);
          mbar_arrive(bar(kSigSent + g));
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t ww[4] = {w[c].x, w[c].y, w[c].z, w[c].w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            x[8 * c + 2 * u] = add_f16_lo(ww[u], x[8 * c + 2 * u]);
            x[8 * c + 2 * u + 1] = add_f16_hi(ww[u], x[8 * c + 2 * u + 1]);
          }
        }
      }
      // Readable rows of this tile and the row maximum over them (log2 units).
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
      // Lazy reference maximum, handed from tile to tile: it moves only when a tile's
      // maximum exceeds it by more than 2^8.
      float m_prev = -INFINITY;
      if (i >= 1) {
        if (!warp_wait(bar(kMref + (i - 1) % kGroups), (uint32_t)((i - 1) / kGroups) & 1u, wait_ns)) {
          aborted = true;
          break;
        }
        m_prev = mref_sh[h];
      }
      const bool grow = mx > m_prev + kRescaleThreshold;
      const float m_new = grow ? mx : m_prev;
      mref_sh[h] = m_new;
      mbar_arrive(bar(kMref + g));
      const float alpha = grow ? ex2_approx(m_prev - m_new) : 1.f;   // 0 when m_prev = -inf
      if (m_g != m_new) {
        l_g *= ex2_approx(m_g - m_new);
        m_g = m_new;
      }
      // p = 2^(s * scale_log2 - m_ref); unreadable rows (s = -inf) give p = 0, and so does
      // every row while no readable row has been seen (m_ref = -inf).
      const float bias = (m_new == -INFINITY) ? 0.f : -m_new;
      uint32_t pw[32];
      float ps = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float a = ex2_approx(fmaf(x[2 * j], p.scale_log2, bias));
        const float d = ex2_approx(fmaf(x[2 * j + 1], p.scale_log2, bias));
        ps += a + d;
        pw[j] = f2_to_bf2(a, d);
      }
      l_g += ps;
      // The P buffer is free, and O stable, once PV(i-1) is done.
      if (i >= 1 && !warp_wait(bar(kPvDone + (i - 1) % kGroups), (uint32_t)((i - 1) / kGroups) & 1u, wait_ns)) {
        aborted = true;
        break;
      }
      {
        const uint32_t prow = s0 + kOffP + (uint32_t)h * 128u;
#pragma unroll
        for (int c = 0; c < 8; ++c)   // 128B swizzle: 16-byte chunk c of row h sits at chunk c ^ (h & 7)
          st_shared_u4(prow + (uint32_t)((c ^ (h & 7)) << 4), pw[4 * c], pw[4 * c + 1], pw[4 * c + 2],
                       pw[4 * c + 3]);
      }
      // Rescale this warp's rows of O to the new reference (PV(i-1) has landed).
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
      // re-read V tile so that 0-weighted rows add exactly 0 (the FP8 widening writes them
      // as zeros).
      if (!kFp8 && valid < kN) {
        const int vs = i % kVStages;
        if (!warp_wait(bar(kVFull + vs), (uint32_t)(i / kVStages) & 1u, wait_ns)) {
          aborted = true;
          break;
        }
        const uint32_t vt = s0 + kOffV + (uint32_t)vs * kLatBytes;
        const int nrow = kN - valid;
        for (int idx = gtid; idx < nrow * 32; idx += kGroupThreads) {
          const int row = valid + idx / 32, c = idx % 32;   // 4 boxes x 8 chunks per row
          st_shared_v4_zero(vt + (uint32_t)(c >> 3) * kBoxBytes + (uint32_t)row * 128u + (uint32_t)(c & 7) * 16u);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(kPFull));
      if (kFp8 && i + kGroups < ntiles && !convert(i + kGroups)) {
        aborted = true;
        break;
      }
    }

    // Epilogue.  The groups' row-sum shares, each moved to the final reference maximum,
    // are summed through shared memory (the receive buffers are idle now); then each
    // group takes the column chunks c = g, g+3, g+6 of the O half, divided by the sum,
    // stages them in shared memory and writes each with one TMA store (full lines,
    // where per-thread row stores would scatter 16 bytes over 32 rows each).  Once the
    // last PV is done no copy is in flight and no MMA reads the rings, which hold the
    // staging.  A CTA that gave up writes its rows directly.
    named_bar_sync(1, kGroups * kGroupThreads);
    const float m_fin = mref_sh[h];
    float* lsh = reinterpret_cast<float*>(smem + kOffRecv);
    lsh[g * 128 + h] = (l_g > 0.f) ? l_g * ex2_approx(m_g - m_fin) : 0.f;
    named_bar_sync(1, kGroups * kGroupThreads);
    const float l = lsh[h] + lsh[128 + h] + lsh[256 + h];
    const int64_t orow = (p.num_splits > 1) ? (int64_t)split * rows_all + qrow : qrow;
    float* out = p.o_out + orow * kDc + 256 * rank;
    if (!aborted) {
      const int last = ntiles - 1;
      if (!warp_wait(bar(kPvDone + last % kGroups), (uint32_t)(last / kGroups) & 1u, wait_ns)) aborted = true;
    }
    const bool have = !aborted && l > 0.f;   // a row with no readable position: exact zeros
    tc_fence_after();
    const float inv = have ? 1.f / l : 0.f;
    // The group stages only if none of its four warps gave up (then no copy is in flight
    // into the rings); otherwise each warp writes its rows directly.
    const bool stage = named_bar_and(2 + g, kGroupThreads, !aborted);
#pragma unroll 1
    for (int c = g; c < 8; c += kGroups) {
      uint32_t r[32];
      if (!aborted) {
        tmem_ld32(tb + lane_off + kTmemO + 32u * c, r);
        tmem_ld_wait();
      }
      const uint32_t row = s0 + kOffStage + (uint32_t)c * kStageChunk + (uint32_t)h * 128u;
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const float4 o4 = have ? make_float4(__uint_as_float(r[4 * v]) * inv, __uint_as_float(r[4 * v + 1]) * inv,
                                             __uint_as_float(r[4 * v + 2]) * inv, __uint_as_float(r[4 * v + 3]) * inv)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        if (stage)   // 128B swizzle: 16-byte chunk v of row h sits at chunk v ^ (h & 7)
          st_shared_u4(row + (uint32_t)((v ^ (h & 7)) << 4), __float_as_uint(o4.x), __float_as_uint(o4.y),
                       __float_as_uint(o4.z), __float_as_uint(o4.w));
        else if (head_ok)
          reinterpret_cast<float4*>(out + 32 * c)[v] = o4;
      }
    }
    if (stage) {
      fence_proxy_async_smem();
      named_bar_sync(2 + g, kGroupThreads);
      if (gtid == 0) {
        const int y = (int)((p.num_splits > 1 ? (int64_t)split * rows_all : 0) + (int64_t)m * p.H);
        for (int c = g; c < 8; c += kGroups)
          tma_store_2d(&maps.o_store, 256 * (int)rank + 32 * c, y, s0 + kOffStage + (uint32_t)c * kStageChunk);
        bulk_commit_group();
        bulk_wait_group_read0();   // the staging outlives its reads; the writes finish with the grid
      }
    }
    if (g == 0 && head_ok && rank == 0)
      p.lse_out[orow] = have ? (m_fin + log2f(l)) * kLn2 : -INFINITY;
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

// Tensor maps and launch of one instance.  The FP8 cache is read through two maps over
// its 640-byte rows: the E4M3 bytes (box 256 bytes x 64 rows, no swizzle) and k^R (the
// rows viewed as 320 bf16, box 32 x 64, 64B swizzle).
template <bool kFp8>
cudaError_t launch_decode_impl(DecodeParams p, cudaStream_t st) {
  Maps maps;
  const uint64_t kv_rows = p.block_table ? (uint64_t)p.num_pages * kPage
                                         : (uint64_t)p.B * (uint64_t)p.kv_seq_stride;
  const uint64_t q_rows = (uint64_t)p.B * p.S * p.H;
  if (kv_rows == 0 || kv_rows > 0x7FFFFFFFull) return cudaErrorInvalidValue;
  const uint64_t o_rows = q_rows * (uint64_t)(p.num_splits > 1 ? p.num_splits : 1);
  const bool kv_ok =
      kFp8 ? encode_tma_2d_u8(&maps.kv_lat, p.kv, kRow8, kv_rows, kRow8, 256, kN, CU_TENSOR_MAP_SWIZZLE_NONE) &&
                 encode_tma_2d(&maps.kv_rope, true, p.kv, kRow8 / 2, kv_rows, kRow8, 32, kN, CU_TENSOR_MAP_SWIZZLE_64B)
           : encode_rows(&maps.kv_lat, p.kv, kv_rows, 64, kN, CU_TENSOR_MAP_SWIZZLE_128B) &&
                 encode_rows(&maps.kv_rope, p.kv, kv_rows, 32, kN, CU_TENSOR_MAP_SWIZZLE_64B);
  // FP8: the scales as one line of kv_rows fp32 (x = the tile's first row, a multiple of 4).
  const bool scale_ok = !kFp8 || encode_tma_2d(&maps.kv_scale, false, p.kv_scale, kv_rows, 1,
                                               (kv_rows * 4 + 15) & ~uint64_t(15), kN, 1, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (!kv_ok || !scale_ok || !encode_rows(&maps.q_rope, p.q_cat, q_rows, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !encode_rows(&maps.q_lat, p.q_cat, q_rows, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tma_2d(&maps.o_store, false, p.o_out, kDc, o_rows, (uint64_t)kDc * 4, 32, (uint32_t)p.H,
                     CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const WaitConfig wc = wait_config(kFaultDecode);
  p.wait_ns = wc.wait_ns;
  p.fault = wc.fault;
  static SmemOptIn opt_in, opt_in_hook;
  cudaError_t e = wc.fault ? ensure_dynamic_smem((const void*)k_decode_sm103<true, kFp8>, (int)kSmemBytes, opt_in_hook)
                           : ensure_dynamic_smem((const void*)k_decode_sm103<false, kFp8>, (int)kSmemBytes, opt_in);
  if (e != cudaSuccess) return e;
  const int units = p.B * p.S * p.num_splits;
  e = wc.fault ? launch_pdl(k_decode_sm103<true, kFp8>, dim3(2 * units), dim3(kThreads), kSmemBytes, st, maps, p)
               : launch_pdl(k_decode_sm103<false, kFp8>, dim3(2 * units), dim3(kThreads), kSmemBytes, st, maps, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(DecodeParams p, cudaStream_t st) { return launch_decode_impl<false>(p, st); }

cudaError_t launch_decode_fp8(DecodeParams p, cudaStream_t st) { return launch_decode_impl<true>(p, st); }

}  // namespace mla
