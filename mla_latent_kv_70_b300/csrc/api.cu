// The C ABI of include/mla.h: argument checks, split planning, launches.
#include <algorithm>
#include <vector>
#include <cmath>
#include <cstdint>

#include "common.cuh"
#include "gemm.cuh"

using mla::kDc;
using mla::kPage;
using mla::kRow;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool heads_ok(int H) { return H >= 16 && H <= 128 && H % 16 == 0; }

// Split count for the CTA-pair decode: each non-empty (query token, split) unit occupies
// two SMs.  A split is a chunk of C = ceil(max_seqlen / s) rows (rounded to 64), so the
// run takes about waves(s) x C row-times, where waves(s) = ceil(units / pair slots) and
// units ~ total_rows / C plus half a chunk per query token for the ragged ends; splitting
// adds a round trip of fp32 partials (513 values per head per unit).  Pick the count with
// the least estimated traffic-time, in bytes moved by the whole GPU.
int auto_splits(int B, int S, int H, int max_seqlen, int64_t total_rows, int sms) {
  if (sms <= 0) sms = 148;
  if (max_seqlen <= 0) return 1;
  const int slots = sms / 2;
  const int tiles = (max_seqlen + 63) / 64;
  const int64_t tokens = (int64_t)B * S;
  const double rows = total_rows > 0 ? (double)total_rows : (double)B * (double)max_seqlen;
  int best = 1;
  double best_cost = 0.0;
  for (int s = 1; s <= MLA_MAX_SPLITS && s <= tiles; ++s) {
    int chunk = (max_seqlen + s - 1) / s;
    chunk = (chunk + 63) & ~63;
    double units = rows * S / chunk + 0.5 * (double)tokens;
    units = units < (double)tokens ? (double)tokens : units;
    const double cap = (double)tokens * s;
    units = units > cap ? cap : units;
    const double waves = ceil(units / slots);
    const double cost = waves * chunk * 1152.0 * slots +
                        (s > 1 ? units * H * (kDc + 1) * 4.0 * 2.0 : 0.0);
    if (s == 1 || cost < best_cost * 0.98) {
      best = s;
      best_cost = cost;
    }
  }
  return best;
}

// Times of the CTA-pair decode on a B300, measured on the DeepSeek-V3 shape (H = 128): a
// unit's fixed cost (set-up, first tiles, drain, epilogue; less for a unit that starts
// after the launch, whose first requests do not queue behind every other pair's) and each
// 64-row tile after it; an empty unit only writes its empty partial; the merge is a launch
// plus one pass over the fp32 partials.
constexpr double kUnitFixedUs = 17.0, kLaterUnitFixedUs = 11.0, kTileUs = 1.036, kEmptyUnitUs = 1.5;
constexpr double kMergeFixedUs = 3.0, kMergeBytesPerUs = 6.0e6;

// Estimated decode time with `s` splits: units are handed to the pair slots in launch
// order ((query token, split), token-major), each to the slot that frees first, as the
// hardware starts a cluster wherever one finishes.
double simulate_splits(const int32_t* seqlens, int B, int S, int H, int causal, int max_seqlen, int s,
                       int slots, std::vector<double>& heap) {
  int chunk = (max_seqlen + s - 1) / s;
  chunk = (chunk + 63) & ~63;
  heap.assign((size_t)slots, 0.0);   // a min-heap of the times the slots free up
  auto cmp = [](double x, double y) { return x > y; };
  for (int b = 0; b < B; ++b) {
    const int T = std::min(std::max(0, seqlens[b]), max_seqlen);
    for (int q = 0; q < S; ++q) {
      const int n_vis = causal ? std::min(T, std::max(0, T - S + q + 1)) : T;
      for (int k = 0; k < s; ++k) {
        const int t0 = std::min(k * chunk, n_vis), t1 = std::min(t0 + chunk, n_vis);
        const int tiles = (t1 - t0 + 63) / 64;
        std::pop_heap(heap.begin(), heap.end(), cmp);
        const double fixed = heap.back() < 3.0 ? kUnitFixedUs : kLaterUnitFixedUs;
        heap.back() += tiles > 0 ? fixed + tiles * kTileUs : kEmptyUnitUs;
        std::push_heap(heap.begin(), heap.end(), cmp);
      }
    }
  }
  double t = *std::max_element(heap.begin(), heap.end());
  if (s > 1) t += kMergeFixedUs + (double)s * B * S * H * (kDc + 1) * 4.0 * 2.0 / kMergeBytesPerUs;
  return t;
}

mla_status launch_status(cudaError_t e) {
  if (e == cudaSuccess) return MLA_OK;
  cudaGetLastError();
  return MLA_ERR_CUDA;
}

}  // namespace

mla_status mla::check_decode_args(const void* q_cat, const void* kv, int64_t kv_seq_stride,
                                  const int32_t* seqlens, const int32_t* block_table, int max_pages,
                                  int page_size, int num_pages, int B, int S, int H, float scale,
                                  int num_splits, int max_seqlen, const float* o_lat, const float* lse) {
  if (!q_cat || !kv || !seqlens || !o_lat || !lse) return MLA_ERR_INVALID;
  if (B < 1 || S < 1 || H < 1 || max_seqlen < 0) return MLA_ERR_INVALID;
  if (!aligned16(q_cat) || !aligned16(kv) || !aligned16(o_lat)) return MLA_ERR_INVALID;
  if (!heads_ok(H) || S > 4) return MLA_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || !std::isfinite(scale)) return MLA_ERR_INVALID;
  if (num_splits < 0 || num_splits > MLA_MAX_SPLITS) return MLA_ERR_INVALID;
  if (block_table) {
    if (page_size != kPage) return MLA_ERR_UNSUPPORTED;
    if (max_pages < 1 || num_pages < 1) return MLA_ERR_INVALID;
    if ((int64_t)max_pages * kPage < max_seqlen) return MLA_ERR_INVALID;
  } else {
    if (kv_seq_stride < max_seqlen || kv_seq_stride < 0) return MLA_ERR_INVALID;
  }
  return MLA_OK;
}

extern "C" {

const char* mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID: return "MLA_ERR_INVALID";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE";
    case MLA_ERR_BLOCK_TABLE: return "MLA_ERR_BLOCK_TABLE";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT";
    default: return "MLA_ERR_UNKNOWN";
  }
}

int mla_device_sm_count(void) { return mla::device_sm_count(); }

mla_status mla_absorb_q(const mla_bf16* q_nope, const mla_bf16* q_rope, const mla_bf16* w_uk,
                        const int32_t* q_pos, float rope_theta, int B, int S, int H,
                        mla_bf16* q_cat, mla_stream stream) {
  if (!q_nope || !q_rope || !w_uk || !q_cat) return MLA_ERR_INVALID;
  if (B < 1 || S < 1 || H < 1) return MLA_ERR_INVALID;
  if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(w_uk) || !aligned16(q_cat))
    return MLA_ERR_INVALID;
  if (!heads_ok(H) || S > 4) return MLA_ERR_UNSUPPORTED;
  if (q_pos && !(rope_theta > 0.f)) return MLA_ERR_INVALID;
  const mla::RopeFreqs f = mla::make_rope_freqs(q_pos ? rope_theta : 10000.f);
  return launch_status(mla::launch_absorb_q(
      reinterpret_cast<const __nv_bfloat16*>(q_nope), reinterpret_cast<const __nv_bfloat16*>(q_rope),
      reinterpret_cast<const __nv_bfloat16*>(w_uk), q_pos, f, B * S, H,
      reinterpret_cast<__nv_bfloat16*>(q_cat), static_cast<cudaStream_t>(stream)));
}

int mla_decode_num_splits(int B, int S, int H, int max_seqlen, int64_t total_rows) {
  if (B < 1 || S < 1 || max_seqlen < 0) return 1;
  return auto_splits(B, S, H, max_seqlen, total_rows, mla::device_sm_count());
}

int mla_decode_plan_splits(const int32_t* seqlens, int B, int S, int H, int causal, int max_seqlen) {
  if (!seqlens || B < 1 || S < 1 || S > 4 || !heads_ok(H) || max_seqlen < 0) return 0;
  int longest = 0;
  for (int b = 0; b < B; ++b) longest = std::max(longest, std::min(std::max(0, seqlens[b]), max_seqlen));
  if (longest == 0) return 1;
  const int sms = mla::device_sm_count() > 0 ? mla::device_sm_count() : 148;
  const int slots = std::max(1, sms / 2);
  const int tiles = (max_seqlen + 63) / 64;
  std::vector<double> heap;
  int best = 1;
  double best_t = 0.0;
  for (int s = 1; s <= MLA_MAX_SPLITS && s <= tiles; ++s) {
    if ((int64_t)B * S * s > (1 << 22)) break;   // bounds the host work
    const double t = simulate_splits(seqlens, B, S, H, causal, max_seqlen, s, slots, heap);
    if (s == 1 || t < best_t * 0.98) {
      best = s;
      best_t = t;
    }
  }
  return best;
}

size_t mla_decode_workspace_bytes(int B, int S, int H, int num_splits, int max_seqlen) {
  if (B < 1 || S < 1 || H < 1 || num_splits < 0 || num_splits > MLA_MAX_SPLITS) return 0;
  const int splits = num_splits ? num_splits : mla_decode_num_splits(B, S, H, max_seqlen, 0);
  if (splits <= 1) return 0;
  const size_t rows = (size_t)B * S * H;
  return (size_t)splits * rows * (kDc + 1) * sizeof(float);
}

namespace {

// The decode over either form of the cache (fp8: kv is the 640-byte-row form, kv_scale
// its scales).
mla_status decode_any(const mla_bf16* q_cat, const void* kv, const float* kv_scale, bool fp8,
                      int64_t kv_seq_stride, const int32_t* seqlens, const int32_t* block_table,
                      int max_pages, int page_size, int num_pages, int B, int S, int H, int causal,
                      float scale, int num_splits, int max_seqlen, float* o_lat, float* lse,
                      void* workspace, size_t workspace_bytes, int32_t* status_dev, mla_stream stream) {
  const mla_status bad = mla::check_decode_args(q_cat, kv, kv_seq_stride, seqlens, block_table,
                                                max_pages, page_size, num_pages, B, S, H, scale,
                                                num_splits, max_seqlen, o_lat, lse);
  if (bad != MLA_OK) return bad;
  // FP8: a tile's 64 scales are one TMA box, so the scale array is 16-byte aligned and a
  // contiguous cache keeps sequences a multiple of 4 rows apart.
  if (fp8 && (!kv_scale || !aligned16(kv_scale) || (!block_table && kv_seq_stride % 4))) return MLA_ERR_INVALID;
  const int splits = num_splits ? num_splits : mla_decode_num_splits(B, S, H, max_seqlen, 0);
  const size_t need = mla_decode_workspace_bytes(B, S, H, splits, max_seqlen);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace)))
    return MLA_ERR_WORKSPACE;

  const int64_t rows = (int64_t)B * S * H;
  mla::DecodeParams p{};
  p.q_cat = reinterpret_cast<const __nv_bfloat16*>(q_cat);
  p.kv = reinterpret_cast<const __nv_bfloat16*>(kv);
  p.kv_scale = kv_scale;
  p.kv_seq_stride = kv_seq_stride;
  p.seqlens = seqlens;
  p.block_table = block_table;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  p.max_seqlen = max_seqlen;
  p.B = B;
  p.S = S;
  p.H = H;
  p.causal = causal ? 1 : 0;
  p.scale_log2 = scale * mla::kLog2e;
  p.num_splits = splits;
  p.status = status_dev;
  float* part_o = static_cast<float*>(workspace);
  float* part_lse = part_o ? part_o + (size_t)splits * rows * kDc : nullptr;
  p.o_out = splits > 1 ? part_o : o_lat;
  p.lse_out = splits > 1 ? part_lse : lse;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  mla_status r = launch_status(fp8 ? mla::launch_decode_fp8(p, st) : mla::launch_decode(p, st));
  if (r != MLA_OK || splits <= 1) return r;
  return launch_status(mla::launch_combine(part_o, part_lse, splits, rows, o_lat, lse, st));
}

}  // namespace

mla_status mla_decode_latent(const mla_bf16* q_cat, const mla_bf16* kv, int64_t kv_seq_stride,
                             const int32_t* seqlens, const int32_t* block_table, int max_pages,
                             int page_size, int num_pages, int B, int S, int H, int causal,
                             float scale, int num_splits, int max_seqlen, float* o_lat,
                             float* lse, void* workspace, size_t workspace_bytes,
                             int32_t* status_dev, mla_stream stream) {
  return decode_any(q_cat, kv, nullptr, false, kv_seq_stride, seqlens, block_table, max_pages, page_size,
                    num_pages, B, S, H, causal, scale, num_splits, max_seqlen, o_lat, lse, workspace,
                    workspace_bytes, status_dev, stream);
}

mla_status mla_decode_latent_fp8(const mla_bf16* q_cat, const uint8_t* kv8, const float* kv_scale,
                                 int64_t kv_seq_stride, const int32_t* seqlens, const int32_t* block_table,
                                 int max_pages, int page_size, int num_pages, int B, int S, int H,
                                 int causal, float scale, int num_splits, int max_seqlen, float* o_lat,
                                 float* lse, void* workspace, size_t workspace_bytes,
                                 int32_t* status_dev, mla_stream stream) {
  return decode_any(q_cat, kv8, kv_scale, true, kv_seq_stride, seqlens, block_table, max_pages, page_size,
                    num_pages, B, S, H, causal, scale, num_splits, max_seqlen, o_lat, lse, workspace,
                    workspace_bytes, status_dev, stream);
}

mla_status mla_quantize_fp8(const mla_bf16* rows, int64_t row_stride, int64_t n_rows, uint8_t* kv8,
                            float* kv_scale, mla_stream stream) {
  if (!rows || !kv8 || !kv_scale || n_rows < 0 || row_stride < kRow || row_stride % 8) return MLA_ERR_INVALID;
  if (!aligned16(rows) || !aligned16(kv8) || (reinterpret_cast<uintptr_t>(kv_scale) & 3u)) return MLA_ERR_INVALID;
  if (n_rows == 0) return MLA_OK;
  return launch_status(mla::launch_quantize_fp8(reinterpret_cast<const __nv_bfloat16*>(rows), row_stride, n_rows,
                                                kv8, kv_scale, static_cast<cudaStream_t>(stream)));
}

mla_status mla_combine_partials(const float* o_part, const float* lse_part, int num_splits,
                                int64_t rows, float* o_lat, float* lse, mla_stream stream) {
  if (!o_part || !lse_part || !o_lat || !lse) return MLA_ERR_INVALID;
  if (num_splits < 1 || num_splits > MLA_MAX_SPLITS || rows < 0) return MLA_ERR_INVALID;
  if (!aligned16(o_part) || !aligned16(o_lat)) return MLA_ERR_INVALID;
  return launch_status(mla::launch_combine(o_part, lse_part, num_splits, rows, o_lat, lse,
                                           static_cast<cudaStream_t>(stream)));
}

mla_status mla_out_proj_uv(const float* o_lat, const mla_bf16* w_uv, int B, int S, int H,
                           float* o, mla_stream stream) {
  if (!o_lat || !w_uv || !o) return MLA_ERR_INVALID;
  if (B < 1 || S < 1 || H < 1) return MLA_ERR_INVALID;
  if (!aligned16(o_lat) || !aligned16(w_uv) || !aligned16(o)) return MLA_ERR_INVALID;
  if (!heads_ok(H) || S > 4) return MLA_ERR_UNSUPPORTED;
  return launch_status(mla::launch_out_proj_uv(o_lat, reinterpret_cast<const __nv_bfloat16*>(w_uv),
                                               B * S, H, o, static_cast<cudaStream_t>(stream)));
}

mla_status mla_append_latent(const mla_bf16* rows, int B, int S, float rope_theta, int32_t* seqlens,
                             mla_bf16* kv, int64_t kv_seq_stride, const int32_t* block_table,
                             int max_pages, int page_size, int num_pages, int32_t* status_dev,
                             mla_stream stream) {
  if (!rows || !seqlens || !kv) return MLA_ERR_INVALID;
  if (B < 1 || S < 1 || rope_theta < 0.f || !std::isfinite(rope_theta)) return MLA_ERR_INVALID;
  if (!aligned16(rows) || !aligned16(kv)) return MLA_ERR_INVALID;
  if (block_table) {
    if (page_size != kPage) return MLA_ERR_UNSUPPORTED;
    if (max_pages < 1 || num_pages < 1) return MLA_ERR_INVALID;
  } else if (kv_seq_stride < 1) {
    return MLA_ERR_INVALID;
  }
  const mla::RopeFreqs f = mla::make_rope_freqs(rope_theta > 0.f ? rope_theta : 10000.f);
  return launch_status(mla::launch_append_latent(
      reinterpret_cast<const __nv_bfloat16*>(rows), B, S, seqlens, reinterpret_cast<__nv_bfloat16*>(kv),
      kv_seq_stride, block_table, max_pages, num_pages, rope_theta > 0.f ? 1 : 0, f, status_dev,
      static_cast<cudaStream_t>(stream)));
}

mla_status mla_append_latent_fp8(const mla_bf16* rows, int B, int S, float rope_theta, int32_t* seqlens,
                                 uint8_t* kv8, float* kv_scale, int64_t kv_seq_stride, const int32_t* block_table,
                                 int max_pages, int page_size, int num_pages, int32_t* status_dev,
                                 mla_stream stream) {
  if (!rows || !seqlens || !kv8 || !kv_scale) return MLA_ERR_INVALID;
  if (B < 1 || S < 1 || S > 4 || rope_theta < 0.f || !std::isfinite(rope_theta)) return MLA_ERR_INVALID;
  if (!aligned16(rows) || !aligned16(kv8) || (reinterpret_cast<uintptr_t>(kv_scale) & 3u)) return MLA_ERR_INVALID;
  if (block_table) {
    if (page_size != kPage) return MLA_ERR_UNSUPPORTED;
    if (max_pages < 1 || num_pages < 1) return MLA_ERR_INVALID;
  } else if (kv_seq_stride < 1) {
    return MLA_ERR_INVALID;
  }
  const mla::RopeFreqs f = mla::make_rope_freqs(rope_theta > 0.f ? rope_theta : 10000.f);
  return launch_status(mla::launch_append_latent_fp8(
      reinterpret_cast<const __nv_bfloat16*>(rows), B, S, seqlens, kv8, kv_scale, kv_seq_stride, block_table,
      max_pages, num_pages, rope_theta > 0.f ? 1 : 0, f, status_dev, static_cast<cudaStream_t>(stream)));
}

static inline int round16(int x) { return (x + 15) & ~15; }

mla_status mla_fuse_weights(const mla_bf16* w_uq, const mla_bf16* w_uk, const mla_bf16* w_uv,
                            const mla_bf16* w_o, int H, int d_cq, int d_model, mla_bf16* w_uqk,
                            mla_bf16* w_uvo, mla_stream stream) {
  if (!w_uq || !w_uk || !w_uv || !w_o || !w_uqk || !w_uvo) return MLA_ERR_INVALID;
  if (!aligned16(w_uq) || !aligned16(w_uk) || !aligned16(w_uv) || !aligned16(w_o) || !aligned16(w_uqk) ||
      !aligned16(w_uvo))
    return MLA_ERR_INVALID;
  if (H < 1 || d_cq < 64 || d_model < 128) return MLA_ERR_INVALID;
  if (!heads_ok(H) || d_cq % 64 || d_model % 128) return MLA_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // W_UQK[h][i, c] = sum_d W_UQ[h][i, d] W_UK[h][c, d]: m = c (512), n = i (d_cq), k = d.
  {
    const mla::GemmOperand a{w_uk, (uint64_t)H * kDc, (uint64_t)mla::kDn, (uint64_t)mla::kDn, 0};
    const mla::GemmOperand b{w_uq, (uint64_t)H * d_cq, (uint64_t)mla::kDn, (uint64_t)mla::kDn, 0};
    mla::GemmShape g{};
    g.M = kDc, g.N = d_cq, g.K = mla::kDn, g.batches = H, g.n_tile = d_cq % 256 ? 64 : 256, g.k_splits = 1;
    g.a_batch_rows = kDc, g.b_batch_rows = d_cq;
    g.c = w_uqk, g.out_bf16 = 1, g.ldc_m = 1, g.ldc_n = kDc, g.ldc_batch = (int64_t)d_cq * kDc;
    const mla_status r = launch_status(mla::launch_gemm(a, b, g, st));
    if (r != MLA_OK) return r;
  }
  // W_UVO[h][c, j] = sum_v W_UV[h][c, v] W_O[h][v, j]: m = j (d_model), n = c (512), k = v.
  const mla::GemmOperand a{w_o, (uint64_t)H * mla::kDv, (uint64_t)d_model, (uint64_t)d_model, 1};
  const mla::GemmOperand b{w_uv, (uint64_t)H * kDc, (uint64_t)mla::kDv, (uint64_t)mla::kDv, 0};
  mla::GemmShape g{};
  g.M = d_model, g.N = kDc, g.K = mla::kDv, g.batches = H, g.n_tile = 256, g.k_splits = 1;
  g.a_batch_rows = mla::kDv, g.b_batch_rows = kDc;
  g.c = w_uvo, g.out_bf16 = 1, g.ldc_m = 1, g.ldc_n = d_model, g.ldc_batch = (int64_t)kDc * d_model;
  return launch_status(mla::launch_gemm(a, b, g, st));
}

mla_status mla_absorb_q_fused(const mla_bf16* c_q, const mla_bf16* q_rope, const mla_bf16* w_uqk,
                              const int32_t* q_pos, float rope_theta, int B, int S, int H, int d_cq,
                              mla_bf16* q_cat, mla_stream stream) {
  if (!c_q || !q_rope || !w_uqk || !q_cat) return MLA_ERR_INVALID;
  if (B < 1 || S < 1 || H < 1 || d_cq < 64) return MLA_ERR_INVALID;
  if (!aligned16(c_q) || !aligned16(q_rope) || !aligned16(w_uqk) || !aligned16(q_cat)) return MLA_ERR_INVALID;
  if (!heads_ok(H) || S > 4 || d_cq % 64) return MLA_ERR_UNSUPPORTED;
  if (q_pos && !(rope_theta > 0.f)) return MLA_ERR_INVALID;
  const int rows = B * S;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // q~[r, h, c] = sum_i c_q[r, i] W_UQK[h][i, c]: m = c (512), n = r, k = i (d_cq).
  const mla::GemmOperand a{w_uqk, (uint64_t)H * d_cq, (uint64_t)kDc, (uint64_t)kDc, 1};
  const mla::GemmOperand b{c_q, (uint64_t)rows, (uint64_t)d_cq, (uint64_t)d_cq, 0};
  mla::GemmShape g{};
  g.M = kDc, g.N = rows, g.K = d_cq, g.batches = H, g.n_tile = rows >= 256 ? 256 : round16(rows), g.k_splits = 1;
  g.a_batch_rows = d_cq, g.b_batch_rows = 0;
  g.c = q_cat, g.out_bf16 = 1, g.ldc_m = 1, g.ldc_n = (int64_t)H * kRow, g.ldc_batch = kRow;
  mla_status r = launch_status(mla::launch_gemm(a, b, g, st));
  if (r != MLA_OK) return r;
  const mla::RopeFreqs f = mla::make_rope_freqs(q_pos ? rope_theta : 10000.f);
  return launch_status(mla::launch_rope_slice(reinterpret_cast<const __nv_bfloat16*>(q_rope), q_pos, f, rows, H,
                                              reinterpret_cast<__nv_bfloat16*>(q_cat), st));
}

size_t mla_out_proj_fused_workspace_bytes(int B, int S, int H) {
  if (B < 1 || S < 1 || H < 1) return 0;
  return (size_t)B * S * H * kDc * 2;
}

mla_status mla_out_proj_fused(const float* o_lat, const mla_bf16* w_uvo, int B, int S, int H, int d_model,
                              float* out, void* workspace, size_t workspace_bytes, mla_stream stream) {
  if (!o_lat || !w_uvo || !out) return MLA_ERR_INVALID;
  if (B < 1 || S < 1 || H < 1 || d_model < 128) return MLA_ERR_INVALID;
  if (!aligned16(o_lat) || !aligned16(w_uvo) || !aligned16(out)) return MLA_ERR_INVALID;
  if (!heads_ok(H) || S > 4 || d_model % 128) return MLA_ERR_UNSUPPORTED;
  const size_t need = mla_out_proj_fused_workspace_bytes(B, S, H);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return MLA_ERR_WORKSPACE;
  const int rows = B * S;
  const int K = H * kDc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The tensor core takes o_lat in bf16 (as mla_out_proj_uv does).
  mla_status r = launch_status(mla::launch_f32_to_bf16(o_lat, (int64_t)rows * K,
                                                       static_cast<__nv_bfloat16*>(workspace), st));
  if (r != MLA_OK) return r;
  // out[r, j] = sum_(h,c) o_lat[r, h, c] W_UVO[h][c, j]: m = j (d_model), n = r, k = (h, c),
  // split along k to fill the device, the parts added into the zeroed output.
  const mla::GemmOperand a{w_uvo, (uint64_t)K, (uint64_t)d_model, (uint64_t)d_model, 1};
  const mla::GemmOperand b{workspace, (uint64_t)rows, (uint64_t)K, (uint64_t)K, 0};
  mla::GemmShape g{};
  g.M = d_model, g.N = rows, g.K = K, g.batches = 1, g.n_tile = rows >= 256 ? 256 : round16(rows);
  const int tiles = (d_model / 128) * ((rows + g.n_tile - 1) / g.n_tile);
  const int sms = mla::device_sm_count() > 0 ? mla::device_sm_count() : 148;
  g.k_splits = std::max(1, std::min(K / 64, 2 * sms / tiles));
  g.a_batch_rows = 0, g.b_batch_rows = 0;
  g.c = out, g.out_bf16 = 0, g.ldc_m = 1, g.ldc_n = d_model, g.ldc_batch = 0;
  if (g.k_splits > 1 && cudaMemsetAsync(out, 0, (size_t)rows * d_model * sizeof(float), st) != cudaSuccess)
    return launch_status(cudaErrorUnknown);
  return launch_status(mla::launch_gemm(a, b, g, st));
}

size_t mla_prefill_workspace_bytes(int B, int64_t kv_seq_stride, int H) {
  if (B < 1 || kv_seq_stride < 1 || H < 1) return 0;
  return 2 * (size_t)B * (size_t)kv_seq_stride * (size_t)H * mla::kDn * 2;
}

mla_status mla_prefill(const mla_bf16* q_nope, const mla_bf16* q_rope, const mla_bf16* kv, int64_t kv_seq_stride,
                       int T_kv, const mla_bf16* w_uk, const mla_bf16* w_uv, int B, int T_q, int H, float scale,
                       float* o, float* lse, void* workspace, size_t workspace_bytes, int32_t* status_dev,
                       mla_stream stream) {
  if (!q_nope || !q_rope || !kv || !w_uk || !w_uv || !o || !lse) return MLA_ERR_INVALID;
  if (B < 1 || H < 1 || T_q < 1 || T_kv < T_q || kv_seq_stride < T_kv) return MLA_ERR_INVALID;
  if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(kv) || !aligned16(w_uk) || !aligned16(w_uv) ||
      !aligned16(o))
    return MLA_ERR_INVALID;
  if (!(scale > 0.f) || !std::isfinite(scale)) return MLA_ERR_INVALID;
  if (!heads_ok(H)) return MLA_ERR_UNSUPPORTED;
  if ((uint64_t)B * (uint64_t)kv_seq_stride > 0x7FFFFFFFull || (int64_t)B * T_q > 0x7FFFFFFF) return MLA_ERR_UNSUPPORTED;
  const size_t need = mla_prefill_workspace_bytes(B, kv_seq_stride, H);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return MLA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const uint64_t rows = (uint64_t)B * (uint64_t)kv_seq_stride;
  __nv_bfloat16* k_exp = static_cast<__nv_bfloat16*>(workspace);
  __nv_bfloat16* v_exp = k_exp + rows * (uint64_t)H * mla::kDn;
  // K_h[t] = c_t W_UK[h], V_h[t] = c_t W_UV[h] for every row of the cache (rows past T_kv
  // included; the attention never reads them).
  const mla_status r = launch_status(mla::launch_expand_kv(reinterpret_cast<const __nv_bfloat16*>(kv), rows,
                                                           reinterpret_cast<const __nv_bfloat16*>(w_uk),
                                                           reinterpret_cast<const __nv_bfloat16*>(w_uv), H,
                                                           k_exp, v_exp, status_dev, st));
  if (r != MLA_OK) return r;
  return launch_status(mla::launch_prefill_attn(
      reinterpret_cast<const __nv_bfloat16*>(q_nope), reinterpret_cast<const __nv_bfloat16*>(q_rope),
      reinterpret_cast<const __nv_bfloat16*>(kv), kv_seq_stride, k_exp, v_exp, B, T_q, T_kv, H, scale, o, lse,
      status_dev, st));
}

mla_status mla_copy_from_host(void* dst, const void* src_host, size_t bytes, mla_stream stream) {
  if (!dst || !src_host || bytes % 16 || !aligned16(dst) || !aligned16(src_host)) return MLA_ERR_INVALID;
  if (bytes == 0) return MLA_OK;
  void* alias = nullptr;
  if (cudaHostGetDevicePointer(&alias, const_cast<void*>(src_host), 0) != cudaSuccess || !alias) {
    cudaGetLastError();
    return MLA_ERR_INVALID;   // not pinned (page-locked) host memory
  }
  return launch_status(mla::launch_copy_from_host(alias, dst, (int64_t)bytes, static_cast<cudaStream_t>(stream)));
}

mla_status mla_rope_inplace(mla_bf16* x, int64_t row_stride, int64_t rows, int col_offset,
                            const int32_t* pos, float theta, mla_stream stream) {
  if (!x || !pos || rows < 0 || col_offset < 0 || row_stride < col_offset + mla::kDr)
    return MLA_ERR_INVALID;
  if ((col_offset & 1) || (row_stride & 1) || !(theta > 0.f)) return MLA_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(x) & 3u) return MLA_ERR_INVALID;
  const mla::RopeFreqs f = mla::make_rope_freqs(theta);
  return launch_status(mla::launch_rope_inplace(reinterpret_cast<__nv_bfloat16*>(x), row_stride,
                                                rows, col_offset, pos, f,
                                                static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
