/*
 * mla.h -- C ABI of libmla.so: Multi-Head Latent Attention decode with weight absorption
 * on one B300 (sm_103a).
 *
 * The calls follow the steps of the decode computation described on the page
 * "MLA의 계산: KV를 펼치지 않고 Attention하기" (ai-systems-engineering.com), cited below as
 * [CALC], with dimensions from "Multi-Head Latent Attention (MLA)" (molayo1419.me), [MLA],
 * and the cache row of "DeepSeek Multi-Head Latent Attention(MLA) 아키텍처 해부"
 * (blog.huny.dev), [ANATOMY]:
 *
 *   mla_absorb_q       key absorption: q~ = q_nope W_UK^T per head, q_rope appended
 *   mla_decode_latent  scores against the latent cache, softmax, latent aggregation
 *                      (optionally split along the cache and merged by log-sum-exp)
 *   mla_out_proj_uv    value up-projection of the aggregated latent, once per head
 *   mla_rope_inplace   RoPE on the 64-wide rope slice of cache rows or queries
 *   mla_append_latent  the step's new latent rows into the cache (k^R rotated), before
 *                      the decode reads it
 *   mla_fuse_weights, mla_absorb_q_fused, mla_out_proj_fused
 *                      the projections multiplied together ahead of time, and the two
 *                      decode-time products that use them
 *   mla_prefill        prefill / chunked prefill in the expanded order (per-head K, V built)
 *   mla_quantize_fp8, mla_append_latent_fp8, mla_decode_latent_fp8
 *                      the FP8 (E4M3, a power-of-two scale per row) form of the latent
 *                      cache: quantize rows, append a step's rows, decode over it
 *   mla_decode_num_splits, mla_decode_plan_splits
 *                      split counts for the decode (from max_seqlen, or from the
 *                      batch's host-side lengths)
 *   mla_copy_from_host the host-to-device leg of a serving loop, by SM loads
 *
 * Conventions shared by every call
 *   - Dimensions are fixed: d_c = 512 (latent), d_r = 64 (decoupled RoPE key),
 *     d_nope = d_v = 128.  A cache row is 576 bf16 = [c^KV (512) | k^R (64)], 1152 bytes.
 *   - H (heads) must be a multiple of 16 and at most 128; S (query tokens per
 *     sequence) is 1..4; B >= 1.
 *   - Every pointer is a DEVICE pointer unless stated otherwise, 16-byte aligned.
 *     The caller owns every buffer; no call allocates device memory.  Between calls
 *     the library keeps only what it looks up once per device (SM count, the kernels'
 *     shared-memory opt-in, the scratch address of mla_decode_latent_noalloc) and the
 *     driver entry point it looks up once per process; these look-ups are safe from
 *     several host threads and devices.  Every device that loads the library also
 *     holds the fixed MLA_NOALLOC_SCRATCH_BYTES array that only
 *     mla_decode_latent_noalloc uses.
 *   - bf16 values are passed as raw 16-bit patterns (mla_bf16).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  The return value reports host-side argument checks and launch
 *     errors only.  Errors found on the device (a block-table entry outside the
 *     pool, a pipeline wait that timed out) are OR-ed as bit flags
 *     (1 << MLA_ERR_BLOCK_TABLE, 1 << MLA_ERR_TIMEOUT) into *status_dev when the
 *     caller passes one; the affected rows are skipped, never read out of bounds.
 *   - Argument checks run before any CUDA call, so a rejected call never touches
 *     the GPU.
 *   - The kernels are launched with programmatic dependent launch: each may start
 *     while the previous kernel on the stream is still running, and waits for it
 *     before reading what that kernel writes (q_cat, o_lat, partials).  The latent
 *     decode reads seqlens, block_table and its first cache rows BEFORE that wait.
 *     So the cache rows, seqlens and block_table of a decode must not be written by
 *     the kernel issued just before it on the stream if that kernel lets its
 *     dependents start early (griddepcontrol.launch_dependents); an ordinary
 *     kernel, a copy, or mla_append_latent / mla_rope_inplace (which do not) are
 *     safe.
 */
#ifndef MLA_H
#define MLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_D_C 512
#define MLA_D_R 64
#define MLA_D_NOPE 128
#define MLA_D_V 128
#define MLA_ROW 576
#define MLA_MAX_SPLITS 128

typedef uint16_t mla_bf16;   /* raw bfloat16 bits */
typedef void* mla_stream;    /* cudaStream_t */

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID = 1,      /* null pointer, bad size, misaligned pointer */
  MLA_ERR_UNSUPPORTED = 2,  /* a shape outside the supported set (H, S, page size) */
  MLA_ERR_CUDA = 3,         /* a CUDA runtime/driver error at launch */
  MLA_ERR_WORKSPACE = 4,    /* workspace missing or smaller than mla_decode_workspace_bytes */
  MLA_ERR_BLOCK_TABLE = 5,  /* device flag: a block-table entry outside [0, num_pages) */
  MLA_ERR_TIMEOUT = 6       /* device flag: a bounded pipeline wait expired */
} mla_status;

/* Human-readable name of a status code (static storage, never NULL). */
const char* mla_status_string(int status);

/* Number of SMs of the current device (0 when no device is usable). */
int mla_device_sm_count(void);

/*
 * mla_absorb_q -- key absorption, [CALC] "Key 투영을 Query 쪽으로 옮기기" (Fig. 3):
 * q (c_j U^K)^T = (q U^K^T) c_j^T, so each head's content query is mapped once into
 * the latent space instead of expanding every cached latent.
 *
 *   q_cat[b,s,h, 0:512]   = bf16( sum_k q_nope[b,s,h,k] * W_UK[h, :, k] )   (fp32 accumulate)
 *   q_cat[b,s,h, 512:576] = bf16( RoPE(q_rope[b,s,h,:], q_pos[b,s]) )  if q_pos != NULL
 *                         = q_rope[b,s,h,:]                            otherwise
 *
 *   q_nope  bf16 [B,S,H,128]     q_rope bf16 [B,S,H,64]
 *   w_uk    bf16 [H,512,128]     (W_UK[h] is d_c x d_nope; K_h = C W_UK[h], [MLA] "공식 정의")
 *   q_pos   int32 [B,S] or NULL  (position of each query token)
 *   rope_theta                   RoPE base (10000 for DeepSeek-V3); ignored without q_pos
 *   q_cat   bf16 [B,S,H,576]     output, the query row matched to a 576-wide cache row
 *
 * RoPE pairs interleaved elements (2i, 2i+1) and turns them by pos * theta^(-2i/64)
 * ([MLA] "구현", _apply_rope).  The product runs on the tensor core (bf16 inputs, fp32
 * accumulation).  If a pipeline wait inside the kernel expires, the affected q~ values
 * are NaN.
 */
mla_status mla_absorb_q(const mla_bf16* q_nope, const mla_bf16* q_rope, const mla_bf16* w_uk,
                        const int32_t* q_pos, float rope_theta, int B, int S, int H,
                        mla_bf16* q_cat, mla_stream stream);

/*
 * Workspace needed by mla_decode_latent for `num_splits` splits (0 = the automatic
 * choice for this shape, mla_decode_num_splits with total_rows = 0).  0 when one split
 * is used.
 * Layout: fp32 partial o_lat [splits,B,S,H,512] then fp32 partial lse [splits,B,S,H].
 */
size_t mla_decode_workspace_bytes(int B, int S, int H, int num_splits, int max_seqlen);

/*
 * A split count for mla_decode_latent.  Split k of a sequence covers its rows
 * [k*C, (k+1)*C), C = ceil(max_seqlen / num_splits) rounded up to 64 (the same C for
 * every sequence), so short sequences leave their trailing splits empty.  The count is
 * chosen to fill the device's SMs with (query token, split) units of two SMs each while
 * limiting the extra traffic of split partials, never more splits than 64-row tiles in
 * the longest sequence, at most MLA_MAX_SPLITS.  max_seqlen is the caller's bound on
 * seqlens[] (a host value); total_rows, if > 0, is the sum of seqlens[] (a host value
 * a serving scheduler knows), which lets a ragged batch split its long sequences more;
 * 0 assumes every sequence is max_seqlen long.  mla_decode_latent with num_splits = 0
 * uses this function with total_rows = 0.
 */
int mla_decode_num_splits(int B, int S, int H, int max_seqlen, int64_t total_rows);

/*
 * A split count for mla_decode_latent from the batch's own lengths, for callers that
 * know them on the host (a serving scheduler does).  For each candidate count s (1 ..
 * MLA_MAX_SPLITS, at most the 64-row tiles of max_seqlen) it lays out the (query token,
 * split) units exactly as mla_decode_latent will (C = ceil(max_seqlen / s) rounded up to
 * 64, causal visibility per query token), hands them in launch order to the device's
 * CTA-pair slots (each to the slot that frees first, as the hardware starts a cluster
 * where one finishes), with each unit's time from measured costs (a fixed part plus one
 * per 64-row tile; near nothing for an empty unit), adds the merge of the partials for
 * s > 1, and returns the s with the least estimated time (a larger s must win by 2%).
 *   seqlens    HOST int32 [B]; entries are clamped to [0, max_seqlen] as the decode does
 *   B, S, H    as for mla_decode_latent (S <= 4, H a multiple of 16 in [16,128])
 *   causal     as for mla_decode_latent
 *   max_seqlen the bound that will be passed to mla_decode_latent
 * Returns 0 on invalid arguments (null seqlens, bad sizes), 1 when no row is readable.
 * Host work grows with B*S*s; candidates past B*S*s = 2^22 units are not tried.
 */
int mla_decode_plan_splits(const int32_t* seqlens, int B, int S, int H, int causal, int max_seqlen);

/*
 * mla_decode_latent -- attention of the absorbed queries straight over the latent
 * cache, [CALC] "Content 점수와 위치 점수 합치기" (eq. s_j, Fig. 2) and
 * "Value 투영을 가중합 뒤로 옮기기" (Fig. 4):
 *
 *   x_j   = scale * ( q_cat[b,s,h,:] . row_j[:] )          (= q~.c_j + q^R.k^R_j, scaled)
 *   a_j   = softmax_j(x_j) over the rows query s may read  (all j < seqlens[b]; with
 *           causal != 0 query s is the row at position T-S+s and reads j <= T-S+s)
 *   o_lat[b,s,h,:] = sum_j a_j row_j[0:512]                (the k^R tail is not aggregated)
 *   lse[b,s,h]     = ln sum_j exp(x_j)
 *
 * A sequence with no readable row gives o_lat = 0 and lse = -inf.
 *
 *   q_cat        bf16 [B,S,H,576] from mla_absorb_q
 *   kv           bf16 cache rows of 576:
 *                  block_table == NULL: contiguous, row t of sequence b at
 *                                       kv + (b*kv_seq_stride + t)*576
 *                  block_table != NULL: a pool [num_pages, page_size, 576]; row t of
 *                                       sequence b is row t % page_size of page
 *                                       block_table[b*max_pages + t/page_size]
 *                Rows at or past seqlens[b] are never used, whatever they hold.
 *   kv_seq_stride rows between sequences (contiguous layout only), >= max seqlen
 *   seqlens      int32 [B] device, cached rows per sequence (>= 0)
 *   block_table  int32 [B, max_pages] device or NULL; page_size must be 64
 *   scale        softmax scale, 1/sqrt(d_nope + d_r) = 1/sqrt(192) for DeepSeek-V3
 *                ([CALC] "RoPE 경로를 분리한 이유": not 1/sqrt(d_c + d_r))
 *   num_splits   0 = automatic; 1..MLA_MAX_SPLITS splits the cache axis into chunks
 *                of ceil(max_seqlen / num_splits) rows (rounded up to 64), merged by
 *                log-sum-exp (see mla_decode_num_splits)
 *   max_seqlen   host-side bound on seqlens[] (used to plan splits; rows past it
 *                are never read)
 *   o_lat        fp32 [B,S,H,512] output;   lse fp32 [B,S,H] output
 *   workspace    device scratch of mla_decode_workspace_bytes(...) bytes (may be
 *                NULL when that is 0)
 *   status_dev   int32 device word for device-side error flags, or NULL
 */
mla_status mla_decode_latent(const mla_bf16* q_cat, const mla_bf16* kv, int64_t kv_seq_stride,
                             const int32_t* seqlens, const int32_t* block_table, int max_pages,
                             int page_size, int num_pages, int B, int S, int H, int causal,
                             float scale, int num_splits, int max_seqlen, float* o_lat,
                             float* lse, void* workspace, size_t workspace_bytes,
                             int32_t* status_dev, mla_stream stream);

/*
 * FP8 latent cache ("DeepSeek Multi-Head Latent Attention(MLA) 아키텍처 해부", section 5,
 * the checklist item on FP8 mixed precision: E4M3 over the 512-wide latent space with a
 * per-token scale).  A row is 640 bytes: the 512 latent values as E4M3 codes (OCP 8-bit
 * floating point, E4M3: bias 7, largest 448, no infinities) of c / s, then k^R as 64
 * bf16, unchanged; s, the row's scale, is a separate fp32.  Rows sit like bf16 rows:
 * contiguous (row t of sequence b at kv8 + (b*kv_seq_stride + t)*640) or a page pool
 * [num_pages, 64, 640] with the same block table; scale i belongs to row i of the same
 * layout.
 *
 * mla_quantize_fp8 -- bf16 cache rows of 576 (n_rows of them, row_stride bf16 apart, a
 * multiple of 8) to that form: s = the least power of two 2^e with max|c| / s <= 448,
 * e clamped to [-126, 15] (an all-zero row takes 1); codes = E4M3 of c / s rounded to
 * nearest even, saturating at +-448.  Latent values must be finite.  Writes kv8
 * [n_rows, 640] and kv_scale [n_rows] (both device; kv8 16-byte aligned, kv_scale 4-byte
 * aligned here and 16-byte aligned for mla_decode_latent_fp8).
 */
mla_status mla_quantize_fp8(const mla_bf16* rows, int64_t row_stride, int64_t n_rows, uint8_t* kv8,
                            float* kv_scale, mla_stream stream);

/*
 * mla_append_latent_fp8 -- mla_append_latent into the FP8 form of the cache: row s of
 * sequence b (bf16 [B,S,576], S <= 4) goes to position seqlens[b] + s of kv8 / kv_scale
 * (laid out as for mla_decode_latent_fp8), its latent values quantized exactly as by
 * mla_quantize_fp8, its k^R rotated at that position as by mla_append_latent (when
 * rope_theta > 0) and stored as bf16; seqlens[b] += S.  A row with no place is skipped
 * and 1 << MLA_ERR_BLOCK_TABLE is OR-ed into *status_dev.  No early start for the next
 * kernel, as for mla_append_latent.
 */
mla_status mla_append_latent_fp8(const mla_bf16* rows, int B, int S, float rope_theta, int32_t* seqlens,
                                 uint8_t* kv8, float* kv_scale, int64_t kv_seq_stride, const int32_t* block_table,
                                 int max_pages, int page_size, int num_pages, int32_t* status_dev,
                                 mla_stream stream);

/*
 * mla_decode_latent_fp8 -- mla_decode_latent over the FP8 form of the cache: the same
 * result as mla_decode_latent on rows whose latent part is s * E4M3(code) (exact in
 * bf16 for the power-of-two scales mla_quantize_fp8 writes; other scales are rounded
 * once to bf16 after the product) and whose k^R is the stored one.  Arguments as for
 * mla_decode_latent, with kv8 (640-byte rows, 16-byte aligned) and kv_scale (fp32, one
 * per row, 16-byte aligned) in place of kv; scales must lie in [2^-126, 2^15].  For a
 * contiguous cache kv_seq_stride is a multiple of 4 (a tile's 64 scales are read as one
 * 256-byte block).  Same workspace, split planning, status flags and early-start contract.
 */
mla_status mla_decode_latent_fp8(const mla_bf16* q_cat, const uint8_t* kv8, const float* kv_scale,
                                 int64_t kv_seq_stride, const int32_t* seqlens, const int32_t* block_table,
                                 int max_pages, int page_size, int num_pages, int B, int S, int H,
                                 int causal, float scale, int num_splits, int max_seqlen, float* o_lat,
                                 float* lse, void* workspace, size_t workspace_bytes,
                                 int32_t* status_dev, mla_stream stream);

/*
 * mla_decode_latent_noalloc -- mla_decode_latent without a caller-provided workspace.
 * The pages have no counterpart: this is a convenience for callers that cannot allocate
 * device memory themselves, such as plugins that are handed only their input and output
 * buffers by a host runtime with no allocator hook, or loops that must not call
 * cudaMalloc (it can synchronise the device).  The split-KV partials go to a fixed
 * array of MLA_NOALLOC_SCRATCH_BYTES compiled into libmla.so, which every device that
 * loads the library keeps until the process exits; this call allocates nothing.
 *
 * Arguments and results are those of mla_decode_latent (same layouts, same ownership of
 * the inputs and outputs), minus `workspace` / `workspace_bytes`.  If the partials of
 * the chosen split count (mla_decode_workspace_bytes) exceed MLA_NOALLOC_SCRATCH_BYTES
 * the call returns MLA_ERR_WORKSPACE and launches nothing; pick fewer splits.
 *
 * The first call on a device looks up the array's device address on that device
 * (cudaGetSymbolAddress); make that first call before any stream capture.  All calls
 * share the one array and each fully rewrites the part it reads, so no clearing is
 * needed between calls, but calls that overlap on the GPU (other streams, other host
 * threads) race on it: order them.
 */
#define MLA_NOALLOC_SCRATCH_BYTES (32u << 20)
mla_status mla_decode_latent_noalloc(const mla_bf16* q_cat, const mla_bf16* kv,
                                     int64_t kv_seq_stride, const int32_t* seqlens,
                                     const int32_t* block_table, int max_pages, int page_size,
                                     int num_pages, int B, int S, int H, int causal, float scale,
                                     int num_splits, int max_seqlen, float* o_lat, float* lse,
                                     int32_t* status_dev, mla_stream stream);

/*
 * mla_combine_partials -- merge attention computed over disjoint row ranges:
 *   lse = ln sum_k exp(lse_part[k]),  o = sum_k exp(lse_part[k] - lse) * o_part[k]
 * (the log-sum-exp merge that split-KV and a cross-GPU gather of partials both use;
 * not on the pages).
 *   o_part fp32 [num_splits, rows, 512], lse_part fp32 [num_splits, rows];
 *   o_lat fp32 [rows, 512], lse fp32 [rows].  Parts with lse = -inf count as empty.
 */
mla_status mla_combine_partials(const float* o_part, const float* lse_part, int num_splits,
                                int64_t rows, float* o_lat, float* lse, mla_stream stream);

/*
 * mla_out_proj_uv -- value up-projection, [CALC] "Value 투영을 가중합 뒤로 옮기기":
 * a (C U^V) = (a C) U^V, applied once per head after the latents are mixed.
 *   o[b,s,h,:] = sum_i bf16(o_lat[b,s,h,i]) * W_UV[h,i,:]   (tensor core, fp32 accumulate)
 *   o_lat fp32 [B,S,H,512]; w_uv bf16 [H,512,128]; o fp32 [B,S,H,128]
 * o_lat is rounded to bf16 on its way to the tensor core (unit roundoff 2^-8), so each
 * output differs from the exact product by at most 2^-8 * sum_i |o_lat_i W_UV[h,i,n]|
 * plus fp32 rounding.
 * If a pipeline wait inside the kernel expires, the affected outputs are NaN.
 */
mla_status mla_out_proj_uv(const float* o_lat, const mla_bf16* w_uv, int B, int S, int H,
                           float* o, mla_stream stream);

/*
 * mla_append_latent -- add the latent rows of this step's S tokens per sequence to the
 * cache, before mla_decode_latent reads it ([CALC] "계산 재배치의 효과와 한계": the current
 * token's latent is appended first and the token then reads itself; [ANATOMY] section 2:
 * the cached k^R carries RoPE, applied once when the row is written).
 *
 *   rows        bf16 [B,S,576] new rows [c^KV (512) | k^R (64), not yet rotated]
 *   rope_theta  RoPE base; > 0 rotates k^R of the row at position t by t * theta^(-2i/64)
 *               (interleaved pairs, as mla_rope_inplace), 0 stores k^R as given
 *   seqlens     int32 [B] device: row s of sequence b goes to position seqlens[b] + s;
 *               afterwards seqlens[b] += S (read and advanced by the same kernel)
 *   kv, kv_seq_stride, block_table, max_pages, page_size, num_pages: the cache, laid out
 *               as for mla_decode_latent (contiguous when block_table is NULL)
 *   status_dev  int32 device word or NULL: a row whose position has no place (past
 *               kv_seq_stride, past max_pages pages, or a page outside [0, num_pages)) is
 *               not written and 1 << MLA_ERR_BLOCK_TABLE is OR-ed in
 *
 * The c^KV part is copied bit for bit; k^R is rotated in fp32 (angle reduced as in
 * mla_rope_inplace) and stored as bf16.  The kernel does not let the next kernel on the
 * stream start before it completes, so a mla_decode_latent issued right after it sees
 * the appended rows and the advanced seqlens (see the convention on early starts above).
 */
mla_status mla_append_latent(const mla_bf16* rows, int B, int S, float rope_theta, int32_t* seqlens,
                             mla_bf16* kv, int64_t kv_seq_stride, const int32_t* block_table,
                             int max_pages, int page_size, int num_pages, int32_t* status_dev,
                             mla_stream stream);

/*
 * mla_rope_inplace -- rotate the 64 values x[r, col_offset : col_offset+64] of each of
 * `rows` rows (row r starts at x + r*row_stride elements) by position pos[r]:
 * interleaved pairs (2i, 2i+1) turn by pos * theta^(-2i/64) ([MLA] "구현").  Used to
 * put k^R of cache rows at their positions when they are written
 * ([ANATOMY] section 2: the cached k^R carries RoPE).  The angle pos * theta^(-2i/64)
 * is reduced modulo 2 pi in fp32 with two-term arithmetic (within about 1e-6 rad for
 * positions 0 <= pos < 2^24, the range this call and mla_absorb_q accept for exact
 * angles); the rotation runs in fp32 and is stored as bf16.
 */
mla_status mla_rope_inplace(mla_bf16* x, int64_t row_stride, int64_t rows, int col_offset,
                            const int32_t* pos, float theta, mla_stream stream);

/*
 * Pre-fused weights, [CALC] "Query·출력 투영과 합치기": once the key projection is moved to
 * the query side and the value projection behind the weighted sum, each can be multiplied
 * ahead of time into its neighbour: the query projection (U^Q (U^K)^T, so the content
 * query comes straight from the query latent c^Q) and the output projection (U^V W^O per
 * head; the heads' contributions are summed).  The RoPE query path stays separate.
 *
 * mla_fuse_weights -- the offline products, bf16 out (fp32 accumulation):
 *   W_UQK[h] = W_UQ[h] W_UK[h]^T   [d_cq x 512]      W_UVO[h] = W_UV[h] W_O[h]   [512 x d_model]
 *   w_uq  bf16 [H, d_cq, 128]   (q_nope[h] = c^Q W_UQ[h])
 *   w_uk  bf16 [H, 512, 128]    w_uv bf16 [H, 512, 128]   (as for mla_absorb_q / mla_out_proj_uv)
 *   w_o   bf16 [H, 128, d_model] (the head-h rows of the output projection W^O)
 *   w_uqk bf16 [H, d_cq, 512] out;   w_uvo bf16 [H, 512, d_model] out
 *   d_cq a multiple of 64 (1536 for DeepSeek-V3), d_model a multiple of 128.
 */
mla_status mla_fuse_weights(const mla_bf16* w_uq, const mla_bf16* w_uk, const mla_bf16* w_uv,
                            const mla_bf16* w_o, int H, int d_cq, int d_model, mla_bf16* w_uqk,
                            mla_bf16* w_uvo, mla_stream stream);

/*
 * mla_absorb_q_fused -- key absorption from the query latent with the fused weights:
 *   q_cat[b,s,h, 0:512]   = bf16( c_q[b,s,:] W_UQK[h] )                   (fp32 accumulate)
 *   q_cat[b,s,h, 512:576] = bf16( RoPE(q_rope[b,s,h,:], q_pos[b,s]) ), or q_rope as given
 *   c_q bf16 [B,S,d_cq]; q_rope bf16 [B,S,H,64]; w_uqk bf16 [H,d_cq,512]; q_cat as mla_absorb_q.
 */
mla_status mla_absorb_q_fused(const mla_bf16* c_q, const mla_bf16* q_rope, const mla_bf16* w_uqk,
                              const int32_t* q_pos, float rope_theta, int B, int S, int H, int d_cq,
                              mla_bf16* q_cat, mla_stream stream);

/* Device scratch mla_out_proj_fused needs: a bf16 copy of o_lat, B*S*H*512*2 bytes. */
size_t mla_out_proj_fused_workspace_bytes(int B, int S, int H);

/*
 * mla_out_proj_fused -- the attention output through the fused output weights, summed over
 * the heads:  out[b,s,:] = sum_h bf16(o_lat[b,s,h,:]) W_UVO[h]   (fp32 accumulate)
 *   o_lat fp32 [B,S,H,512]; w_uvo bf16 [H,512,d_model]; out fp32 [B,S,d_model]
 *   workspace: mla_out_proj_fused_workspace_bytes(B,S,H) bytes of device scratch.
 * The sum over the H*512 products is split into parts added with fp32 atomics, so the
 * last bits of `out` may differ between calls.
 */
mla_status mla_out_proj_fused(const float* o_lat, const mla_bf16* w_uvo, int B, int S, int H, int d_model,
                              float* out, void* workspace, size_t workspace_bytes, mla_stream stream);

/*
 * mla_prefill -- attention of T_q query tokens per sequence (a whole prompt, or a chunk
 * of one) in the expanded order: [MLA] (prefill vs. decode) and [CALC]
 * "계산 재배치의 효과와 한계": when many queries share the keys, building the per-head keys
 * and values once costs less than d_c-wide absorbed dot products, so prefill may keep
 * that order.  For each sequence b and head h:
 *   K_h[t] = c_t W_UK[h],  V_h[t] = c_t W_UV[h]          (bf16, fp32 accumulation)
 *   x_ij = scale * (q_nope[b,i,h] . K_h[j] + q_rope[b,i,h] . k^R_j)
 *   query i is the row at position T_kv - T_q + i and reads rows j <= T_kv - T_q + i
 *   o[b,i,h,:] = sum_j softmax_j(x_ij) V_h[j],  lse[b,i,h] = ln sum_j exp(x_ij)
 *
 *   q_nope bf16 [B,T_q,H,128]; q_rope bf16 [B,T_q,H,64], already rotated at the query
 *   positions (mla_rope_inplace); kv the contiguous cache [B, kv_seq_stride, 576] whose
 *   first T_kv rows per sequence are read (k^R already rotated); w_uk, w_uv [H,512,128];
 *   o fp32 [B,T_q,H,128]; lse fp32 [B,T_q,H]; 1 <= T_q <= T_kv <= kv_seq_stride.
 *   workspace: mla_prefill_workspace_bytes(B, kv_seq_stride, H) bytes, which hold K_h and
 *   V_h of every cache row of the B sequences (bf16 [B * kv_seq_stride][H][128], K_h first;
 *   rows past T_kv hold whatever their cache rows give and are never read).
 */
size_t mla_prefill_workspace_bytes(int B, int64_t kv_seq_stride, int H);
mla_status mla_prefill(const mla_bf16* q_nope, const mla_bf16* q_rope, const mla_bf16* kv, int64_t kv_seq_stride,
                       int T_kv, const mla_bf16* w_uk, const mla_bf16* w_uv, int B, int T_q, int H, float scale,
                       float* o, float* lse, void* workspace, size_t workspace_bytes, int32_t* status_dev,
                       mla_stream stream);

/*
 * mla_copy_from_host -- copy `bytes` (a multiple of 16; both pointers 16-byte aligned) from
 * pinned (page-locked) host memory `src_host` to device memory `dst`, asynchronously on
 * `stream`, by a kernel whose threads read the host buffer through its device-mapped
 * address.  Not a step of the method: the host-to-device leg of a serving loop, for hosts
 * whose copy engines move host-to-device data slowly.  Returns MLA_ERR_INVALID if src_host
 * is not pinned memory.  The host buffer must stay unchanged until the copy has run.
 */
mla_status mla_copy_from_host(void* dst, const void* src_host, size_t bytes, mla_stream stream);

/*
 * mla_debug_inject_timeout -- test hook for the device-side failure path (not a step of
 * the method).  For the kernels named in `kernels` (bit 0: the latent decode, bit 1: the
 * key absorption, bit 2: the W_UV projection; 0 turns the hook off) every later launch
 * from this process shortens its mbarrier wait limit from 2 s to `wait_ms` and withholds
 * one completion signal of its own (the decode: the score MMAs of each unit's first tile;
 * the projections: the copy of one weight chunk).  A wait then runs out: the kernel
 * records MLA_ERR_TIMEOUT in *status_dev (the decode; the projections write NaN), waits
 * for its own copies and MMAs, frees its tensor memory and exits.  Nothing faults and the
 * device stays usable; results of the affected calls are documented above (the decode
 * writes o_lat = 0 and lse = -inf for the units that gave up).  Process-wide; returns
 * MLA_ERR_INVALID for unknown bits or wait_ms outside (0, 2000].
 */
mla_status mla_debug_inject_timeout(int kernels, double wait_ms);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H */
