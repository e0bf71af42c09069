// Declarations of the batched GEMM (gemm_sm103.cu) and of the calls built on it
// (internal; the public ABI is include/mla.h).
#pragma once

#include "common.cuh"

namespace mla {

// Batched GEMM (gemm_sm103.cu): D[m, n] = sum_k A[m, k] B[n, k] for each batch z, tiles of
// 128 m x n_tile n, k in blocks of 64, written as C[z * ldc_batch + m * ldc_m + n * ldc_n].
struct GemmOperand {
  const void* ptr;       // bf16 2D array the TMA map covers
  uint64_t rows, cols;   // its extent; K-major: rows (z, m or n), cols k; MN-major: rows (z, k), cols m or n
  uint64_t row_stride;   // elements between rows
  int mn;                // 1: MN-major (m or n contiguous), 0: K-major (k contiguous)
};
struct GemmShape {
  int M, N, K, batches, n_tile, k_splits;
  int stages;                       // shared-memory stages of the k ring, 2..4 (0: 4)
  int a_batch_rows, b_batch_rows;   // batch z starts at map row z * this (0: shared by all)
  int a_mn, b_mn;                   // filled in by launch_gemm
  void* c;                          // output: bf16, or fp32 (atomically added when k_splits > 1)
  int out_bf16;
  int64_t ldc_m, ldc_n, ldc_batch;
  int32_t* status;                  // device flag word or null
};
cudaError_t launch_gemm(const GemmOperand& a, const GemmOperand& b, GemmShape g, cudaStream_t st);
// K_h = C W_UK[h] and V_h = C W_UV[h] for every cache row and head, bf16 [rows][H][128]
// (expand_sm103.cu).
cudaError_t launch_expand_kv(const __nv_bfloat16* kv, uint64_t rows, const __nv_bfloat16* w_uk,
                             const __nv_bfloat16* w_uv, int H, __nv_bfloat16* k_exp, __nv_bfloat16* v_exp,
                             int32_t* status, cudaStream_t st);
cudaError_t launch_f32_to_bf16(const float* x, int64_t n, __nv_bfloat16* y, cudaStream_t st);
cudaError_t launch_copy_from_host(const void* src_dev_alias, void* dst, int64_t bytes, cudaStream_t st);
cudaError_t launch_rope_slice(const __nv_bfloat16* q_rope, const int32_t* q_pos, const RopeFreqs& f, int M,
                              int H, __nv_bfloat16* q_cat, cudaStream_t st);

}  // namespace mla
