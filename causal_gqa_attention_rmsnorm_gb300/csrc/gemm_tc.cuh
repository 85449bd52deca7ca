// Host interface of the bf16 tcgen05 GEMMs and the TMA tensor-map helper.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace tb {

// Encode a 2-D row-major bf16 tensor [rows, cols] with a (box_cols × box_rows)
// box and the 128-byte swizzle (box_cols · 2 must be 128).  Out-of-range
// elements of a box read as zero.
cudaError_t make_tmap_2d_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                              uint64_t row_stride_elems, uint32_t box_cols, uint32_t box_rows);
// 3-D variant: [planes, rows, cols] with plane stride plane_stride_elems.
cudaError_t make_tmap_3d_bf16(CUtensorMap* m, const void* base, uint64_t planes, uint64_t rows, uint64_t cols,
                              uint64_t row_stride_elems, uint64_t plane_stride_elems, uint32_t box_cols,
                              uint32_t box_rows);
// 3-D byte tensor (int8 codes), strides in bytes, same box rules (box_cols must be 128).
cudaError_t make_tmap_3d_u8(CUtensorMap* m, const void* base, uint64_t planes, uint64_t rows, uint64_t cols,
                            uint64_t row_stride, uint64_t plane_stride, uint32_t box_cols, uint32_t box_rows);
int sm_count();

cudaError_t gemm_tc_qkv(const void* A, const void* B, int M, int N, int K, const Dims& D, const QKVArgs& e,
                        cudaStream_t s);
// row_parts: Σh² partials per row the launch writes (one per column tile)
cudaError_t gemm_tc_wo(const void* A, const void* B, int M, int N, int K, const Dims& D, const WoArgs& e,
                       cudaStream_t s, int* row_parts);
cudaError_t gemm_tc_w13(const void* A, const void* B, int M, int N, int K, const Dims& D, const W13Args& e,
                        cudaStream_t s);
cudaError_t gemm_tc_w2(const void* A, const void* B, int M, int N, int K, const Dims& D, const W2Args& e,
                       cudaStream_t s);
// Plain C = A·Bᵀ in fp32 with the same main loop (test hook); mt = 2 takes the
// CTA-pair tiles (256 rows over two CTAs, M = 256 MMAs).
cudaError_t gemm_tc_f32out(const void* A, const void* B, float* C, int M, int N, int K, int bn, int mt,
                           cudaStream_t s);

}  // namespace tb
