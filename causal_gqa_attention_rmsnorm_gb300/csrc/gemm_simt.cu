// fp32 SIMT GEMM of the fp32 path: C = A·Bᵀ with A [M, K] and the packed
// weight B [N, K] (reduction axis contiguous), 64×64 tiles, fp32 FMA, and the
// block's fused epilogues.  tf32 tensor cores would not hold the fp32 path's
// 1e-4 bound (10-bit mantissa), so this path stays on the FMA pipes.
#include "common.cuh"
#include "epilogues.cuh"

namespace tb {
namespace {

constexpr int BM = 64, BN = 64, BK = 16;

template <typename T, class Epi>
__global__ void __launch_bounds__(256) k_gemm_simt(const T* __restrict__ A, const T* __restrict__ B, int M, int N,
                                                   int K, Epi epi) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  for (int k0 = 0; k0 < K; k0 += BK) {
    for (int i = threadIdx.x; i < BM * BK; i += 256) {
      const int r = i / BK, c = i % BK;
      const int gk = k0 + c;
      const int gm = m0 + r, gn = n0 + r;
      As[c][r] = (gm < M && gk < K) ? to_f(A[(size_t)gm * K + gk]) : 0.f;
      Bs[c][r] = (gn < N && gk < K) ? to_f(B[(size_t)gn * K + gk]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][ty * 4 + i];
        b[i] = Bs[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }

  const int col = n0 + tx * 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = m0 + ty * 4 + i;
    float part = 0.f;
    if (row < M && col < N) {
      const auto ra = epi.row_aux(row);
      part = epi(row, col, acc[i], ra, epi.aux(row, col, ra));
    }
    if constexpr (Epi::kRowReduce) {
      // the 16 threads of a half-warp share this row: its partial blockIdx.x
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      if (tx == 0 && row < M) epi.row_sums().part[(size_t)row * epi.row_sums().stride + blockIdx.x] = part;
    }
  }
}

template <typename T, class Epi>
cudaError_t run(const void* A, const void* B, int M, int N, int K, const Epi& e, cudaStream_t s) {
  const dim3 grid((N + BN - 1) / BN, (M + BM - 1) / BM);
  k_gemm_simt<T, Epi><<<grid, 256, 0, s>>>((const T*)A, (const T*)B, M, N, K, e);
  return cudaGetLastError();
}

}  // namespace

cudaError_t gemm_simt_qkv(int dtype, const void* A, const void* B, int M, int N, int K, const Dims& D,
                          const QKVArgs& e, cudaStream_t s) {
  if (dtype == TB_F32) return run<float>(A, B, M, N, K, EpiQKV<float>{e, D.H, D.Hkv, D.dh, log2_dh(D.dh)}, s);
  return run<bf16>(A, B, M, N, K, EpiQKV<bf16>{e, D.H, D.Hkv, D.dh, log2_dh(D.dh)}, s);
}
cudaError_t gemm_simt_wo(int dtype, const void* A, const void* B, int M, int N, int K, const Dims& D,
                         const WoArgs& e, cudaStream_t s, int* row_parts) {
  if (row_parts) *row_parts = (N + BN - 1) / BN;     // one Σh² partial per row and column block
  if (dtype == TB_F32) return run<float>(A, B, M, N, K, EpiWo<float>{e, D.d}, s);
  return run<bf16>(A, B, M, N, K, EpiWo<bf16>{e, D.d}, s);
}
cudaError_t gemm_simt_w13(int dtype, const void* A, const void* B, int M, int N, int K, const Dims& D,
                          const W13Args& e, cudaStream_t s) {
  if (dtype == TB_F32) return run<float>(A, B, M, N, K, EpiW13<float>{e, D.d, D.f, D.eps}, s);
  return run<bf16>(A, B, M, N, K, EpiW13<bf16>{e, D.d, D.f, D.eps}, s);
}
cudaError_t gemm_simt_w2(int dtype, const void* A, const void* B, int M, int N, int K, const Dims& D,
                         const W2Args& e, cudaStream_t s) {
  if (dtype == TB_F32) return run<float>(A, B, M, N, K, EpiW2<>{e, D.d}, s);
  return run<bf16>(A, B, M, N, K, EpiW2<>{e, D.d}, s);
}

cudaError_t gemm_simt_logits(int dtype, const void* A, const void* B, int M, int N, int K, const LogitsArgs& e,
                             cudaStream_t s) {
  if (dtype == TB_F32) return run<float>(A, B, M, N, K, EpiLogits{e}, s);
  return run<bf16>(A, B, M, N, K, EpiLogits{e}, s);
}

}  // namespace tb
