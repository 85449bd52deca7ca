// The steps either side of the block ("Transformer block" page, tirogla.com,
// "How it works", steps 1 and 4): the embedding gather, and the reductions of
// the LM head's logits into a per-token loss.
#include <math.h>

#include <algorithm>

#include "common.cuh"

namespace tb {
namespace {

// x[t] = table[ids[t]]: one CTA per token row, 16-byte vectors.  An id outside
// [0, V) gives a zero row and sets TB_DEVERR_BAD_TOKEN.
__global__ void k_embed(const uint4* __restrict__ table, int V, int row_vecs, const int32_t* __restrict__ ids,
                        uint4* __restrict__ x, int* __restrict__ err) {
  const long long t = blockIdx.x;
  const int id = ids[t];
  const bool ok = id >= 0 && id < V;
  if (!ok && threadIdx.x == 0) atomicOr(err, TB_DEVERR_BAD_TOKEN);
  for (int i = threadIdx.x; i < row_vecs; i += blockDim.x)
    x[t * row_vecs + i] = ok ? table[(size_t)id * row_vecs + i] : make_uint4(0, 0, 0, 0);
}

// nll[r] = logsumexp(logits[r]) - logits[r, targets[r]], the row maximum taken
// first ("The Transformer" page, GenerativeAIDocs, §5 pitfalls: a softmax
// without the max subtraction overflows).  One CTA of 256 threads per row.
__global__ void __launch_bounds__(256) k_lse_nll(const float* __restrict__ logits, int ld, int V,
                                                 const int32_t* __restrict__ targets, float* __restrict__ nll,
                                                 int* __restrict__ err) {
  __shared__ float red[8];
  const int r = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float* z = logits + (size_t)r * ld;
  float m = -INFINITY;
  for (int i = threadIdx.x; i < V; i += 256) m = fmaxf(m, z[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  m = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) m = fmaxf(m, red[i]);
  __syncthreads();
  float sum = 0.f;
  for (int i = threadIdx.x; i < V; i += 256) sum += expf(z[i] - m);
  sum = warp_sum(sum);
  if (lane == 0) red[warp] = sum;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) tot += red[i];
    const int t = targets[r];
    if (t < 0 || t >= V) {
      atomicOr(err, TB_DEVERR_BAD_TOKEN);
      nll[r] = NAN;
    } else {
      nll[r] = m + logf(tot) - z[t];
    }
  }
}

// nll[r] = M + log S - logit[r, targets[r]] from a row's (max, Σ exp) pairs,
// one per 256-column tile of the fused head GEMM: lane l merges pairs l, l+32,
// ... in order, then the lanes merge in a fixed tree.  One warp per row.
__device__ __forceinline__ void lse_fold(float& m, float& s, float m2, float s2) {
  const float mn = fmaxf(m, m2);
  s = mn == -INFINITY ? 0.f : s * expf(m - mn) + s2 * expf(m2 - mn);
  m = mn;
}

__global__ void __launch_bounds__(256) k_lse_merge(const float2* __restrict__ part, int n_parts,
                                                   const float* __restrict__ tgt, const int32_t* __restrict__ targets,
                                                   int V, int M, float* __restrict__ nll, int* __restrict__ err) {
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= M) return;
  float m = -INFINITY, s = 0.f;
  for (int p = lane; p < n_parts; p += 32) {
    const float2 q = part[(size_t)r * n_parts + p];
    lse_fold(m, s, q.x, q.y);
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
    lse_fold(m, s, m2, s2);
  }
  if (lane == 0) {
    const int t = targets[r];
    if (t < 0 || t >= V) {
      atomicOr(err, TB_DEVERR_BAD_TOKEN);
      nll[r] = NAN;
    } else {
      nll[r] = m + logf(s) - tgt[r];
    }
  }
}

// dst[r][c] = src[r][c] · gain[c]: a tied LM head packs the embedding table
// [V, d] with the final norm's gain folded into its columns.
template <typename T>
__global__ void k_scale_cols(const T* __restrict__ src, const T* __restrict__ gain, long long rows, int cols,
                             T* __restrict__ dst) {
  const long long n = rows * cols;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    dst[i] = from_f<T>(to_f(src[i]) * to_f(gain[i % cols]));
}

}  // namespace

cudaError_t launch_embed(int dtype, const void* table, int V, int d, const int32_t* ids, long long n, void* x,
                         int* err, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  if (n > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int row_vecs = d * (dtype == TB_F32 ? 4 : 2) / 16;
  k_embed<<<(unsigned)n, 128, 0, s>>>((const uint4*)table, V, row_vecs, ids, (uint4*)x, err);
  return cudaGetLastError();
}

cudaError_t launch_lse_nll(const float* logits, int ld, int M, int V, const int32_t* targets, float* nll, int* err,
                           cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  k_lse_nll<<<M, 256, 0, s>>>(logits, ld, V, targets, nll, err);
  return cudaGetLastError();
}

cudaError_t launch_lse_merge(const float2* part, int n_parts, const float* tgt, const int32_t* targets, int V, int M,
                             float* nll, int* err, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  k_lse_merge<<<(M + 7) / 8, 256, 0, s>>>(part, n_parts, tgt, targets, V, M, nll, err);
  return cudaGetLastError();
}

cudaError_t launch_scale_cols(int dtype, const void* src, const void* gain, int rows, int cols, void* dst,
                              cudaStream_t s) {
  const long long n = (long long)rows * cols;
  const unsigned blocks = (unsigned)std::min<long long>((n + 255) / 256, 65535LL * 8);
  if (dtype == TB_F32)
    k_scale_cols<float><<<blocks, 256, 0, s>>>((const float*)src, (const float*)gain, rows, cols, (float*)dst);
  else
    k_scale_cols<bf16><<<blocks, 256, 0, s>>>((const bf16*)src, (const bf16*)gain, rows, cols, (bf16*)dst);
  return cudaGetLastError();
}

}  // namespace tb
