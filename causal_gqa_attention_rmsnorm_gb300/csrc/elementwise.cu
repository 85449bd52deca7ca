// Weight packing, RoPE table, per-token RMS statistics and KV-cache appends.
//
// RMSNorm ("Transformer block" page, tirogla.com, step 2; Go rmsnorm of
// "09 The Transformer"): xn = x / sqrt(mean(x²) + eps) ⊙ g.  The gain is folded
// into the packed weights, so the only per-token work left is the inverse RMS
// r = 1/sqrt(mean(x²) + eps), which the GEMM epilogues apply as a row scale.
#include <algorithm>

#include "common.cuh"

namespace tb {
namespace {

// dst row (n·row_mul + row_add), length K  <-  column n of src [K, N], times gain[k].
template <typename T>
__global__ void k_pack_transpose(const T* __restrict__ src, int K, int N, const T* __restrict__ gain,
                                 T* __restrict__ dst, int row_mul, int row_add) {
  __shared__ float tile[32][33];
  const int n0 = blockIdx.x * 32, k0 = blockIdx.y * 32;
  const int tx = threadIdx.x, ty = threadIdx.y;
  for (int i = ty; i < 32; i += 8) {
    const int k = k0 + i, n = n0 + tx;
    float v = 0.f;
    if (k < K && n < N) {
      v = to_f(src[(size_t)k * N + n]);
      if (gain) v *= to_f(gain[k]);
    }
    tile[i][tx] = v;
  }
  __syncthreads();
  for (int i = ty; i < 32; i += 8) {
    const int n = n0 + i, k = k0 + tx;
    if (n < N && k < K) dst[((size_t)n * row_mul + row_add) * K + k] = from_f<T>(tile[tx][i]);
  }
}

// (cos, sin) of t·base^(-2i/dh) for t < max_pos, i < dh/2, computed in fp64.
__global__ void k_rope_table(float2* __restrict__ tab, int max_pos, int half, int dh, double base) {
  const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (size_t)max_pos * half) return;
  const int t = (int)(idx / half), i = (int)(idx % half);
  const double phi = (double)t * pow(base, -2.0 * i / dh);
  double s, c;
  sincos(phi, &s, &c);
  tab[idx] = make_float2((float)c, (float)s);
}

// One warp per token row: r = 1/sqrt(mean(x²) + eps).  Side duties, done by
// lane 0 of the row: set the cache length after a prefill (lens_set), or take
// the decode position and advance the cache length (lens_bump -> pos_out, -1
// when the cache is full), and zero a counter a later kernel of the step uses
// (zero_word).
template <typename T>
__global__ void k_row_stats(const T* __restrict__ x, int M, int d, float eps, float* __restrict__ r, int Tseq,
                            int32_t* __restrict__ lens_set,
                            int32_t* __restrict__ lens_bump, int32_t* __restrict__ pos_out, int T_max,
                            int* __restrict__ zero_word, int* __restrict__ err) {
  pdl_trigger();
  pdl_wait();
  const int row = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  const T* xr = x + (size_t)row * d;
  float s = 0.f;
  constexpr int V = Vec16<T>::N;
  if ((d % V) == 0) {
    // four 16-byte loads in flight per lane
    const uint4* p = reinterpret_cast<const uint4*>(xr);
    const int nv = d / V;
    int i = lane;
    for (; i + 96 < nv; i += 128) {
      Vec16<T> v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u].raw = __ldg(p + i + 32 * u);
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int j = 0; j < V; ++j) {
          const float f = v[u].get(j);
          s = fmaf(f, f, s);
        }
    }
    for (; i < nv; i += 32) {
      Vec16<T> v;
      v.raw = __ldg(p + i);
#pragma unroll
      for (int j = 0; j < V; ++j) {
        const float f = v.get(j);
        s = fmaf(f, f, s);
      }
    }
  } else {
    for (int i = lane; i < d; i += 32) {
      const float f = to_f(xr[i]);
      s = fmaf(f, f, s);
    }
  }
  s = warp_sum(s);
  if (lane == 0) {
    r[row] = 1.0f / sqrtf(s / (float)d + eps);
    if (zero_word && row == 0) *zero_word = 0;
    if (lens_set && (row % Tseq) == 0) lens_set[row / Tseq] = Tseq;
    if (lens_bump) {
      const int p = lens_bump[row];
      if (p >= 0 && p < T_max) {
        pos_out[row] = p;
        lens_bump[row] = p + 1;
      } else {
        pos_out[row] = -1;
        atomicOr(err, TB_DEVERR_CACHE_FULL);
      }
    }
  }
}

// Copy n new rows of every (b, kv head) to cache rows [lens[b], lens[b]+n).
// 16-byte vectors; grid.y = b.  Rows of a full sequence are skipped here and
// flagged by k_append_bump, which reads the same unchanged lens[b].
__global__ void k_append_copy(uint4* __restrict__ kc, uint4* __restrict__ vc, const int32_t* __restrict__ lens,
                              int Hkv, int T_max, int row_vecs, const uint4* __restrict__ kn,
                              const uint4* __restrict__ vn, int n, PagedKV pg) {
  const int b = blockIdx.y;
  const int L = lens[b];
  if (L < 0 || L + n > T_max) return;
  const size_t per_head = (size_t)n * row_vecs;
  const size_t total = (size_t)Hkv * per_head;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const size_t h = i / per_head, rem = i % per_head;
    const int r = (int)(rem / row_vecs), piece = (int)(rem % row_vecs);
    size_t dst;
    if (pg.bt) {                     // paged: the page holding row L + r
      const long long row = paged_row(pg, Hkv, b, (int)h, L + r);
      if (row < 0) continue;
      dst = (size_t)row * row_vecs + piece;
    } else {
      dst = (((size_t)b * Hkv + h) * T_max + L) * row_vecs + rem;
    }
    const size_t src = ((size_t)b * Hkv + h) * per_head + rem;
    kc[dst] = kn[src];
    vc[dst] = vn[src];
  }
}

__global__ void k_append_bump(int32_t* __restrict__ lens, int B, int T_max, int n, int* __restrict__ err) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int L = lens[b];
  if (L < 0 || L + n > T_max) {
    atomicOr(err, TB_DEVERR_CACHE_FULL);
    return;
  }
  lens[b] = L + n;
}

// int8 cache rows ("The Transformer Architecture", thegeniusblogs, pitfalls:
// the KV cache itself can be quantised to int8).  Each row of dh = 128 values
// gets the scale s = max|x| / 127 and codes round-half-even(x / s) clamped to
// [-127, 127]; s and x / s are fp32 operations (IEEE division), and a zero
// row keeps s = 0 and zero codes.  One warp per row, four values per lane.
__device__ __forceinline__ void quantize_row128(const bf16* __restrict__ x, int8_t* __restrict__ q,
                                                float* __restrict__ s_out, int lane) {
  const uint2 raw = *reinterpret_cast<const uint2*>(x + lane * 4);
  const float v[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xffff0000u),
                      __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xffff0000u)};
  float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float s = m / 127.0f;
  uint32_t packed = 0;
  if (s > 0.f) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = min(127, max(-127, __float2int_rn(v[i] / s)));
      packed |= (uint32_t)(c & 0xff) << (8 * i);
    }
  }
  *reinterpret_cast<uint32_t*>(q + lane * 4) = packed;
  if (lane == 0) *s_out = s;
}

// k and v rows [B, Hkv, rows, 128] -> cache rows start[b] + r of codes
// [B, Hkv, T_max, 128] and scales [B, Hkv, T_max], or, paged (pg.bt set), of
// the page pools [num_pages, Hkv, page_size, 128] and [num_pages, Hkv,
// page_size] at the pages the block table names.  A sequence whose start is
// negative (a skipped decode row) or whose rows would pass T_max is left
// alone; a page id outside the pool is never written through and sets
// TB_DEVERR_BAD_PAGE.
__global__ void k_quantize_kv(const bf16* __restrict__ kn, const bf16* __restrict__ vn, int rows,
                              const int32_t* __restrict__ start, int Hkv, int T_max, int8_t* __restrict__ kq,
                              float* __restrict__ ks, int8_t* __restrict__ vq, float* __restrict__ vs, PagedKV pg) {
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * (blockDim.x >> 5) + warp, h = blockIdx.y, b = blockIdx.z;
  if (r >= rows) return;
  const int t0 = start ? start[b] : 0;
  if (t0 < 0 || t0 + rows > T_max) return;
  const size_t src = (((size_t)b * Hkv + h) * rows + r) * 128;
  size_t row;
  if (pg.bt) {
    const long long pr = paged_row(pg, Hkv, b, h, t0 + r);
    if (pr < 0) return;
    row = (size_t)pr;
  } else {
    row = ((size_t)b * Hkv + h) * T_max + t0 + r;
  }
  quantize_row128(kn + src, kq + row * 128, ks + row, lane);
  quantize_row128(vn + src, vq + row * 128, vs + row, lane);
}

template <typename T>
void pack_all(const Dims& D, const tb_block_weights& w, const Packed& P, float rope_base, cudaStream_t s) {
  const dim3 blk(32, 8);
  auto grid = [](int K, int N) { return dim3((N + 31) / 32, (K + 31) / 32); };
  const int d = D.d, qn = D.H * D.dh, kn = D.Hkv * D.dh;
  T* qkv = (T*)P.wqkv;
  const T* ga = (const T*)w.g_attn;
  const T* gm = (const T*)w.g_mlp;
  k_pack_transpose<T><<<grid(d, qn), blk, 0, s>>>((const T*)w.wq, d, qn, ga, qkv, 1, 0);
  k_pack_transpose<T><<<grid(d, kn), blk, 0, s>>>((const T*)w.wk, d, kn, ga, qkv, 1, qn);
  k_pack_transpose<T><<<grid(d, kn), blk, 0, s>>>((const T*)w.wv, d, kn, ga, qkv, 1, qn + kn);
  k_pack_transpose<T><<<grid(qn, d), blk, 0, s>>>((const T*)w.wo, qn, d, nullptr, (T*)P.wo, 1, 0);
  k_pack_transpose<T><<<grid(d, D.f), blk, 0, s>>>((const T*)w.w1, d, D.f, gm, (T*)P.w13, 2, 0);
  k_pack_transpose<T><<<grid(d, D.f), blk, 0, s>>>((const T*)w.w3, d, D.f, gm, (T*)P.w13, 2, 1);
  k_pack_transpose<T><<<grid(D.f, d), blk, 0, s>>>((const T*)w.w2, D.f, d, nullptr, (T*)P.w2, 1, 0);
  const size_t n = (size_t)D.max_pos * (D.dh / 2);
  k_rope_table<<<(unsigned)((n + 255) / 256), 256, 0, s>>>((float2*)P.rope, D.max_pos, D.dh / 2, D.dh,
                                                           (double)rope_base);
}

}  // namespace

cudaError_t launch_pack(int dtype, const Dims& D, const tb_block_weights& w, void* /*packed*/,
                        const Packed& P, float rope_base, cudaStream_t s) {
  if (dtype == TB_F32)
    pack_all<float>(D, w, P, rope_base, s);
  else
    pack_all<bf16>(D, w, P, rope_base, s);
  return cudaGetLastError();
}

cudaError_t launch_row_stats(int dtype, const void* x, int M, int d, float eps, float* r, int T, int32_t* lens_set,
                             int32_t* lens_bump, int32_t* pos_out, int T_max, int* zero_word, int* err,
                             cudaStream_t s) {
  const int threads = 256;
  const unsigned blocks = (unsigned)(((size_t)M * 32 + threads - 1) / threads);
  if (dtype == TB_F32)
    return launch_pdl(k_row_stats<float>, dim3(blocks), dim3(threads), 0, s, (const float*)x, M, d, eps, r, T,
                      lens_set, lens_bump, pos_out, T_max, zero_word, err);
  return launch_pdl(k_row_stats<bf16>, dim3(blocks), dim3(threads), 0, s, (const bf16*)x, M, d, eps, r, T, lens_set,
                    lens_bump, pos_out, T_max, zero_word, err);
}

cudaError_t launch_pack_transpose(int dtype, const void* src, int K, int N, const void* gain, void* dst,
                                  cudaStream_t s) {
  const dim3 blk(32, 8), grid((N + 31) / 32, (K + 31) / 32);
  if (grid.y > 65535) return cudaErrorInvalidValue;
  if (dtype == TB_F32)
    k_pack_transpose<float><<<grid, blk, 0, s>>>((const float*)src, K, N, (const float*)gain, (float*)dst, 1, 0);
  else
    k_pack_transpose<bf16><<<grid, blk, 0, s>>>((const bf16*)src, K, N, (const bf16*)gain, (bf16*)dst, 1, 0);
  return cudaGetLastError();
}

cudaError_t launch_quantize_kv(const tb_kvcache& kv, const void* k_new, const void* v_new, int rows,
                               const int32_t* start, cudaStream_t s) {
  if (rows <= 0 || kv.B <= 0) return cudaSuccess;
  if (kv.B > 65535 || kv.Hkv > 65535) return cudaErrorInvalidValue;
  const int warps = std::min(rows, 8);
  const dim3 grid((unsigned)((rows + warps - 1) / warps), kv.Hkv, kv.B);
  PagedKV pg;
  if (kv.block_table) {
    pg.k = kv.k;
    pg.v = kv.v;
    pg.bt = kv.block_table;
    pg.ps = kv.page_size;
    pg.max_pages = kv.T_max / kv.page_size;
    pg.num_pages = kv.num_pages;
    pg.err = device_error_word();
  }
  return launch_pdl(k_quantize_kv, grid, dim3(32 * warps), 0, s, (const bf16*)k_new, (const bf16*)v_new, rows,
                    start, kv.Hkv, kv.T_max, (int8_t*)kv.k, kv.k_scale, (int8_t*)kv.v, kv.v_scale, pg);
}

cudaError_t launch_kv_append(int dtype, const tb_kvcache& kv, const void* k_new, const void* v_new, int n,
                             int* err, cudaStream_t s) {
  if (kv.dtype == TB_I8) {      // quantise the bf16 rows into place, then grow lens
    const cudaError_t e = launch_quantize_kv(kv, k_new, v_new, n, kv.lens, s);
    if (e != cudaSuccess) return e;
    k_append_bump<<<(kv.B + 127) / 128, 128, 0, s>>>(kv.lens, kv.B, kv.T_max, n, err);
    return cudaGetLastError();
  }
  const int esz = dtype == TB_F32 ? 4 : 2;
  const int row_vecs = kv.dh * esz / 16;
  const size_t per_seq = (size_t)kv.Hkv * n * row_vecs;
  const unsigned gx = (unsigned)std::min<size_t>((per_seq + 255) / 256, 1024);
  PagedKV pg;
  if (kv.block_table) {
    pg.k = kv.k;
    pg.v = kv.v;
    pg.bt = kv.block_table;
    pg.ps = kv.page_size;
    pg.max_pages = kv.T_max / kv.page_size;
    pg.num_pages = kv.num_pages;
    pg.err = err;
  }
  k_append_copy<<<dim3(gx, kv.B), 256, 0, s>>>((uint4*)kv.k, (uint4*)kv.v, kv.lens, kv.Hkv, kv.T_max,
                                               row_vecs, (const uint4*)k_new, (const uint4*)v_new, n, pg);
  k_append_bump<<<(kv.B + 127) / 128, 128, 0, s>>>(kv.lens, kv.B, kv.T_max, n, err);
  return cudaGetLastError();
}

}  // namespace tb
