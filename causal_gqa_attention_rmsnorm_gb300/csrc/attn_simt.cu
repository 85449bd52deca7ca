// Causal GQA attention of the fp32 path, one warp per query row.
//
// o_i = Σ_{j≤i} softmax_j(q_i·k_j/√dh) v_j per query head h, with KV head
// h / (H/Hkv) ("Transformer block" page, tirogla.com, step 2 and the GQA
// paragraph; "Transformers", engineering.msaqlain.com, 1.3 and 5.1); with a
// sliding window W > 0 the sum starts at j = i - W + 1 ("09 The Transformer",
// infra.pidoku.co.in, §5, sliding-window attention).  The
// softmax is computed online in fp32 (running max m, running sum l), the
// exact flash-style reformulation the "Transformers" page (section 6)
// describes, with the max subtracted before every exponential.
#include <math.h>

#include "common.cuh"

namespace tb {
namespace {

template <typename T, int DH>
__global__ void __launch_bounds__(128) k_attn_prefill_simt(const T* __restrict__ q, const T* __restrict__ k,
                                                           const T* __restrict__ v, T* __restrict__ o, int Tn,
                                                           int H, int Hkv, int kv_stride, int window,
                                                           float scale_log2) {
  constexpr int PER = (DH + 31) / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 4 + warp;
  if (t >= Tn) return;
  const int h = blockIdx.y, b = blockIdx.z;
  const int kvh = h / (H / Hkv);
  const T* qr = q + (((size_t)b * H + h) * Tn + t) * DH;
  const T* kb = k + ((size_t)b * Hkv + kvh) * kv_stride * DH;
  const T* vb = v + ((size_t)b * Hkv + kvh) * kv_stride * DH;
  float qv[PER], acc[PER];
#pragma unroll
  for (int p = 0; p < PER; ++p) {
    const int e = lane + 32 * p;
    qv[p] = e < DH ? to_f(qr[e]) * scale_log2 : 0.f;
    acc[p] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  for (int j = window > 0 && t >= window ? t - window + 1 : 0; j <= t; ++j) {
    float s = 0.f;
#pragma unroll
    for (int p = 0; p < PER; ++p) {
      const int e = lane + 32 * p;
      if (e < DH) s = fmaf(qv[p], to_f(kb[(size_t)j * DH + e]), s);
    }
    s = warp_sum(s);
    const float mn = fmaxf(m, s);
    const float c = exp2f(m - mn), pj = exp2f(s - mn);
    l = l * c + pj;
#pragma unroll
    for (int p = 0; p < PER; ++p) {
      const int e = lane + 32 * p;
      if (e < DH) acc[p] = fmaf(pj, to_f(vb[(size_t)j * DH + e]), acc[p] * c);
    }
    m = mn;
  }
  const float inv = 1.0f / l;
  T* orow = o + ((size_t)b * Tn + t) * H * DH + (size_t)h * DH;
#pragma unroll
  for (int p = 0; p < PER; ++p) {
    const int e = lane + 32 * p;
    if (e < DH) orow[e] = from_f<T>(acc[p] * inv);
  }
}

template <typename T, int DH>
cudaError_t run(const void* q, const void* k, const void* v, void* o, int B, int Tn, int H, int Hkv,
                int kv_stride, int window, cudaStream_t s) {
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)DH);
  const dim3 grid((Tn + 3) / 4, H, B);
  k_attn_prefill_simt<T, DH><<<grid, 128, 0, s>>>((const T*)q, (const T*)k, (const T*)v, (T*)o, Tn, H, Hkv,
                                                  kv_stride, window, scale_log2);
  return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch(const void* q, const void* k, const void* v, void* o, int B, int Tn, int H, int Hkv,
                     int dh, int kv_stride, int window, cudaStream_t s) {
  switch (dh) {
    case 16: return run<T, 16>(q, k, v, o, B, Tn, H, Hkv, kv_stride, window, s);
    case 32: return run<T, 32>(q, k, v, o, B, Tn, H, Hkv, kv_stride, window, s);
    case 64: return run<T, 64>(q, k, v, o, B, Tn, H, Hkv, kv_stride, window, s);
    case 128: return run<T, 128>(q, k, v, o, B, Tn, H, Hkv, kv_stride, window, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t attn_prefill_simt(int dtype, const void* q, const void* k, const void* v, void* o, int B, int T,
                              int H, int Hkv, int dh, int kv_stride, int window, cudaStream_t s) {
  if (dtype == TB_F32) return dispatch<float>(q, k, v, o, B, T, H, Hkv, dh, kv_stride, window, s);
  return dispatch<bf16>(q, k, v, o, B, T, H, Hkv, dh, kv_stride, window, s);
}

}  // namespace tb
