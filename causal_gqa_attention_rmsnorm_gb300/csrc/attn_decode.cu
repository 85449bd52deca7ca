// Split-K decode attention over the KV cache (one new query per sequence).
//
// A decode step attends the new token's G = H/Hkv query heads over the
// lens[b]+1 post-RoPE keys and values of its KV head ("Transformer block"
// page, tirogla.com, KV-cache paragraph; "Transformers" 5.2).  The work is
// bound by reading the cache (4 FLOPs per byte for G = 4), so the kernel is
// built for bandwidth, not for tensor cores:
//  * one CTA per (chunk of kChunk keys, KV head, sequence), so every KV row is
//    read exactly once and the G heads of a group share it;
//  * lanes read 16-byte pieces of consecutive key rows, so a warp load covers
//    whole rows contiguously, and K and V loads of several keys are issued
//    before any of them is used;
//  * fp32 online softmax per head (running max, running sum) inside the chunk,
//    then a log-sum-exp merge of the chunks in a second kernel.
// Rows at or beyond lens[b]+1 are never read: they may hold anything.
#include <math.h>

#include "common.cuh"

namespace tb {
namespace {

constexpr int kChunk = 256;  // keys per CTA
constexpr int kWarps = 4;

template <int DH>
struct PartLayout {
  static constexpr int stride = DH + 4;  // m, l, pad, pad, acc[DH]  (16-byte rows)
};

template <typename T, int DH, int G>
__global__ void __launch_bounds__(kWarps * 32) k_decode_split(const T* __restrict__ q, const T* __restrict__ kc,
                                                              const T* __restrict__ vc,
                                                              const int32_t* __restrict__ pos_arr, int Hkv,
                                                              int T_max, float* __restrict__ part, int nchunk_max,
                                                              float scale_log2) {
  constexpr int VEC = 16 / sizeof(T);
  constexpr int LPK = DH / VEC;   // lanes per key row
  static_assert(LPK >= 1 && LPK <= 32 && (32 % LPK) == 0, "row must split evenly over lanes");
  constexpr int KPW = 32 / LPK;   // key rows per warp load
  constexpr int KB = G <= 4 ? 4 : 2;
  constexpr int H_STEP = KPW * KB;

  const int c = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int pos = pos_arr[b];
  if (pos < 0) return;
  const int n = pos + 1;
  const int j0 = c * kChunk;
  if (j0 >= n) return;
  const int j1 = min(n, j0 + kChunk);
  const int H = Hkv * G;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane / LPK, li = lane % LPK;

  float qv[G][VEC];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    Vec16<T> v;
    v.raw = *reinterpret_cast<const uint4*>(q + ((size_t)b * H + kvh * G + g) * DH + li * VEC);
#pragma unroll
    for (int e = 0; e < VEC; ++e) qv[g][e] = v.get(e) * scale_log2;
  }
  float m[G], l[G], acc[G][VEC];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[g][e] = 0.f;
  }

  const size_t head_off = ((size_t)b * Hkv + kvh) * T_max;
  const uint4* kb = reinterpret_cast<const uint4*>(kc + head_off * DH) + li;
  const uint4* vb = reinterpret_cast<const uint4*>(vc + head_off * DH) + li;
  constexpr int ROWV = DH / VEC;  // uint4 per row

  for (int base = j0 + warp * H_STEP; base < j1; base += kWarps * H_STEP) {
    Vec16<T> kr[KB], vr[KB];
    bool ok[KB];
#pragma unroll
    for (int u = 0; u < KB; ++u) {
      const int j = base + u * KPW + grp;
      ok[u] = j < j1;
      if (ok[u]) {
        kr[u].raw = __ldcs(kb + (size_t)j * ROWV);
        vr[u].raw = __ldcs(vb + (size_t)j * ROWV);
      } else {
        kr[u].raw = make_uint4(0, 0, 0, 0);
        vr[u].raw = make_uint4(0, 0, 0, 0);
      }
    }
    float s[KB][G];
#pragma unroll
    for (int u = 0; u < KB; ++u)
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) a = fmaf(qv[g][e], kr[u].get(e), a);
        s[u][g] = a;
      }
#pragma unroll
    for (int o = LPK / 2; o > 0; o >>= 1)
#pragma unroll
      for (int u = 0; u < KB; ++u)
#pragma unroll
        for (int g = 0; g < G; ++g) s[u][g] += __shfl_xor_sync(0xffffffffu, s[u][g], o);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float mx = -INFINITY;
#pragma unroll
      for (int u = 0; u < KB; ++u) mx = ok[u] ? fmaxf(mx, s[u][g]) : mx;
      const float mn = fmaxf(m[g], mx);
      if (mn == -INFINITY) continue;   // no visible key yet in this lane group
      const float corr = exp2f(m[g] - mn);
      l[g] *= corr;
#pragma unroll
      for (int e = 0; e < VEC; ++e) acc[g][e] *= corr;
#pragma unroll
      for (int u = 0; u < KB; ++u) {
        const float p = ok[u] ? exp2f(s[u][g] - mn) : 0.f;
        l[g] += p;
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[g][e] = fmaf(p, vr[u].get(e), acc[g][e]);
      }
      m[g] = mn;
    }
  }

  // merge the lane groups of the warp (same li, different keys)
#pragma unroll
  for (int o = LPK; o < 32; o <<= 1) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m[g], o);
      const float l2 = __shfl_xor_sync(0xffffffffu, l[g], o);
      const float mn = fmaxf(m[g], m2);
      const float e1 = mn == -INFINITY ? 0.f : exp2f(m[g] - mn);
      const float e2 = mn == -INFINITY ? 0.f : exp2f(m2 - mn);
      l[g] = l[g] * e1 + l2 * e2;
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const float a2 = __shfl_xor_sync(0xffffffffu, acc[g][e], o);
        acc[g][e] = acc[g][e] * e1 + a2 * e2;
      }
      m[g] = mn;
    }
  }

  // merge the warps through shared memory
  __shared__ float sm_m[kWarps][G], sm_l[kWarps][G];
  __shared__ float sm_acc[kWarps][G][DH];
  if (grp == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if (li == 0) {
        sm_m[warp][g] = m[g];
        sm_l[warp][g] = l[g];
      }
#pragma unroll
      for (int e = 0; e < VEC; ++e) sm_acc[warp][g][li * VEC + e] = acc[g][e];
    }
  }
  __syncthreads();
  constexpr int P = PartLayout<DH>::stride;
  for (int idx = threadIdx.x; idx < G * DH; idx += blockDim.x) {
    const int g = idx / DH, e = idx % DH;
    float mn = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) mn = fmaxf(mn, sm_m[w][g]);
    float L = 0.f, A = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float sc = sm_m[w][g] == -INFINITY ? 0.f : exp2f(sm_m[w][g] - mn);
      L += sm_l[w][g] * sc;
      A += sm_acc[w][g][e] * sc;
    }
    float* pr = part + (((size_t)b * H + kvh * G + g) * nchunk_max + c) * P;
    pr[4 + e] = A;
    if (e == 0) {
      pr[0] = mn;
      pr[1] = L;
    }
  }
}

// o[b, h·DH + e] = Σ_c acc_c[e]·2^(m_c - M) / Σ_c l_c·2^(m_c - M), M = max_c m_c.
template <typename T, int DH>
__global__ void k_decode_combine(const float* __restrict__ part, const int32_t* __restrict__ pos_arr, int H,
                                 int nchunk_max, T* __restrict__ o) {
  const int h = blockIdx.x, b = blockIdx.y;
  const int pos = pos_arr[b];
  T* orow = o + ((size_t)b * H + h) * DH;
  if (pos < 0) {
    for (int e = threadIdx.x; e < DH; e += blockDim.x) orow[e] = from_f<T>(0.f);
    return;
  }
  const int nc = (pos + 1 + kChunk - 1) / kChunk;
  constexpr int P = PartLayout<DH>::stride;
  const float* pr = part + ((size_t)b * H + h) * nchunk_max * P;
  float M = -INFINITY;
  for (int c = 0; c < nc; ++c) M = fmaxf(M, pr[(size_t)c * P]);
  for (int e = threadIdx.x; e < DH; e += blockDim.x) {
    float L = 0.f, A = 0.f;
    for (int c = 0; c < nc; ++c) {
      const float sc = exp2f(pr[(size_t)c * P] - M);
      L += pr[(size_t)c * P + 1] * sc;
      A += pr[(size_t)c * P + 4 + e] * sc;
    }
    orow[e] = from_f<T>(A / L);
  }
}

template <typename T, int DH, int G>
cudaError_t run(const void* q, const void* kc, const void* vc, const int32_t* pos, int B, int Hkv, int T_max,
                float* part, int nchunk_max, void* o, cudaStream_t s) {
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)DH);
  k_decode_split<T, DH, G><<<dim3(nchunk_max, Hkv, B), kWarps * 32, 0, s>>>(
      (const T*)q, (const T*)kc, (const T*)vc, pos, Hkv, T_max, part, nchunk_max, scale_log2);
  k_decode_combine<T, DH><<<dim3(Hkv * G, B), DH < 128 ? DH : 128, 0, s>>>(part, pos, Hkv * G, nchunk_max,
                                                                          (T*)o);
  return cudaGetLastError();
}

template <typename T, int DH>
cudaError_t by_g(int G, const void* q, const void* kc, const void* vc, const int32_t* pos, int B, int Hkv,
                 int T_max, float* part, int nchunk_max, void* o, cudaStream_t s) {
  switch (G) {
    case 1: return run<T, DH, 1>(q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, o, s);
    case 2: return run<T, DH, 2>(q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, o, s);
    case 4: return run<T, DH, 4>(q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, o, s);
    case 8: return run<T, DH, 8>(q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, o, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t by_dh(int dh, int G, const void* q, const void* kc, const void* vc, const int32_t* pos, int B,
                  int Hkv, int T_max, float* part, int nchunk_max, void* o, cudaStream_t s) {
  switch (dh) {
    case 16: return by_g<T, 16>(G, q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, o, s);
    case 32: return by_g<T, 32>(G, q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, o, s);
    case 64: return by_g<T, 64>(G, q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, o, s);
    case 128: return by_g<T, 128>(G, q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, o, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int decode_chunk_keys() { return kChunk; }

size_t decode_part_floats(int B, int H, int dh, int nchunk_max) {
  return (size_t)B * H * nchunk_max * (dh + 4);
}

cudaError_t attn_decode(int dtype, const void* q, const void* kc, const void* vc, const int32_t* pos, int B,
                        int H, int Hkv, int dh, int T_max, float* part, int nchunk_max, void* o,
                        cudaStream_t s) {
  const int G = H / Hkv;
  if (dtype == TB_F32) return by_dh<float>(dh, G, q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, o, s);
  return by_dh<bf16>(dh, G, q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, o, s);
}

}  // namespace tb
