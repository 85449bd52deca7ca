// Split-K decode attention over the KV cache (one new query per sequence).
//
// A decode step attends the new token's G = H/Hkv query heads over the
// lens[b]+1 post-RoPE keys and values of its KV head ("Transformer block"
// page, tirogla.com, KV-cache paragraph; "Transformers" 5.2).  The work is
// bound by reading the cache (4 FLOPs per byte for G = 4), so the kernels are
// built for bandwidth, not for tensor cores.  Every KV row is read once and
// the G query heads of a group share it; each (sequence, KV head) is cut into
// chunks whose partial softmax states (running max m, sum l, unnormalised o)
// a second kernel merges by log-sum-exp.
//
// bf16 (k_decode_stream): persistent warps take 256-key chunks from a global
// counter, so the grid has no idle CTAs and the tail is one chunk.  Each warp
// streams its chunk in 32-key stages through two shared-memory slots with
// TMA (128-byte swizzle), the next stage always in flight while the current
// one is computed.  q·k: lane = key, the swizzle makes the 32 rows' reads
// conflict-free and q is a broadcast; p·v: lane = 4 (or 2) head dimensions,
// p a broadcast; all products as packed fp32x2 FMAs.
// fp32 (k_decode_split): one CTA per 256-key chunk, lanes read 16-byte pieces
// of consecutive rows straight from global memory.
// Rows at or beyond lens[b]+1 never reach the result.
#include <math.h>

#include "gemm_tc.cuh"
#include "common.cuh"
#include "sm100_ptx.cuh"

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
                                 int nchunk_max, int chunk, T* __restrict__ o) {
  const int h = blockIdx.x, b = blockIdx.y;
  const int pos = pos_arr[b];
  T* orow = o + ((size_t)b * H + h) * DH;
  if (pos < 0) {
    for (int e = threadIdx.x; e < DH; e += blockDim.x) orow[e] = from_f<T>(0.f);
    return;
  }
  const int nc = (pos + 1 + chunk - 1) / chunk;
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

// ---------------------------------------------------------------------------
// bf16 streaming kernel
// ---------------------------------------------------------------------------

constexpr int kSChunk = 256;   // keys per work item
constexpr int kSKeys = 32;     // keys per stage (one per lane)
constexpr int kSWarps = 6;

template <int DH, int G> struct StreamCfg {
  static constexpr int NB = DH / 64;                           // 128-byte boxes per row
  static constexpr uint32_t HALF_BYTES = kSKeys * 128;         // one box: 32 rows x 128 B
  static constexpr uint32_t KV_BYTES = NB * HALF_BYTES;        // K (or V) of one stage
  static constexpr uint32_t SLOT_BYTES = 2 * KV_BYTES;         // K then V
  static constexpr uint32_t WARP_SLOTS = 2 * SLOT_BYTES;
  static constexpr uint32_t Q_FLOATS = G * DH;
  static constexpr uint32_t OFF_Q = kSWarps * WARP_SLOTS;
  static constexpr uint32_t OFF_P = OFF_Q + kSWarps * Q_FLOATS * 4;
  static constexpr uint32_t OFF_BAR = OFF_P + kSWarps * kSKeys * G * 4;
  static constexpr uint32_t OFF_PRE = OFF_BAR + kSWarps * 2 * 8;
};

__device__ __forceinline__ float2 bf2_to_f2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

template <int DH, int G>
__global__ void __launch_bounds__(kSWarps * 32, 1)
    k_decode_stream(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const bf16* __restrict__ q, const int32_t* __restrict__ pos_arr, int B, int Hkv,
                    float* __restrict__ part, int nchunk_max, int* __restrict__ counter, float scale_log2,
                    int* err) {
  using C = StreamCfg<DH, G>;
  using namespace ptx;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* pre = reinterpret_cast<int*>(smem + C::OFF_PRE);       // [B+1] item prefix over sequences
  __shared__ int abort_word;

  // items of sequence b: Hkv x ceil((pos+1)/chunk), in (b, kv head, chunk) order
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int b = 0; b < B; ++b) {
      pre[b] = acc;
      const int p = pos_arr[b];
      acc += p < 0 ? 0 : Hkv * ((p + kSChunk) / kSChunk);
    }
    pre[B] = acc;
    abort_word = 0;
  }
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR) + warp * 2;
  if (lane == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    fence_barrier_init();
  }
  __syncthreads();
  volatile int* abort_flag = &abort_word;
  const int total = pre[B];
  const int H = Hkv * G;

  uint8_t* slots = smem + warp * C::WARP_SLOTS;
  float* qs = reinterpret_cast<float*>(smem + C::OFF_Q) + warp * C::Q_FLOATS;
  float* ps = reinterpret_cast<float*>(smem + C::OFF_P) + warp * kSKeys * G;

  struct Item { int b, kvh, c, key0, nkeys; };
  auto decode = [&](int t) {
    int lo = 0, hi = B - 1;                 // last b with pre[b] <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const int n = pos_arr[b] + 1;
    const int nch = (n + kSChunk - 1) / kSChunk;
    const int r = t - pre[b];
    Item it;
    it.b = b;
    it.kvh = r / nch;
    it.c = r - it.kvh * nch;
    it.key0 = it.c * kSChunk;
    it.nkeys = min(kSChunk, n - it.key0);
    return it;
  };
  // lane 0: TMA of stage `st` of item `it` into slot `sl` (K and V, all boxes)
  auto issue = [&](const Item& it, int st, int sl) {
    uint8_t* base = slots + sl * C::SLOT_BYTES;
    mbar_arrive_expect_tx(&full[sl], C::SLOT_BYTES);
    const int y = it.key0 + st * kSKeys, z = it.b * Hkv + it.kvh;
#pragma unroll
    for (int h = 0; h < C::NB; ++h) {
      tma_load_3d(&tmK, base + h * C::HALF_BYTES, &full[sl], h * 64, y, z);
      tma_load_3d(&tmV, base + C::KV_BYTES + h * C::HALF_BYTES, &full[sl], h * 64, y, z);
    }
  };

  int cur = 0, nxt = 0;
  if (lane == 0) {
    cur = atomicAdd(counter, 1);
    nxt = atomicAdd(counter, 1);
  }
  cur = __shfl_sync(0xffffffffu, cur, 0);
  nxt = __shfl_sync(0xffffffffu, nxt, 0);
  uint32_t use = 0;            // stages consumed so far by this warp
  int pending = -1;            // slot with a load in flight that no one will consume (abort path)
  if (cur < total && lane == 0) issue(decode(cur), 0, 0);
  bool ok = true;

  while (ok && cur < total) {
    const Item it = decode(cur);
    const int nst = (it.nkeys + kSKeys - 1) / kSKeys;
    // q of the G heads of this KV head, in fp32, pre-scaled to base-2 logits
    for (int i = lane; i < G * DH / 8; i += 32) {
      const int g = i / (DH / 8), e = (i % (DH / 8)) * 8;
      const uint4 raw = *reinterpret_cast<const uint4*>(q + ((size_t)it.b * H + it.kvh * G + g) * DH + e);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = bf2_to_f2(w[k]);
        qs[g * DH + e + 2 * k] = f.x * scale_log2;
        qs[g * DH + e + 2 * k + 1] = f.y * scale_log2;
      }
    }
    __syncwarp();
    float m[G], lsum[G];
    float2 o[G][DH / 64];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m[g] = -INFINITY;
      lsum[g] = 0.f;
#pragma unroll
      for (int k = 0; k < DH / 64; ++k) o[g][k] = make_float2(0.f, 0.f);
    }
    for (int st = 0; st < nst; ++st, ++use) {
      const int sl = use & 1;
      if (lane == 0) {             // prefetch the next stage of the stream into the other slot
        if (st + 1 < nst) {
          issue(it, st + 1, sl ^ 1);
          pending = sl ^ 1;
        } else if (nxt < total) {
          issue(decode(nxt), 0, sl ^ 1);
          pending = sl ^ 1;
        } else {
          pending = -1;
        }
      }
      if (!mbar_wait_warp(&full[sl], (use >> 1) & 1, abort_flag, err)) {
        ok = false;
        break;
      }
      const uint8_t* ks = slots + sl * C::SLOT_BYTES;
      const uint8_t* vs = ks + C::KV_BYTES;
      const int nvalid = min(kSKeys, it.nkeys - st * kSKeys);

      // q·k, lane = key
      float2 acc[G];
#pragma unroll
      for (int g = 0; g < G; ++g) acc[g] = make_float2(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < DH / 8; ++c) {
        const int h = c >> 3, cc = c & 7;
        const uint4 kr = *reinterpret_cast<const uint4*>(ks + h * C::HALF_BYTES + lane * 128 + ((cc ^ (lane & 7)) << 4));
        const float2 k0 = bf2_to_f2(kr.x), k1 = bf2_to_f2(kr.y), k2 = bf2_to_f2(kr.z), k3 = bf2_to_f2(kr.w);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float4 qa = *reinterpret_cast<const float4*>(qs + g * DH + c * 8);
          const float4 qb = *reinterpret_cast<const float4*>(qs + g * DH + c * 8 + 4);
          acc[g] = __ffma2_rn(make_float2(qa.x, qa.y), k0, acc[g]);
          acc[g] = __ffma2_rn(make_float2(qa.z, qa.w), k1, acc[g]);
          acc[g] = __ffma2_rn(make_float2(qb.x, qb.y), k2, acc[g]);
          acc[g] = __ffma2_rn(make_float2(qb.z, qb.w), k3, acc[g]);
        }
      }
      // online softmax over the stage: lane = key
      float pv[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float sc = lane < nvalid ? acc[g].x + acc[g].y : -INFINITY;
        float mx = sc;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float mn = fmaxf(m[g], mx);             // finite: the stage has a visible key
        const float corr = ex2_approx(m[g] - mn);
        pv[g] = ex2_approx(sc - mn);
        lsum[g] = lsum[g] * corr + pv[g];
#pragma unroll
        for (int k = 0; k < DH / 64; ++k) o[g][k] = __fmul2_rn(o[g][k], make_float2(corr, corr));
        m[g] = mn;
      }
#pragma unroll
      for (int g = 0; g < G; ++g) ps[lane * G + g] = pv[g];
      __syncwarp();
      // p·v, lane = head dimensions [lane·DH/32, +DH/32)
      const int vh = (lane * (DH / 32)) >> 6;               // which 64-column box
      const int vc = ((lane * (DH / 32)) & 63) >> 3;        // 16-byte chunk in the row
      const int vo = ((lane * (DH / 32)) & 7) * 2;          // byte offset in the chunk
      for (int jj = 0; jj < nvalid; ++jj) {
        const uint8_t* vrow = vs + vh * C::HALF_BYTES + jj * 128 + ((vc ^ (jj & 7)) << 4) + vo;
        float2 v[DH / 64];
        if constexpr (DH == 128) {
          const uint2 raw = *reinterpret_cast<const uint2*>(vrow);
          v[0] = bf2_to_f2(raw.x);
          v[1] = bf2_to_f2(raw.y);
        } else {
          v[0] = bf2_to_f2(*reinterpret_cast<const uint32_t*>(vrow));
        }
        float pj[G];
        if constexpr (G % 4 == 0) {
#pragma unroll
          for (int g = 0; g < G; g += 4) {
            const float4 t = *reinterpret_cast<const float4*>(ps + jj * G + g);
            pj[g] = t.x; pj[g + 1] = t.y; pj[g + 2] = t.z; pj[g + 3] = t.w;
          }
        } else {
#pragma unroll
          for (int g = 0; g < G; ++g) pj[g] = ps[jj * G + g];
        }
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int k = 0; k < DH / 64; ++k) o[g][k] = __ffma2_rn(make_float2(pj[g], pj[g]), v[k], o[g][k]);
      }
      __syncwarp();                // the slot and p may be rewritten after this
    }
    if (!ok) break;
    // write this chunk's partial states
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float l = lsum[g];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
      float* pr = part + (((size_t)it.b * H + it.kvh * G + g) * nchunk_max + it.c) * PartLayout<DH>::stride;
      float* po = pr + 4 + lane * (DH / 32);
      if constexpr (DH == 128) {
        *reinterpret_cast<float4*>(po) = make_float4(o[g][0].x, o[g][0].y, o[g][1].x, o[g][1].y);
      } else {
        *reinterpret_cast<float2*>(po) = o[g][0];
      }
      if (lane == 0) {
        pr[0] = m[g];
        pr[1] = l;
      }
    }
    cur = nxt;
    if (lane == 0 && cur < total) nxt = atomicAdd(counter, 1);
    nxt = __shfl_sync(0xffffffffu, nxt, 0);
    pending = -1;
  }
  // on an aborted wait, the copies in flight (the stage waited for and the one
  // issued ahead) must land before the CTA exits
  pending = __shfl_sync(0xffffffffu, pending, 0);
  if (!ok && lane == 0) {
    volatile int no_abort = 0;
    mbar_wait(&full[use & 1], (use >> 1) & 1, &no_abort, err);
    if (pending >= 0) mbar_wait(&full[pending], ((use + 1) >> 1) & 1, &no_abort, err);
  }
}

template <int DH, int G>
cudaError_t run_stream(const void* q, const void* kc, const void* vc, const int32_t* pos, int B, int Hkv, int T_max,
                       float* part, int nchunk_max, int* counter, void* o, cudaStream_t s) {
  using C = StreamCfg<DH, G>;
  CUtensorMap tk, tv;
  cudaError_t e = make_tmap_3d_bf16(&tk, kc, (uint64_t)B * Hkv, T_max, DH, DH, (uint64_t)T_max * DH, 64, kSKeys);
  if (e != cudaSuccess) return e;
  e = make_tmap_3d_bf16(&tv, vc, (uint64_t)B * Hkv, T_max, DH, DH, (uint64_t)T_max * DH, 64, kSKeys);
  if (e != cudaSuccess) return e;
  const size_t smem = C::OFF_PRE + (size_t)(B + 1) * 4 + 1024;
  if (smem > 232448) return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(k_decode_stream<DH, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)DH);
  k_decode_stream<DH, G><<<sm_count(), kSWarps * 32, smem, s>>>(tk, tv, (const bf16*)q, pos, B, Hkv, part,
                                                                nchunk_max, counter, scale_log2,
                                                                device_error_word());
  k_decode_combine<bf16, DH><<<dim3(Hkv * G, B), DH < 128 ? DH : 128, 0, s>>>(part, pos, Hkv * G, nchunk_max,
                                                                             kSChunk, (bf16*)o);
  return cudaGetLastError();
}

template <int DH>
cudaError_t stream_by_g(int G, const void* q, const void* kc, const void* vc, const int32_t* pos, int B, int Hkv,
                        int T_max, float* part, int nchunk_max, int* counter, void* o, cudaStream_t s) {
  switch (G) {
    case 1: return run_stream<DH, 1>(q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, counter, o, s);
    case 2: return run_stream<DH, 2>(q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, counter, o, s);
    case 4: return run_stream<DH, 4>(q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, counter, o, s);
    case 8: return run_stream<DH, 8>(q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, counter, o, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T, int DH, int G>
cudaError_t run(const void* q, const void* kc, const void* vc, const int32_t* pos, int B, int Hkv, int T_max,
                float* part, int nchunk_max, void* o, cudaStream_t s) {
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)DH);
  k_decode_split<T, DH, G><<<dim3(nchunk_max, Hkv, B), kWarps * 32, 0, s>>>(
      (const T*)q, (const T*)kc, (const T*)vc, pos, Hkv, T_max, part, nchunk_max, scale_log2);
  k_decode_combine<T, DH><<<dim3(Hkv * G, B), DH < 128 ? DH : 128, 0, s>>>(part, pos, Hkv * G, nchunk_max,
                                                                          kChunk, (T*)o);
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
                        int H, int Hkv, int dh, int T_max, float* part, int nchunk_max, int* work_counter,
                        void* o, cudaStream_t s) {
  const int G = H / Hkv;
  if (dtype == TB_F32) return by_dh<float>(dh, G, q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, o, s);
  if (dh == 128) return stream_by_g<128>(G, q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, work_counter, o, s);
  if (dh == 64) return stream_by_g<64>(G, q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, work_counter, o, s);
  return cudaErrorInvalidValue;
}

}  // namespace tb
