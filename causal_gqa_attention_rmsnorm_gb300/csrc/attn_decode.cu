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
// bf16 (k_decode_mma): persistent warps take chunks (256 keys, or 128 / 64
// for small batches, see decode_chunk_keys) from a global counter, so the
// grid has no idle CTAs and the tail is one chunk.  Each warp
// streams its chunks in 16-key stages through three shared-memory slots with
// TMA (128-byte swizzle), two stages always in flight while one is computed.
// The two small contractions (G query heads against 16 keys) run as
// warp-level m16n8k16 MMAs on fragments read with ldmatrix, which keeps the
// instruction count per key far below the SIMT form so the kernel can run at
// the rate the cache streams in; the softmax stays in fp32 registers.
// int8 caches (k_decode_i8): the same scheme over int8 codes, see below.
// fp32 (k_decode_split): one CTA per 256-key chunk, lanes read 16-byte pieces
// of consecutive rows straight from global memory.
// Rows at or beyond lens[b]+1 never reach the result.
#include <math.h>

#include "gemm_tc.cuh"
#include "common.cuh"
#include "sm100_ptx.cuh"

namespace tb {
namespace {

constexpr int kChunk = 256;  // keys per CTA (fp32 kernel) and per work item (bf16 kernel)
constexpr float kRescaleLog2 = 8.0f;  // rescale O only when the running max grows by more than 2^8
constexpr int kWarps = 4;

template <int DH>
struct PartLayout {
  static constexpr int stride = DH + 4;  // m, l, pad, pad, acc[DH]  (16-byte rows)
};

// First key a decode query at position n-1 attends: 0, or n - W with a
// sliding window W > 0 ("09 The Transformer", infra.pidoku.co.in, §5,
// sliding-window attention: the query sees its W most recent positions).
// Chunk c of a sequence covers keys [first + c·chunk, ...).
__device__ __forceinline__ int window_first(int n, int window) { return window > 0 && n > window ? n - window : 0; }
// First key of a sequence's first chunk: the window start rounded down to
// `align` keys (keys below the window start are masked).
__device__ __forceinline__ int chunk_base(int n, int window, int align) {
  return window_first(n, window) / align * align;
}

template <typename T, int DH, int G>
__global__ void __launch_bounds__(kWarps * 32) k_decode_split(const T* __restrict__ q, const T* __restrict__ kc,
                                                              const T* __restrict__ vc,
                                                              const int32_t* __restrict__ pos_arr, int Hkv,
                                                              int T_max, float* __restrict__ part, int nchunk_max,
                                                              int window, PagedKV pg, float scale_log2) {
  pdl_trigger();
  pdl_wait();
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
  const int j0 = window_first(n, window) + c * kChunk;
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
  // row j of this (sequence, KV head): -1 for a bad page id
  auto row_of = [&](int j) -> long long { return pg.bt ? paged_row(pg, Hkv, b, kvh, j) : (long long)j; };
  const uint4* kpool = pg.bt ? reinterpret_cast<const uint4*>(pg.k) + li : kb;
  const uint4* vpool = pg.bt ? reinterpret_cast<const uint4*>(pg.v) + li : vb;

  for (int base = j0 + warp * H_STEP; base < j1; base += kWarps * H_STEP) {
    Vec16<T> kr[KB], vr[KB];
    bool ok[KB];
#pragma unroll
    for (int u = 0; u < KB; ++u) {
      const int j = base + u * KPW + grp;
      const long long row = j < j1 ? row_of(j) : -1;
      ok[u] = row >= 0;
      if (ok[u]) {
        kr[u].raw = __ldcs(kpool + (size_t)row * ROWV);
        vr[u].raw = __ldcs(vpool + (size_t)row * ROWV);
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
// One CTA per (head, sequence).  Every global load is issued first: each
// thread reads the (m, l) pair of a chunk and, for output column e, the values
// of up to kCombineRegs of its chunks into registers; after one block
// reduction of the maxima and one of the sums, the weighted sums need no
// further global round trip (chunks beyond what the registers hold are read in
// a second pass).  All sums run in a fixed order.
constexpr int kCombineMaxChunks = 1024;
constexpr int kCombineRegs = 32;

template <typename T, int DH>
__global__ void __launch_bounds__(256) k_decode_combine(const float* __restrict__ part,
                                                        const int32_t* __restrict__ pos_arr, int H, int nchunk_max,
                                                        int chunk, int window, int align, T* __restrict__ o) {
  pdl_trigger();
  pdl_wait();
  static_assert(256 % DH == 0, "head width must divide the block");
  constexpr int NG = 256 / DH;      // thread groups, each covering the DH columns
  __shared__ float w_s[kCombineMaxChunks], l_s[kCombineMaxChunks];
  __shared__ float red[256 / 32];
  __shared__ float acc_s[NG][DH];
  const int h = blockIdx.x, b = blockIdx.y;
  const int pos = pos_arr[b];
  T* orow = o + ((size_t)b * H + h) * DH;
  if (pos < 0) {
    for (int e = threadIdx.x; e < DH; e += blockDim.x) orow[e] = from_f<T>(0.f);
    return;
  }
  const int nkeys = pos + 1 - chunk_base(pos + 1, window, align);
  const int nc = min((nkeys + chunk - 1) / chunk, kCombineMaxChunks);
  constexpr int P = PartLayout<DH>::stride;
  const float* pr = part + ((size_t)b * H + h) * nchunk_max * P;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int e = threadIdx.x % DH, g = threadIdx.x / DH;
  // thread (e, g) holds column e of chunks g, g + NG, ...
  float v[kCombineRegs];
#pragma unroll
  for (int u = 0; u < kCombineRegs; ++u) {
    const int c = g + NG * u;
    v[u] = c < nc ? pr[(size_t)c * P + 4 + e] : 0.f;
  }
  float mx = -INFINITY;
  for (int c = threadIdx.x; c < nc; c += blockDim.x) {
    const float2 ml = *reinterpret_cast<const float2*>(pr + (size_t)c * P);
    w_s[c] = ml.x;
    l_s[c] = ml.y;
    mx = fmaxf(mx, ml.x);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  float M = red[0];
#pragma unroll
  for (int i = 1; i < 256 / 32; ++i) M = fmaxf(M, red[i]);
  __syncthreads();
  // weights w_c = 2^(m_c - M) and L = Σ_c l_c·w_c
  float Lp = 0.f;
  for (int c = threadIdx.x; c < nc; c += blockDim.x) {
    const float w = exp2f(w_s[c] - M);
    w_s[c] = w;
    Lp += l_s[c] * w;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) Lp += __shfl_xor_sync(0xffffffffu, Lp, off);
  if (lane == 0) red[warp] = Lp;
  __syncthreads();
  float L = 0.f;
#pragma unroll
  for (int i = 0; i < 256 / 32; ++i) L += red[i];
  float a = 0.f;
#pragma unroll
  for (int u = 0; u < kCombineRegs; ++u) {
    const int c = g + NG * u;
    if (c < nc) a = fmaf(v[u], w_s[c], a);
  }
  for (int c = g + NG * kCombineRegs; c < nc; c += NG) a = fmaf(pr[(size_t)c * P + 4 + e], w_s[c], a);
  acc_s[g][e] = a;
  __syncthreads();
  if (g == 0) {
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < NG; ++i) sum += acc_s[i][e];
    orow[e] = from_f<T>(sum / L);
  }
}

// ---------------------------------------------------------------------------
// bf16 streaming kernel
// ---------------------------------------------------------------------------

constexpr int kMChunk = 256;   // keys per work item at most (one partial state per head)
constexpr int kMKeys = 16;     // keys per stage
constexpr int kMSlots = 3;     // stages in shared memory per warp: the current one + 2 in flight
constexpr int kMWarps = 8;

template <int DH> struct MCfg {
  static constexpr int NB = DH / 64;                          // 128-byte boxes per row
  static constexpr uint32_t BOX = kMKeys * 128;               // 16 rows x 128 B
  static constexpr uint32_t KV_BYTES = NB * BOX;              // K (or V) of one stage
  static constexpr uint32_t SLOT = 2 * KV_BYTES;              // K then V
  static constexpr uint32_t WARP_BYTES = kMSlots * SLOT;
  static constexpr uint32_t OFF_BAR = kMWarps * WARP_BYTES;
  static constexpr uint32_t OFF_PRE = OFF_BAR + kMWarps * kMSlots * 8;
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&t);
}

// D = A·B + D, m16n8k16, bf16 inputs, fp32 accumulators (warp-level MMA).
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// Address of the 16-byte piece holding dims [8·chunk, 8·chunk+8) of stage row
// `row` in a K or V stage written by TMA with the 128-byte swizzle.
template <int DH>
__device__ __forceinline__ uint32_t swz(uint32_t base, int row, int chunk) {
  return base + (chunk >> 3) * MCfg<DH>::BOX + row * 128 + (((chunk & 7) ^ (row & 7)) << 4);
}

// Each warp owns a stream of work items (a sequence, a KV head, 256 keys) taken
// from a global counter, and walks it in 16-key stages.  Per stage:
//   S[16 × 16] = Q·Kᵀ with Q the G query heads padded to 16 rows (held as
//   bf16 MMA fragments in registers for the whole item) and K fragments read
//   with ldmatrix from the swizzled stage; lane (g, t) then holds four scores
//   of head g, so the row max is a two-step shuffle within its quad;
//   O[16 × dh] += P·V with P built in registers from the score fragments and
//   V fragments read with ldmatrix.trans.
// The tensor cores only shrink the instruction count; the kernel is bound by
// reading K and V from HBM.
template <int DH, int G>
__global__ void __launch_bounds__(kMWarps * 32, 1)
    k_decode_mma(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const bf16* __restrict__ q, const int32_t* __restrict__ pos_arr, int B, int Hkv,
                 float* __restrict__ part, int nchunk_max, int chunk, int* __restrict__ counter, int window,
                 PagedKV pg, float scale_log2, int* err, L2Prefetch pf) {
  pdl_trigger();
  pdl_wait();
  using C = MCfg<DH>;
  using namespace ptx;
  static_assert(G <= 8, "at most 8 query heads per KV head");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;     // MMA fragment row (query head) and column pair
  int* pre = reinterpret_cast<int*>(smem + C::OFF_PRE);
  int* nlen = pre + B + 1;           // keys of sequence b this step (0: skipped)
  __shared__ int abort_word;

  if (threadIdx.x == 0) {
    int acc = 0;
    for (int b = 0; b < B; ++b) {
      pre[b] = acc;
      const int p = pos_arr[b];
      nlen[b] = p < 0 ? 0 : p + 1;
      acc += p < 0 ? 0 : Hkv * ((p + 1 - chunk_base(p + 1, window, kMKeys) + chunk - 1) / chunk);
    }
    pre[B] = acc;
    abort_word = 0;
  }
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR) + warp * kMSlots;
  if (lane == 0) {
    for (int i = 0; i < kMSlots; ++i) mbar_init(&full[i], 1);
    fence_barrier_init();
  }
  __syncthreads();
  volatile int* abort_flag = &abort_word;
  const int total = pre[B];
  const int H = Hkv * G;
  uint8_t* slots = smem + warp * C::WARP_BYTES;
  const uint32_t slots_u32 = smem_u32(slots);

  struct Item { int b, kvh, c, key0, nkeys, first; };
  auto decode = [&](int id) {
    int lo = 0, hi = B - 1;                    // last b with pre[b] <= id
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= id) lo = mid; else hi = mid - 1;
    }
    const int n = nlen[lo];
    const int base = chunk_base(n, window, kMKeys);     // 16-key stages never straddle a page
    const int nch = (n - base + chunk - 1) / chunk;
    const int r = id - pre[lo];
    Item it;
    it.b = lo;
    it.kvh = r / nch;
    it.c = r - it.kvh * nch;
    it.key0 = base + it.c * chunk;
    it.nkeys = min(chunk, n - it.key0);
    it.first = window_first(n, window);
    return it;
  };

  // ---- lane 0: item queue and stage producer ----
  int queue[4] = {0, 0, 0, 0};
  int qn = 0, reserve = 0, pidx = 0, pst = 0;
  uint32_t issued = 0, consumed = 0;
  bool stream_done = false;
  auto push = [&]() {
    queue[qn++] = reserve;
    reserve = atomicAdd(counter, 1);          // the reply is needed only at the next push
  };
  Item pit{};                  // the producer's current item, decoded once
  int pit_id = -1, pit_nst = 0;
  const uint64_t pol = policy_evict_first();   // the cache is read once per step
  auto issue_one = [&]() {
    while (!stream_done) {
      if (pidx >= qn) push();
      const int id = queue[pidx];
      if (id >= total) {
        stream_done = true;
        return;
      }
      if (id != pit_id) {        // ids are unique: a new id is a new item
        pit = decode(id);
        pit_id = id;
        pit_nst = (pit.nkeys + kMKeys - 1) / kMKeys;
      }
      const Item& it = pit;
      if (pst < pit_nst) {
        const int sl = issued % kMSlots;
        uint8_t* base = slots + sl * C::SLOT;
        fence_proxy_async();       // earlier generic writes to the slot, before the TMA overwrite
        mbar_arrive_expect_tx(&full[sl], C::SLOT);
        const int key = it.key0 + pst * kMKeys;
        int y = key, z = it.b * Hkv + it.kvh;
        if (pg.bt) {                 // paged: the stage lies inside one page
          const int page = pg.bt[(size_t)it.b * pg.max_pages + key / pg.ps];
          y = key % pg.ps;
          if (page < 0 || page >= pg.num_pages) {
            atomicOr(err, TB_DEVERR_BAD_PAGE);
            z = pg.num_pages * Hkv;   // outside the pool: the copy reads zeros
          } else {
            z = page * Hkv + it.kvh;
          }
        }
#pragma unroll
        for (int hb = 0; hb < C::NB; ++hb) {
          tma_load_3d_hint(&tmK, base + hb * C::BOX, &full[sl], hb * 64, y, z, pol);
          tma_load_3d_hint(&tmV, base + C::KV_BYTES + hb * C::BOX, &full[sl], hb * 64, y, z, pol);
        }
        ++pst;
        ++issued;
        return;
      }
      ++pidx;
      pst = 0;
    }
  };
  if (lane == 0) {
    reserve = atomicAdd(counter, 1);
    push();
  }

  bool ok = true;
  while (ok) {
    const int cur = __shfl_sync(0xffffffffu, queue[0], 0);
    if (cur >= total) break;
    const Item it = decode(cur);
    const int nst = (it.nkeys + kMKeys - 1) / kMKeys;
    // Q fragments: rows = query heads of this KV head (rows >= G are zero)
    uint32_t qa0[DH / 16], qa2[DH / 16];
    {
      const bf16* qrow = q + ((size_t)it.b * H + it.kvh * G + (g < G ? g : 0)) * DH;
#pragma unroll
      for (int ks = 0; ks < DH / 16; ++ks) {
        qa0[ks] = g < G ? *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 2 * t) : 0u;
        qa2[ks] = g < G ? *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 8 + 2 * t) : 0u;
      }
    }
    float o[DH / 8][4];
#pragma unroll
    for (int i = 0; i < DH / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_used = -INFINITY, lsum = 0.f;

    for (int st = 0; st < nst; ++st) {
      if (lane == 0)
        while (!stream_done && issued < consumed + kMSlots) issue_one();
      const int sl = consumed % kMSlots;
      if (!mbar_wait_warp(&full[sl], (consumed / kMSlots) & 1, abort_flag, err)) {
        ok = false;
        break;
      }
      const uint32_t ks_base = slots_u32 + sl * C::SLOT, vs_base = ks_base + C::KV_BYTES;
      const int nvalid = min(kMKeys, it.nkeys - st * kMKeys);
      if (nvalid < kMKeys) {
        // V rows past the sequence hold whatever the cache holds there; P is 0
        // for them, but 0·NaN is NaN inside an MMA, so zero them first
        uint8_t* vrows = slots + sl * C::SLOT + C::KV_BYTES;
        for (int i = lane; i < (kMKeys - nvalid) * C::NB * 8; i += 32) {
          const int row = nvalid + i / (C::NB * 8), piece = i % (C::NB * 8);
          *reinterpret_cast<uint4*>(vrows + (piece >> 3) * C::BOX + row * 128 + (piece & 7) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }

      // S = Q·Kᵀ for two 8-key column tiles
      float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
      {
        const int mi = lane >> 3, row = 8 * (mi >> 1) + (lane & 7);
#pragma unroll
        for (int ks = 0; ks < DH / 16; ++ks) {
          uint32_t kb[4];
          ldsm_x4(swz<DH>(ks_base, row, 2 * ks + (mi & 1)), kb);
          mma16816(s0, qa0[ks], 0u, qa2[ks], 0u, kb[0], kb[1]);
          mma16816(s1, qa0[ks], 0u, qa2[ks], 0u, kb[2], kb[3]);
        }
      }
      // online softmax of head g over the stage's keys (raw scores; scale folded into the exponent)
      const int k0 = 2 * t, k1 = 2 * t + 1, k2 = 8 + 2 * t, k3 = 9 + 2 * t;
      const int lead = it.first - (it.key0 + st * kMKeys);   // keys below lead precede the window
      float r0 = k0 < nvalid && k0 >= lead ? s0[0] : -INFINITY, r1 = k1 < nvalid && k1 >= lead ? s0[1] : -INFINITY;
      float r2 = k2 < nvalid && k2 >= lead ? s1[0] : -INFINITY, r3 = k3 < nvalid && k3 >= lead ? s1[1] : -INFINITY;
      float mx = fmaxf(fmaxf(r0, r1), fmaxf(r2, r3));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_used, mx * scale_log2);     // finite: the stage has a visible key
      if (m_new > m_used + kRescaleLog2 || m_used == -INFINITY) {
        const float f = m_used == -INFINITY ? 0.f : ex2_approx(m_used - m_new);
        lsum *= f;
#pragma unroll
        for (int i = 0; i < DH / 8; ++i) {
          o[i][0] *= f;
          o[i][1] *= f;
        }
        m_used = m_new;
      }
      const float p0 = ex2_approx(fmaf(r0, scale_log2, -m_used)), p1 = ex2_approx(fmaf(r1, scale_log2, -m_used));
      const float p2 = ex2_approx(fmaf(r2, scale_log2, -m_used)), p3 = ex2_approx(fmaf(r3, scale_log2, -m_used));
      lsum += (p0 + p1) + (p2 + p3);
      const uint32_t pa0 = pack_bf16(p0, p1), pa2 = pack_bf16(p2, p3);
      // O += P·V over eight-dimension column tiles, two per ldmatrix
      {
        const int mi = lane >> 3, row = 8 * (mi & 1) + (lane & 7);
#pragma unroll
        for (int dt = 0; dt < DH / 8; dt += 2) {
          uint32_t vb[4];
          ldsm_x4_t(swz<DH>(vs_base, row, dt + (mi >> 1)), vb);
          mma16816(o[dt], pa0, 0u, pa2, 0u, vb[0], vb[1]);
          mma16816(o[dt + 1], pa0, 0u, pa2, 0u, vb[2], vb[3]);
        }
      }
      __syncwarp();           // the slot may be refilled after this
      ++consumed;
    }
    if (!ok) break;
    // partial state of each query head of this chunk
    float l = lsum;
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    if (g < G) {
      float* pr = part + (((size_t)it.b * H + it.kvh * G + g) * nchunk_max + it.c) * PartLayout<DH>::stride;
#pragma unroll
      for (int i = 0; i < DH / 8; ++i)
        *reinterpret_cast<float2*>(pr + 4 + 8 * i + 2 * t) = make_float2(o[i][0], o[i][1]);
      if (t == 0) {
        pr[0] = m_used;
        pr[1] = l;
      }
    }
    if (lane == 0) {          // drop the finished item from the queue
      queue[0] = queue[1];
      queue[1] = queue[2];
      queue[2] = queue[3];
      --qn;
      --pidx;
    }
  }
  // this warp's share of the next kernel's weights, pulled into L2 while the
  // other warps finish their last items
  if (ok && lane == 0 && pf.bytes)
    prefetch_l2_part(pf.p, pf.bytes, blockIdx.x * kMWarps + warp, gridDim.x * kMWarps);
  // copies issued but not consumed (only after an aborted wait) must land before the CTA exits
  issued = __shfl_sync(0xffffffffu, issued, 0);
  if (!ok && lane == 0) {
    volatile int no_abort = 0;
    for (uint32_t k = consumed; k < issued; ++k)
      mbar_wait(&full[k % kMSlots], (k / kMSlots) & 1, &no_abort, err);
  }
}

// ---------------------------------------------------------------------------
// int8-cache streaming kernel (dh = 128)
// ---------------------------------------------------------------------------
//
// The same work items and chunk states as k_decode_mma, over a cache of int8
// codes with one fp32 scale per row (a row reads back as code·scale).  A
// 32-key stage is 4 KB of K codes and 4 KB of V codes, as much as a 16-key
// bf16 stage, plus the stage's 64 row scales.
//
// Twelve warps per CTA (the transposed layout below keeps a warp at 155
// registers), each with a ring of two stage slots; as in the bf16 kernel,
// lane 0 of each warp takes work items from the global counter and issues the
// warp's own copies (two TMA boxes of codes, two 128-byte bulk copies of
// scales), writing beside each slot which item and stage it holds so that the
// warp never decodes an item.  Producers in every warp keep the copies spread
// over all four schedulers; one producer warp for the whole CTA could not
// issue them fast enough.  (Sixteen warps with three 16-key slots each ran
// 2.5% slower.)
//
// Both contractions run transposed, on fp16 m16n8k16 MMAs with fp32
// accumulators, so that the query heads sit on the MMA's n side (8 columns)
// instead of padding its 16 rows:
//   Sᵀ[16 keys × 8 heads] = K·Qᵀ for each 16-key half of a stage.  ldmatrix
//     gives lane (g, t) four consecutive codes of key g (dims 16p+4t ..
//     16p+4t+3); the MMA's k index is mapped onto dims so that those four are
//     its two k pairs, and Q's fragment uses the same map (a dot product does
//     not depend on the order of its terms).
//   Oᵀ[16 dims × 8 heads] += Vᵀ·Pᵀ.  ldmatrix.trans on 16-bit units gives
//     lane (g, t) the codes of keys 2t, 2t+1 at dims 2g, 2g+1: one word is the
//     A fragment of rows g (dim 16p+2g) and g+8 (dim 16p+2g+1).  Pᵀ comes from
//     Sᵀ's accumulator layout by one movmatrix transpose per 8 keys.
// A code c enters the MMA as the fp16 number 1152 + c: after XOR 0x80 its
// byte is u = c + 128, and the fp16 bit pattern 0x6400 | u is 1024 + u.  The
// bias is removed after the products, exactly in the algebra and to fp32
// rounding in the arithmetic: Σ_d q_d(c_d + 1152) - 1152·Σ_d q_d for the
// scores, Σ_j P_j(c_j + 1152) - 1152·Σ_j P_j for the output, with the sums
// taken over the fp16 values the MMA multiplies.
// Q is converted to fp16 once per item with a power-of-two scale per head that
// puts its largest element in [0.5, 1), so every bf16 query fits.  The K
// scales multiply the fp32 scores.  The V scales multiply P before P is
// rounded to fp16, inside a power-of-two frame vf (the accumulators hold
// vf·O) chosen so that the stage's largest visible scale times vf lies in
// [1/16, 16]: P·scale·vf then stays far from fp16's overflow and underflow
// whatever the magnitude of V.  The frame moves like the softmax maximum,
// rarely, and both rescale O by exact factors.
constexpr int kQKeys = 32;       // keys per stage
constexpr int kQWarps = 12;      // warps per CTA, each its own producer
constexpr int kQSlots = 2;       // stage slots per warp
struct QDesc {
  int4 a;                        // sequence, KV head, chunk, stage
  int4 b;                        // first key of the chunk, its keys, first visible key, item id (-1: no more)
};
struct QCfg {
  static constexpr uint32_t BOX = kQKeys * 128;        // 32 rows x 128 codes
  static constexpr uint32_t SLOT = 2 * BOX;            // K codes, then V codes
  static constexpr uint32_t WARP_BYTES = kQSlots * SLOT;
  static constexpr uint32_t SC = 2 * kQKeys * 4;       // K then V scales of one stage
  static constexpr uint32_t TX = SLOT + SC;            // bytes one stage brings in
  static constexpr uint32_t OFF_SC = kQWarps * WARP_BYTES;
  static constexpr uint32_t OFF_DESC = OFF_SC + kQWarps * kQSlots * SC;
  static constexpr uint32_t OFF_BAR = OFF_DESC + kQWarps * kQSlots * sizeof(QDesc);
  static constexpr uint32_t OFF_PRE = OFF_BAR + kQWarps * kQSlots * 8;   // then pre[B + 1], nlen[B]
};
static_assert(QCfg::OFF_SC % 1024 == 0 && QCfg::OFF_DESC % 16 == 0 && QCfg::OFF_BAR % 8 == 0, "layout");

// D = A·B + D, m16n8k16, fp16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma16816_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ float2 unpack_f16(uint32_t h) {
  float2 r;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "r"(h));
  return r;
}

// The two codes of `w` (already XORed with 0x80808080) that `sel` picks, as the
// fp16 pair 1152 + code (sel's nibbles 4 insert the byte 0x64).
__device__ __forceinline__ uint32_t biased_f16x2(uint32_t w, uint32_t sel) { return __byte_perm(w, 0x64646464u, sel); }

// Transpose of an 8x8 matrix of 16-bit elements held as MMA fragments.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// 2^-e with x·2^-e in [0.5, 1) for a normal x > 0 (read off the exponent
// field), clamped to normal powers of two; 1 for x <= 0 or NaN.
__device__ __forceinline__ float pow2_frame(float x) {
  if (!(x > 0.f)) return 1.f;
  int e = (int)((__float_as_uint(x) >> 23) & 0xffu) - 126;
  e = max(-126, min(126, e));
  return __uint_as_float((uint32_t)(127 - e) << 23);
}

// 16-byte piece `chunk` of row `row` of a 16-row x 128-byte stage written by
// TMA with the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz128(uint32_t base, int row, int chunk) {
  return base + row * 128 + (((chunk ^ row) & 7) << 4);
}

template <int G>
__global__ void __launch_bounds__(kQWarps * 32, 1)
    k_decode_i8(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                const float* __restrict__ kscale, const float* __restrict__ vscale, const bf16* __restrict__ q,
                const int32_t* __restrict__ pos_arr, int B, int Hkv, int T_max, float* __restrict__ part,
                int nchunk_max, int chunk, int* __restrict__ counter, int window, PagedKV pg, float scale_log2,
                int* err, L2Prefetch pf) {
  pdl_trigger();
  pdl_wait();
  constexpr int DH = 128, S = kQSlots;
  using C = QCfg;
  using namespace ptx;
  static_assert(G <= 8, "at most 8 query heads per KV head");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* pre = reinterpret_cast<int*>(smem + C::OFF_PRE);
  int* nlen = pre + B + 1;           // keys of sequence b this step (0: skipped)
  QDesc* desc = reinterpret_cast<QDesc*>(smem + C::OFF_DESC);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);   // [warp][slot]
  __shared__ int abort_word;

  if (threadIdx.x == 0) {
    int acc = 0;
    for (int b = 0; b < B; ++b) {
      pre[b] = acc;
      const int p = pos_arr[b];
      nlen[b] = p < 0 ? 0 : p + 1;
      acc += p < 0 ? 0 : Hkv * ((p + 1 - chunk_base(p + 1, window, kQKeys) + chunk - 1) / chunk);
    }
    pre[B] = acc;
    abort_word = 0;
    for (int i = 0; i < kQWarps * S; ++i) mbar_init(&full[i], 1);
    fence_barrier_init();
  }
  __syncthreads();
  volatile int* abort_flag = &abort_word;
  const int total = pre[B];
  const int H = Hkv * G;

  // ---------------- lane 0 of each warp fills the warp's own slots ----------------
  const int pw = warp;
  int pb = 0, pkvh = 0, pc = 0, pkey0 = 0, pnkeys = 0, pfirst = 0, pst = 0, pnst = 0, pid = 0;
  uint32_t issued = 0;
  bool pdone = false;
  int next = lane == 0 ? atomicAdd(counter, 1) : 0;
  const uint64_t pol = policy_evict_first();   // the cache is read once per step
  auto produce = [&](uint32_t consumed) {
    while (!pdone && issued < consumed + S) {
      const int sl = issued % S, bi = pw * S + sl;
      if (pst == pnst) {
        if (next >= total) {
          desc[bi].b = make_int4(0, 0, 0, -1);
          mbar_arrive(&full[bi]);
          pdone = true;
          ++issued;
          return;
        }
        pid = next;
        next = atomicAdd(counter, 1);
        int lo = pb;
        if (pre[lo + 1] <= pid) {
          int l2 = lo + 1, hi = B - 1;
          while (l2 < hi) {
            const int mid = (l2 + hi + 1) >> 1;
            if (pre[mid] <= pid) l2 = mid; else hi = mid - 1;
          }
          lo = l2;
        }
        const int n = nlen[lo];
        const int base = chunk_base(n, window, kQKeys);
        const int nch = (n - base + chunk - 1) / chunk;
        const int r = pid - pre[lo];
        pb = lo;
        pkvh = r / nch;
        pc = r - pkvh * nch;
        pkey0 = base + pc * chunk;
        pnkeys = min(chunk, n - pkey0);
        pfirst = window_first(n, window);
        pst = 0;
        pnst = (pnkeys + kQKeys - 1) / kQKeys;
      }
      desc[bi].a = make_int4(pb, pkvh, pc, pst);
      desc[bi].b = make_int4(pkey0, pnkeys, pfirst, pid);
      uint8_t* dst = smem + pw * C::WARP_BYTES + sl * C::SLOT;
      float* sc = reinterpret_cast<float*>(smem + C::OFF_SC + bi * C::SC);
      mbar_arrive_expect_tx(&full[bi], C::TX);
      const int key = pkey0 + pst * kQKeys;
      int plane = pb * Hkv + pkvh, y = key;
      size_t srow = (size_t)plane * T_max + key;
      if (pg.bt) {       // paged: a 32-key stage lies inside one page (page_size a multiple of 32)
        const int page = pg.bt[(size_t)pb * pg.max_pages + key / pg.ps];
        y = key % pg.ps;
        if (page < 0 || page >= pg.num_pages) {
          atomicOr(err, TB_DEVERR_BAD_PAGE);
          plane = pg.num_pages * Hkv;   // outside the pool: the code copies read zeros
          srow = 0;                     // and the scales come from the pool's first row
        } else {
          plane = page * Hkv + pkvh;
          srow = (size_t)plane * pg.ps + y;
        }
      }
      tma_load_3d_hint(&tmK, dst, &full[bi], 0, y, plane, pol);
      tma_load_3d_hint(&tmV, dst + C::BOX, &full[bi], 0, y, plane, pol);
      bulk_load_hint(sc, kscale + srow, kQKeys * 4, &full[bi], pol);
      bulk_load_hint(sc + kQKeys, vscale + srow, kQKeys * 4, &full[bi], pol);
      ++pst;
      ++issued;
    }
  };

  // ---------------- consumers ----------------
  const int w = warp;
  const int g = lane >> 2, t = lane & 3;
  const int mi = lane >> 3, lrow = (lane & 7) + 8 * (mi & 1);
  const uint32_t slots_u32 = smem_u32(smem + w * C::WARP_BYTES);
  const float* scw = reinterpret_cast<const float*>(smem + C::OFF_SC + w * S * C::SC);
  uint32_t qb0[DH / 16], qb1[DH / 16];
  float A0 = 0.f, A1 = 0.f, Bc0 = 0.f, Bc1 = 0.f;   // per head 2t, 2t+1: score scale and bias term
  float o[DH / 16][4];
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f, lv0 = 0.f, lv1 = 0.f, vf = 1.f;
  int ib = 0, ikvh = 0, ic = 0, ikey0 = 0, inkeys = 0, ifirst = 0;
  bool ok = true;
  uint32_t k = 0;
  for (;; ++k) {
    if (lane == 0) produce(k);
    const int sl = k % S, bi = w * S + sl;
    if (!mbar_wait_warp(&full[bi], (k / S) & 1, abort_flag, err)) {
      ok = false;
      break;
    }
    const int4 da = desc[bi].a, db = desc[bi].b;
    if (db.w < 0) break;
    const int st = da.w;
    if (st == 0) {
      // a new item: Q fragments of head g (rows >= G zero), dims 16p + 4t .. 16p + 4t + 3 of slice p
      ib = da.x;
      ikvh = da.y;
      ic = da.z;
      ikey0 = db.x;
      inkeys = db.y;
      ifirst = db.z;
      const bf16* qrow = q + ((size_t)ib * H + ikvh * G + (g < G ? g : 0)) * DH + 4 * t;
      float qv[DH / 16][4];
      float amax = 0.f;
#pragma unroll
      for (int p = 0; p < DH / 16; ++p) {
        const uint2 raw = g < G ? *reinterpret_cast<const uint2*>(qrow + 16 * p) : make_uint2(0u, 0u);
        qv[p][0] = __uint_as_float(raw.x << 16);
        qv[p][1] = __uint_as_float(raw.x & 0xffff0000u);
        qv[p][2] = __uint_as_float(raw.y << 16);
        qv[p][3] = __uint_as_float(raw.y & 0xffff0000u);
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(qv[p][0]), fabsf(qv[p][1])), fmaxf(fabsf(qv[p][2]), fabsf(qv[p][3]))));
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      const float qf = pow2_frame(amax);
      float qs = 0.f;                   // Σ of the fp16 query values, for the score bias
#pragma unroll
      for (int p = 0; p < DH / 16; ++p) {
        qb0[p] = pack_f16(qv[p][0] * qf, qv[p][1] * qf);
        qb1[p] = pack_f16(qv[p][2] * qf, qv[p][3] * qf);
        const float2 a = unpack_f16(qb0[p]), c = unpack_f16(qb1[p]);
        qs += (a.x + a.y) + (c.x + c.y);
      }
      qs += __shfl_xor_sync(0xffffffffu, qs, 1);
      qs += __shfl_xor_sync(0xffffffffu, qs, 2);
      const float cq = scale_log2 / qf, cb = 1152.f * qs * cq;
      A0 = __shfl_sync(0xffffffffu, cq, 8 * t);         // lane 8t holds head 2t, lane 8t+4 head 2t+1
      A1 = __shfl_sync(0xffffffffu, cq, 8 * t + 4);
      Bc0 = __shfl_sync(0xffffffffu, cb, 8 * t);
      Bc1 = __shfl_sync(0xffffffffu, cb, 8 * t + 4);
#pragma unroll
      for (int p = 0; p < DH / 16; ++p) o[p][0] = o[p][1] = o[p][2] = o[p][3] = 0.f;
      m0 = m1 = -INFINITY;
      l0 = l1 = lv0 = lv1 = 0.f;
      vf = 1.f;
    }
    const uint32_t kbase = slots_u32 + sl * C::SLOT, vbase = kbase + C::BOX;
    const float* sc = scw + sl * (C::SC / 4);
    const int nvalid = min(kQKeys, inkeys - st * kQKeys);
    const int lead = ifirst - (ikey0 + st * kQKeys);   // keys below lead precede the window

    // Sᵀ = K·Qᵀ (biased codes) for keys 16h .. 16h+15, h = 0, 1; even and odd
    // slices in separate accumulators
    float sa[2][4], sb[2][4];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int j = 0; j < 4; ++j) sa[h][j] = sb[h][j] = 0.f;
#pragma unroll
    for (int pp = 0; pp < DH / 32; ++pp)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t kb[4];
        ldsm_x4(swz128(kbase, lrow + 16 * h, 2 * pp + (mi >> 1)), kb);
#pragma unroll
        for (int j = 0; j < 4; ++j) kb[j] ^= 0x80808080u;
        mma16816_f16(sa[h], biased_f16x2(kb[0], 0x4140), biased_f16x2(kb[1], 0x4140), biased_f16x2(kb[0], 0x4342),
                     biased_f16x2(kb[1], 0x4342), qb0[2 * pp], qb1[2 * pp]);
        mma16816_f16(sb[h], biased_f16x2(kb[2], 0x4140), biased_f16x2(kb[3], 0x4140), biased_f16x2(kb[2], 0x4342),
                     biased_f16x2(kb[3], 0x4342), qb0[2 * pp + 1], qb1[2 * pp + 1]);
      }
    // lane (g, t): keys 16h + 8s + g (h, s = 0, 1), heads 2t and 2t+1
    float r[2][2][2], wv[2][2];
    float mx0 = -INFINITY, mx1 = -INFINITY, vmax = 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int sk = 0; sk < 2; ++sk) {
        const int key = 16 * h + 8 * sk + g;
        const bool ok = key < nvalid && key >= lead;
        const float ks = sc[key], vs = sc[kQKeys + key];
        r[h][sk][0] = ok ? ks * fmaf(sa[h][2 * sk] + sb[h][2 * sk], A0, -Bc0) : -INFINITY;
        r[h][sk][1] = ok ? ks * fmaf(sa[h][2 * sk + 1] + sb[h][2 * sk + 1], A1, -Bc1) : -INFINITY;
        wv[h][sk] = ok ? vs : 0.f;
        mx0 = fmaxf(mx0, r[h][sk][0]);
        mx1 = fmaxf(mx1, r[h][sk][1]);
        vmax = fmaxf(vmax, wv[h][sk]);
      }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, off));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);   // finite: the stage has a visible key
    const bool nm0 = m0 == -INFINITY || mn0 > m0 + kRescaleLog2;
    const bool nm1 = m1 == -INFINITY || mn1 > m1 + kRescaleLog2;
    const float vr = vmax * vf;
    const bool nf = vr > 16.f || (vmax > 0.f && vr < 0.0625f);
    if (nm0 || nm1 || nf) {
      float f0 = 1.f, f1 = 1.f;
      if (nm0) {
        f0 = m0 == -INFINITY ? 0.f : ex2_approx(m0 - mn0);
        l0 *= f0;
        m0 = mn0;
      }
      if (nm1) {
        f1 = m1 == -INFINITY ? 0.f : ex2_approx(m1 - mn1);
        l1 *= f1;
        m1 = mn1;
      }
      if (nf) {
        const float vf_new = pow2_frame(vmax);
        const float rr = vf_new / vf;            // both powers of two: exact
        vf = vf_new;
        if (f0 != 0.f) f0 *= rr;
        if (f1 != 0.f) f1 *= rr;
      }
      lv0 *= f0;
      lv1 *= f1;
#pragma unroll
      for (int p = 0; p < DH / 16; ++p) {
        o[p][0] *= f0;
        o[p][2] *= f0;
        o[p][1] *= f1;
        o[p][3] *= f1;
      }
    }
    // P·scale·vf in fp16, then the Pᵀ fragments of each 16-key half by movmatrix
    uint32_t pb0[2], pb1[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float p00 = ex2_approx(r[h][0][0] - m0), p01 = ex2_approx(r[h][0][1] - m1);
      const float p10 = ex2_approx(r[h][1][0] - m0), p11 = ex2_approx(r[h][1][1] - m1);
      l0 += p00 + p10;
      l1 += p01 + p11;
      const float wl = wv[h][0] * vf, wh = wv[h][1] * vf;
      const uint32_t pk_lo = pack_f16(p00 * wl, p01 * wl), pk_hi = pack_f16(p10 * wh, p11 * wh);
      const float2 a = unpack_f16(pk_lo), c = unpack_f16(pk_hi);
      lv0 += a.x + c.x;
      lv1 += a.y + c.y;
      pb0[h] = movmatrix_t(pk_lo);
      pb1[h] = movmatrix_t(pk_hi);
    }
    // Oᵀ += Vᵀ·Pᵀ: m-tile p = dims 16p + 2g (rows g) and 16p + 2g + 1 (rows g+8), k = the two key halves
#pragma unroll
    for (int pp = 0; pp < DH / 32; ++pp)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t vb[4];
        ldsm_x4_t(swz128(vbase, lrow + 16 * h, 2 * pp + (mi >> 1)), vb);
#pragma unroll
        for (int j = 0; j < 4; ++j) vb[j] ^= 0x80808080u;
        mma16816_f16(o[2 * pp], biased_f16x2(vb[0], 0x4240), biased_f16x2(vb[0], 0x4341),
                     biased_f16x2(vb[1], 0x4240), biased_f16x2(vb[1], 0x4341), pb0[h], pb1[h]);
        mma16816_f16(o[2 * pp + 1], biased_f16x2(vb[2], 0x4240), biased_f16x2(vb[2], 0x4341),
                     biased_f16x2(vb[3], 0x4240), biased_f16x2(vb[3], 0x4341), pb0[h], pb1[h]);
      }
    __syncwarp();             // the slot may be refilled after this
    if ((st + 1) * kQKeys >= inkeys) {
      // the item's partial state for heads 2t and 2t+1: sums over the eight key rows g
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        lv0 += __shfl_xor_sync(0xffffffffu, lv0, off);
        lv1 += __shfl_xor_sync(0xffffffffu, lv1, off);
      }
      const float inv = 1.0f / vf, c0 = 1152.f * lv0, c1 = 1152.f * lv1;
      const int h0 = 2 * t, h1 = 2 * t + 1;
      constexpr int P = PartLayout<DH>::stride;
      if (h0 < G) {
        float* pr = part + (((size_t)ib * H + ikvh * G + h0) * nchunk_max + ic) * P;
#pragma unroll
        for (int p = 0; p < DH / 16; ++p)
          *reinterpret_cast<float2*>(pr + 4 + 16 * p + 2 * g) = make_float2((o[p][0] - c0) * inv, (o[p][2] - c0) * inv);
        if (g == 0) {
          pr[0] = m0;
          pr[1] = l0;
        }
      }
      if (h1 < G) {
        float* pr = part + (((size_t)ib * H + ikvh * G + h1) * nchunk_max + ic) * P;
#pragma unroll
        for (int p = 0; p < DH / 16; ++p)
          *reinterpret_cast<float2*>(pr + 4 + 16 * p + 2 * g) = make_float2((o[p][1] - c1) * inv, (o[p][3] - c1) * inv);
        if (g == 0) {
          pr[0] = m1;
          pr[1] = l1;
        }
      }
    }
  }
  if (ok && lane == 0 && pf.bytes)     // this warp's share of the next kernel's weights, into L2
    prefetch_l2_part(pf.p, pf.bytes, blockIdx.x * kQWarps + warp, gridDim.x * kQWarps);
  issued = __shfl_sync(0xffffffffu, issued, 0);
  if (!ok && lane == 0) {      // copies issued but not consumed must land before the CTA exits
    volatile int no_abort = 0;
    for (uint32_t j = k; j < issued; ++j) mbar_wait(&full[pw * S + j % S], (j / S) & 1, &no_abort, err);
  }
}

template <int G>
cudaError_t run_stream_i8(const void* q, const void* kc, const void* vc, const float* ks, const float* vs,
                          const int32_t* pos, int B, int Hkv, int T_max, float* part, int nchunk_max, int chunk,
                          int* counter, int window, const PagedKV& pg, void* o, cudaStream_t s,
                          const L2Prefetch& pf) {
  using C = QCfg;
  CUtensorMap tk, tv;
  // contiguous: (sequence, KV head) planes of T_max rows; paged: (page, KV head) planes of page_size rows
  const uint64_t planes = pg.bt ? (uint64_t)pg.num_pages * Hkv : (uint64_t)B * Hkv;
  const uint64_t rows = pg.bt ? (uint64_t)pg.ps : (uint64_t)T_max;
  cudaError_t e = make_tmap_3d_u8(&tk, kc, planes, rows, 128, 128, rows * 128, 128, kQKeys);
  if (e != cudaSuccess) return e;
  e = make_tmap_3d_u8(&tv, vc, planes, rows, 128, 128, rows * 128, 128, kQKeys);
  if (e != cudaSuccess) return e;
  const size_t smem = C::OFF_PRE + (size_t)(2 * B + 1) * 4 + 1024;
  if (smem > 232448) return cudaErrorInvalidValue;
  static size_t attr_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || attr_set[dev] < smem) {
    e = cudaFuncSetAttribute(k_decode_i8<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = smem;
  }
  const float scale_log2 = 1.4426950408889634f / sqrtf(128.f);
  e = launch_pdl(k_decode_i8<G>, dim3(sm_count()), dim3(kQWarps * 32), smem, s, tk, tv, ks, vs, (const bf16*)q, pos, B,
                 Hkv, T_max, part, nchunk_max, chunk, counter, window, pg, scale_log2, device_error_word(), pf);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_decode_combine<bf16, 128>, dim3(Hkv * G, B), dim3(256), 0, s, (const float*)part, pos, Hkv * G,
                    nchunk_max, chunk, window, kQKeys, (bf16*)o);
}

template <int DH, int G>
cudaError_t run_stream(const void* q, const void* kc, const void* vc, const int32_t* pos, int B, int Hkv, int T_max,
                       float* part, int nchunk_max, int chunk, int* counter, int window, const PagedKV& pg, void* o,
                       cudaStream_t s, const L2Prefetch& pf) {
  using C = MCfg<DH>;
  CUtensorMap tk, tv;
  // planes of rows: (sequence, KV head) planes of T_max rows, or (page, KV head) planes of page_size rows
  const uint64_t planes = pg.bt ? (uint64_t)pg.num_pages * Hkv : (uint64_t)B * Hkv;
  const uint64_t rows = pg.bt ? (uint64_t)pg.ps : (uint64_t)T_max;
  cudaError_t e = make_tmap_3d_bf16(&tk, pg.bt ? pg.k : kc, planes, rows, DH, DH, rows * DH, 64, kMKeys);
  if (e != cudaSuccess) return e;
  e = make_tmap_3d_bf16(&tv, pg.bt ? pg.v : vc, planes, rows, DH, DH, rows * DH, 64, kMKeys);
  if (e != cudaSuccess) return e;
  const size_t smem = C::OFF_PRE + (size_t)(2 * B + 1) * 4 + 1024;
  if (smem > 232448) return cudaErrorInvalidValue;
  // raise the kernel's dynamic shared-memory limit only when a launch needs
  // more than this device has been given so far (no attribute call in the
  // steady state, e.g. while a stream is being captured)
  static size_t attr_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || attr_set[dev] < smem) {
    e = cudaFuncSetAttribute(k_decode_mma<DH, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = smem;
  }
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)DH);
  e = launch_pdl(k_decode_mma<DH, G>, dim3(sm_count()), dim3(kMWarps * 32), smem, s, tk, tv, (const bf16*)q, pos, B,
                 Hkv, part, nchunk_max, chunk, counter, window, pg, scale_log2, device_error_word(), pf);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_decode_combine<bf16, DH>, dim3(Hkv * G, B), dim3(256), 0, s, (const float*)part, pos, Hkv * G,
                    nchunk_max, chunk, window, kMKeys, (bf16*)o);
}

template <int DH>
cudaError_t stream_by_g(int G, const void* q, const void* kc, const void* vc, const int32_t* pos, int B, int Hkv,
                        int T_max, float* part, int nchunk_max, int chunk, int* counter, int window, const PagedKV& pg,
                        void* o, cudaStream_t s, const L2Prefetch& pf) {
  switch (G) {
    case 1: return run_stream<DH, 1>(q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, chunk, counter, window, pg, o,
                                         s, pf);
    case 2: return run_stream<DH, 2>(q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, chunk, counter, window, pg, o,
                                         s, pf);
    case 4: return run_stream<DH, 4>(q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, chunk, counter, window, pg, o,
                                         s, pf);
    case 8: return run_stream<DH, 8>(q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, chunk, counter, window, pg, o,
                                         s, pf);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T, int DH, int G>
cudaError_t run(const void* q, const void* kc, const void* vc, const int32_t* pos, int B, int Hkv, int T_max,
                float* part, int nchunk_max, int window, const PagedKV& pg, void* o, cudaStream_t s) {
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)DH);
  const cudaError_t e = launch_pdl(k_decode_split<T, DH, G>, dim3(nchunk_max, Hkv, B), dim3(kWarps * 32), 0, s,
                                   (const T*)q, (const T*)kc, (const T*)vc, pos, Hkv, T_max, part, nchunk_max, window,
                                   pg, scale_log2);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_decode_combine<T, DH>, dim3(Hkv * G, B), dim3(256), 0, s, (const float*)part, pos, Hkv * G,
                    nchunk_max, kChunk, window, 1, (T*)o);
}

template <typename T, int DH>
cudaError_t by_g(int G, const void* q, const void* kc, const void* vc, const int32_t* pos, int B, int Hkv,
                 int T_max, float* part, int nchunk_max, int window, const PagedKV& pg, void* o, cudaStream_t s) {
  switch (G) {
    case 1: return run<T, DH, 1>(q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, window, pg, o, s);
    case 2: return run<T, DH, 2>(q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, window, pg, o, s);
    case 4: return run<T, DH, 4>(q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, window, pg, o, s);
    case 8: return run<T, DH, 8>(q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, window, pg, o, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t by_dh(int dh, int G, const void* q, const void* kc, const void* vc, const int32_t* pos, int B,
                  int Hkv, int T_max, float* part, int nchunk_max, int window, const PagedKV& pg, void* o, cudaStream_t s) {
  switch (dh) {
    case 16: return by_g<T, 16>(G, q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, window, pg, o, s);
    case 32: return by_g<T, 32>(G, q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, window, pg, o, s);
    case 64: return by_g<T, 64>(G, q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, window, pg, o, s);
    case 128: return by_g<T, 128>(G, q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, window, pg, o, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

// Keys per work item.  The fp32 kernel takes 256 per CTA.  The streaming
// kernels take 256 unless a full cache would give fewer items than there are
// warps on the GPU; then 128 or 64 (small batches: more, shorter items, so
// that every SM streams), while a sequence of T_max rows stays within the
// merge's 1024 chunks.  Shorter items cost more per key (each carries its own
// query setup and partial state), so the chunk is halved only that far.  The
// workspace and the launch both use this value.
int decode_chunk_keys(int dtype, int B, int Hkv, int T_max) {
  return decode_chunk_keys_sms(dtype, B, Hkv, T_max, sm_count());
}

int decode_chunk_keys_sms(int dtype, int B, int Hkv, int T_max, int sms) {
  if (dtype == TB_F32) return kChunk;
  const long long target = (long long)sms * kMWarps;
  int c = kMChunk;
  while (c > 64 && (long long)B * Hkv * ((T_max + c - 1) / c) < target &&
         (T_max + c / 2 - 1) / (c / 2) <= kCombineMaxChunks)
    c /= 2;
  return c;
}

cudaError_t attn_decode_i8(const void* q, const void* kc, const void* vc, const float* ks, const float* vs,
                           const int32_t* pos, int B, int H, int Hkv, int T_max, float* part, int nchunk_max, int chunk,
                           int* work_counter, int window, const PagedKV& pg, void* o, cudaStream_t s,
                           const L2Prefetch& pf) {
  if (chunk % kQKeys || (pg.bt && pg.ps % kQKeys)) return cudaErrorInvalidValue;
  switch (H / Hkv) {
    case 1: return run_stream_i8<1>(q, kc, vc, ks, vs, pos, B, Hkv, T_max, part, nchunk_max, chunk, work_counter,
                                         window, pg, o, s, pf);
    case 2: return run_stream_i8<2>(q, kc, vc, ks, vs, pos, B, Hkv, T_max, part, nchunk_max, chunk, work_counter,
                                         window, pg, o, s, pf);
    case 4: return run_stream_i8<4>(q, kc, vc, ks, vs, pos, B, Hkv, T_max, part, nchunk_max, chunk, work_counter,
                                         window, pg, o, s, pf);
    case 8: return run_stream_i8<8>(q, kc, vc, ks, vs, pos, B, Hkv, T_max, part, nchunk_max, chunk, work_counter,
                                         window, pg, o, s, pf);
    default: return cudaErrorInvalidValue;
  }
}

size_t decode_part_floats(int B, int H, int dh, int nchunk_max) {
  return (size_t)B * H * nchunk_max * (dh + 4);
}

cudaError_t attn_decode(int dtype, const void* q, const void* kc, const void* vc, const int32_t* pos, int B,
                        int H, int Hkv, int dh, int T_max, float* part, int nchunk_max, int chunk, int* work_counter,
                        int window, const PagedKV& pg, void* o, cudaStream_t s, const L2Prefetch& pf) {
  const int G = H / Hkv;
  if (dtype == TB_F32) return by_dh<float>(dh, G, q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, window, pg, o, s);
  if (chunk % kMKeys) return cudaErrorInvalidValue;
  if (dh == 128)
    return stream_by_g<128>(G, q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, chunk, work_counter, window, pg, o, s,
                            pf);
  if (dh == 64)
    return stream_by_g<64>(G, q, kc, vc, pos, B, Hkv, T_max, part, nchunk_max, chunk, work_counter, window, pg, o, s,
                           pf);
  return cudaErrorInvalidValue;
}

}  // namespace tb
