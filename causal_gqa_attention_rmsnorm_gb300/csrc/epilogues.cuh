// GEMM epilogues of the block, shared by the fp32 SIMT GEMM and the bf16
// tcgen05 GEMM.  Each functor receives 4 consecutive output columns
// [col, col+4) of one row with col % 4 == 0, in fp32, and returns a value the
// caller sums over its share of the row's columns when kRowReduce is set, as
// one partial of the RowSum that row_sums() names.  kRowSumIn marks an
// epilogue whose row inputs start from such a RowSum (row_sum_in), so that the
// tile GEMM can form each row's sum once per warp.
//
// Steps ("Transformer block" page, tirogla.com, "How it works" step 2-3):
//   QKV  : × r (RMSNorm-1 row scale), RoPE on q and k, scatter q / k / v
//   Wo   : h = x + o·Wo  (first residual add), Σ h² for RMSNorm-2
//   W1W3 : a = SiLU(r2·gate) ⊙ (r2·up)  (columns come interleaved gate, up)
//   W2   : y = h + a·W2 (second residual add)
#pragma once

#include "common.cuh"

namespace tb {

template <typename T> __device__ __forceinline__ void store4(T* p, const float v[4]);
template <> __device__ __forceinline__ void store4<float>(float* p, const float v[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
template <> __device__ __forceinline__ void store4<bf16>(bf16* p, const float v[4]) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
  __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}
template <typename T> __device__ __forceinline__ void load4(const T* p, float v[4]);
template <> __device__ __forceinline__ void load4<float>(const float* p, float v[4]) {
  const float4 f = *reinterpret_cast<const float4*>(p);
  v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
}
template <> __device__ __forceinline__ void load4<bf16>(const bf16* p, float v[4]) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  v[0] = __uint_as_float(u.x << 16); v[1] = __uint_as_float(u.x & 0xffff0000u);
  v[2] = __uint_as_float(u.y << 16); v[3] = __uint_as_float(u.y & 0xffff0000u);
}
template <typename T> __device__ __forceinline__ void store2(T* p, float a, float b);
template <> __device__ __forceinline__ void store2<float>(float* p, float a, float b) {
  *reinterpret_cast<float2*>(p) = make_float2(a, b);
}
template <> __device__ __forceinline__ void store2<bf16>(bf16* p, float a, float b) {
  *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(a, b);
}

// Streaming forms (ld/st.global.cs: evict-first in L2) for the outputs and
// residual inputs of a prefill-sized GEMM, which pass through once and are
// larger than L2; they would otherwise push the GEMM's operand tiles out.
// Chosen at compile time (kStream): a run-time choice in the epilogue's inner
// loop measured slower than either form.
template <typename T> __device__ __forceinline__ void store4cs(T* p, const float v[4]);
template <> __device__ __forceinline__ void store4cs<float>(float* p, const float v[4]) {
  __stcs(reinterpret_cast<float4*>(p), make_float4(v[0], v[1], v[2], v[3]));
}
template <> __device__ __forceinline__ void store4cs<bf16>(bf16* p, const float v[4]) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
  __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  __stcs(reinterpret_cast<uint2*>(p), u);
}
template <typename T> __device__ __forceinline__ void load4cs(const T* p, float v[4]);
template <> __device__ __forceinline__ void load4cs<float>(const float* p, float v[4]) {
  const float4 f = __ldcs(reinterpret_cast<const float4*>(p));
  v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
}
template <> __device__ __forceinline__ void load4cs<bf16>(const bf16* p, float v[4]) {
  const uint2 u = __ldcs(reinterpret_cast<const uint2*>(p));
  v[0] = __uint_as_float(u.x << 16); v[1] = __uint_as_float(u.x & 0xffff0000u);
  v[2] = __uint_as_float(u.y << 16); v[3] = __uint_as_float(u.y & 0xffff0000u);
}
template <typename T> __device__ __forceinline__ void store2cs(T* p, float a, float b);
template <> __device__ __forceinline__ void store2cs<float>(float* p, float a, float b) {
  __stcs(reinterpret_cast<float2*>(p), make_float2(a, b));
}
template <> __device__ __forceinline__ void store2cs<bf16>(bf16* p, float a, float b) {
  __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
  __stcs(reinterpret_cast<unsigned int*>(p), *reinterpret_cast<unsigned int*>(&t));
}
template <bool CS, typename T> __device__ __forceinline__ void st4(T* p, const float v[4]) {
  if constexpr (CS) store4cs<T>(p, v); else store4<T>(p, v);
}
template <bool CS, typename T> __device__ __forceinline__ void ld4(const T* p, float v[4]) {
  if constexpr (CS) load4cs<T>(p, v); else load4<T>(p, v);
}
template <bool CS, typename T> __device__ __forceinline__ void st2(T* p, float a, float b) {
  if constexpr (CS) store2cs<T>(p, a, b); else store2<T>(p, a, b);
}

// RoPE rotation of one adjacent pair by the angle whose (cos, sin) is cs.
__device__ __forceinline__ void rope_pair(float& a, float& b, float2 cs) {
  const float x = a, y = b;
  a = x * cs.x - y * cs.y;
  b = x * cs.y + y * cs.x;
}

// Every epilogue reads its global inputs in two steps ahead of any store, so a
// caller processing several (row, 4-column) items can issue all their loads
// before the first store.  kStream (the prefill tile GEMM's instances) turns
// the once-through traffic into streaming loads and stores:
//   RowAux row_aux(row)            inputs that depend on the row only (once per tile)
//   Aux    aux(row, col, RowAux)   inputs of the 4 columns
//   float  operator()(row, col, v, RowAux, Aux)   compute and store; returns the
//                                  item's share of a row reduction (kRowReduce)

template <typename T, bool kStream = false>
struct EpiQKV {
  static constexpr bool kRowReduce = false;
  static constexpr bool kRowLse = false;
  static constexpr bool kRowSumIn = false;
  static constexpr bool kRowStats = true;           // can form RMSNorm-1 statistics (a.st.x != nullptr)
  static constexpr bool kRowDone = false;
  static constexpr bool kTileStats = true;          // the tile GEMM may form them (a.ts.x != nullptr)
  QKVArgs a;
  int H, Hkv, dh, dh_shift;             // dh = 1 << dh_shift
  struct RowAux { float r; int b, t, qt, kt; };
  struct Aux { float2 c0, c1; };
  __device__ __forceinline__ RowAux row_aux_nor(int row) const {
    RowAux ra;
    if (a.pos) {
      ra.b = row; ra.t = a.pos[row]; ra.qt = 0;
    } else {
      ra.b = row / a.T; ra.t = row - ra.b * a.T; ra.qt = ra.t;
    }
    ra.kt = a.kv_dense ? ra.qt : ra.t;
    ra.r = 0.f;
    return ra;
  }
  __device__ __forceinline__ RowAux row_aux(int row) const {
    RowAux ra = row_aux_nor(row);
    ra.r = __ldcg(a.r + row);       // L2: with a.ts.x set, another CTA of this kernel wrote it
    return ra;
  }
  // The row inputs with the row scale r given (the tile GEMM's epilogue when
  // it formed r itself).
  __device__ __forceinline__ RowAux row_aux_r(int row, float r) const {
    RowAux ra = row_aux_nor(row);
    ra.r = r;
    return ra;
  }
  // The tile GEMM's statistics warp: Σx² of token row m over its 32 lanes
  // (16-byte vectors lane, lane + 32, ...), added across the warp in a fixed
  // order ("Transformer block" page, RMSNorm: eps inside the root).  Sixteen
  // loads per lane are in flight at once (a whole 8 KB row at d = 4096), so
  // that one warp per CTA keeps ahead of the tiles that wait for its rows.
  __device__ __forceinline__ float tile_row_scale(int m, int lane) const {
    const int d = a.ts.d;
    const T* xr = (const T*)a.ts.x + (size_t)m * d;
    constexpr int V = 16 / sizeof(T), U = 16;
    float s = 0.f;
    if (d % V == 0) {
      const uint4* p = reinterpret_cast<const uint4*>(xr);
      const int nv = d / V;
      int i = lane;
      for (; i + 32 * (U - 1) < nv; i += 32 * U) {
        Vec16<T> v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) v[u].raw = __ldcs(p + i + 32 * u);
#pragma unroll
        for (int u = 0; u < U; ++u)
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
    return 1.0f / sqrtf(s / (float)d + a.ts.eps);
  }
  // Few-token decode with a.st.x set, one warp: Σx² of token rows t_first,
  // t_first + t_step, ... (below M, at most TPW of them) over columns
  // [k0, k1), k0 and k1 multiples of 64; each row's 16-byte vectors are taken
  // by lanes lane, lane + 32, ..., then summed across the warp in a fixed
  // order.  The loads of all the rows are issued together.  The cluster adds
  // the ranges in order, and the root is taken as the "Transformer block"
  // page's RMSNorm has it: mean of squares, eps inside the root.
  template <int TPW>
  __device__ __forceinline__ void row_stats_ranges(int t_first, int t_step, int M, int k0, int k1, int lane,
                                                   float (&ss)[TPW]) const {
    constexpr int V = 16 / sizeof(T);
    const int nv = (k1 - k0) / V;
#pragma unroll
    for (int j = 0; j < TPW; ++j) ss[j] = 0.f;
    for (int i = lane; i < nv; i += 32) {
      Vec16<T> v[TPW];
#pragma unroll
      for (int j = 0; j < TPW; ++j) {
        const int t = t_first + j * t_step;
        if (t < M) v[j].raw = __ldg(reinterpret_cast<const uint4*>((const T*)a.st.x + (size_t)t * a.st.d + k0) + i);
      }
#pragma unroll
      for (int j = 0; j < TPW; ++j) {
        if (t_first + j * t_step < M) {
#pragma unroll
          for (int e = 0; e < V; ++e) {
            const float f = v[j].get(e);
            ss[j] = fmaf(f, f, ss[j]);
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < TPW; ++j) ss[j] = warp_sum(ss[j]);
  }
  // The row inputs of decode token m from lens (the scale r follows from Σx²).
  __device__ __forceinline__ RowAux row_aux_pos(int m) const {
    RowAux ra;
    const int p = a.st.lens[m];
    ra.b = m;
    ra.t = (p >= 0 && p < a.st.T_max) ? p : -1;
    ra.qt = 0;
    ra.kt = a.kv_dense ? ra.qt : ra.t;
    ra.r = 0.f;
    return ra;
  }
  // The scale r from Σx²; the token's first reducer (first) publishes the
  // position, flags a full cache, and zeroes the step's work counter.
  __device__ __forceinline__ void row_stats_finish(RowAux& ra, int m, float ssq, bool first) const {
    ra.r = 1.0f / sqrtf(ssq / (float)a.st.d + a.st.eps);
    if (first) {
      a.st.pos_out[m] = ra.t;
      if (ra.t < 0) atomicOr(a.st.err, TB_DEVERR_CACHE_FULL);
      if (m == 0 && a.st.zero_word) *a.st.zero_word = 0;
    }
  }
  __device__ __forceinline__ Aux aux(int, int col, const RowAux& ra) const {
    Aux x;
    if (col < (H + Hkv) * dh && ra.t >= 0) {
      const float2* cs = a.rope + (size_t)ra.t * (dh >> 1) + ((col & (dh - 1)) >> 1);
      x.c0 = cs[0];
      x.c1 = cs[1];
    } else {
      x.c0 = x.c1 = make_float2(1.f, 0.f);
    }
    return x;
  }
  __device__ __forceinline__ float operator()(int, int col, float v[4], const RowAux& ra, const Aux& x) const {
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] *= ra.r;
    const int qn = H * dh, kn = Hkv * dh;
    const int e = col & (dh - 1);       // dh is a power of two
    rope_pair(v[0], v[1], x.c0);        // identity rotation for v columns
    rope_pair(v[2], v[3], x.c1);
    if (col < qn) {
      const int h = col >> dh_shift;
      st4<kStream, T>((T*)a.q + (((size_t)ra.b * H + h) * a.T + ra.qt) * dh + e, v);   // K/V: re-read
    } else if (ra.t >= 0) {
      const bool is_k = col < qn + kn;
      const int h = (col - (is_k ? qn : qn + kn)) >> dh_shift;
      if (a.k) {
        T* base = (T*)(is_k ? a.k : a.v);
        store4<T>(base + (((size_t)ra.b * Hkv + h) * a.kv_stride + ra.kt) * dh + e, v);
      }
      if (a.pg.bt) {
        const long long row = paged_row(a.pg, Hkv, ra.b, h, ra.t);
        if (row >= 0) store4<T>((T*)(is_k ? a.pg.k : a.pg.v) + row * dh + e, v);
      }
    }
    return 0.f;
  }
};

template <typename T, bool kStream = false>
struct EpiWo {
  static constexpr bool kRowReduce = true;
  static constexpr bool kRowLse = false;
  static constexpr bool kRowSumIn = false;
  static constexpr bool kRowStats = false;
  static constexpr bool kRowDone = true;            // few-token decode: advances the cache length
  static constexpr bool kTileStats = false;
  WoArgs a;
  int d;
  struct RowAux {};
  struct Aux { float x[4]; };
  __device__ __forceinline__ RowAux row_aux(int) const { return RowAux{}; }
  __device__ __forceinline__ Aux aux(int row, int col, const RowAux&) const {
    Aux x;
    ld4<kStream, T>((const T*)a.x + (size_t)row * d + col, x.x);
    return x;
  }
  __device__ __forceinline__ float operator()(int row, int col, float v[4], const RowAux&, const Aux& x) const {
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] += x.x[i];
    st4<kStream, float>(a.h + (size_t)row * d + col, v);
    if ((void*)a.hb != (void*)a.h) st4<kStream, T>((T*)a.hb + (size_t)row * d + col, v);
    return v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3];
  }
  __device__ __forceinline__ const RowSum& row_sums() const { return a.ssq; }
  // once per token row, after every reader of the old cache length
  __device__ __forceinline__ void row_done(int m) const {
    if (a.lens && a.pos[m] >= 0) a.lens[m] = a.pos[m] + 1;
  }
};

template <typename T, bool kStream = false>
struct EpiW13 {
  static constexpr bool kRowReduce = false;
  static constexpr bool kRowLse = false;
  static constexpr bool kRowSumIn = true;
  static constexpr bool kRowStats = false;
  static constexpr bool kRowDone = false;
  static constexpr bool kTileStats = false;
  W13Args a;
  int d, f;
  float eps;
  struct RowAux { float r2; };
  struct Aux {};
  // Σ h² of a row: the Wo GEMM's partials in order
  __device__ __forceinline__ float row_sum_in(int row) const {
    return ordered_sum(a.ssq.part + (size_t)row * a.ssq.stride, a.ssq.n);
  }
  __device__ __forceinline__ RowAux row_aux_with(float ssq) const {
    return RowAux{1.0f / sqrtf(ssq / (float)d + eps)};
  }
  __device__ __forceinline__ RowAux row_aux(int row) const { return row_aux_with(row_sum_in(row)); }
  __device__ __forceinline__ Aux aux(int, int, const RowAux&) const { return Aux{}; }
  __device__ __forceinline__ float operator()(int row, int col, float v[4], const RowAux& ra, const Aux&) const {
    const float r2 = ra.r2;
    const float o0 = silu_f(v[0] * r2) * (v[1] * r2);
    const float o1 = silu_f(v[2] * r2) * (v[3] * r2);
    st2<kStream, T>((T*)a.a + (size_t)row * f + (col >> 1), o0, o1);
    return 0.f;
  }
};

template <bool kStream = false>
struct EpiW2 {
  static constexpr bool kRowReduce = false;
  static constexpr bool kRowLse = false;
  static constexpr bool kRowSumIn = false;
  static constexpr bool kRowStats = false;
  static constexpr bool kRowDone = false;
  static constexpr bool kTileStats = false;
  W2Args a;
  int d;
  struct RowAux {};
  struct Aux { float h[4]; };
  __device__ __forceinline__ RowAux row_aux(int) const { return RowAux{}; }
  __device__ __forceinline__ Aux aux(int row, int col, const RowAux&) const {
    Aux x;
    ld4<kStream, float>(a.h + (size_t)row * d + col, x.h);
    return x;
  }
  __device__ __forceinline__ float operator()(int row, int col, float v[4], const RowAux&, const Aux& x) const {
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] += x.h[i];
    if (a.y_dtype == TB_F32)
      st4<kStream, float>((float*)a.y + (size_t)row * d + col, v);
    else
      st4<kStream, bf16>((bf16*)a.y + (size_t)row * d + col, v);
    return 0.f;
  }
};

// LM head: logits = (x·r)·W_Uᵀ with the final norm's gain folded into the
// packed W_U and r the final RMSNorm's row scale ("Transformer block" page,
// "How it works", step 4); fp32 logits, row stride ld.
struct EpiLogits {
  static constexpr bool kRowReduce = false;
  static constexpr bool kRowLse = false;
  static constexpr bool kRowSumIn = false;
  static constexpr bool kRowStats = false;
  static constexpr bool kRowDone = false;
  static constexpr bool kTileStats = false;
  LogitsArgs a;
  struct RowAux { float r; };
  struct Aux {};
  __device__ __forceinline__ RowAux row_aux(int row) const { return RowAux{a.r[row]}; }
  __device__ __forceinline__ Aux aux(int, int, const RowAux&) const { return Aux{}; }
  __device__ __forceinline__ float operator()(int row, int col, float v[4], const RowAux& ra, const Aux&) const {
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] *= ra.r;
    store4<float>(a.out + (size_t)row * a.ld + col, v);
    return 0.f;
  }
};

// The LM head's loss with no logits in memory ("The Transformer" page,
// GenerativeAIDocs, §5, step 18: the full fp32 logits are a memory trap).  A
// row's columns of one tile are folded into a running (max, Σ exp(v - max))
// pair, the max subtracted before each exponential; the column that is the
// row's target keeps its logit.  The pairs of a row's tiles are merged by
// launch_lse_merge.
struct EpiLse {
  static constexpr bool kRowReduce = false;
  static constexpr bool kRowLse = true;
  static constexpr bool kRowSumIn = false;
  static constexpr bool kRowStats = false;
  static constexpr bool kRowDone = false;
  static constexpr bool kTileStats = false;
  LseArgs a;
  struct RowAux { float r; int t; };
  struct Aux {};
  __device__ __forceinline__ RowAux row_aux(int row) const { return RowAux{a.r[row], a.targets[row]}; }
  __device__ __forceinline__ Aux aux(int, int, const RowAux&) const { return Aux{}; }
  __device__ __forceinline__ float operator()(int, int, float*, const RowAux&, const Aux&) const { return 0.f; }
  __device__ __forceinline__ void lse(int row, int col, float v[4], const RowAux& ra, float& m, float& s) const {
    float mx = m;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[i] *= ra.r;
      mx = fmaxf(mx, v[i]);
    }
    if (mx > m) {
      s *= expf(m - mx);
      m = mx;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) s += expf(v[i] - m);
    const int dt = ra.t - col;
    if (dt >= 0 && dt < 4) a.tgt[row] = dt == 0 ? v[0] : dt == 1 ? v[1] : dt == 2 ? v[2] : v[3];
  }
  __device__ __forceinline__ void lse_part(int row, int nt, float m, float s) const {
    a.part[(size_t)row * a.n_parts + nt] = make_float2(m, s);
  }
};

}  // namespace tb
