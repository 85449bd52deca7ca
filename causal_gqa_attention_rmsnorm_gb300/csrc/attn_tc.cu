// Causal GQA flash attention of the bf16 prefill on the 5th-generation tensor
// cores.
//
// o_i = Σ_{j≤i} softmax_j(q_i·k_j/√dh) v_j for every query head h, KV head
// h / (H/Hkv) ("Transformer block" page, tirogla.com, step 2 and the GQA
// paragraph; "Transformers", engineering.msaqlain.com, 1.3 and 5.1), computed
// tile by tile with an online softmax — the exact reformulation "Transformers"
// section 6 describes, which never materialises the T×T matrix.
//
// A CTA owns two 128-query tiles ("slots") that read the same K/V tiles:
//   * H/Hkv even: query heads 2p and 2p+1 — one KV group — at one query block,
//     so both slots see the same causal extent and every K/V tile staged in
//     shared memory serves two heads of the group;
//   * H/Hkv odd (e.g. MHA): query blocks 2i and 2i+1 of one head; slot 0 sits
//     out the last key tile, and slot 1 is empty when the block count is odd.
// Roles (320 threads):
//   warp 8      TMA: both Q tiles once, then K and V tiles of 128 keys through
//               two-stage rings (3-D tensor maps: keys past T read as zero);
//   warp 9      MMA issuer: S_g = Q_g·K_jᵀ into slot g's TMEM columns
//               (M = 128, N = 128, K = dh; both operands in shared memory) and
//               O_g += P_g·V_j (M = 128, N = dh, K = 128) with P_g read from
//               tensor memory and V, the MN-major operand, read in place;
//   warps 0..7  softmax: warps 4g..4g+3 serve slot g, one thread per query row
//               (TMEM lane = row), fp32 online softmax in base 2 with the scale
//               and maximum in one FMA; P goes back over S as bf16.
// The MMA order per key tile j is P·V of slot 0, S of slot 0 for tile j+1,
// P·V of slot 1, S of slot 1 for tile j+1: while one slot's softmax runs, the
// tensor pipe works on the other slot, so neither waits on a single softmax.
// Key tiles past a query tile are never loaded or multiplied (causal skip);
// only the diagonal tile is masked element by element.  O is rescaled only when
// a row maximum grows by more than 2^8 over the one in use: with a stale
// maximum every weight stays ≤ 2^8, and O/l is exact either way.
#include <math.h>

#include "gemm_tc.cuh"
#include "sm100_ptx.cuh"

namespace tb {
namespace {

using namespace ptx;

constexpr int kBM = 128, kBN = 128;
constexpr float kRescaleLog2 = 8.0f;

template <int DH> struct AttnCfg {
  static constexpr int NB = DH / 64;                       // 64-column swizzle blocks per row
  static constexpr uint32_t Q_BYTES = kBM * DH * 2;
  static constexpr uint32_t KV_BYTES = kBN * DH * 2;
  static constexpr uint32_t OFF_K = 2 * Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + 2 * KV_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_V + 2 * KV_BYTES;
  static constexpr size_t SMEM = OFF_BAR + 256 + 1024;
  static constexpr uint32_t TMEM_O = 2 * kBN;              // S/P of slot g at g·128, O of slot g at 256 + g·DH
};

template <int DH>
__global__ void __launch_bounds__(320, 1)
    k_attn_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, bf16* __restrict__ out, int T, int H, int Hkv, int n_qtiles,
              int head_pairs, float scale_log2, int* err) {
  using C = AttnCfg<DH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;     // [2]
  uint64_t* k_empty = bars + 3;    // [2]
  uint64_t* v_full = bars + 5;     // [2]
  uint64_t* v_empty = bars + 7;    // [2]
  uint64_t* s_full = bars + 9;     // [slot]
  uint64_t* p_full = bars + 11;    // [slot]
  uint64_t* pv_done = bars + 13;   // [slot]
  uint64_t* o_full = bars + 15;
  uint64_t* drain = bars + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 17);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.y;
  const int G = H / Hkv;
  // the two slots: heads h0, h1 at query blocks qb0, qb1; heaviest work first
  int h0, h1, qb0, qb1;
  if (head_pairs) {
    h0 = 2 * blockIdx.x;
    h1 = h0 + 1;
    qb0 = qb1 = n_qtiles - 1 - (int)blockIdx.z;
  } else {
    h0 = h1 = blockIdx.x;
    qb0 = 2 * ((int)gridDim.z - 1 - (int)blockIdx.z);
    qb1 = qb0 + 1;
  }
  const int kvh = h0 / G;
  const int nkv0 = qb0 + 1;                         // key tiles 0..qb hold every visible key
  const int nkv1 = qb1 < n_qtiles ? qb1 + 1 : 0;    // 0: slot 1 empty
  const int nkv = nkv0 > nkv1 ? nkv0 : nkv1;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(o_full, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      const int nq_slots = nkv1 > 0 ? 2 : 1;
      mbar_arrive_expect_tx(q_full, nq_slots * C::Q_BYTES);
      for (int g = 0; g < nq_slots; ++g)
#pragma unroll
        for (int blk = 0; blk < C::NB; ++blk)
          tma_load_3d(&tmQ, smem + g * C::Q_BYTES + blk * kBM * 128, q_full, blk * 64, (g ? qb1 : qb0) * kBM,
                      b * H + (g ? h1 : h0));
      int last = -1;
      for (int j = 0; j < nkv; ++j) {
        const int st = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (!mbar_wait(&k_empty[st], ph ^ 1u, abort_flag, err)) break;
        mbar_arrive_expect_tx(&k_full[st], C::KV_BYTES);
#pragma unroll
        for (int blk = 0; blk < C::NB; ++blk)
          tma_load_3d(&tmK, smem + C::OFF_K + st * C::KV_BYTES + blk * kBN * 128, &k_full[st], blk * 64, j * kBN,
                      b * Hkv + kvh);
        if (!mbar_wait(&v_empty[st], ph ^ 1u, abort_flag, err)) {
          last = j;
          break;
        }
        mbar_arrive_expect_tx(&v_full[st], C::KV_BYTES);
#pragma unroll
        for (int blk = 0; blk < C::NB; ++blk)
          tma_load_3d(&tmV, smem + C::OFF_V + st * C::KV_BYTES + blk * kBN * 128, &v_full[st], blk * 64, j * kBN,
                      b * Hkv + kvh);
        last = j;
      }
      // every copy issued must land before the CTA may exit
      volatile int no_abort = 0;
      mbar_wait(q_full, 0, &no_abort, err);
      for (int j = last - 1 < 0 ? 0 : last - 1; j <= last; ++j) {
        mbar_wait(&k_full[j & 1], (j >> 1) & 1, &no_abort, err);
        mbar_wait(&v_full[j & 1], (j >> 1) & 1, &no_abort, err);
      }
    }
  } else if (warp == 9) {
    // ---------------- MMA issuer ----------------
    // tcgen05.mma operations of one thread execute in issue order, so S of
    // slot g for tile j+1 may be issued into the columns P_g of tile j
    // occupies once that P·V is issued.
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(kBM, kBN);
      constexpr uint32_t idesc_pv = idesc_bf16(kBM, DH, false, true);
      const uint32_t sQ = smem_u32(smem);
      const uint32_t sK = sQ + C::OFF_K, sV = sQ + C::OFF_V;
      auto issue_s = [&](int g, int j) {
        const uint32_t qb = sQ + g * C::Q_BYTES, kb = sK + (j & 1) * C::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (kBM * 128) + (kk & 3) * 32;
          mma_bf16_ss(tmem + g * kBN, desc_kmajor_sw128(qb + off), desc_kmajor_sw128(kb + off), idesc_qk, kk > 0);
        }
        mma_commit(&s_full[g]);
      };
      auto issue_pv = [&](int g, int j) {
        const uint32_t vb = sV + (j & 1) * C::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_bf16_ts(tmem + C::TMEM_O + g * DH, tmem + g * kBN + kk * 8,
                      desc_mnmajor_sw128(vb + kk * 16 * 128, kBN * 128, 1024), idesc_pv, (j | kk) != 0);
        mma_commit(&pv_done[g]);
      };
      bool ok = mbar_wait(q_full, 0, abort_flag, err) && mbar_wait(&k_full[0], 0, abort_flag, err);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        if (nkv1 > 0) issue_s(1, 0);
        mma_commit(&k_empty[0]);
      }
      for (int j = 0; ok && j < nkv; ++j) {
        const int vst = j & 1;
        const uint32_t vph = (j >> 1) & 1;
        const bool next = j + 1 < nkv;
        if (!mbar_wait(&v_full[vst], vph, abort_flag, err)) break;
        // slot 0: P·V of tile j, then S of tile j+1
        if (j < nkv0) {
          if (!mbar_wait(&p_full[0], j & 1, abort_flag, err)) break;
          tc_fence_after();
          issue_pv(0, j);
        }
        if (next) {
          if (!mbar_wait(&k_full[(j + 1) & 1], ((j + 1) >> 1) & 1, abort_flag, err)) break;
          tc_fence_after();
          if (j + 1 < nkv0) issue_s(0, j + 1);
        }
        // slot 1: P·V of tile j, then S of tile j+1
        if (j < nkv1) {
          if (!mbar_wait(&p_full[1], j & 1, abort_flag, err)) break;
          tc_fence_after();
          issue_pv(1, j);
        }
        if (next) {
          if (j + 1 < nkv1) issue_s(1, j + 1);
          mma_commit(&k_empty[(j + 1) & 1]);
        }
        mma_commit(&v_empty[vst]);
        if (j == nkv - 1) mma_commit(o_full);
      }
      mma_commit(drain);
      volatile int no_abort = 0;
      mbar_wait(drain, 0, &no_abort, err);
    }
  } else {
    // ---------------- softmax (warps 0..7, one query row per thread) ----------------
    const int g = warp >> 2, quad = warp & 3;
    const int r = quad * 32 + lane;
    const int nk = g == 0 ? nkv0 : nkv1;
    const int qb = g ? qb1 : qb0;
    const int qi = qb * kBM + r;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    const uint32_t s_col = lane_base + g * kBN, o_col = lane_base + C::TMEM_O + g * DH;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nk; ++j) {
      if (!mbar_wait_warp(&s_full[g], j & 1, abort_flag, err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[kBN];
#pragma unroll
      for (int c = 0; c < kBN; c += 16) {
        uint32_t u[16];
        tmem_ld16(s_col + c, u);
#pragma unroll
        for (int i = 0; i < 16; ++i) s[c + i] = __uint_as_float(u[i]);
      }
      tmem_wait_ld();
      // raw row maximum, four independent chains; only the diagonal tile masks
      if (j == qb) {
        const int lim = qi - j * kBN;          // column c is a future key iff c > lim
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (c > lim) s[c] = -INFINITY;
      }
      float m4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
      for (int c = 4; c < kBN; c += 4)
#pragma unroll
        for (int i = 0; i < 4; ++i) m4[i] = fmaxf(m4[i], s[c + i]);
      const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      const float m_new = fmaxf(m_used, mx * scale_log2);
      bool need = false;
      if (j == 0) {
        m_used = m_new;
      } else {
        need = m_new > m_used + kRescaleLog2;
      }
      if (__any_sync(0xffffffffu, need)) {
        // the previous P·V of this slot must be finished before O is rewritten
        if (!mbar_wait_warp(&pv_done[g], (j - 1) & 1, abort_flag, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float factor = need ? ex2_approx(m_used - m_new) : 1.f;
#pragma unroll 1
        for (int c = 0; c < DH; c += 8) {
          uint32_t u[8];
          tmem_ld8(o_col + c, u);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 8; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * factor);
          tmem_st8(o_col + c, u);
        }
        tmem_wait_st();
        if (need) {
          l *= factor;
          m_used = m_new;
        }
      }
      const float msub = m_used == -INFINITY ? 0.f : m_used;
      // p = 2^(s·scale − m), in pairs; bf16 P back over the first 64 S columns
      const float2 sc2 = make_float2(scale_log2, scale_log2), nm2 = make_float2(-msub, -msub);
      float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int c = 0; c < kBN; c += 16) {
        uint32_t u[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 arg = __ffma2_rn(make_float2(s[c + 2 * i], s[c + 2 * i + 1]), sc2, nm2);
          const float2 p = make_float2(ex2_approx(arg.x), ex2_approx(arg.y));
          sum2[i & 1] = __fadd2_rn(sum2[i & 1], p);
          __nv_bfloat162 t = __floats2bfloat162_rn(p.x, p.y);
          u[i] = *reinterpret_cast<uint32_t*>(&t);
        }
        tmem_st8(s_col + c / 2, u);
      }
      const float2 s01 = __fadd2_rn(sum2[0], sum2[1]);
      l += s01.x + s01.y;
      tmem_wait_st();
      tc_fence_before();      // P (and any O rescale) before the next MMA
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[g]);
    }
    if (nk > 0 && ok && mbar_wait_warp(o_full, 0, abort_flag, err)) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.0f / l : 0.f;
      bf16* orow = out + ((size_t)b * T + qi) * (size_t)H * DH + (size_t)(g ? h1 : h0) * DH;
#pragma unroll 1
      for (int c = 0; c < DH; c += 16) {
        uint32_t u[16];
        tmem_ld16(o_col + c, u);
        tmem_wait_ld();
        if (qi < T) {
          uint4 w[2];
          uint32_t* wp = reinterpret_cast<uint32_t*>(w);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            __nv_bfloat162 t = __floats2bfloat162_rn(__uint_as_float(u[2 * i]) * inv,
                                                     __uint_as_float(u[2 * i + 1]) * inv);
            wp[i] = *reinterpret_cast<uint32_t*>(&t);
          }
          *reinterpret_cast<uint4*>(orow + c) = w[0];
          *reinterpret_cast<uint4*>(orow + c + 8) = w[1];
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int DH>
cudaError_t run(const void* q, const void* k, const void* v, void* o, int B, int T, int H, int Hkv, int kv_stride,
                cudaStream_t s) {
  using C = AttnCfg<DH>;
  CUtensorMap tq, tk, tv;
  cudaError_t e = make_tmap_3d_bf16(&tq, q, (uint64_t)B * H, T, DH, DH, (uint64_t)T * DH, 64, kBM);
  if (e != cudaSuccess) return e;
  e = make_tmap_3d_bf16(&tk, k, (uint64_t)B * Hkv, T, DH, DH, (uint64_t)kv_stride * DH, 64, kBN);
  if (e != cudaSuccess) return e;
  e = make_tmap_3d_bf16(&tv, v, (uint64_t)B * Hkv, T, DH, DH, (uint64_t)kv_stride * DH, 64, kBN);
  if (e != cudaSuccess) return e;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    e = cudaFuncSetAttribute(k_attn_tc<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int nq = (T + kBM - 1) / kBM;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)DH);
  const int head_pairs = ((H / Hkv) % 2 == 0) ? 1 : 0;
  const dim3 grid = head_pairs ? dim3(H / 2, B, nq) : dim3(H, B, (nq + 1) / 2);
  k_attn_tc<DH><<<grid, 320, C::SMEM, s>>>(tq, tk, tv, (bf16*)o, T, H, Hkv, nq, head_pairs, scale_log2,
                                           device_error_word());
  return cudaGetLastError();
}

}  // namespace

cudaError_t attn_prefill_tc(const void* q, const void* k, const void* v, void* o, int B, int T, int H, int Hkv,
                            int dh, int kv_stride, cudaStream_t s) {
  if (B <= 0 || T <= 0) return cudaSuccess;
  if (dh == 128) return run<128>(q, k, v, o, B, T, H, Hkv, kv_stride, s);
  if (dh == 64) return run<64>(q, k, v, o, B, T, H, Hkv, kv_stride, s);
  return cudaErrorInvalidValue;
}

}  // namespace tb
