// Causal GQA flash attention of the bf16 prefill on CTA pairs: the four query
// heads of a KV group share every K/V tile, and each tile is loaded once per
// group.
//
// The same computation as the single-CTA kernel (attn_tc.cu): o_i =
// Σ_{j≤i} softmax_j(q_i·k_j/√dh) v_j for every query head h, KV head
// h / (H/Hkv) ("Transformer block" page, tirogla.com, step 2 and the GQA
// paragraph, "each group shares one K/V head"; "Transformers",
// engineering.msaqlain.com, 1.3, 4.1 and 5.1), tile by tile with an online
// softmax ("Transformers" section 6).
//
// A cluster of two CTAs owns one work item: query block qb of the four heads
// 4p..4p+3 of KV group kvh (for H/Hkv a multiple of 4, dh = 128).  Each
// matrix product is one M = 256 tcgen05 MMA issued by the even CTA for both:
//   slot s (0, 1) is heads 4p+2s (rows 0..127, the even CTA) and 4p+2s+1
//   (rows 128..255, the odd CTA);
//   S_s = Q_s·K_jᵀ: Q rows from each CTA's own shared memory, the 128-key K
//   tile split by keys (keys 0..63 staged by the even CTA, 64..127 by the odd);
//   O_s += P_s·V_j: P from each CTA's own tensor memory, the V tile split by
//   value columns (0..63 even, 64..127 odd).
// Each CTA thus stages 16 KB of K and 16 KB of V per 128-key tile for two
// heads (the single-CTA kernel: 32 + 32 KB for two heads), and each SM's
// tensor core reads half of every B operand from its own shared memory.
// Roles per CTA (320 threads):
//   warp 8      TMA: this CTA's Q rows of both slots, then its K and V halves
//               through an NS-stage ring; the copies of both CTAs complete on
//               the even CTA's barriers;
//   warp 9      even CTA: the MMA issuer, in the order P·V slot 0, S slot 0
//               (next tile), P·V slot 1, S slot 1 (next tile); its commits
//               arrive on the barriers of both CTAs.  Odd CTA: idle;
//   warps 0..7  softmax, as in the single-CTA kernel (one thread per query
//               row; warps 4g..4g+3 serve slot g); P_g ready is signalled to
//               the even CTA's MMA issuer by all eight warps of the pair.
#include <math.h>

#include "gemm_tc.cuh"
#include "sm100_ptx.cuh"

namespace tb {
namespace {

using namespace ptx;

constexpr int kBM = 128, kBN = 128, kDH = 128;
constexpr int NS = 4;                                      // K/V ring stages
constexpr float kRescaleLog2 = 8.0f;
constexpr float kRescaleBound = 256.0f;                    // 2^kRescaleLog2
constexpr uint32_t Q_BYTES = kBM * kDH * 2;                // one slot's Q rows in this CTA
constexpr uint32_t KH_BYTES = (kBN / 2) * kDH * 2;         // 64 keys x 128 dims
constexpr uint32_t VH_BYTES = kBN * (kDH / 2) * 2;         // 128 keys x 64 dims
constexpr uint32_t OFF_K = 2 * Q_BYTES;
constexpr uint32_t OFF_V = OFF_K + NS * KH_BYTES;
constexpr uint32_t OFF_BAR = OFF_V + NS * VH_BYTES;
constexpr size_t SMEM = OFF_BAR + 512 + 1024;
constexpr uint32_t TMEM_O = 2 * kBN;                      // S/P of slot g at g·128, O of slot g at 256 + g·128

struct Item {
  int b, kvh, h0, qb, lo, hi;      // h0: first of the four heads; key tiles lo..hi
};

__device__ __forceinline__ Item decode_item(int w, int B, int Hkv, int G, int nq, int window) {
  const int quads = G / 4, per = B * Hkv * quads;
  const int level = w / per, r = w - level * per;
  Item it;
  it.qb = nq - 1 - level;
  it.b = r / (Hkv * quads);
  const int rr = r - it.b * Hkv * quads;
  it.kvh = rr / quads;
  it.h0 = it.kvh * G + 4 * (rr - it.kvh * quads);
  it.hi = it.qb;
  it.lo = window > 0 && it.qb * kBM >= window ? (it.qb * kBM - window + 1) / kBN : 0;
  return it;
}

// The k-th item of this cluster: rounds of one item per cluster, alternating
// direction, over items numbered heaviest first.
__device__ __forceinline__ int item_of(int k, int c, int C) { return k * C + ((k & 1) ? (C - 1 - c) : c); }

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(320, 1)
    k_attn_pair(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, bf16* __restrict__ out, int B, int T, int H, int Hkv,
                int n_qtiles, int n_items, int window, float scale_log2, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* q_full = bars;             // even CTA: Q rows of both CTAs
  uint64_t* q_empty = bars + 1;        // both
  uint64_t* k_full = bars + 2;         // [NS] even CTA
  uint64_t* k_empty = k_full + NS;     // [NS] both
  uint64_t* v_full = k_empty + NS;     // [NS] even CTA
  uint64_t* v_empty = v_full + NS;     // [NS] both
  uint64_t* s_full = v_empty + NS;     // [slot] both
  uint64_t* p_full = s_full + 2;       // [slot] even CTA, 8 warps of the pair
  uint64_t* pv_done = p_full + 2;      // [slot] both
  uint64_t* o_full = pv_done + 2;      // [slot] both
  uint64_t* drain = o_full + 2;        // even CTA
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cl = (int)cluster_id_x(), C = (int)nclusters_x();
  const int G = H / Hkv;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(&s_full[g], 1);
      mbar_init(&p_full[g], 8);
      mbar_init(&pv_done[g], 1);
      mbar_init(&o_full[g], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  // both CTAs' barriers exist before either CTA's copies or commits reach them
  __syncthreads();
  cluster_sync();
  if (warp == 9) {
    tmem_alloc_pair(tmem_slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ---------------- TMA producer (both CTAs) ----------------
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      const uint32_t qf = mapa_shared(smem_u32(q_full), 0);
      int n_issued = 0, nq_issued = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int w = item_of(k, cl, C);
        if (w >= n_items) break;
        const Item it = decode_item(w, B, Hkv, G, n_qtiles, window);
        if (k > 0 && !mbar_wait(q_empty, (k - 1) & 1, abort_flag, err)) break;
        if (rank == 0) mbar_arrive_expect_tx(q_full, 2 * 2 * Q_BYTES);
#pragma unroll
        for (int g = 0; g < 2; ++g)
#pragma unroll
          for (int blk = 0; blk < 2; ++blk)
            tma_load_3d_pair(&tmQ, smem + g * Q_BYTES + blk * kBM * 128, qf, blk * 64, it.qb * kBM,
                             it.b * H + it.h0 + 2 * g + (int)rank);
        ++nq_issued;
        for (int j = it.lo; j <= it.hi; ++j) {
          const int t = n_issued, st = t % NS;
          const uint32_t ph = (uint32_t)(t / NS) & 1u;
          if (!mbar_wait(&k_empty[st], ph ^ 1u, abort_flag, err)) {
            ok = false;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(&k_full[st], 2 * KH_BYTES);
          const uint32_t kf = mapa_shared(smem_u32(&k_full[st]), 0);
#pragma unroll
          for (int blk = 0; blk < 2; ++blk)
            tma_load_3d_pair(&tmK, smem + OFF_K + st * KH_BYTES + blk * (kBN / 2) * 128, kf, blk * 64,
                             j * kBN + (int)rank * (kBN / 2), it.b * Hkv + it.kvh);
          if (!mbar_wait(&v_empty[st], ph ^ 1u, abort_flag, err)) {
            ok = false;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(&v_full[st], 2 * VH_BYTES);
          tma_load_3d_pair(&tmV, smem + OFF_V + st * VH_BYTES, mapa_shared(smem_u32(&v_full[st]), 0),
                           (int)rank * 64, j * kBN, it.b * Hkv + it.kvh);
          ++n_issued;
        }
      }
      // The even CTA's full barriers count the bytes of both CTAs: once the
      // last phases armed there are complete, every copy of the pair has
      // landed (earlier phases were consumed, hence complete).
      if (rank == 0) {
        volatile int no_abort = 0;
        if (nq_issued > 0) mbar_wait(q_full, (nq_issued - 1) & 1, &no_abort, err);
        for (int t = n_issued - NS < 0 ? 0 : n_issued - NS; t < n_issued; ++t) {
          mbar_wait(&k_full[t % NS], (uint32_t)(t / NS) & 1u, &no_abort, err);
          mbar_wait(&v_full[t % NS], (uint32_t)(t / NS) & 1u, &no_abort, err);
        }
      }
    }
  } else if (warp == 9) {
    // ---------------- MMA issuer (even CTA) ----------------
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(2 * kBM, kBN);
      constexpr uint32_t idesc_pv = idesc_bf16(2 * kBM, kDH, false, true);
      const uint32_t sQ = smem_u32(smem);
      // A descriptor's address field is the byte address / 16 and no stage
      // crosses 256 KB, so a stage's descriptor is the first one plus an offset.
      const uint64_t dq0 = desc_kmajor_sw128(sQ), dq1 = desc_kmajor_sw128(sQ + Q_BYTES);
      const uint64_t dk0 = desc_kmajor_sw128(sQ + OFF_K);
      const uint64_t dv0 = desc_mnmajor_sw128(sQ + OFF_V, VH_BYTES, 1024);
      auto issue_s = [&](int g, int t) {
        mma2_tile_ss128(tmem + g * kBN, g ? dq1 : dq0, dk0 + (uint64_t)((t % NS) * (KH_BYTES >> 4)), idesc_qk);
        mma_commit_pair(&s_full[g]);
      };
      auto issue_pv = [&](int g, int t, bool acc) {
        mma2_tile_ts128(tmem + TMEM_O + g * kDH, tmem + g * kBN, dv0 + (uint64_t)((t % NS) * (VH_BYTES >> 4)),
                        idesc_pv, acc ? 1u : 0u);
        mma_commit_pair(&pv_done[g]);
      };
      int kt = 0, c = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int w = item_of(k, cl, C);
        if (w >= n_items) break;
        const Item it = decode_item(w, B, Hkv, G, n_qtiles, window);
        const int nkv = it.hi - it.lo + 1;
        if (!mbar_wait(q_full, k & 1, abort_flag, err) ||
            !mbar_wait(&k_full[kt % NS], (uint32_t)(kt / NS) & 1u, abort_flag, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_s(0, kt);
        issue_s(1, kt);
        mma_commit_pair(&k_empty[kt % NS]);
        if (nkv == 1) mma_commit_pair(q_empty);
        for (int jj = 0; jj < nkv; ++jj) {
          const int t = kt + jj;
          const bool next = jj + 1 < nkv;
          if (!mbar_wait(&v_full[t % NS], (uint32_t)(t / NS) & 1u, abort_flag, err)) {
            ok = false;
            break;
          }
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            if (!mbar_wait(&p_full[g], c & 1, abort_flag, err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_pv(g, t, jj > 0);
            if (!next) mma_commit_pair(&o_full[g]);
            if (next) {
              if (g == 0 &&
                  !mbar_wait(&k_full[(t + 1) % NS], (uint32_t)((t + 1) / NS) & 1u, abort_flag, err)) {
                ok = false;
                break;
              }
              tc_fence_after();
              issue_s(g, t + 1);
            }
          }
          if (!ok) break;
          ++c;
          if (next) {
            mma_commit_pair(&k_empty[(t + 1) % NS]);
            if (jj + 2 == nkv) mma_commit_pair(q_empty);     // the item's last S is issued
          }
          mma_commit_pair(&v_empty[t % NS]);
        }
        if (!ok) break;
        kt += nkv;
      }
      mma_commit_pair(drain);     // arrives on both CTAs' drain; only the even CTA waits
      volatile int no_abort = 0;
      mbar_wait(drain, 0, &no_abort, err);
    }
  } else {
    // ---------------- softmax (warps 0..7 of both CTAs) ----------------
    const int g = warp >> 2, quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    const uint32_t s_col = lane_base + g * kBN, o_col = lane_base + TMEM_O + g * kDH;
    const uint32_t pf = mapa_shared(smem_u32(&p_full[g]), 0);
    int c = 0;                                  // running tile count (both slots see every tile)
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int w = item_of(k, cl, C);
      if (w >= n_items) break;
      const Item it = decode_item(w, B, Hkv, G, n_qtiles, window);
      const int qi = it.qb * kBM + r;
      float m_used = -INFINITY, l = 0.f;
      for (int j = it.lo; j <= it.hi; ++j, ++c) {
        if (!mbar_wait_warp(&s_full[g], c & 1, abort_flag, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float s[kBN];
#pragma unroll
        for (int cc = 0; cc < kBN; cc += 16) {
          uint32_t u[16];
          tmem_ld16(s_col + cc, u);
#pragma unroll
          for (int i = 0; i < 16; ++i) s[cc + i] = __uint_as_float(u[i]);
        }
        tmem_wait_ld();
        // only the diagonal tile masks future keys; with a window, only tiles
        // reaching back past a row's oldest visible key mask older ones.  A
        // row whose first tile holds none of its keys gets m = -inf there and
        // weights 0; its next tile rescales O and l by 2^-inf = 0.
        if (j == it.qb) {
          const int lim = qi - j * kBN;
#pragma unroll
          for (int cc = 0; cc < kBN; ++cc)
            if (cc > lim) s[cc] = -INFINITY;
        }
        if (window > 0 && (it.qb - j + 1) * kBN > window) {
          const int wlim = qi - window + 1 - j * kBN;
#pragma unroll
          for (int cc = 0; cc < kBN; ++cc)
            if (cc < wlim) s[cc] = -INFINITY;
        }
        // P = 2^(s·scale − m) in pairs, written as bf16 over the first 64 S
        // columns; returns Σ P (fp32, before the rounding).
        auto p_pass = [&](float msub) -> float {
          const float2 sc2 = make_float2(scale_log2, scale_log2), nm2 = make_float2(-msub, -msub);
          float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
          for (int cc = 0; cc < kBN; cc += 16) {
            uint32_t u[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float2 arg = __ffma2_rn(make_float2(s[cc + 2 * i], s[cc + 2 * i + 1]), sc2, nm2);
              const float2 p = make_float2(ex2_approx(arg.x), ex2_approx(arg.y));
              sum2[i & 1] = __fadd2_rn(sum2[i & 1], p);
              __nv_bfloat162 t = __floats2bfloat162_rn(p.x, p.y);
              u[i] = *reinterpret_cast<uint32_t*>(&t);
            }
            tmem_st8(s_col + cc / 2, u);
          }
          const float2 s01 = __fadd2_rn(sum2[0], sum2[1]);
          return s01.x + s01.y;
        };
        // The tile's raw row maximum: four chains of three-input maxima.
        auto row_max = [&]() -> float {
          float m4[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float m = fmaxf(s[2 * i], s[2 * i + 1]);
#pragma unroll
            for (int cc = 8 + 2 * i; cc < kBN; cc += 8) m = fmax3(m, s[cc], s[cc + 1]);
            m4[i] = m;
          }
          return fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        };
        // O ← O · 2^(m_used − m_new) on the lanes that need it, once the
        // previous P·V of this slot has finished with O.
        auto rescale_o = [&](bool need, float m_new) -> bool {
          if (!mbar_wait_warp(&pv_done[g], (c - 1) & 1, abort_flag, err)) return false;
          tc_fence_after();
          const float factor = need ? ex2_approx(m_used - m_new) : 1.f;
#pragma unroll 1
          for (int cc = 0; cc < kDH; cc += 8) {
            uint32_t u[8];
            tmem_ld8(o_col + cc, u);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 8; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * factor);
            tmem_st8(o_col + cc, u);
          }
          tmem_wait_st();
          if (need) {
            l *= factor;
            m_used = m_new;
          }
          return true;
        };
        // A row's first tile takes its maximum first.  After that P is formed
        // against the maximum in use, so the maximum is off the path from S
        // to P.  Every weight is at most Σ P, so Σ P ≤ 2^kRescaleLog2 proves
        // that no weight exceeds 2^kRescaleLog2, i.e. that the tile does not
        // raise the row's maximum by more than that, and P stands; otherwise
        // the tile's exact maximum decides, and a row it raises by more makes
        // the warp rescale O and form P again from the scores it holds.
        if (j != it.lo && !__any_sync(0xffffffffu, m_used == -INFINITY)) {
          const float sum = p_pass(m_used);
          float m_new = m_used;
          if (!(sum <= kRescaleBound)) m_new = fmaxf(m_used, row_max() * scale_log2);
          const bool need = m_new > m_used + kRescaleLog2;
          if (__any_sync(0xffffffffu, need)) {
            tmem_wait_st();
            if (!rescale_o(need, m_new)) {
              ok = false;
              break;
            }
            l += p_pass(m_used);
          } else {
            l += sum;
          }
        } else {
          const float m_new = fmaxf(m_used, row_max() * scale_log2);
          bool need = false;
          if (j == it.lo) {
            m_used = m_new;
          } else {
            need = m_new > m_used + kRescaleLog2;
          }
          if (__any_sync(0xffffffffu, need) && !rescale_o(need, m_new)) {
            ok = false;
            break;
          }
          l += p_pass(m_used == -INFINITY ? 0.f : m_used);
        }
        tmem_wait_st();
        tc_fence_before();      // P (and any O rescale) before the next MMA
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(pf);
      }
      if (!ok || !mbar_wait_warp(&o_full[g], k & 1, abort_flag, err)) {
        ok = false;
        break;
      }
      // O of this item; the next item's first P·V into these columns waits for
      // this slot's next P, which these warps write only after this drain
      tc_fence_after();
      const float inv = l > 0.f ? 1.0f / l : 0.f;
      const int h = it.h0 + 2 * g + (int)rank;
      bf16* orow = out + ((size_t)it.b * T + qi) * (size_t)H * kDH + (size_t)h * kDH;
      uint32_t u[kDH];
#pragma unroll
      for (int cc = 0; cc < kDH; cc += 16) tmem_ld16(o_col + cc, *reinterpret_cast<uint32_t(*)[16]>(u + cc));
      tmem_wait_ld();
      if (qi < T) {
#pragma unroll
        for (int cc = 0; cc < kDH; cc += 8) {
          uint4 wv;
          uint32_t* wp = reinterpret_cast<uint32_t*>(&wv);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 t = __floats2bfloat162_rn(__uint_as_float(u[cc + 2 * i]) * inv,
                                                     __uint_as_float(u[cc + 2 * i + 1]) * inv);
            wp[i] = *reinterpret_cast<uint32_t*>(&t);
          }
          *reinterpret_cast<uint4*>(orow + cc) = wv;
        }
      }
      tc_fence_before();
    }
  }

  // Teardown: every MMA of the pair has completed (the even CTA's issuer waited
  // on its drain) before either CTA releases the pair's tensor memory.
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

}  // namespace

// Pair kernel launch: H/Hkv a multiple of 4, dh = 128.  Returns
// cudaErrorNotSupported when the shape does not fit it.
cudaError_t attn_prefill_pair(const void* q, const void* k, const void* v, void* o, int B, int T, int H, int Hkv,
                              int dh, int kv_stride, int window, cudaStream_t s) {
  if (B <= 0 || T <= 0) return cudaSuccess;
  if (dh != kDH || Hkv <= 0 || H % Hkv != 0 || (H / Hkv) % 4 != 0) return cudaErrorNotSupported;
  CUtensorMap tq, tk, tv;
  cudaError_t e = make_tmap_3d_bf16(&tq, q, (uint64_t)B * H, T, kDH, kDH, (uint64_t)T * kDH, 64, kBM);
  if (e != cudaSuccess) return e;
  e = make_tmap_3d_bf16(&tk, k, (uint64_t)B * Hkv, T, kDH, kDH, (uint64_t)kv_stride * kDH, 64, kBN / 2);
  if (e != cudaSuccess) return e;
  e = make_tmap_3d_bf16(&tv, v, (uint64_t)B * Hkv, T, kDH, kDH, (uint64_t)kv_stride * kDH, 64, kBN);
  if (e != cudaSuccess) return e;
  static bool attr_set[64] = {false};
  static int max_clusters[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(k_attn_pair, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * (sm_count() / 2), 1, 1);
    cfg.blockDim = dim3(320, 1, 1);
    cfg.dynamicSmemBytes = SMEM;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, k_attn_pair, &cfg);
    if (e != cudaSuccess) return e;
    if (n <= 0) return cudaErrorNotSupported;
    max_clusters[dev] = n;
    attr_set[dev] = true;
  }
  const int nq = (T + kBM - 1) / kBM;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)kDH);
  const long long items = (long long)nq * B * Hkv * (H / Hkv / 4);
  if (items > 0x7fffffff) return cudaErrorInvalidValue;
  const int n_items = (int)items;
  const int clusters = n_items < max_clusters[dev] ? n_items : max_clusters[dev];
  k_attn_pair<<<2 * clusters, 320, SMEM, s>>>(tq, tk, tv, (bf16*)o, B, T, H, Hkv, nq, n_items, window, scale_log2,
                                              device_error_word());
  return cudaGetLastError();
}

}  // namespace tb
