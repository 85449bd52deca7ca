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

// One work item: two query tiles of one sequence that share a KV head.  Slot
// g attends key tiles lo_g..hi_g (hi_g = its query block, -1: slot empty);
// the item streams key tiles j0 .. j0 + nkv - 1, their union.
struct Item {
  int b, h0, h1, qb0, qb1, kvh;
  int lo0, lo1, hi0, hi1;
  int j0, nkv;
};

// Items are numbered heaviest first: all items of the last query block (or
// block pair) come first, then the next one down.  With a sliding window W the
// first key tile of query block qb holds key qb·128 - W + 1, the oldest key
// its first row sees.
__device__ __forceinline__ Item decode_item(int w, int B, int H, int Hkv, int nq, int head_pairs, int window) {
  Item it;
  if (head_pairs) {
    const int P = H / 2, per = B * P;
    const int level = w / per, r = w - level * per;
    it.b = r / P;
    it.h0 = 2 * (r - it.b * P);
    it.h1 = it.h0 + 1;
    it.qb0 = it.qb1 = nq - 1 - level;
  } else {
    const int per = B * H, npair = (nq + 1) / 2;
    const int level = w / per, r = w - level * per;
    it.b = r / H;
    it.h0 = it.h1 = r - it.b * H;
    it.qb0 = 2 * (npair - 1 - level);
    it.qb1 = it.qb0 + 1;
  }
  it.kvh = it.h0 / (H / Hkv);
  auto first_tile = [&](int qb) { return window > 0 && qb * kBM >= window ? (qb * kBM - window + 1) / kBN : 0; };
  it.hi0 = it.qb0;                                 // key tiles past a query block hold no visible key
  it.hi1 = it.qb1 < nq ? it.qb1 : -1;              // -1: slot 1 empty
  it.lo0 = first_tile(it.qb0);
  it.lo1 = first_tile(it.qb1);
  it.j0 = it.lo0;                                  // qb0 <= qb1, so lo0 <= lo1
  it.nkv = (it.hi1 > it.hi0 ? it.hi1 : it.hi0) - it.j0 + 1;
  return it;
}

// The k-th item of CTA c: rounds of gridDim.x items, alternating direction, so
// every CTA gets a near-equal share of the decreasing item sizes.
__device__ __forceinline__ int item_of(int k) {
  const int G = gridDim.x, c = blockIdx.x;
  return k * G + ((k & 1) ? (G - 1 - c) : c);
}

template <int DH>
__global__ void __launch_bounds__(320, 1)
    k_attn_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, bf16* __restrict__ out, int B, int T, int H, int Hkv,
              int n_qtiles, int head_pairs, int n_items, int window, float scale_log2, int* err) {
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
  uint64_t* o_full = bars + 15;    // [slot]
  uint64_t* drain = bars + 17;
  uint64_t* q_empty = bars + 18;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 19);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
      mbar_init(&pv_done[i], 1);
      mbar_init(&o_full[i], 1);
    }
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

  // Barrier phases run on across items: K/V stages by the CTA's running key
  // tile count, s_full / p_full / pv_done by each slot's running tile count,
  // q_full / q_empty by the item count, o_full by the count of items in which
  // the slot has work.
  if (warp == 8) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      int nk_issued = 0, nv_issued = 0, nq_issued = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int w = item_of(k);
        if (w >= n_items) break;
        const Item it = decode_item(w, B, H, Hkv, n_qtiles, head_pairs, window);
        // the previous item's last S must be done with the Q tiles
        if (k > 0 && !mbar_wait(q_empty, (k - 1) & 1, abort_flag, err)) break;
        const int nq_slots = it.hi1 >= 0 ? 2 : 1;
        mbar_arrive_expect_tx(q_full, nq_slots * C::Q_BYTES);
        for (int g = 0; g < nq_slots; ++g)
#pragma unroll
          for (int blk = 0; blk < C::NB; ++blk)
            tma_load_3d(&tmQ, smem + g * C::Q_BYTES + blk * kBM * 128, q_full, blk * 64,
                        (g ? it.qb1 : it.qb0) * kBM, it.b * H + (g ? it.h1 : it.h0));
        ++nq_issued;
        for (int j = 0; j < it.nkv; ++j) {
          const int t = nk_issued, st = t & 1;
          const uint32_t ph = (t >> 1) & 1;
          if (!mbar_wait(&k_empty[st], ph ^ 1u, abort_flag, err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&k_full[st], C::KV_BYTES);
#pragma unroll
          for (int blk = 0; blk < C::NB; ++blk)
            tma_load_3d(&tmK, smem + C::OFF_K + st * C::KV_BYTES + blk * kBN * 128, &k_full[st], blk * 64,
                        (it.j0 + j) * kBN, it.b * Hkv + it.kvh);
          ++nk_issued;
          if (!mbar_wait(&v_empty[st], ph ^ 1u, abort_flag, err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&v_full[st], C::KV_BYTES);
#pragma unroll
          for (int blk = 0; blk < C::NB; ++blk)
            tma_load_3d(&tmV, smem + C::OFF_V + st * C::KV_BYTES + blk * kBN * 128, &v_full[st], blk * 64,
                        (it.j0 + j) * kBN, it.b * Hkv + it.kvh);
          ++nv_issued;
        }
      }
      // every copy issued must land before the CTA may exit (earlier copies
      // into the same buffers were consumed, hence complete)
      volatile int no_abort = 0;
      if (nq_issued > 0) mbar_wait(q_full, (nq_issued - 1) & 1, &no_abort, err);
      for (int t = nk_issued - 2 < 0 ? 0 : nk_issued - 2; t < nk_issued; ++t)
        mbar_wait(&k_full[t & 1], (t >> 1) & 1, &no_abort, err);
      for (int t = nv_issued - 2 < 0 ? 0 : nv_issued - 2; t < nv_issued; ++t)
        mbar_wait(&v_full[t & 1], (t >> 1) & 1, &no_abort, err);
    }
  } else if (warp == 9) {
    // ---------------- MMA issuer ----------------
    // tcgen05.mma operations of one thread execute in issue order, so S of
    // slot g for tile j+1 may be issued into the columns P_g of tile j
    // occupies once that P·V is issued.
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(kBM, kBN);
      constexpr uint32_t idesc_pv = idesc_bf16(kBM, DH, false, true);
      // Every operand descriptor is formed once: the issuing thread shares its
      // sub-partition with two softmax warps, so each MMA must cost it as few
      // instructions as possible.  A descriptor's address field is the byte
      // address / 16, and no block crosses 256 KB, so offsetting a block is a
      // plain add to the descriptor.
      const uint32_t sQ = smem_u32(smem);
      const uint64_t dq0 = desc_kmajor_sw128(sQ), dq1 = desc_kmajor_sw128(sQ + C::Q_BYTES);
      const uint64_t dk0 = desc_kmajor_sw128(sQ + C::OFF_K), dk1 = desc_kmajor_sw128(sQ + C::OFF_K + C::KV_BYTES);
      const uint64_t dv0 = desc_mnmajor_sw128(sQ + C::OFF_V, kBN * 128, 1024);
      const uint64_t dv1 = desc_mnmajor_sw128(sQ + C::OFF_V + C::KV_BYTES, kBN * 128, 1024);
      auto issue_s = [&](int g, int t) {
        const uint64_t qd = g ? dq1 : dq0, kd = (t & 1) ? dk1 : dk0;
        mma_tile_ss<DH / 16>(tmem + g * kBN, qd, kd, idesc_qk);
        mma_commit(&s_full[g]);
      };
      auto issue_pv = [&](int g, int t, bool acc) {
        const uint64_t vd = (t & 1) ? dv1 : dv0;
        mma_tile_ts128(tmem + C::TMEM_O + g * DH, tmem + g * kBN, vd, idesc_pv, acc ? 1u : 0u);
        mma_commit(&pv_done[g]);
      };
      int kt = 0, c0 = 0, c1 = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int w = item_of(k);
        if (w >= n_items) break;
        const Item it = decode_item(w, B, H, Hkv, n_qtiles, head_pairs, window);
        if (!mbar_wait(q_full, k & 1, abort_flag, err) ||
            !mbar_wait(&k_full[kt & 1], (kt >> 1) & 1, abort_flag, err)) {
          ok = false;
          break;
        }
        // slot g works on key tile j iff lo_g <= j <= hi_g
        auto on0 = [&](int j) { return j >= it.lo0 && j <= it.hi0; };
        auto on1 = [&](int j) { return j >= it.lo1 && j <= it.hi1; };
        tc_fence_after();
        if (on0(it.j0)) issue_s(0, kt);
        if (on1(it.j0)) issue_s(1, kt);
        mma_commit(&k_empty[kt & 1]);
        if (it.nkv == 1) mma_commit(q_empty);
        for (int jj = 0; jj < it.nkv; ++jj) {
          const int t = kt + jj, j = it.j0 + jj;
          const bool next = jj + 1 < it.nkv;
          if (!mbar_wait(&v_full[t & 1], (t >> 1) & 1, abort_flag, err)) {
            ok = false;
            break;
          }
          // slot 0: P·V of tile j, then S of tile j+1
          if (on0(j)) {
            if (!mbar_wait(&p_full[0], c0 & 1, abort_flag, err)) {
              ok = false;
              break;
            }
            ++c0;
            tc_fence_after();
            issue_pv(0, t, j > it.lo0);
            if (j == it.hi0) mma_commit(&o_full[0]);
          }
          if (next) {
            if (!mbar_wait(&k_full[(t + 1) & 1], ((t + 1) >> 1) & 1, abort_flag, err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            if (on0(j + 1)) issue_s(0, t + 1);
          }
          // slot 1: P·V of tile j, then S of tile j+1
          if (on1(j)) {
            if (!mbar_wait(&p_full[1], c1 & 1, abort_flag, err)) {
              ok = false;
              break;
            }
            ++c1;
            tc_fence_after();
            issue_pv(1, t, j > it.lo1);
            if (j == it.hi1) mma_commit(&o_full[1]);
          }
          if (next) {
            if (on1(j + 1)) issue_s(1, t + 1);
            mma_commit(&k_empty[(t + 1) & 1]);
            if (jj + 2 == it.nkv) mma_commit(q_empty);     // the item's last S is issued
          }
          mma_commit(&v_empty[t & 1]);
        }
        if (!ok) break;
        kt += it.nkv;
      }
      mma_commit(drain);
      volatile int no_abort = 0;
      mbar_wait(drain, 0, &no_abort, err);
    }
  } else {
    // ---------------- softmax (warps 0..7, one query row per thread) ----------------
    const int g = warp >> 2, quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    const uint32_t s_col = lane_base + g * kBN, o_col = lane_base + C::TMEM_O + g * DH;
    int c = 0;                                  // this slot's running tile count
    int nitem = 0;                              // items in which this slot had work
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int w = item_of(k);
      if (w >= n_items) break;
      const Item it = decode_item(w, B, H, Hkv, n_qtiles, head_pairs, window);
      const int lo = g ? it.lo1 : it.lo0, hi = g ? it.hi1 : it.hi0;
      if (hi < 0) continue;
      const int qb = g ? it.qb1 : it.qb0;
      const int qi = qb * kBM + r;
      float m_used = -INFINITY, l = 0.f;
      for (int j = lo; j <= hi; ++j, ++c) {
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
        // raw row maximum, four chains of three-input maxima; only the
        // diagonal tile masks future keys, and with a window only the tiles
        // that reach back past a row's oldest visible key mask older ones.  A
        // row whose first tile holds none of its keys gets m = -inf there and
        // weights 0; its next tile rescales O and l by 2^-inf = 0.
        if (j == qb) {
          const int lim = qi - j * kBN;          // column cc is a future key iff cc > lim
#pragma unroll
          for (int cc = 0; cc < kBN; ++cc)
            if (cc > lim) s[cc] = -INFINITY;
        }
        if (window > 0 && (qb - j + 1) * kBN > window) {
          const int wlim = qi - window + 1 - j * kBN;   // column cc is too old iff cc < wlim
#pragma unroll
          for (int cc = 0; cc < kBN; ++cc)
            if (cc < wlim) s[cc] = -INFINITY;
        }
        float m4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float m = fmaxf(s[2 * i], s[2 * i + 1]);
#pragma unroll
          for (int cc = 8 + 2 * i; cc < kBN; cc += 8) m = fmax3(m, s[cc], s[cc + 1]);
          m4[i] = m;
        }
        const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        const float m_new = fmaxf(m_used, mx * scale_log2);
        bool need = false;
        if (j == lo) {
          m_used = m_new;
        } else {
          need = m_new > m_used + kRescaleLog2;
        }
        if (__any_sync(0xffffffffu, need)) {
          // the previous P·V of this slot must be finished before O is rewritten
          if (!mbar_wait_warp(&pv_done[g], (c - 1) & 1, abort_flag, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float factor = need ? ex2_approx(m_used - m_new) : 1.f;
#pragma unroll 1
          for (int cc = 0; cc < DH; cc += 8) {
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
        }
        const float msub = m_used == -INFINITY ? 0.f : m_used;
        // p = 2^(s·scale − m), in pairs; bf16 P back over the first 64 S columns
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
        l += s01.x + s01.y;
        tmem_wait_st();
        tc_fence_before();      // P (and any O rescale) before the next MMA
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[g]);
      }
      if (!ok || !mbar_wait_warp(&o_full[g], nitem & 1, abort_flag, err)) {
        ok = false;
        break;
      }
      ++nitem;
      // O of this item; the next item's first P·V into these columns waits for
      // this slot's next P, which these warps write only after this drain
      tc_fence_after();
      const float inv = l > 0.f ? 1.0f / l : 0.f;
      bf16* orow = out + ((size_t)it.b * T + qi) * (size_t)H * DH + (size_t)(g ? it.h1 : it.h0) * DH;
      uint32_t u[DH];
#pragma unroll
      for (int cc = 0; cc < DH; cc += 16) tmem_ld16(o_col + cc, *reinterpret_cast<uint32_t(*)[16]>(u + cc));
      tmem_wait_ld();
      if (qi < T) {
#pragma unroll
        for (int cc = 0; cc < DH; cc += 8) {
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

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int DH>
cudaError_t run(const void* q, const void* k, const void* v, void* o, int B, int T, int H, int Hkv, int kv_stride,
                int window, cudaStream_t s) {
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
  const long long items = head_pairs ? (long long)nq * B * (H / 2) : (long long)((nq + 1) / 2) * B * H;
  if (items > 0x7fffffff) return cudaErrorInvalidValue;
  const int n_items = (int)items;
  const int grid = n_items < sm_count() ? n_items : sm_count();
  k_attn_tc<DH><<<grid, 320, C::SMEM, s>>>(tq, tk, tv, (bf16*)o, B, T, H, Hkv, nq, head_pairs, n_items, window,
                                           scale_log2, device_error_word());
  return cudaGetLastError();
}

}  // namespace

cudaError_t attn_prefill_tc(const void* q, const void* k, const void* v, void* o, int B, int T, int H, int Hkv,
                            int dh, int kv_stride, int window, cudaStream_t s) {
  if (B <= 0 || T <= 0) return cudaSuccess;
  // four query heads per KV group and dh 128: one CTA pair per head quad
  if (dh == 128 && Hkv > 0 && H % Hkv == 0 && (H / Hkv) % 4 == 0)
    return attn_prefill_pair(q, k, v, o, B, T, H, Hkv, dh, kv_stride, window, s);
  if (dh == 128) return run<128>(q, k, v, o, B, T, H, Hkv, kv_stride, window, s);
  if (dh == 64) return run<64>(q, k, v, o, B, T, H, Hkv, kv_stride, window, s);
  return cudaErrorInvalidValue;
}

}  // namespace tb
