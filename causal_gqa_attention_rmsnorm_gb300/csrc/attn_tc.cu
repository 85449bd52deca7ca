// Causal GQA flash attention of the bf16 prefill on the 5th-generation tensor
// cores.
//
// o_i = Σ_{j≤i} softmax_j(q_i·k_j/√dh) v_j for every query head h, KV head
// h / (H/Hkv) ("Transformer block" page, tirogla.com, step 2 and the GQA
// paragraph; "Transformers", engineering.msaqlain.com, 1.3 and 5.1), computed
// tile by tile with an online softmax — the exact reformulation "Transformers"
// section 6 describes, which never materialises the T×T matrix.
//
// One CTA per (query head, sequence, 128-query tile), heaviest tiles first:
//   warp 8      TMA: the Q tile once, then K and V tiles of 128 keys through a
//               two-stage ring (3-D tensor maps, so keys past T read as zero);
//   warp 9      MMA issuer: S_j = Q·K_jᵀ into one of two TMEM buffers
//               (M = 128, N = 128, K = dh; both operands in shared memory),
//               then O += P_j·V_j into a TMEM accumulator (M = 128, N = dh,
//               K = 128) with P read from tensor memory and V, the MN-major
//               operand, read in place from its [keys, dh] tile;
//   warps 0..7  softmax: query row i is TMEM lane i; warps w and w+4 share the
//               32 rows of lane quarter w%4, each taking half of the 128 key
//               columns and half of O's columns, and agree on the row maximum
//               through shared memory.  fp32 online softmax in base 2 with
//               the scale and maximum in one FMA; P goes back to tensor
//               memory as bf16 over the S columns it came from.
// P never touches shared memory, which leaves shared-memory bandwidth to the
// operands of Q·Kᵀ and to V.  Key tiles past the query tile are never loaded
// (causal skip); only the diagonal tile is masked element by element.  O is
// rescaled only when a row maximum grows by more than 2^8 over the one in use:
// with a stale maximum every weight stays ≤ 2^8, and O/l is exact either way.
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
  static constexpr uint32_t OFF_K = Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + 2 * KV_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_V + 2 * KV_BYTES;
  static constexpr uint32_t OFF_RED = OFF_BAR + 256;      // [2 buffers][2 halves][128 rows] fp32
  static constexpr size_t SMEM = OFF_RED + 2 * 2 * 128 * 4 + 1024;
  static constexpr uint32_t TMEM_O = 2 * kBN;              // S/P buffers at columns 0 and 128
};

// Named barrier for the 64 threads of one softmax warp pair.
__device__ __forceinline__ void pair_sync(int id) { asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory"); }

template <int DH>
__global__ void __launch_bounds__(320, 1)
    k_attn_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, bf16* __restrict__ out, int T, int H, int Hkv, int n_qtiles,
              float scale_log2, int* err) {
  using C = AttnCfg<DH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = bars + 3;
  uint64_t* v_full = bars + 5;
  uint64_t* v_empty = bars + 7;
  uint64_t* s_full = bars + 9;
  uint64_t* p_full = bars + 11;
  uint64_t* pv_done = bars + 13;
  uint64_t* o_full = bars + 15;
  uint64_t* drain = bars + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 17);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x, b = blockIdx.y;
  const int qb = n_qtiles - 1 - (int)blockIdx.z;     // heaviest query tiles first
  const int q0 = qb * kBM;
  const int kvh = h / (H / Hkv);
  const int nkv = qb + 1;                             // key tiles 0..qb hold every visible key

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 8);
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
      mbar_arrive_expect_tx(q_full, C::Q_BYTES);
#pragma unroll
      for (int blk = 0; blk < C::NB; ++blk)
        tma_load_3d(&tmQ, smem + blk * kBM * 128, q_full, blk * 64, q0, b * H + h);
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
    // tcgen05.mma operations of one thread execute in issue order, so S_{j+1}
    // may be issued into the columns P_{j-1} occupied once P·V_{j-1} is issued.
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(kBM, kBN);
      constexpr uint32_t idesc_pv = idesc_bf16(kBM, DH, false, true);
      const uint32_t sQ = smem_u32(smem);
      const uint32_t sK = sQ + C::OFF_K, sV = sQ + C::OFF_V;
      bool ok = mbar_wait(q_full, 0, abort_flag, err);
      auto issue_s = [&](int j) -> bool {
        const int st = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (!mbar_wait(&k_full[st], ph, abort_flag, err)) return false;
        tc_fence_after();
        const uint32_t kb = sK + st * C::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (kBM * 128) + (kk & 3) * 32;
          mma_bf16_ss(tmem + st * kBN, desc_kmajor_sw128(sQ + off), desc_kmajor_sw128(kb + off), idesc_qk, kk > 0);
        }
        mma_commit(&s_full[st]);
        mma_commit(&k_empty[st]);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; ok && j < nkv; ++j) {
        if (j + 1 < nkv && !issue_s(j + 1)) break;
        const int st = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (!mbar_wait(&p_full[st], ph, abort_flag, err)) break;
        if (!mbar_wait(&v_full[st], ph, abort_flag, err)) break;
        tc_fence_after();
        const uint32_t vb = sV + st * C::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_bf16_ts(tmem + C::TMEM_O, tmem + st * kBN + kk * 8,
                      desc_mnmajor_sw128(vb + kk * 16 * 128, kBN * 128, 1024), idesc_pv, (j | kk) != 0);
        mma_commit(&pv_done[st]);
        mma_commit(&v_empty[st]);
        if (j == nkv - 1) mma_commit(o_full);
      }
      mma_commit(drain);
      volatile int no_abort = 0;
      mbar_wait(drain, 0, &no_abort, err);
    }
  } else {
    // ---------------- softmax (warps 0..7, half a query row per thread) ----------------
    constexpr int HC = kBN / 2;          // key columns per thread
    constexpr int HO = DH / 2;           // O columns per thread
    const int quad = warp & 3, half = warp >> 2;
    const int r = quad * 32 + lane;
    const int qi = q0 + r;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const int st = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      if (!mbar_wait_warp(&s_full[st], ph, abort_flag, err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[HC];
#pragma unroll
      for (int c = 0; c < HC; c += 16) {
        uint32_t u[16];
        tmem_ld16(lane_base + st * kBN + half * HC + c, u);
#pragma unroll
        for (int i = 0; i < 16; ++i) s[c + i] = __uint_as_float(u[i]);
      }
      tmem_wait_ld();
      // raw maximum of this thread's columns; only the diagonal tile masks
      float mx = -INFINITY;
      if (j == nkv - 1) {
        const int lim = qi - (j * kBN + half * HC);     // column c is a future key iff c > lim
#pragma unroll
        for (int c = 0; c < HC; ++c) {
          if (c > lim) s[c] = -INFINITY;
          mx = fmaxf(mx, s[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < HC; ++c) mx = fmaxf(mx, s[c]);
      }
      // agree with the partner thread on the row maximum; the barrier also
      // orders both threads' reads of S before either writes P over it
      red[(st * 2 + half) * 128 + r] = mx;
      tc_fence_before();
      pair_sync(1 + quad);
      tc_fence_after();
      mx = fmaxf(mx, red[(st * 2 + (half ^ 1)) * 128 + r]);
      const float m_new = fmaxf(m_used, mx * scale_log2);
      bool need = false;
      if (j == 0) {
        m_used = m_new;
      } else {
        need = m_new > m_used + kRescaleLog2;
      }
      if (__any_sync(0xffffffffu, need)) {
        // the previous P·V must be finished before O is read and rewritten
        if (!mbar_wait_warp(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float factor = need ? ex2_approx(m_used - m_new) : 1.f;
#pragma unroll 1
        for (int c = 0; c < HO; c += 16) {
          uint32_t u[16];
          tmem_ld16(lane_base + C::TMEM_O + half * HO + c, u);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * factor);
          tmem_st16(lane_base + C::TMEM_O + half * HO + c, u);
        }
        tmem_wait_st();
        if (need) {
          l *= factor;
          m_used = m_new;
        }
      }
      const float msub = m_used == -INFINITY ? 0.f : m_used;
      // p = 2^(s·scale − m), in pairs; bf16 P back into this S buffer's columns
      const float2 sc2 = make_float2(scale_log2, scale_log2), nm2 = make_float2(-msub, -msub);
      float2 sum2 = make_float2(0.f, 0.f);
      uint32_t pk[HC / 2];
#pragma unroll
      for (int c = 0; c < HC; c += 2) {
        const float2 arg = __ffma2_rn(make_float2(s[c], s[c + 1]), sc2, nm2);
        const float2 p = make_float2(ex2_approx(arg.x), ex2_approx(arg.y));
        sum2 = __fadd2_rn(sum2, p);
        __nv_bfloat162 t = __floats2bfloat162_rn(p.x, p.y);
        pk[c / 2] = *reinterpret_cast<uint32_t*>(&t);
      }
      l += sum2.x + sum2.y;
#pragma unroll
      for (int c = 0; c < HC / 2; c += 16) {
        uint32_t u[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) u[i] = pk[c + i];
        tmem_st16(lane_base + st * kBN + half * (HC / 2) + c, u);
      }
      tmem_wait_st();
      tc_fence_before();      // P (and any O rescale) before the next MMA
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[st]);
    }
    const bool have_o = ok && mbar_wait_warp(o_full, 0, abort_flag, err);
    // both halves' sums share the same maximum: add them.  Every softmax
    // thread reaches the pair barrier, whether or not its waits succeeded.
    if (have_o) red[half * 128 + r] = l;
    pair_sync(1 + quad);
    if (have_o) {
      tc_fence_after();
      l += red[(half ^ 1) * 128 + r];
      const float inv = l > 0.f ? 1.0f / l : 0.f;
      bf16* orow = out + ((size_t)b * T + qi) * (size_t)H * DH + (size_t)h * DH + half * HO;
#pragma unroll 1
      for (int c = 0; c < HO; c += 16) {
        uint32_t u[16];
        tmem_ld16(lane_base + C::TMEM_O + half * HO + c, u);
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
  k_attn_tc<DH><<<dim3(H, B, nq), 320, C::SMEM, s>>>(tq, tk, tv, (bf16*)o, T, H, Hkv, nq, scale_log2,
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
