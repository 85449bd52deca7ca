// bf16 GEMM for few tokens (M ≤ 64, e.g. the decode step's one token per
// sequence) on the 5th-generation tensor cores, split over K.
//
// With M tokens and N outputs, C = X·Wᵀ is bound by streaming the weight
// matrix W [N, K] from HBM.  The product is computed transposed, Cᵀ = W·Xᵀ, so
// that 128 weight rows form the MMA's M dimension and the (padded) tokens its N
// dimension: no MMA lane is wasted on padding rows.  A work item is one
// 128-row weight tile over one contiguous range of K; persistent CTAs, two per
// SM, walk the items with one continuous stage ring, so every SM streams
// weights from the first cycle to the last.
//   warp 0      TMA: the weight tile [128, 64] and the token tile [NT, 64]
//               of each K block into a ring of shared-memory stages;
//   warp 1      MMA issuer: D[128, NT] += W_blk · X_blkᵀ (tcgen05, fp32 in
//               tensor memory);
//   warps 2..5  drain: each warp's 32 TMEM lanes are 32 output features; the
//               fp32 partial sums go to part[split][token][feature] while the
//               next item accumulates into the other TMEM buffer.
// A second kernel adds the K-range partials (from L2) and applies the block's
// fused epilogue, the same functors as the large GEMMs, to 4 outputs per
// thread.
#include "epilogues.cuh"
#include "gemm_tc.cuh"
#include "sm100_ptx.cuh"

namespace tb {
namespace {

using namespace ptx;

constexpr int kRows = 128;       // weight rows per CTA: the MMA's M
constexpr int kBK = 64;          // K per stage (one 128-byte swizzle row)
constexpr int kMaxTok = 64;
constexpr int kMaxItems = 1024;  // (weight tile, K range) items; sizes the partial buffer

template <int NT> struct SkCfg {
  static constexpr int STAGES = NT <= 32 ? 5 : 4;           // two CTAs per SM
  static constexpr uint32_t W_BYTES = kRows * kBK * 2;       // 16 KB
  static constexpr uint32_t X_BYTES = NT * kBK * 2;          // a multiple of 1 KB
  static constexpr uint32_t STAGE_BYTES = W_BYTES + X_BYTES;
  static constexpr uint32_t OFF_BAR = STAGES * STAGE_BYTES;
  static constexpr size_t SMEM = OFF_BAR + 256 + 1024;
  static constexpr uint32_t ACC_COLS = 64;                   // two accumulators of NT ≤ 64 columns
  static constexpr uint32_t TMEM_COLS = 2 * ACC_COLS;
};

// Persistent: CTA c takes work items c, c + gridDim.x, ...; item w is weight
// tile w % tiles over K range w / tiles.  The stage ring runs on across items
// and the accumulators alternate, so one item's drain overlaps the next
// item's loads and MMAs.
template <int NT>
__global__ void __launch_bounds__(192)
    k_gemm_skinny(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, int M, int N,
                  int tiles, int kblocks, int splits, float* __restrict__ part, int* err) {
  using C = SkCfg<NT>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;     // [2]
  uint64_t* tempty = tfull + 2;         // [2]
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int items = tiles * splits;
  auto krange = [&](int sp, int& kb0, int& nkb) {
    kb0 = (int)((long long)kblocks * sp / splits);
    nkb = (int)((long long)kblocks * (sp + 1) / splits) - kb0;   // ≥ 1: splits ≤ kblocks
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmX);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // The weights do not depend on earlier kernels: the first STAGES weight
      // tiles are requested before the wait for the previous kernel, so they
      // stream while it drains; their token tiles follow the wait.
      const uint64_t pol = policy_evict_first();   // weights are read once per call
      int held_kb[STAGES];
      int held = 0;
      bool dep = false;
      auto release = [&]() {
        pdl_wait();
        dep = true;
        for (int h = 0; h < held; ++h)       // stage h holds the h-th K block issued
          tma_load_2d(&tmX, smem + h * C::STAGE_BYTES + C::W_BYTES, &full[h], held_kb[h] * kBK, 0);
      };
      int i = 0;                                  // running K-block count: stage i % STAGES
      bool ok = true;
      for (int w = blockIdx.x; ok && w < items; w += gridDim.x) {
        const int tile = w % tiles;
        int kb0, nkb;
        krange(w / tiles, kb0, nkb);
        for (int j = 0; j < nkb; ++j, ++i) {
          const int st = i % STAGES;
          if (!mbar_wait(&empty[st], ((i / STAGES) & 1) ^ 1u, abort_flag, err)) {
            ok = false;
            break;
          }
          uint8_t* sw = smem + st * C::STAGE_BYTES;
          mbar_arrive_expect_tx(&full[st], C::STAGE_BYTES);
          tma_load_2d_hint(&tmW, sw, &full[st], (kb0 + j) * kBK, tile * kRows, pol);
          if (dep) {
            tma_load_2d(&tmX, sw + C::W_BYTES, &full[st], (kb0 + j) * kBK, 0);
          } else {
            held_kb[held++] = kb0 + j;
            if (held == STAGES) release();
          }
        }
      }
      if (!dep) release();
      // every copy issued must land before the CTA may exit (earlier copies
      // into the same stages were consumed, hence complete)
      volatile int no_abort = 0;
      for (int t = i - STAGES < 0 ? 0 : i - STAGES; t < i; ++t)
        mbar_wait(&full[t % STAGES], (t / STAGES) & 1, &no_abort, err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kRows, NT);
      int i = 0, local = 0;
      bool ok = true;
      for (int w = blockIdx.x; ok && w < items; w += gridDim.x, ++local) {
        int kb0, nkb;
        krange(w / tiles, kb0, nkb);
        const int acc = local & 1;
        if (!mbar_wait(&tempty[acc], ((local >> 1) & 1) ^ 1u, abort_flag, err)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * C::ACC_COLS;
        for (int j = 0; j < nkb; ++j, ++i) {
          const int st = i % STAGES;
          if (!mbar_wait(&full[st], (i / STAGES) & 1, abort_flag, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t w0 = smem_u32(smem + st * C::STAGE_BYTES), x0 = w0 + C::W_BYTES;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            mma_bf16_ss(d, desc_kmajor_sw128(w0 + k * 32), desc_kmajor_sw128(x0 + k * 32), idesc, (j | k) != 0);
          mma_commit(&empty[st]);
        }
        if (ok) mma_commit(&tfull[acc]);
      }
      mma_commit(drain);
      volatile int no_abort = 0;
      mbar_wait(drain, 0, &no_abort, err);
    }
  } else {
    // lane l of warp w holds output feature 32·(w%4) + l of the tile for all
    // NT tokens; the accumulator is released as soon as it is in registers
    const int quad = warp & 3;
    int local = 0;
    for (int w = blockIdx.x; w < items; w += gridDim.x, ++local) {
      const int acc = local & 1;
      if (!mbar_wait_warp(&tfull[acc], (local >> 1) & 1, abort_flag, err)) break;
      tc_fence_after();
      uint32_t u[NT];
#pragma unroll
      for (int c = 0; c < NT; c += 16)
        tmem_ld16(tmem + ((uint32_t)(quad * 32) << 16) + acc * C::ACC_COLS + c,
                  *reinterpret_cast<uint32_t(*)[16]>(u + c));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      const int n = (w % tiles) * kRows + quad * 32 + lane;
      if (n < N) {
        float* dst = part + (size_t)(w / tiles) * M * N + n;
#pragma unroll
        for (int m = 0; m < NT; ++m)
          if (m < M) dst[(size_t)m * N] = __uint_as_float(u[m]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// Sum of the K-range partials of 4 consecutive outputs of one token, then the
// fused epilogue.  Rows (tokens) are blockIdx.y, so a row reduction (Σh² of
// the Wo epilogue) is one partial per warp.  With RMSNorm-1 statistics in the
// QKV epilogue (kRowStats, a.st.x set) every CTA of row m first forms the
// row's Σx² itself (the row is a few KB, read from L2 by each of the row's
// CTAs) in a fixed order: per thread, per warp, then warps in order.
constexpr int kEpiWarps = 8;                 // warps per CTA of the partial-sum epilogue (256 threads)

template <class Epi>
__global__ void __launch_bounds__(256)
    k_splitk_epilogue(const float* __restrict__ part, int splits, int M, int N, Epi epi) {
  pdl_trigger();
  pdl_wait();
  const int m = blockIdx.y;
  const int col = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
  float r = 0.f;
  typename Epi::RowAux ra_stats{};
  bool have_stats = false;
  if constexpr (Epi::kRowStats) {
    if (epi.a.st.x) {
      __shared__ float s_part[kEpiWarps];
      __shared__ typename Epi::RowAux s_ra;
      const float ss = warp_sum(epi.row_stats_partial(m, threadIdx.x, blockDim.x));
      if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = ss;
      __syncthreads();
      if (threadIdx.x == 0) {
        float t = 0.f;
        for (int w = 0; w < kEpiWarps; ++w) t += s_part[w];
        s_ra = epi.row_aux_stats(m, t, blockIdx.x == 0);
      }
      __syncthreads();
      ra_stats = s_ra;
      have_stats = true;
    }
  }
  if constexpr (Epi::kRowDone) {
    if (blockIdx.x == 0 && threadIdx.x == 0) epi.row_done(m);
  }
  if (col < N) {
    // the first eight partials are requested before the epilogue's own inputs
    // (which may depend on one another), so all of them are in flight together
    constexpr int U = 8;
    float4 a[U];
    const float* p = part + (size_t)m * N + col;
    const size_t stride = (size_t)M * N;
#pragma unroll
    for (int u = 0; u < U; ++u)
      a[u] = u < splits ? *reinterpret_cast<const float4*>(p + (size_t)u * stride) : make_float4(0.f, 0.f, 0.f, 0.f);
    const auto ra = have_stats ? ra_stats : epi.row_aux(m);
    const auto ax = epi.aux(m, col, ra);
    int sp = U;
    for (; sp + U <= splits; sp += U) {
      float4 t[U];
#pragma unroll
      for (int u = 0; u < U; ++u) t[u] = *reinterpret_cast<const float4*>(p + (size_t)(sp + u) * stride);
#pragma unroll
      for (int u = 0; u < U; ++u) a[u] = make_float4(a[u].x + t[u].x, a[u].y + t[u].y, a[u].z + t[u].z, a[u].w + t[u].w);
    }
    for (int u = 0; sp < splits; ++sp, ++u) {
      const float4 t = *reinterpret_cast<const float4*>(p + (size_t)sp * stride);
      a[u] = make_float4(a[u].x + t.x, a[u].y + t.y, a[u].z + t.z, a[u].w + t.w);
    }
    float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int u = 0; u < U; ++u) {
      v[0] += a[u].x;
      v[1] += a[u].y;
      v[2] += a[u].z;
      v[3] += a[u].w;
    }
    r = epi(m, col, v, ra, ax);
  }
  if constexpr (Epi::kRowReduce) {
    // each warp's share of row m is one partial
    const RowSum& rs = epi.row_sums();
    r = warp_sum(r);
    if ((threadIdx.x & 31) == 0) rs.part[(size_t)m * rs.stride + blockIdx.x * kEpiWarps + (threadIdx.x >> 5)] = r;
  }
}

int split_count(int tiles, int kblocks) { return skinny_split_count(tiles, kblocks, 2 * sm_count()); }

template <int NT, class Epi>
cudaError_t run_nt(const void* X, const void* W, int M, int N, int K, const Epi& epi, float* part, cudaStream_t s) {
  using C = SkCfg<NT>;
  CUtensorMap tw, tx;
  cudaError_t e = make_tmap_2d_bf16(&tw, W, (uint64_t)N, (uint64_t)K, (uint64_t)K, kBK, kRows);
  if (e != cudaSuccess) return e;
  e = make_tmap_2d_bf16(&tx, X, (uint64_t)M, (uint64_t)K, (uint64_t)K, kBK, NT);
  if (e != cudaSuccess) return e;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    e = cudaFuncSetAttribute(k_gemm_skinny<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int tiles = (N + kRows - 1) / kRows, kblocks = K / kBK;
  const int splits = split_count(tiles, kblocks);
  const int items = tiles * splits, slots = 2 * sm_count();
  e = launch_pdl(k_gemm_skinny<NT>, dim3(items < slots ? items : slots), dim3(192), C::SMEM, s, tw, tx, M, N, tiles,
                 kblocks, splits, part, device_error_word());
  if (e != cudaSuccess) return e;
  return launch_pdl(k_splitk_epilogue<Epi>, dim3((N / 4 + 255) / 256, M), dim3(32 * kEpiWarps), 0, s,
                    (const float*)part, splits, M, N, epi);
}

template <class Epi>
cudaError_t run(const void* X, const void* W, int M, int N, int K, const Epi& epi, float* part, cudaStream_t s) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  if (M > kMaxTok || K % kBK != 0 || N % 4 != 0 || !part) return cudaErrorInvalidValue;
  if (M <= 16) return run_nt<16>(X, W, M, N, K, epi, part, s);
  if (M <= 32) return run_nt<32>(X, W, M, N, K, epi, part, s);
  if (M <= 48) return run_nt<48>(X, W, M, N, K, epi, part, s);
  return run_nt<64>(X, W, M, N, K, epi, part, s);
}

}  // namespace

// K ranges per weight tile.  Items are equal in size, so the time is the
// number of item waves over the resident CTAs (two per SM): take the split
// count whose item count fills its last wave best (fewest splits on a tie),
// with at least 4 K blocks (64 KB of weights) per item and at most kMaxItems
// items.  The partials (items × 128 × M floats) stay in L2 between the two
// kernels.
int skinny_split_count(int tiles, int kblocks, int slots) {
  if (tiles <= 0 || kblocks <= 0 || slots <= 0) return -1;
  int spmax = kblocks / 4;
  if (spmax > kMaxItems / tiles) spmax = kMaxItems / tiles;
  int best = 1;
  double best_fill = 0.0;
  for (int sp = 1; sp <= spmax; ++sp) {
    const long long items = (long long)tiles * sp, waves = (items + slots - 1) / slots;
    const double fill = (double)items / (double)(waves * slots);
    if (fill > best_fill + 1e-3) best = sp, best_fill = fill;
  }
  return best;
}

int skinny_max_tokens() { return kMaxTok; }

size_t skinny_part_floats(int M, int max_n) {
  const size_t tiles = (size_t)(max_n + kRows - 1) / kRows;
  return (size_t)M * kRows * (tiles > (size_t)kMaxItems ? tiles : (size_t)kMaxItems);
}

cudaError_t gemm_skinny_qkv(const void* A, const void* B, int M, int N, int K, const Dims& D, const QKVArgs& e,
                            float* part, cudaStream_t s) {
  return run(A, B, M, N, K, EpiQKV<bf16>{e, D.H, D.Hkv, D.dh, log2_dh(D.dh)}, part, s);
}
cudaError_t gemm_skinny_wo(const void* A, const void* B, int M, int N, int K, const Dims& D, const WoArgs& e,
                           float* part, cudaStream_t s, int* row_parts) {
  // one Σh² partial per row and epilogue warp (128 columns)
  if (row_parts) *row_parts = (N / 4 + 255) / 256 * kEpiWarps;
  return run(A, B, M, N, K, EpiWo<bf16>{e, D.d}, part, s);
}
cudaError_t gemm_skinny_w13(const void* A, const void* B, int M, int N, int K, const Dims& D, const W13Args& e,
                            float* part, cudaStream_t s) {
  return run(A, B, M, N, K, EpiW13<bf16>{e, D.d, D.f, D.eps}, part, s);
}
cudaError_t gemm_skinny_w2(const void* A, const void* B, int M, int N, int K, const Dims& D, const W2Args& e,
                           float* part, cudaStream_t s) {
  return run(A, B, M, N, K, EpiW2<>{e, D.d}, part, s);
}

cudaError_t gemm_skinny_logits(const void* A, const void* B, int M, int N, int K, const LogitsArgs& e, float* part,
                               cudaStream_t s) {
  return run(A, B, M, N, K, EpiLogits{e}, part, s);
}

}  // namespace tb
