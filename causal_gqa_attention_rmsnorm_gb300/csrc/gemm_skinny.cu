// bf16 GEMM for few tokens (M ≤ 64, e.g. the decode step's one token per
// sequence) on the 5th-generation tensor cores, split over K, with the split
// reduced inside a thread-block cluster.
//
// With M tokens and N outputs, C = X·Wᵀ is bound by streaming the weight
// matrix W [N, K] from HBM.  The product is computed transposed, Cᵀ = W·Xᵀ, so
// that 128 weight rows form the MMA's M dimension and the (padded) tokens its N
// dimension: no MMA lane is wasted on padding rows.  The `splits` CTAs of one
// 128-row weight tile form a cluster, CTA rank r taking K range r:
//   warp 0      TMA: the weight tile [128, 64] and the token tile [NT, 64]
//               of each K block of the range into a ring of shared-memory
//               stages (the first weight stages before the wait for the
//               previous kernel, which they do not depend on);
//   warp 1      MMA issuer: D[128, NT] += W_blk · X_blkᵀ (tcgen05, fp32 in
//               tensor memory);
//   warps 2..5  epilogue: the accumulator to shared memory as
//               part[token][feature] (the stage ring is free by then); after a
//               cluster barrier, the tokens [r·tpr, (r+1)·tpr) summed over the
//               cluster's partials in rank order through distributed shared
//               memory, then the block's fused epilogue (the functors of the
//               tile GEMM), one warp per token and four features per lane.
// No partial sums go through global memory and no second kernel runs.  With
// RMSNorm-1's statistics (the decode QKV epilogue) each CTA also forms Σx² of
// every token over its own K range while its MMAs run, and the same reduction
// adds those in rank order.
#include "epilogues.cuh"
#include "gemm_tc.cuh"
#include "sm100_ptx.cuh"

namespace tb {
namespace {

using namespace ptx;

constexpr int kRows = 128;       // weight rows per CTA: the MMA's M
constexpr int kBK = 64;          // K per stage (one 128-byte swizzle row)
constexpr int kMaxTok = 64;

// Shared-memory plan: the stage ring, whose first NT × 128 floats hold the
// partial tile after the main loop, then the barriers and Σx² partials.
template <int NT, int CPS = 2> struct SkCfg {
  // CPS CTAs per SM: two with a 4-5 stage ring, or three with a 3-stage one
  static constexpr int STAGES = CPS == 3 ? 3 : (NT <= 32 ? 5 : 4);
  static constexpr uint32_t W_BYTES = kRows * kBK * 2;       // 16 KB
  static constexpr uint32_t X_BYTES = NT * kBK * 2;
  static constexpr uint32_t STAGE_BYTES = W_BYTES + X_BYTES;
  static constexpr uint32_t OFF_BAR = STAGES * STAGE_BYTES;
  static constexpr uint32_t OFF_SSQ = OFF_BAR + 128;         // NT floats: Σx² over this CTA's K range
  static constexpr uint32_t OFF_RA = OFF_SSQ + 256;          // the row inputs of the tokens this CTA reduces
  static constexpr uint32_t RA_BYTES = 2048;
  static constexpr uint32_t OFF_MISC = OFF_RA + RA_BYTES;    // TMEM address, abort flag
  static constexpr size_t SMEM = OFF_MISC + 16 + 1024;
  static constexpr uint32_t TMEM_COLS = NT <= 32 ? 32 : 64;
  static_assert(NT * kRows * 4 <= OFF_BAR, "the partial tile reuses the stage ring");
};

template <int NT, class Epi, int CPS>
__global__ void __launch_bounds__(192, CPS)
    k_gemm_skinny(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, int M, int N,
                  int kblocks, int splits, Epi epi, int* err) {
  using C = SkCfg<NT, CPS>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* drain = tfull + 1;
  float* ssq_s = reinterpret_cast<float*>(smem + C::OFF_SSQ);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* part_s = reinterpret_cast<float*>(smem);             // [NT][kRows] after the main loop
  using RowAux = typename Epi::RowAux;
  static_assert(sizeof(RowAux) * NT <= C::RA_BYTES, "row inputs");
  RowAux* ra_s = reinterpret_cast<RowAux*>(smem + C::OFF_RA);

  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x / splits;
  const int rank = (int)cluster_ctarank();                    // blockIdx.x % splits
  const int kb0 = (int)((long long)kblocks * rank / splits);
  const int nkb = (int)((long long)kblocks * (rank + 1) / splits) - kb0;   // ≥ 1: splits ≤ kblocks
  const int tpr = (M + splits - 1) / splits;                   // tokens each CTA of the cluster reduces
  const int t0 = min(M, rank * tpr), t1 = min(M, t0 + tpr);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
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
      bool dep = false;
      auto release = [&]() {
        pdl_wait();
        dep = true;
        const int held = nkb < STAGES ? nkb : STAGES;
        for (int h = 0; h < held; ++h)
          tma_load_2d(&tmX, smem + h * C::STAGE_BYTES + C::W_BYTES, &full[h], (kb0 + h) * kBK, 0);
      };
      int j = 0;
      for (; j < nkb; ++j) {
        const int st = j % STAGES;
        if (!mbar_wait(&empty[st], ((j / STAGES) & 1) ^ 1u, abort_flag, err)) break;
        uint8_t* sw = smem + st * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&full[st], C::STAGE_BYTES);
        tma_load_2d_hint(&tmW, sw, &full[st], (kb0 + j) * kBK, tile * kRows, pol);
        if (dep) tma_load_2d(&tmX, sw + C::W_BYTES, &full[st], (kb0 + j) * kBK, 0);
        else if (j + 1 == STAGES) release();
      }
      if (!dep) release();
      // every copy issued must land before the CTA may exit (earlier copies
      // into the same stages were consumed, hence complete)
      volatile int no_abort = 0;
      for (int t = j - STAGES < 0 ? 0 : j - STAGES; t < j; ++t)
        mbar_wait(&full[t % STAGES], (t / STAGES) & 1, &no_abort, err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kRows, NT);
      bool ok = true;
      for (int j = 0; j < nkb; ++j) {
        const int st = j % STAGES;
        if (!mbar_wait(&full[st], (j / STAGES) & 1, abort_flag, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t w0 = smem_u32(smem + st * C::STAGE_BYTES), x0 = w0 + C::W_BYTES;
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          mma_bf16_ss(tmem, desc_kmajor_sw128(w0 + k * 32), desc_kmajor_sw128(x0 + k * 32), idesc, (j | k) != 0);
        mma_commit(&empty[st]);
      }
      if (ok) mma_commit(tfull);
      // all MMAs must be done before TMEM is released
      mma_commit(drain);
      volatile int no_abort = 0;
      mbar_wait(drain, 0, &no_abort, err);
    }
  } else {
    pdl_wait();
    const int ew = warp - 2;                 // 0..3
    // While the MMAs run: the row inputs of the tokens this CTA will reduce,
    // one thread per token (positions; the second norm's scale from the Σh²
    // partials; ...), and with RMSNorm-1's statistics Σx² of every token
    // over this CTA's K range.
    for (int t = t0 + (int)threadIdx.x - 64; t < t1; t += 128) {
      bool have = false;
      if constexpr (Epi::kRowStats) {
        if (epi.a.st.x) {
          ra_s[t - t0] = epi.row_aux_pos(t);
          have = true;
        }
      }
      if (!have) ra_s[t - t0] = epi.row_aux(t);
    }
    if constexpr (Epi::kRowStats) {
      if (epi.a.st.x) {
        constexpr int TPW = NT / 4;
        float ss[TPW];
        epi.template row_stats_ranges<TPW>(ew, 4, M, kb0 * kBK, (kb0 + nkb) * kBK, lane, ss);
#pragma unroll
        for (int j = 0; j < TPW; ++j)
          if (lane == 0 && ew + 4 * j < M) ssq_s[ew + 4 * j] = ss[j];
      }
    }
    // lane l of warp w holds output feature 32·(w%4) + l of the tile for all NT tokens
    const int quad = warp & 3;
    if (mbar_wait_warp(tfull, 0, abort_flag, err)) {
      tc_fence_after();
      uint32_t u[NT];
#pragma unroll
      for (int c = 0; c < NT; c += 16)
        tmem_ld16(tmem + ((uint32_t)(quad * 32) << 16) + c, *reinterpret_cast<uint32_t(*)[16]>(u + c));
      tmem_wait_ld();
      const int f = quad * 32 + lane;
#pragma unroll
      for (int t = 0; t < NT; ++t) part_s[t * kRows + f] = __uint_as_float(u[t]);
    }
  }

  // the partials of every CTA of the cluster are in shared memory
  tc_fence_before();
  __syncwarp();
  cluster_sync();

  if (warp >= 2) {
    const int col = tile * kRows + 4 * lane;
    const uint32_t part_base = smem_u32(part_s) + 16u * lane, ssq_base = smem_u32(ssq_s);
    constexpr int kMaxSplits = 8;
    for (int m = t0 + (warp - 2); m < t1; m += 4) {
      // the epilogue's global inputs first (they do not depend on the sums),
      // then this token's four columns from every CTA of the cluster
      RowAux ra = ra_s[m - t0];
      typename Epi::Aux ax{};
      if (col < N) ax = epi.aux(m, col, ra);
      float4 p[kMaxSplits];
      float q[kMaxSplits];
#pragma unroll
      for (int r = 0; r < kMaxSplits; ++r) {
        if (r < splits) {
          p[r] = ld_dsmem_f4(mapa_shared(part_base + (uint32_t)(m * kRows * 4), (uint32_t)r));
          q[r] = 0.f;
          if constexpr (Epi::kRowStats) {
            if (epi.a.st.x) q[r] = ld_dsmem_f32(mapa_shared(ssq_base + (uint32_t)(m * 4), (uint32_t)r));
          }
        }
      }
      // summed in rank order
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      float ss = 0.f;
#pragma unroll
      for (int r = 0; r < kMaxSplits; ++r) {
        if (r < splits) {
          acc.x += p[r].x;
          acc.y += p[r].y;
          acc.z += p[r].z;
          acc.w += p[r].w;
          ss += q[r];
        }
      }
      if constexpr (Epi::kRowStats) {
        // the token's reducer in the cluster of tile 0 publishes its position and flags
        if (epi.a.st.x) epi.row_stats_finish(ra, m, ss, tile == 0 && lane == 0);
      }
      if constexpr (Epi::kRowDone) {
        if (tile == 0 && lane == 0) epi.row_done(m);
      }
      float rsum = 0.f;
      if (col < N) {
        float v[4] = {acc.x, acc.y, acc.z, acc.w};
        rsum = epi(m, col, v, ra, ax);
      }
      if constexpr (Epi::kRowReduce) {
        // this tile's share of the token's row sum is partial `tile`
        const RowSum& rs = epi.row_sums();
        rsum = warp_sum(rsum);
        if (lane == 0) rs.part[(size_t)m * rs.stride + tile] = rsum;
      }
    }
  }

  // no CTA leaves (and frees its shared memory) while another still reads it
  tc_fence_before();
  __syncwarp();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace

// K ranges per weight tile (the cluster size): the largest power of two that
// one wave of the resident CTAs (two per SM) allows, at most 8 (a portable
// cluster), with at least 4 K blocks (64 KB of weights) per CTA.  (Measured on
// the decode QKV GEMM, 48 tiles at 152 SMs: clusters of 4, 6 and 8 took 18.6,
// 25.0 and 22.9 us.)
int skinny_split_count(int tiles, int kblocks, int slots) {
  if (tiles <= 0 || kblocks <= 0 || slots <= 0) return -1;
  int lim = slots / tiles;
  if (lim > kblocks / 4) lim = kblocks / 4;
  int sp = 1;
  while (2 * sp <= lim && 2 * sp <= 8) sp *= 2;
  return sp;
}

namespace {

template <int NT, class Epi, int CPS>
cudaError_t launch_nt(const CUtensorMap& tw, const CUtensorMap& tx, int M, int N, int tiles, int kblocks, int sp,
                      const Epi& epi, cudaStream_t s) {
  using C = SkCfg<NT, CPS>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    const cudaError_t e =
        cudaFuncSetAttribute(k_gemm_skinny<NT, Epi, CPS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  // a cluster of sp CTAs per weight tile, launched as a programmatic
  // dependent of the previous kernel
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles * sp);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = sp;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k_gemm_skinny<NT, Epi, CPS>, tw, tx, M, N, kblocks, sp, epi, device_error_word());
}

template <int NT, class Epi>
cudaError_t run_nt(const void* X, const void* W, int M, int N, int K, const Epi& epi, cudaStream_t s) {
  CUtensorMap tw, tx;
  cudaError_t e = make_tmap_2d_bf16(&tw, W, (uint64_t)N, (uint64_t)K, (uint64_t)K, kBK, kRows);
  if (e != cudaSuccess) return e;
  e = make_tmap_2d_bf16(&tx, X, (uint64_t)M, (uint64_t)K, (uint64_t)K, kBK, NT);
  if (e != cudaSuccess) return e;
  const int tiles = (N + kRows - 1) / kRows, kblocks = K / kBK;
  // Three CTAs per SM (3-stage rings) when that allows a larger split in one
  // wave: more weight bytes in flight over the GPU (decode W1/W3: 224 tiles,
  // one CTA each on two per SM, two each on three per SM).  Measured on the
  // decode step of 32 tokens at d = 4096: 266.6 -> 263.8 us as a graph.
  const int sp2 = skinny_split_count(tiles, kblocks, 2 * sm_count());
  if constexpr (NT <= 32) {
    const int sp3 = skinny_split_count(tiles, kblocks, 3 * sm_count());
    if (sp3 > sp2) return launch_nt<NT, Epi, 3>(tw, tx, M, N, tiles, kblocks, sp3, epi, s);
  }
  return launch_nt<NT, Epi, 2>(tw, tx, M, N, tiles, kblocks, sp2, epi, s);
}

template <class Epi>
cudaError_t run(const void* X, const void* W, int M, int N, int K, const Epi& epi, cudaStream_t s) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  if (M > kMaxTok || K % kBK != 0 || N % 4 != 0) return cudaErrorInvalidValue;
  if (M <= 16) return run_nt<16>(X, W, M, N, K, epi, s);
  if (M <= 32) return run_nt<32>(X, W, M, N, K, epi, s);
  if (M <= 48) return run_nt<48>(X, W, M, N, K, epi, s);
  return run_nt<64>(X, W, M, N, K, epi, s);
}

}  // namespace

int skinny_max_tokens() { return kMaxTok; }

cudaError_t gemm_skinny_qkv(const void* A, const void* B, int M, int N, int K, const Dims& D, const QKVArgs& e,
                            cudaStream_t s) {
  return run(A, B, M, N, K, EpiQKV<bf16>{e, D.H, D.Hkv, D.dh, log2_dh(D.dh)}, s);
}
cudaError_t gemm_skinny_wo(const void* A, const void* B, int M, int N, int K, const Dims& D, const WoArgs& e,
                           cudaStream_t s, int* row_parts) {
  // one Σh² partial per row and 128-column weight tile
  if (row_parts) *row_parts = (N + kRows - 1) / kRows;
  return run(A, B, M, N, K, EpiWo<bf16>{e, D.d}, s);
}
cudaError_t gemm_skinny_w13(const void* A, const void* B, int M, int N, int K, const Dims& D, const W13Args& e,
                            cudaStream_t s) {
  return run(A, B, M, N, K, EpiW13<bf16>{e, D.d, D.f, D.eps}, s);
}
cudaError_t gemm_skinny_w2(const void* A, const void* B, int M, int N, int K, const Dims& D, const W2Args& e,
                           cudaStream_t s) {
  return run(A, B, M, N, K, EpiW2<>{e, D.d}, s);
}

cudaError_t gemm_skinny_logits(const void* A, const void* B, int M, int N, int K, const LogitsArgs& e,
                               cudaStream_t s) {
  return run(A, B, M, N, K, EpiLogits{e}, s);
}

}  // namespace tb
