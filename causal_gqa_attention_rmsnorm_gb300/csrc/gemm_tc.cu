// bf16 GEMM on the 5th-generation tensor cores: C = A·Bᵀ, A [M, K] (tokens ×
// reduction), B [N, K] (packed weights, reduction axis contiguous), fp32
// accumulation in tensor memory, and the block's fused epilogues.
//
// Persistent, warp-specialised, one CTA per SM:
//   warp 0      TMA producer: A and B tiles (128-byte swizzle) into a ring of
//               shared-memory stages, completion tracked by mbarriers;
//   warp 1      MMA issuer: one thread issues tcgen05.mma (M = 128, N = BN,
//               K = 16) into one of two TMEM accumulators, and commits each
//               stage back to the producer when the tensor core is done with it;
//   warps 2..5  epilogue: tcgen05.ld of the finished accumulator (each warp
//               owns its 32-lane quarter of TMEM, i.e. 32 rows), released as
//               soon as its last columns are in registers, so the next tile's
//               MMAs overlap this tile's fused epilogue and global stores (the
//               prefill instances stream their once-through loads and stores,
//               see epilogues.cuh).
// Tiles are visited n-fastest so that the CTAs running together share the A
// row block and the weight panel stays resident in L2, or, when the weight
// panel is larger than L2 and K short, in groups of row blocks (see run).
// The Wo, W1/W3 and W2 GEMMs of a prefill with enough 256-row tiles run on
// CTA pairs (PAIR, see TcCfg): M = 256 MMAs issued by the even CTA of a
// cluster, each CTA staging its own A block and half of the weight tile.
#include <cudaTypedefs.h>

#include <mutex>

#include "epilogues.cuh"
#include "gemm_tc.cuh"
#include "sm100_ptx.cuh"

namespace tb {
namespace {

using namespace ptx;

constexpr int BM = 128, BK = 64;

// Shared-memory plan of a CTA tile of 128 rows × BN columns.
//
// PAIR: a cluster of two CTAs computes a 256 × BN tile with M = 256 MMAs
// (tcgen05 cta_group::2) that the even CTA issues: each CTA stages its own
// 128-row A block and half of the weight tile (BN/2 rows), the tensor cores
// read B from both CTAs' shared memory, and each CTA's tensor memory holds
// its 128 rows of the accumulator.  Per CTA a k-block stages 32 KB instead
// of 48 KB for the same MMA work, and each weight tile is fetched once per
// pair of row blocks.
template <int BN, bool PAIR = false> struct TcCfg {
  static constexpr int STAGES = PAIR ? 6 : (BN == 256 ? 4 : 6);
  static constexpr uint32_t A_BYTES = BM * BK * 2;
  static constexpr uint32_t B_BYTES = (PAIR ? BN / 2 : BN) * BK * 2;     // this CTA's share of the weight tile
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t TMEM_COLS = 2 * BN;
  static constexpr uint32_t OFF_BAR = STAGES * STAGE_BYTES;
  static constexpr uint32_t OFF_EPI = OFF_BAR + 256;                // 4 warps x [32 rows][36] fp32
  static constexpr uint32_t EPI_STRIDE = 36;                        // 32 columns + 4 pad: conflict-free both ways
  static constexpr size_t SMEM = OFF_EPI + 4 * 32 * EPI_STRIDE * 4 + 1024;
};

// fp32 output of the raw product (test hook).
#pragma nv_diag_suppress 177
struct EpiF32 {
  static constexpr bool kRowReduce = false;
  static constexpr bool kRowLse = false;
  static constexpr bool kRowSumIn = false;
  static constexpr bool kRowStats = false;
  static constexpr bool kRowDone = false;
  static constexpr bool kTileStats = false;
  float* C;
  int N;
  struct RowAux {};
  struct Aux {};
  __device__ __forceinline__ RowAux row_aux(int) const { return RowAux{}; }
  __device__ __forceinline__ Aux aux(int, int, const RowAux&) const { return Aux{}; }
  __device__ __forceinline__ float operator()(int row, int col, float v[4], const RowAux&, const Aux&) const {
    *reinterpret_cast<float4*>(C + (size_t)row * N + col) = make_float4(v[0], v[1], v[2], v[3]);
    return 0.f;
  }
};

// Tile index -> (m, n) tile.  group_m == 0 walks n fastest (CTAs running
// together share one A row block and stream the whole B panel, best when B
// is reused from L2 or K is long).  Otherwise tiles go in groups of group_m
// row blocks, m fastest inside a group, so the CTAs running together touch
// group_m A blocks and a few B blocks: both stay in L2 even when the B panel
// is larger than L2.
__device__ __forceinline__ void tile_coords(int tile, int m_tiles, int n_tiles, int group_m, int& mt, int& nt) {
  if (group_m <= 0) {
    mt = tile / n_tiles;
    nt = tile - mt * n_tiles;
    return;
  }
  const int per_group = group_m * n_tiles;
  const int g = tile / per_group;
  const int first_m = g * group_m;
  const int gm = min(group_m, m_tiles - first_m);
  const int local = tile - g * per_group;
  mt = first_m + local % gm;
  nt = local / gm;
}

// Threads per CTA: producer, MMA issuer, four epilogue warps, and for an
// epilogue that can take RMSNorm-1 statistics (kTileStats) a statistics warp.
template <class Epi> constexpr int tc_threads() { return Epi::kTileStats ? 224 : 192; }

template <int BN, class Epi, bool PAIR = false>
__global__ void __launch_bounds__(224, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, int M, int N, int K,
              uint32_t a_box_bytes, int group_m, Epi epi, int* err) {
  using C = TcCfg<BN, PAIR>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tiles = (M + BM - 1) / BM, n_tiles = (N + BN - 1) / BN;
  constexpr int MU = PAIR ? 2 : 1;                  // row blocks per (pair or CTA) tile
  const int m_units = (m_tiles + MU - 1) / MU;     // tiles along M
  const int tiles = m_units * n_tiles;
  const int kblocks = K / BK;
  // PAIR: the cluster walks the tiles; rank 0 issues the MMAs
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int tile0 = PAIR ? (int)cluster_id_x() : (int)blockIdx.x;
  const int tstep = PAIR ? (int)nclusters_x() : (int)gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], PAIR ? 8 : 4);     // PAIR: the epilogue warps of both CTAs, on rank 0's
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if constexpr (PAIR) {
    // both CTAs' barriers exist before either CTA's copies or commits reach them
    __syncthreads();
    cluster_sync();
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, C::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued[STAGES];
      uint32_t last_phase[STAGES];
      for (int s = 0; s < STAGES; ++s) issued[s] = 0, last_phase[s] = 0;
      bool ok = true;
      for (int tile = tile0; ok && tile < tiles; tile += tstep) {
        int mu, nt;
        tile_coords(tile, m_units, n_tiles, group_m, mu, nt);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, err)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * C::STAGE_BYTES;
          if constexpr (PAIR) {
            // both CTAs' copies complete on rank 0's barrier, which counts them all
            const uint32_t fb = mapa_shared(smem_u32(&full[stage]), 0);
            if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * (a_box_bytes + C::B_BYTES));
            tma_load_2d_pair(&tmA, sa, fb, kb * BK, (mu * 2 + (int)rank) * BM);     // a block past M reads zeros
            tma_load_2d_pair(&tmB, sa + C::A_BYTES, fb, kb * BK, nt * BN + (int)rank * (BN / 2));
          } else {
            // the A box is shorter than the tile when M < 128; rows past it are never stored
            mbar_arrive_expect_tx(&full[stage], a_box_bytes + C::B_BYTES);
            tma_load_2d(&tmA, sa, &full[stage], kb * BK, mu * BM);
            tma_load_2d(&tmB, sa + C::A_BYTES, &full[stage], kb * BK, nt * BN);
          }
          issued[stage] = 1;
          last_phase[stage] = phase;
          if (++stage == STAGES) stage = 0, phase ^= 1u;
        }
      }
      // every copy issued must have landed before the CTA may exit (PAIR:
      // rank 0's barriers count both CTAs' copies, and the peer waits for
      // rank 0 at the cluster barrier before it exits)
      for (int s = 0; s < STAGES; ++s)
        if (issued[s] && rank == 0) {
          volatile int no_abort = 0;
          mbar_wait(&full[s], last_phase[s], &no_abort, err);
        }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_bf16(PAIR ? 2 * BM : BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      for (int tile = tile0; ok && tile < tiles; tile += tstep, ++local) {
        // two accumulators in turn
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, err)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t b0 = a0 + C::A_BYTES;
          if constexpr (PAIR) {
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              mma2_bf16_ss(d_tmem, desc_kmajor_sw128(a0 + k * 32), desc_kmajor_sw128(b0 + k * 32), idesc,
                           (kb | k) != 0);
            mma_commit_pair(&empty[stage]);     // frees the stage in both CTAs
          } else {
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              mma_bf16_ss(d_tmem, desc_kmajor_sw128(a0 + k * 32), desc_kmajor_sw128(b0 + k * 32), idesc,
                          (kb | k) != 0);
            mma_commit(&empty[stage]);
          }
          if (++stage == STAGES) stage = 0, phase ^= 1u;
        }
        if (ok) {
          if constexpr (PAIR) mma_commit_pair(&tfull[acc]);
          else mma_commit(&tfull[acc]);
        }
      }
      // all MMAs must be done before TMEM is released
      if constexpr (PAIR) mma_commit_pair(drain);     // arrives on both CTAs' drain; rank 0 waits
      else mma_commit(drain);
      volatile int no_abort = 0;
      mbar_wait(drain, 0, &no_abort, err);
    }
  } else if (warp == 6) {
    // Statistics warp (kTileStats with a.ts.x set): r = 1/sqrt(mean(x²) + eps)
    // for rows g·kStatRows + blockIdx.x + k·gridDim.x of every group g in
    // order, each group counted in done[g] once this CTA's rows are written.
    if constexpr (Epi::kTileStats) {
      const TileStats& ts = epi.a.ts;
      if (ts.x) {
        const int ngroups = (M + kStatRows - 1) / kStatRows;
        for (int g = 0; g < ngroups; ++g) {
          const int end = min(M, (g + 1) * kStatRows);
          for (int row = g * kStatRows + (int)blockIdx.x; row < end; row += (int)gridDim.x) {
            const float r = epi.tile_row_scale(row, lane);
            if (lane == 0) {
              ts.r[row] = r;
              if (ts.lens_set && row % ts.T == 0) ts.lens_set[row / ts.T] = ts.T;
            }
          }
          __syncwarp();
          if (lane == 0) {
            __threadfence();
            atomicAdd(ts.done + g, 1);
          }
        }
      }
    }
  } else {
    // Epilogue: each warp reads its 32 TMEM lanes (32 rows) 32 columns at a
    // time, turns the chunk around in shared memory, and then lets lane l
    // handle columns [4·(l%8), +4) of rows (l/8) + 4·i, so every global access
    // of a warp instruction covers four contiguous row segments.
    const int quad = warp & 3;
    int stats_ready = -1;          // groups ≤ this one have their row scales (kTileStats)
    float* stage = reinterpret_cast<float*>(smem + C::OFF_EPI) + (warp - 2) * 32 * C::EPI_STRIDE;
    const int sub_row = lane >> 3, sub_col = 4 * (lane & 7);
    int local = 0;
    // PAIR: this CTA's epilogue frees an accumulator on rank 0's barrier
    const uint32_t tempty_cl[2] = {PAIR ? mapa_shared(smem_u32(&tempty[0]), 0) : 0u,
                                   PAIR ? mapa_shared(smem_u32(&tempty[1]), 0) : 0u};
    for (int tile = tile0; tile < tiles; tile += tstep, ++local) {
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      if (!mbar_wait_warp(&tfull[acc], acc_phase, abort_flag, err)) break;
      tc_fence_after();
      int mu, nt;
      tile_coords(tile, m_units, n_tiles, group_m, mu, nt);
      // kTileStats: the row scales of this tile's group come from every CTA's
      // statistics warp.  A group is complete once all CTAs counted it, and each
      // statistics warp takes the groups in order, so a complete group means that
      // all earlier ones are.  If the group is still incomplete after a bounded
      // poll (a CTA of the grid not resident yet), the warp forms r for its own
      // rows with the same function, hence the same bits.
      bool own_stats = false;
      if constexpr (Epi::kTileStats) {
        if (epi.a.ts.x) {
          const int g = (PAIR ? mu * 2 + (int)rank : mu) * BM / kStatRows;
          if (g > stats_ready) {
            int ready = 0;
            if (lane == 0) ready = poll_count(epi.a.ts.done + g, (int)gridDim.x, epi.a.ts.poll_ns) ? 1 : 0;
            if (__shfl_sync(0xffffffffu, ready, 0)) stats_ready = g;
            else own_stats = true;
          }
        }
      }
      {
        const int mt = PAIR ? mu * 2 + (int)rank : mu;
        const int row0 = mt * BM + quad * 32;
        const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + acc * BN;
        float rsum[8];
        float lm[8], ls[8];        // running (max, Σ exp) of each row (kRowLse)
        typename Epi::RowAux ra[8];
        // kRowSumIn: lane l forms the input row sum of row row0 + l, and each
        // lane takes those of its rows from the lane that owns them; likewise
        // the row scale r of the warp's own rows when it forms them (kTileStats)
        float rs_in = 0.f;
        if constexpr (Epi::kRowSumIn) {
          if (row0 + lane < M) rs_in = epi.row_sum_in(row0 + lane);
        }
        if constexpr (Epi::kTileStats) {
          if (own_stats) {
            for (int j = 0; j < 32 && row0 + j < M; ++j) {
              const float rj = epi.tile_row_scale(row0 + j, lane);
              if (lane == j) rs_in = rj;
            }
          }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          rsum[i] = 0.f;
          lm[i] = -INFINITY;
          ls[i] = 0.f;
          const int row = row0 + sub_row + 4 * i;
          if constexpr (Epi::kRowSumIn) {
            const float ss = __shfl_sync(0xffffffffu, rs_in, sub_row + 4 * i);
            if (row < M) ra[i] = epi.row_aux_with(ss);
          } else if constexpr (Epi::kTileStats) {
            const float rr = __shfl_sync(0xffffffffu, rs_in, sub_row + 4 * i);
            if (row < M) ra[i] = own_stats ? epi.row_aux_r(row, rr) : epi.row_aux(row);
          } else {
            if (row < M) ra[i] = epi.row_aux(row);
          }
        }
        // the global inputs of chunk c0 are requested while chunk c0 - 32 is
        // computed and stored, so their latency overlaps that chunk's stores
        typename Epi::Aux ax_next[8];
        {
          const int col = nt * BN + sub_col;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int row = row0 + sub_row + 4 * i;
            if (row < M && col < N) ax_next[i] = epi.aux(row, col, ra[i]);
          }
        }
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          uint32_t r0[16], r1[16];
          tmem_ld16(taddr + c0, r0);
          tmem_ld16(taddr + c0 + 16, r1);
          tmem_wait_ld();
          if (c0 + 32 == BN) {   // the accumulator is free once its last columns are in registers
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if constexpr (PAIR) mbar_arrive_cluster(tempty_cl[acc]);
              else mbar_arrive(&tempty[acc]);
            }
          }
          float* my = stage + lane * C::EPI_STRIDE;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            *reinterpret_cast<float4*>(my + 4 * i) =
                make_float4(__uint_as_float(r0[4 * i]), __uint_as_float(r0[4 * i + 1]), __uint_as_float(r0[4 * i + 2]),
                            __uint_as_float(r0[4 * i + 3]));
            *reinterpret_cast<float4*>(my + 16 + 4 * i) =
                make_float4(__uint_as_float(r1[4 * i]), __uint_as_float(r1[4 * i + 1]), __uint_as_float(r1[4 * i + 2]),
                            __uint_as_float(r1[4 * i + 3]));
          }
          __syncwarp();
          const int col = nt * BN + c0 + sub_col;
          typename Epi::Aux ax[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) ax[i] = ax_next[i];
          if (c0 + 32 < BN) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int row = row0 + sub_row + 4 * i;
              if (row < M && col + 32 < N) ax_next[i] = epi.aux(row, col + 32, ra[i]);
            }
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rl = sub_row + 4 * i;
            const float4 t = *reinterpret_cast<const float4*>(stage + rl * C::EPI_STRIDE + sub_col);
            float v[4] = {t.x, t.y, t.z, t.w};
            const int row = row0 + rl;
            if (row < M && col < N) {
              if constexpr (Epi::kRowLse)
                epi.lse(row, col, v, ra[i], lm[i], ls[i]);
              else
                rsum[i] += epi(row, col, v, ra[i], ax[i]);
            }
          }
          __syncwarp();            // before the next chunk overwrites the stage
        }
        if constexpr (Epi::kRowLse) {
          // the 8 lanes of a row merge their pairs in a fixed tree
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float m = lm[i], sv = ls[i];
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
              const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, sv, o);
              const float mn = fmaxf(m, m2);
              sv = mn == -INFINITY ? 0.f : sv * expf(m - mn) + s2 * expf(m2 - mn);
              m = mn;
            }
            const int row = row0 + sub_row + 4 * i;
            if ((lane & 7) == 0 && row < M) epi.lse_part(row, nt, m, sv);
          }
        }
        if constexpr (Epi::kRowReduce) {
          // this tile's share of each of the warp's 32 rows is partial nt
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float t = rsum[i];
            t += __shfl_xor_sync(0xffffffffu, t, 1);
            t += __shfl_xor_sync(0xffffffffu, t, 2);
            t += __shfl_xor_sync(0xffffffffu, t, 4);
            const int row = row0 + sub_row + 4 * i;
            if ((lane & 7) == 0 && row < M) epi.row_sums().part[(size_t)row * epi.row_sums().stride + nt] = t;
          }
        }
      }
    }
  }

  // Teardown (PAIR: every MMA of the pair has completed, rank 0's issuer
  // waited on its drain, before either CTA releases the pair's tensor memory)
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    else tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

template <int BN, class Epi, bool PAIR = false>
cudaError_t run(const void* A, const void* B, int M, int N, int K, const Epi& epi, cudaStream_t s,
                int* n_tiles_out = nullptr) {
  using C = TcCfg<BN, PAIR>;
  constexpr int MU = PAIR ? 2 : 1;
  if (n_tiles_out) *n_tiles_out = (N + BN - 1) / BN;
  if (M <= 0 || N <= 0) return cudaSuccess;
  if (PAIR && M < BM) return cudaErrorInvalidValue;
  CUtensorMap ta, tbm;
  const uint32_t a_rows = M >= BM ? BM : (uint32_t)((M + 7) / 8 * 8);
  cudaError_t e = make_tmap_2d_bf16(&ta, A, (uint64_t)M, (uint64_t)K, (uint64_t)K, BK, a_rows);
  if (e != cudaSuccess) return e;
  e = make_tmap_2d_bf16(&tbm, B, (uint64_t)N, (uint64_t)K, (uint64_t)K, BK, PAIR ? BN / 2 : BN);
  if (e != cudaSuccess) return e;
  static bool attr_set[64] = {false};
  static int max_clusters[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(k_gemm_tc<BN, Epi, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::SMEM);
    if (e != cudaSuccess) return e;
    if constexpr (PAIR) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(2 * (sm_count() / 2), 1, 1);
      cfg.blockDim = dim3(tc_threads<Epi>(), 1, 1);
      cfg.dynamicSmemBytes = C::SMEM;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, k_gemm_tc<BN, Epi, PAIR>, &cfg);
      if (e != cudaSuccess) return e;
      if (n <= 0) return cudaErrorNotSupported;
      max_clusters[dev] = n;
    }
    attr_set[dev] = true;
  }
  const int m_units = ((M + BM - 1) / BM + MU - 1) / MU;
  const int tiles = m_units * ((N + BN - 1) / BN);
  const int grid = tiles < sm_count() ? tiles : sm_count();
  // Short K with a B panel beyond what L2 keeps: group up to 48 row blocks (48
  // MB of A at K = 4096; 32 on CTA pairs), m fastest inside a group, so each B
  // tile is read from HBM once per group rather than once per row block.
  // Otherwise n fastest.  (Measured on the W1/W3 GEMM of 32768 tokens: single
  // CTAs with groups of 32, 48 and 64 row blocks ran at 1775-1790, 1835 and
  // 1622 TFLOP/s; CTA pairs with 16, 32, 48, 64 and 96 at 1715, 1793, 1775,
  // 1759 and 1673 TFLOP/s, reading 12.6, 6.6, 8.0, 10.5 and 16.3 GB from DRAM.)
  const size_t b_bytes = (size_t)N * K * 2;
  const int gmax = (PAIR ? 32 : 48) / MU;          // tiles along M per group
  const int group_m =
      (K <= 8192 && b_bytes > (size_t(48) << 20) && m_units > 1) ? (m_units < gmax ? m_units : gmax) : 0;
  if constexpr (PAIR) {
    const int clusters = tiles < max_clusters[dev] ? tiles : max_clusters[dev];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(tc_threads<Epi>());
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_gemm_tc<BN, Epi, PAIR>, ta, tbm, M, N, K, a_rows * BK * 2, group_m, epi,
                              device_error_word());
  }
  k_gemm_tc<BN, Epi><<<grid, tc_threads<Epi>(), C::SMEM, s>>>(ta, tbm, M, N, K, a_rows * BK * 2, group_m, epi,
                                                                   device_error_word());
  return cudaGetLastError();
}

// CTA pairs when the 256-row tiles fill at least two waves of clusters (one
// cluster per two SMs).  Measured on the prefill of 32768 tokens at d = 4096
// against single-CTA tiles: Wo 1445-1463 -> 1671-1680 TFLOP/s, W2 (single CTAs
// with two row blocks each) 1698-1712 -> 1832-1844, W1/W3 1758-1775 ->
// 1780-1789; on 4096 tokens (256 tiles of Wo and of W2): Wo 1165 -> 1325, W2
// 1367 -> 1586.  With 96 tiles (768 columns, 8192 tokens) Wo ran slower on pairs
// (277 -> 220), so fewer tiles keep single CTAs.
bool pair_fits(int M, int N) {
  const long tiles = (long)((M + 2 * BM - 1) / (2 * BM)) * ((N + 255) / 256);
  return M >= 2 * BM && tiles >= (long)sm_count();
}

// Narrow N tiles when the grid would not fill the GPU.
template <class Epi>
cudaError_t run_auto(const void* A, const void* B, int M, int N, int K, const Epi& epi, cudaStream_t s,
                     int* n_tiles_out = nullptr) {
  const long tiles256 = (long)((M + BM - 1) / BM) * ((N + 255) / 256);
  if (tiles256 >= 2L * sm_count()) return run<256, Epi>(A, B, M, N, K, epi, s, n_tiles_out);
  return run<128, Epi>(A, B, M, N, K, epi, s, n_tiles_out);
}

}  // namespace

int sm_count() {
  static int n[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 1;
  if (!n[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    n[dev] = v > 0 ? v : 1;
  }
  return n[dev];
}

cudaError_t make_tmap_2d_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                              uint64_t row_stride_elems, uint32_t box_cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {row_stride_elems * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

namespace {
cudaError_t make_tmap_3d(CUtensorMap* m, CUtensorMapDataType type, uint32_t esize, const void* base,
                         uint64_t planes, uint64_t rows, uint64_t cols, uint64_t row_stride_elems,
                         uint64_t plane_stride_elems, uint32_t box_cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {cols, rows, planes};
  const cuuint64_t strides[2] = {row_stride_elems * esize, plane_stride_elems * esize};
  const cuuint32_t box[3] = {box_cols, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(m, type, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}
}  // namespace

cudaError_t make_tmap_3d_bf16(CUtensorMap* m, const void* base, uint64_t planes, uint64_t rows, uint64_t cols,
                              uint64_t row_stride_elems, uint64_t plane_stride_elems, uint32_t box_cols,
                              uint32_t box_rows) {
  return make_tmap_3d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, planes, rows, cols, row_stride_elems,
                      plane_stride_elems, box_cols, box_rows);
}

cudaError_t make_tmap_3d_u8(CUtensorMap* m, const void* base, uint64_t planes, uint64_t rows, uint64_t cols,
                            uint64_t row_stride, uint64_t plane_stride, uint32_t box_cols, uint32_t box_rows) {
  return make_tmap_3d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, planes, rows, cols, row_stride, plane_stride,
                      box_cols, box_rows);
}

cudaError_t gemm_tc_qkv(const void* A, const void* B, int M, int N, int K, const Dims& D, const QKVArgs& e,
                        cudaStream_t s) {
  const EpiQKV<bf16, true> epi{e, D.H, D.Hkv, D.dh, log2_dh(D.dh)};
  if (pair_fits(M, N)) return run<256, EpiQKV<bf16, true>, true>(A, B, M, N, K, epi, s);
  return run_auto(A, B, M, N, K, epi, s);
}
cudaError_t gemm_tc_wo(const void* A, const void* B, int M, int N, int K, const Dims& D, const WoArgs& e,
                       cudaStream_t s, int* row_parts) {
  // one Σh² partial per row and column tile
  if (pair_fits(M, N)) return run<256, EpiWo<bf16, true>, true>(A, B, M, N, K, EpiWo<bf16, true>{e, D.d}, s, row_parts);
  return run_auto(A, B, M, N, K, EpiWo<bf16, true>{e, D.d}, s, row_parts);
}
cudaError_t gemm_tc_w13(const void* A, const void* B, int M, int N, int K, const Dims& D, const W13Args& e,
                        cudaStream_t s) {
  if (pair_fits(M, N))
    return run<256, EpiW13<bf16, true>, true>(A, B, M, N, K, EpiW13<bf16, true>{e, D.d, D.f, D.eps}, s);
  return run_auto(A, B, M, N, K, EpiW13<bf16, true>{e, D.d, D.f, D.eps}, s);
}
cudaError_t gemm_tc_w2(const void* A, const void* B, int M, int N, int K, const Dims& D, const W2Args& e,
                       cudaStream_t s) {
  if (pair_fits(M, N)) return run<256, EpiW2<true>, true>(A, B, M, N, K, EpiW2<true>{e, D.d}, s);
  return run_auto(A, B, M, N, K, EpiW2<true>{e, D.d}, s);
}
cudaError_t gemm_tc_logits(const void* A, const void* B, int M, int N, int K, const LogitsArgs& e, cudaStream_t s) {
  return run_auto(A, B, M, N, K, EpiLogits{e}, s);
}
int lse_tile_cols() { return 256; }
cudaError_t gemm_tc_lse(const void* A, const void* B, int M, int N, int K, const LseArgs& e, cudaStream_t s) {
  return run<256>(A, B, M, N, K, EpiLse{e}, s);
}
cudaError_t gemm_tc_f32out(const void* A, const void* B, float* Cp, int M, int N, int K, int bn, int mt,
                           cudaStream_t s) {
  if (mt == 2) return run<256, EpiF32, true>(A, B, M, N, K, EpiF32{Cp, N}, s);
  if (bn == 256) return run<256>(A, B, M, N, K, EpiF32{Cp, N}, s);
  return run<128>(A, B, M, N, K, EpiF32{Cp, N}, s);
}

}  // namespace tb
