// bf16 GEMM for few tokens (M ≤ 64, e.g. the decode step's one token per
// sequence) on the 5th-generation tensor cores, split over K.
//
// With M tokens and N outputs, C = X·Wᵀ is bound by streaming the weight
// matrix W [N, K] from HBM.  The product is computed transposed, Cᵀ = W·Xᵀ, so
// that 128 weight rows form the MMA's M dimension and the (padded) tokens its N
// dimension: no MMA lane is wasted on padding rows.  Each CTA owns one
// 128-row weight tile and one contiguous range of K; enough K ranges are used
// that about two CTAs per SM stream weights at once.
//   warp 0      TMA: the weight tile [128, 64] and the token tile [NT, 64]
//               of each K block into a ring of shared-memory stages;
//   warp 1      MMA issuer: D[128, NT] += W_blk · X_blkᵀ (tcgen05, fp32 in
//               tensor memory);
//   warps 2..5  drain: each warp's 32 TMEM lanes are 32 output features; the
//               fp32 partial sums go to part[split][token][feature].
// A second kernel adds the K-range partials and applies the block's fused
// epilogue (the same functors as the large GEMMs) to 4 outputs per thread.
#include "epilogues.cuh"
#include "gemm_tc.cuh"
#include "sm100_ptx.cuh"

namespace tb {
namespace {

using namespace ptx;

constexpr int kRows = 128;       // weight rows per CTA: the MMA's M
constexpr int kBK = 64;          // K per stage (one 128-byte swizzle row)
constexpr int kMaxTok = 64;
constexpr int kMaxCtas = 320;    // tiles × splits target bound; sizes the partial buffer

template <int NT> struct SkCfg {
  static constexpr int STAGES = NT <= 32 ? 5 : 4;           // two CTAs per SM
  static constexpr uint32_t W_BYTES = kRows * kBK * 2;       // 16 KB
  static constexpr uint32_t X_BYTES = NT * kBK * 2;          // a multiple of 1 KB
  static constexpr uint32_t STAGE_BYTES = W_BYTES + X_BYTES;
  static constexpr uint32_t OFF_BAR = STAGES * STAGE_BYTES;
  static constexpr size_t SMEM = OFF_BAR + 256 + 1024;
  static constexpr uint32_t TMEM_COLS = NT <= 32 ? 32 : 64;
};

template <int NT>
__global__ void __launch_bounds__(192)
    k_gemm_skinny(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, int M, int N,
                  int kblocks, int splits, float* __restrict__ part, int* err) {
  using C = SkCfg<NT>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* drain = tfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kRows, sp = blockIdx.y;
  const int kb0 = (int)((long long)kblocks * sp / splits);
  const int nkb = (int)((long long)kblocks * (sp + 1) / splits) - kb0;   // ≥ 1: splits ≤ kblocks

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
      int issued = 0;
      for (int i = 0; i < nkb; ++i) {
        const int st = i % STAGES;
        const uint32_t ph = (i / STAGES) & 1;
        if (!mbar_wait(&empty[st], ph ^ 1u, abort_flag, err)) break;
        uint8_t* sw = smem + st * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&full[st], C::STAGE_BYTES);
        tma_load_2d(&tmW, sw, &full[st], (kb0 + i) * kBK, n0);
        tma_load_2d(&tmX, sw + C::W_BYTES, &full[st], (kb0 + i) * kBK, 0);
        ++issued;
      }
      // every copy issued must land before the CTA may exit
      volatile int no_abort = 0;
      for (int i = issued - STAGES < 0 ? 0 : issued - STAGES; i < issued; ++i)
        mbar_wait(&full[i % STAGES], (i / STAGES) & 1, &no_abort, err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kRows, NT);
      bool ok = true;
      for (int i = 0; i < nkb; ++i) {
        const int st = i % STAGES;
        if (!mbar_wait(&full[st], (i / STAGES) & 1, abort_flag, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t w0 = smem_u32(smem + st * C::STAGE_BYTES), x0 = w0 + C::W_BYTES;
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          mma_bf16_ss(tmem, desc_kmajor_sw128(w0 + k * 32), desc_kmajor_sw128(x0 + k * 32), idesc, (i | k) != 0);
        mma_commit(&empty[st]);
      }
      if (ok) mma_commit(tfull);
      mma_commit(drain);
      volatile int no_abort = 0;
      mbar_wait(drain, 0, &no_abort, err);
    }
  } else {
    // lane l of warp w holds output feature n0 + 32·(w%4) + l for all NT tokens
    const int quad = warp & 3;
    if (mbar_wait_warp(tfull, 0, abort_flag, err)) {
      tc_fence_after();
      uint32_t u[NT];
#pragma unroll
      for (int c = 0; c < NT; c += 16)
        tmem_ld16(tmem + ((uint32_t)(quad * 32) << 16) + c, *reinterpret_cast<uint32_t(*)[16]>(u + c));
      tmem_wait_ld();
      const int n = n0 + quad * 32 + lane;
      if (n < N) {
        float* dst = part + (size_t)sp * M * N + n;
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
// the Wo epilogue) is a warp sum and one atomic per warp.
template <class Epi>
__global__ void __launch_bounds__(256)
    k_splitk_epilogue(const float* __restrict__ part, int splits, int M, int N, Epi epi) {
  const int m = blockIdx.y;
  const int col = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
  float r = 0.f;
  if (col < N) {
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    const float* p = part + (size_t)m * N + col;
    for (int s = 0; s < splits; ++s) {
      const float4 t = *reinterpret_cast<const float4*>(p + (size_t)s * M * N);
      v[0] += t.x;
      v[1] += t.y;
      v[2] += t.z;
      v[3] += t.w;
    }
    const auto ra = epi.row_aux(m);
    r = epi(m, col, v, ra, epi.aux(m, col, ra));
  }
  if constexpr (Epi::kRowReduce) {
    r = warp_sum(r);
    if ((threadIdx.x & 31) == 0) epi.row_reduce(m, r);
  }
}

int split_count(int tiles, int kblocks) {
  int target = 2 * sm_count();
  if (target > kMaxCtas) target = kMaxCtas;
  int sp = target / tiles;
  const int cap = kblocks / 8 > 0 ? kblocks / 8 : 1;     // at least 8 K blocks (1 MB of W) per CTA
  if (sp > cap) sp = cap;
  return sp < 1 ? 1 : sp;
}

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
  k_gemm_skinny<NT><<<dim3(tiles, splits), 192, C::SMEM, s>>>(tw, tx, M, N, kblocks, splits, part,
                                                              device_error_word());
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_splitk_epilogue<Epi><<<dim3((N / 4 + 255) / 256, M), 256, 0, s>>>(part, splits, M, N, epi);
  return cudaGetLastError();
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

int skinny_max_tokens() { return kMaxTok; }

size_t skinny_part_floats(int M, int max_n) {
  const int tiles = (max_n + kRows - 1) / kRows;
  return (size_t)M * kRows * (size_t)(tiles > kMaxCtas ? tiles : kMaxCtas);
}

cudaError_t gemm_skinny_qkv(const void* A, const void* B, int M, int N, int K, const Dims& D, const QKVArgs& e,
                            float* part, cudaStream_t s) {
  return run(A, B, M, N, K, EpiQKV<bf16>{e, D.H, D.Hkv, D.dh}, part, s);
}
cudaError_t gemm_skinny_wo(const void* A, const void* B, int M, int N, int K, const Dims& D, const WoArgs& e,
                           float* part, cudaStream_t s) {
  return run(A, B, M, N, K, EpiWo<bf16>{e, D.d}, part, s);
}
cudaError_t gemm_skinny_w13(const void* A, const void* B, int M, int N, int K, const Dims& D, const W13Args& e,
                            float* part, cudaStream_t s) {
  return run(A, B, M, N, K, EpiW13<bf16>{e, D.d, D.f, D.eps}, part, s);
}
cudaError_t gemm_skinny_w2(const void* A, const void* B, int M, int N, int K, const Dims& D, const W2Args& e,
                           float* part, cudaStream_t s) {
  return run(A, B, M, N, K, EpiW2{e, D.d}, part, s);
}

}  // namespace tb
