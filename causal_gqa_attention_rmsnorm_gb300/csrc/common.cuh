// Shared device helpers and the internal launcher interface of libtb.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/tb.h"

namespace tb {

using bf16 = __nv_bfloat16;

template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<bf16>(bf16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float v) { return __float2bfloat16_rn(v); }

// log2 of a head width (a power of two: 16, 32, 64 or 128).
inline int log2_dh(int dh) {
  int s = 0;
  while ((1 << s) < dh) ++s;
  return s;
}

// Programmatic dependent launch.  The kernels of a decode step are launched
// (launch_pdl) so that each may be scheduled while the one before it drains:
// a kernel calls pdl_trigger() at its start, which lets the next launch as
// soon as every CTA of this one has started, and pdl_wait() before it touches
// any global memory an earlier kernel of the stream writes or reads — the wait
// returns once the previous grid has completed and its writes are visible.
// Every CTA passes pdl_wait() before it exits, so completion is ordered along
// the whole chain.  Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// 16-byte vector of T: 4 floats or 8 bf16.
template <typename T> struct Vec16 {
  static constexpr int N = 16 / sizeof(T);
  uint4 raw;
  __device__ __forceinline__ float get(int i) const {
    if constexpr (sizeof(T) == 4) {
      return __uint_as_float((&raw.x)[i]);
    } else {
      uint32_t w = (&raw.x)[i >> 1];
      return __uint_as_float((i & 1) ? (w & 0xffff0000u) : (w << 16));
    }
  }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// Everything a launcher needs to know about one block call.
struct Dims {
  int d, H, Hkv, dh, f;
  float eps;
  int max_pos;
};

// Views into the packed weight blob (device pointers).
struct Packed {
  const void* wqkv;   // [(H+2Hkv)·dh, d]  gain-folded, transposed
  const void* wo;     // [d, H·dh]
  const void* w13;    // [2f, d]           gain-folded, rows 2j = W1[:,j], 2j+1 = W3[:,j]
  const void* w2;     // [d, f]
  const float2* rope; // [max_pos, dh/2]   (cos, sin)
};

}  // namespace tb

// ---------------------------------------------------------------------------
// Launchers (host functions, one translation unit each group).  All return a
// cudaError_t from cudaGetLastError after their launches.
// ---------------------------------------------------------------------------
namespace tb {

// tb_api.cu: device address of the per-device error word (TB_DEVERR_* bits)
int* device_error_word();
// tb_api.cu: record the message tb_last_error_message() returns; returns st.
tb_status report(tb_status st, const char* fmt, ...);

// elementwise.cu
cudaError_t launch_pack(int dtype, const Dims& D, const tb_block_weights& w, void* packed,
                        const Packed& P, float rope_base, cudaStream_t s);
cudaError_t launch_row_stats(int dtype, const void* x, int M, int d, float eps, float* r,
                             int T, int32_t* lens_set, int32_t* lens_bump,
                             int32_t* pos_out, int T_max, int* zero_word, int* err, cudaStream_t s);
cudaError_t launch_kv_append(int dtype, const tb_kvcache& kv, const void* k_new, const void* v_new,
                             int n, int* err, cudaStream_t s);
// Quantise bf16 rows k_new, v_new [B, Hkv, rows, 128] into the int8 cache kv
// at rows start[b] + r (start == nullptr: 0).  A sequence whose start is
// negative or whose rows would pass T_max is skipped.
cudaError_t launch_quantize_kv(const tb_kvcache& kv, const void* k_new, const void* v_new, int rows,
                               const int32_t* start, cudaStream_t s);

// A paged cache as kernels see it (bt == nullptr: none).  Row t of sequence b
// lives in page bt[b·max_pages + t/ps] at offset t % ps of pools
// [num_pages, Hkv, ps, dh]; a page id outside [0, num_pages) is never
// dereferenced and sets TB_DEVERR_BAD_PAGE.
struct PagedKV {
  void* k = nullptr;
  void* v = nullptr;
  const int32_t* bt = nullptr;
  int ps = 0, max_pages = 0, num_pages = 0;
  int* err = nullptr;
};

// A byte range that a kernel pulls into L2 after its own work, for the next
// kernel on the stream (p 16-byte aligned; bytes 0: none).
struct L2Prefetch {
  const void* p = nullptr;
  unsigned long long bytes = 0;
};

// Row offset (in rows of dh values) of key t of (sequence b, KV head h) in a
// paged pool, or -1 for a bad page id (flagged in the error word).
__device__ __forceinline__ long long paged_row(const PagedKV& p, int Hkv, int b, int h, int t) {
  const int page = p.bt[(size_t)b * p.max_pages + t / p.ps];
  if (page < 0 || page >= p.num_pages) {
    atomicOr(p.err, TB_DEVERR_BAD_PAGE);
    return -1;
  }
  return ((long long)page * Hkv + h) * p.ps + t % p.ps;
}

// Row sums in a fixed order, so that a run is reproducible bit for bit: each
// of a row's producers (one per column tile or column range of the GEMM that
// forms the row) stores its partial at part[row·stride + p], p < n; the
// consumer, a later kernel that sees every partial, adds them in the order
// p = 0, 1, ..., n-1.  No fence, counter or atomic sits on the producer's
// path.
struct RowSum {
  float* part;             // [M, stride]
  int stride;              // partials per row the buffer holds
  int n;                   // partials per row the producing GEMM writes (set by its launcher)
};

// Σ_{p < n} part[p] added in the order p = 0, 1, ..., with the loads issued
// eight at a time (read-only: the partials come from an earlier kernel).
__device__ __forceinline__ float ordered_sum(const float* part, int n) {
  float sum = 0.f;
  int p = 0;
  for (; p + 8 <= n; p += 8) {
    float t[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) t[u] = __ldg(part + p + u);
#pragma unroll
    for (int u = 0; u < 8; ++u) sum += t[u];
  }
  for (; p < n; ++p) sum += __ldg(part + p);
  return sum;
}

// GEMM epilogue argument bundles.

// RMSNorm-1 statistics and the decode step's bookkeeping taken by the
// few-token QKV GEMM's epilogue: each CTA forms Σx² of every token over its K
// range, the cluster adds them, and the token's reducer reads its position
// from lens.  x == nullptr: r and
// the positions come from the row-statistics kernel instead.
struct QKVStats {
  const void* x = nullptr;   // [M, d] block input (the block's dtype)
  int d = 0;
  float eps = 0.f;
  const int32_t* lens = nullptr;   // token m sits at lens[m] (advanced later, by the Wo epilogue)
  int32_t* pos_out = nullptr;      // [M] the positions, -1 for a full cache, for the step's later kernels
  int T_max = 0;
  int* zero_word = nullptr;        // zeroed for a later kernel of the step
  int* err = nullptr;
};
// RMSNorm-1 statistics formed inside the tile QKV GEMM (prefill): one extra
// warp per CTA computes r for its share of each group of kStatRows rows, in
// group order, and counts the finished group in done[group] (zeroed before the
// launch).  A tile's epilogue polls its group's count for a bounded time; if
// the group is not complete by then (a CTA of the grid not yet resident), the
// epilogue warps form r for their own rows with the same function, which gives
// the same bits, so no launch guarantee is needed.
// x == nullptr: r comes from the row-statistics kernel.
constexpr int kStatRows = 2048;
struct TileStats {
  const void* x = nullptr;   // [M, d] block input (the block's dtype)
  int d = 0;
  float eps = 0.f;
  float* r = nullptr;        // [M] the row scales (the epilogue reads them as QKVArgs::r)
  int* done = nullptr;       // [ceil(M / kStatRows)] arrival counts
  int32_t* lens_set = nullptr;   // prefill with a cache: lens[b] = T
  int T = 0;
  unsigned long long poll_ns = 0;   // how long an epilogue polls for its group before forming r itself
};
// The poll limit the prefill passes (stat_poll_ns(); a test hook may shorten it).
unsigned long long stat_poll_ns();
struct QKVArgs {
  const float* r;          // [M] RMSNorm-1 inverse RMS of each token
  const float2* rope;      // [max_pos, dh/2]
  void* q;                 // [B, H, Tq, dh]
  void* k;                 // [B, Hkv, kv_stride, dh]
  void* v;
  int T;                   // tokens per sequence (1 for decode)
  int kv_stride;           // rows per (b, kv head) in k/v
  const int32_t* pos;      // decode: position of sequence b (-1: skip); prefill: nullptr
  PagedKV pg;              // also (or, with k == nullptr, only) store k and v rows into this paged cache
  bool kv_dense = false;   // k/v take the call's rows densely: row = token index in the call, not its position
  QKVStats st;             // few-token decode: statistics and positions formed in the epilogue
  TileStats ts;            // tile GEMM (prefill): statistics formed by the GEMM's statistics warp
};
struct WoArgs {
  const void* x;           // [M, d] residual input (cfg dtype)
  float* h;                // [M, d] fp32 residual stream after attention
  void* hb;                // [M, d] cfg dtype copy of h (A operand of W1/W3), may be == h for f32
  RowSum ssq;              // Σ h² of each row, as partials
  const int32_t* pos = nullptr;   // few-token decode: lens[m] = pos[m] + 1 for pos[m] ≥ 0, here
  int32_t* lens = nullptr;
};
struct W13Args {
  RowSum ssq;              // Σ h² of each row: the Wo GEMM's partials, summed here in order
  void* a;                 // [M, f] SiLU(gate)·up
};
struct LogitsArgs {
  const float* r;          // [M] final-norm inverse RMS of each row
  float* out;              // [M, ld] fp32 logits
  int ld;
};
struct LseArgs {
  const float* r;          // [M] final-norm inverse RMS of each row
  const int32_t* targets;  // [M] target token of each row
  float2* part;            // [M, n_parts] running (max, Σ exp(v - max)) of each column tile
  float* tgt;              // [M] the target's logit
  int n_parts;
};
struct W2Args {
  const float* h;          // [M, d]
  void* y;                 // [M, d]
  int y_dtype;
};

// LM head GEMMs (logits = (x·r)·Wᵀ, W [N, K] packed): tile, few-token and fp32 forms
cudaError_t gemm_tc_logits(const void* A, const void* B, int M, int N, int K, const LogitsArgs& e, cudaStream_t s);
// The per-token loss without logits in memory: per row and 256-column tile a
// (max, Σ exp) pair and the target's logit (ceil(N / 256) pairs per row).
cudaError_t gemm_tc_lse(const void* A, const void* B, int M, int N, int K, const LseArgs& e, cudaStream_t s);
int lse_tile_cols();
cudaError_t gemm_skinny_logits(const void* A, const void* B, int M, int N, int K, const LogitsArgs& e,
                               cudaStream_t s);
cudaError_t gemm_simt_logits(int dtype, const void* A, const void* B, int M, int N, int K, const LogitsArgs& e,
                             cudaStream_t s);

// head.cu: embedding gather, LM-head reductions
cudaError_t launch_embed(int dtype, const void* table, int V, int d, const int32_t* ids, long long n, void* x,
                         int* err, cudaStream_t s);
// nll[m] = logsumexp - target logit from the (max, Σ exp) pairs of gemm_tc_lse
cudaError_t launch_lse_merge(const float2* part, int n_parts, const float* tgt, const int32_t* targets, int V, int M,
                             float* nll, int* err, cudaStream_t s);
cudaError_t launch_lse_nll(const float* logits, int ld, int M, int V, const int32_t* targets, float* nll, int* err,
                           cudaStream_t s);
cudaError_t launch_scale_cols(int dtype, const void* src, const void* gain, int rows, int cols, void* dst,
                              cudaStream_t s);
cudaError_t launch_pack_transpose(int dtype, const void* src, int K, int N, const void* gain, void* dst,
                                  cudaStream_t s);

// gemm_simt.cu (fp32 path)
cudaError_t gemm_simt_qkv(int dtype, const void* A, const void* B, int M, int N, int K, const Dims& D,
                          const QKVArgs& e, cudaStream_t s);
cudaError_t gemm_simt_wo(int dtype, const void* A, const void* B, int M, int N, int K, const Dims& D,
                         const WoArgs& e, cudaStream_t s, int* row_parts);
cudaError_t gemm_simt_w13(int dtype, const void* A, const void* B, int M, int N, int K, const Dims& D,
                          const W13Args& e, cudaStream_t s);
cudaError_t gemm_simt_w2(int dtype, const void* A, const void* B, int M, int N, int K, const Dims& D,
                         const W2Args& e, cudaStream_t s);

// gemm_skinny.cu (bf16, M ≤ skinny_max_tokens(): K-split tcgen05 GEMM whose
// split is reduced inside a cluster, with the fused epilogue)
int skinny_max_tokens();
// K ranges per weight tile (the cluster size) for `tiles` 128-row weight tiles
// of `kblocks` K blocks over `slots` resident CTAs (-1 for a non-positive argument)
int skinny_split_count(int tiles, int kblocks, int slots);
cudaError_t gemm_skinny_qkv(const void* A, const void* B, int M, int N, int K, const Dims& D, const QKVArgs& e,
                            cudaStream_t s);
cudaError_t gemm_skinny_wo(const void* A, const void* B, int M, int N, int K, const Dims& D, const WoArgs& e,
                           cudaStream_t s, int* row_parts);
cudaError_t gemm_skinny_w13(const void* A, const void* B, int M, int N, int K, const Dims& D, const W13Args& e,
                            cudaStream_t s);
cudaError_t gemm_skinny_w2(const void* A, const void* B, int M, int N, int K, const Dims& D, const W2Args& e,
                           cudaStream_t s);

// attn_simt.cu (fp32 path)
cudaError_t attn_prefill_simt(int dtype, const void* q, const void* k, const void* v, void* o, int B,
                              int T, int H, int Hkv, int dh, int kv_stride, int window, cudaStream_t s);

// Attention launchers take the sliding-window width (0: full causal).
// attn_tc.cu (bf16 path, dh 64 or 128): CTA pairs (attn_pair.cu) where H/Hkv
// is a multiple of 4 and dh = 128, single CTAs otherwise.
cudaError_t attn_prefill_tc(const void* q, const void* k, const void* v, void* o, int B, int T, int H, int Hkv,
                            int dh, int kv_stride, int window, cudaStream_t s);
// attn_pair.cu: cudaErrorNotSupported for shapes it does not take.
cudaError_t attn_prefill_pair(const void* q, const void* k, const void* v, void* o, int B, int T, int H, int Hkv,
                              int dh, int kv_stride, int window, cudaStream_t s);

// attn_decode.cu
// Keys per decode work item (chunk) for a step of B sequences over a T_max-row
// cache; the workspace holds ceil(T_max / chunk) partial states per head.
int decode_chunk_keys(int dtype, int B, int Hkv, int T_max);
int decode_chunk_keys_sms(int dtype, int B, int Hkv, int T_max, int sms);   // the same rule for `sms` SMs
size_t decode_part_floats(int B, int H, int dh, int nchunk_max);
cudaError_t attn_decode(int dtype, const void* q, const void* kc, const void* vc, const int32_t* pos,
                        int B, int H, int Hkv, int dh, int T_max, float* part, int nchunk_max, int chunk,
                        int* work_counter, int window, const PagedKV& pg, void* o, cudaStream_t s,
                        const L2Prefetch& pf = L2Prefetch());
// Decode over an int8 cache (dh 128): codes kc, vc [B, Hkv, T_max, 128], row
// scales ks, vs [B, Hkv, T_max]; bf16 q and o.
cudaError_t attn_decode_i8(const void* q, const void* kc, const void* vc, const float* ks, const float* vs,
                           const int32_t* pos, int B, int H, int Hkv, int T_max, float* part, int nchunk_max,
                           int chunk, int* work_counter, int window, const PagedKV& pg, void* o, cudaStream_t s,
                           const L2Prefetch& pf = L2Prefetch());

}  // namespace tb
