// C ABI of libtb: argument checks, buffer carving and the launch sequences of
// the prefill and decode steps.  Declarations and contracts are in tb.h.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <vector>

#include "common.cuh"
#include "gemm_tc.cuh"

namespace tb {
namespace {

__device__ int g_device_error;  // TB_DEVERR_* bits

thread_local char g_msg[512] = "";

tb_status fail(tb_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

tb_status cuda_fail(cudaError_t e, const char* where) {
  return fail(TB_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

}  // namespace

tb_status report(tb_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

namespace {
std::atomic<unsigned long long> g_stat_poll_ns{200000};
}  // namespace
unsigned long long stat_poll_ns() { return g_stat_poll_ns.load(); }

// Device address of the error word on the current device.
int* device_error_word() {
  static int* ptrs[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    ptrs[dev] = (int*)p;
  }
  return ptrs[dev];
}

namespace {

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
size_t esize(int dtype) { return dtype == TB_F32 ? 4 : 2; }

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// The bf16 and int8 decode attention kernels keep two ints per sequence in
// shared memory beside their stage rings.
constexpr int kDecodeMaxBatch = 2048;
// The decode merge takes at most 1024 chunks of at most 256 keys.
constexpr int kDecodeMaxRows = 1024 * 256;

tb_status check_cfg(const tb_block_cfg* c) {
  if (!c) return fail(TB_ERR_INVALID_ARG, "cfg is NULL");
  if (c->d <= 0 || c->H <= 0 || c->Hkv <= 0 || c->dh <= 0 || c->f <= 0)
    return fail(TB_ERR_INVALID_ARG, "d, H, Hkv, dh and f must be positive");
  if (c->H % c->Hkv) return fail(TB_ERR_INVALID_ARG, "H (%d) must be a multiple of Hkv (%d)", c->H, c->Hkv);
  if ((long long)c->H * c->dh != c->d)
    return fail(TB_ERR_INVALID_ARG, "dh (%d) must equal d/H (%d/%d)", c->dh, c->d, c->H);
  if (c->dh % 2) return fail(TB_ERR_INVALID_ARG, "dh must be even (RoPE rotates pairs)");
  if (c->max_pos <= 0) return fail(TB_ERR_INVALID_ARG, "max_pos must be positive");
  if (!(c->rope_base > 0.f)) return fail(TB_ERR_INVALID_ARG, "rope_base must be positive");
  if (!(c->eps >= 0.f)) return fail(TB_ERR_INVALID_ARG, "eps must be non-negative");
  if (c->dtype != TB_F32 && c->dtype != TB_BF16) return fail(TB_ERR_INVALID_ARG, "unknown dtype %d", c->dtype);
  if (c->window < 0) return fail(TB_ERR_INVALID_ARG, "window (%d) must be non-negative", c->window);
  if (c->dh != 16 && c->dh != 32 && c->dh != 64 && c->dh != 128)
    return fail(TB_ERR_UNSUPPORTED, "dh %d: attention kernels exist for 16, 32, 64 and 128", c->dh);
  const int G = c->H / c->Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8)
    return fail(TB_ERR_UNSUPPORTED, "H/Hkv = %d: decode kernels exist for 1, 2, 4 and 8", G);
  if (c->f % 2) return fail(TB_ERR_UNSUPPORTED, "f must be even");
  if (c->dtype == TB_BF16) {
    if (c->d % 64 || c->f % 64)
      return fail(TB_ERR_UNSUPPORTED, "bf16 tensor-core path needs d and f multiples of 64 (d=%d f=%d)", c->d,
                  c->f);
    if (c->dh != 64 && c->dh != 128)
      return fail(TB_ERR_UNSUPPORTED, "bf16 tensor-core attention needs dh 64 or 128 (dh=%d)", c->dh);
  }
  return TB_OK;
}

Dims dims_of(const tb_block_cfg* c) { return Dims{c->d, c->H, c->Hkv, c->dh, c->f, c->eps, c->max_pos}; }

// Packed weight blob: four matrices and the RoPE table, 1 KiB aligned.
struct PackedLayout {
  size_t wqkv, wo, w13, w2, rope, total;
};
PackedLayout packed_layout(const tb_block_cfg* c) {
  const size_t es = esize(c->dtype);
  PackedLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 1024);
    return o;
  };
  const size_t nqkv = (size_t)(c->H + 2 * c->Hkv) * c->dh;
  L.wqkv = take(nqkv * c->d * es);
  L.wo = take((size_t)c->d * c->H * c->dh * es);
  L.w13 = take((size_t)2 * c->f * c->d * es);
  L.w2 = take((size_t)c->d * c->f * es);
  L.rope = take((size_t)c->max_pos * (c->dh / 2) * sizeof(float2));
  L.total = off;
  return L;
}

Packed packed_views(const tb_block_cfg* c, const void* blob) {
  const PackedLayout L = packed_layout(c);
  const char* b = (const char*)blob;
  return Packed{b + L.wqkv, b + L.wo, b + L.w13, b + L.w2, (const float2*)(b + L.rope)};
}

// Workspace carving.  Prefill keeps K/V in the workspace when no cache is given.
struct Work {
  float* r;
  float* ssq_part;           // [M, ssq_stride] ordered partials of Σ h² (the second norm) of each row
  int ssq_stride;
  int32_t* pos;
  int* counter;
  int* stat_done;            // [ceil(M / kStatRows)] group counts of the tile QKV GEMM's statistics warps
  void* q;
  void* k;
  void* v;
  void* o;
  float* h;
  void* hb;
  void* a;
  float* part;
  int nchunk_max;
  int chunk;                 // keys per decode work item
  bool few;                  // bf16 with M ≤ 64 tokens: the few-token GEMM
  size_t total;
};

Work carve(const tb_block_cfg* c, int B, int T, int mode, void* base) {
  const size_t es = esize(c->dtype);
  char* p = (char*)base;
  size_t off = 0;
  auto take = [&](size_t bytes) -> void* {
    void* r = p ? (void*)(p + off) : nullptr;
    off = align_up(off + bytes, 256);
    return r;
  };
  Work w{};
  const size_t M = (size_t)B * (mode == 0 ? T : 1);
  const size_t hd = (size_t)c->H * c->dh, kvd = (size_t)c->Hkv * c->dh;
  w.r = (float*)take(M * 4);
  // partials per row: one per column tile (tile GEMM, ≥ 128 columns; few-token
  // GEMM, 128 columns) or per 64 columns (fp32 GEMM)
  w.ssq_stride = (c->d + 63) / 64 + 8;
  w.ssq_part = (float*)take(M * w.ssq_stride * 4);
  w.pos = (int32_t*)take((size_t)B * 4);
  w.counter = (int*)take(4);
  w.stat_done = (int*)take((M + kStatRows - 1) / kStatRows * 4);
  w.q = take(M * hd * es);
  // prefill: K/V of the call when no contiguous cache of the block's type
  // takes them in place; decode: the new rows on their way into an int8 cache
  w.k = take(M * kvd * es);
  w.v = take(M * kvd * es);
  w.o = take(M * hd * es);
  w.h = (float*)take(M * c->d * 4);
  w.hb = c->dtype == TB_F32 ? (void*)w.h : take(M * c->d * es);
  w.a = take(M * c->f * es);
  if (mode == 1) {
    w.chunk = decode_chunk_keys(c->dtype, B, c->Hkv, T);
    w.nchunk_max = (T + w.chunk - 1) / w.chunk;
    w.part = (float*)take(decode_part_floats(B, c->H, c->dh, w.nchunk_max) * 4);
  }
  w.few = c->dtype == TB_BF16 && M <= (size_t)skinny_max_tokens();
  w.total = off;
  return w;
}

// bf16 GEMMs: few tokens go to the K-split GEMM, which streams the weights
// with every SM; more tokens to the persistent tile GEMM.
cudaError_t mm_qkv(const Work& W, const void* A, const void* Bw, int M, int N, int K, const Dims& D,
                   const QKVArgs& e, cudaStream_t s) {
  return W.few ? gemm_skinny_qkv(A, Bw, M, N, K, D, e, s) : gemm_tc_qkv(A, Bw, M, N, K, D, e, s);
}
cudaError_t mm_wo(const Work& W, const void* A, const void* Bw, int M, int N, int K, const Dims& D, const WoArgs& e,
                  cudaStream_t s, int* row_parts) {
  return W.few ? gemm_skinny_wo(A, Bw, M, N, K, D, e, s, row_parts) : gemm_tc_wo(A, Bw, M, N, K, D, e, s, row_parts);
}
cudaError_t mm_w13(const Work& W, const void* A, const void* Bw, int M, int N, int K, const Dims& D,
                   const W13Args& e, cudaStream_t s) {
  return W.few ? gemm_skinny_w13(A, Bw, M, N, K, D, e, s) : gemm_tc_w13(A, Bw, M, N, K, D, e, s);
}
cudaError_t mm_w2(const Work& W, const void* A, const void* Bw, int M, int N, int K, const Dims& D, const W2Args& e,
                  cudaStream_t s) {
  return W.few ? gemm_skinny_w2(A, Bw, M, N, K, D, e, s) : gemm_tc_w2(A, Bw, M, N, K, D, e, s);
}

// The int8 layout's own rules (dh 128, contiguous, 32-row stages, scales).
tb_status check_i8(const tb_kvcache* kv) {
  if (kv->dh != 128) return fail(TB_ERR_UNSUPPORTED, "an int8 cache needs dh 128 (dh=%d)", kv->dh);
  if (kv->T_max % 32) return fail(TB_ERR_UNSUPPORTED, "an int8 cache needs T_max a multiple of 32 (%d)", kv->T_max);
  if (kv->block_table && kv->page_size % 32)
    return fail(TB_ERR_UNSUPPORTED, "a paged int8 cache needs page_size a multiple of 32 (%d)", kv->page_size);
  if (!kv->k_scale || !kv->v_scale || !aligned16(kv->k_scale) || !aligned16(kv->v_scale))
    return fail(TB_ERR_INVALID_ARG, "an int8 cache needs 16-byte aligned k_scale and v_scale");
  return TB_OK;
}

tb_status check_kv(const tb_block_cfg* c, const tb_kvcache* kv, int B) {
  if (!kv->k || !kv->v || !kv->lens) return fail(TB_ERR_INVALID_ARG, "kv cache pointers must be non-NULL");
  if (kv->B != B) return fail(TB_ERR_INVALID_ARG, "kv->B (%d) differs from B (%d)", kv->B, B);
  if (kv->Hkv != c->Hkv || kv->dh != c->dh)
    return fail(TB_ERR_INVALID_ARG, "kv cache heads/width (%d, %d) differ from cfg (%d, %d)", kv->Hkv, kv->dh,
                c->Hkv, c->dh);
  if (kv->T_max <= 0) return fail(TB_ERR_INVALID_ARG, "kv->T_max must be positive");
  if (kv->dtype == TB_I8) {
    const tb_status st = check_i8(kv);
    if (st != TB_OK) return st;
    if (c->dtype != TB_BF16) return fail(TB_ERR_UNSUPPORTED, "an int8 cache needs a bf16 block");
  } else if (kv->dtype != c->dtype) {
    return fail(TB_ERR_INVALID_ARG, "kv cache dtype differs from cfg dtype");
  }
  if (!aligned16(kv->k) || !aligned16(kv->v) || ((uintptr_t)kv->lens & 3u))
    return fail(TB_ERR_INVALID_ARG, "kv cache pointers must be 16-byte aligned (lens 4-byte)");
  if (kv->block_table) {
    if (kv->page_size <= 0 || kv->page_size % 16)
      return fail(TB_ERR_INVALID_ARG, "page_size (%d) must be a positive multiple of 16", kv->page_size);
    if (kv->T_max % kv->page_size)
      return fail(TB_ERR_INVALID_ARG, "page_size (%d) must divide T_max (%d)", kv->page_size, kv->T_max);
    if (kv->num_pages <= 0) return fail(TB_ERR_INVALID_ARG, "num_pages must be positive");
    if ((uintptr_t)kv->block_table & 3u) return fail(TB_ERR_INVALID_ARG, "block_table must be 4-byte aligned");
  }
  return TB_OK;
}

// The paged view kernels use (bt == nullptr for a contiguous cache).
PagedKV paged_of(const tb_kvcache* kv, int* err) {
  PagedKV p;
  if (kv && kv->block_table) {
    p.k = kv->k;
    p.v = kv->v;
    p.bt = kv->block_table;
    p.ps = kv->page_size;
    p.max_pages = kv->T_max / kv->page_size;
    p.num_pages = kv->num_pages;
    p.err = err;
  }
  return p;
}

// Per-stage CUDA-event trace (test and benchmark hook).  When enabled, each
// prefill/decode call takes the next slot of a ring of `slots` calls and
// records one event before each of its stages and one after the last, on the
// call's own stream, so stage durations are device times of exactly those
// launches.
struct Trace {
  bool on = false;
  int slots = 0, next = 0, stages = 0;
  std::vector<cudaEvent_t> ev;       // slots × (kMaxStages + 1)
  std::vector<int> used;             // stages recorded per slot
  std::vector<const char*> names;    // stage names of the last traced call
};
constexpr int kMaxStages = 8;
Trace g_trace;

struct StageRecorder {
  cudaStream_t s;
  int slot = -1, n = 0;
  explicit StageRecorder(cudaStream_t st) : s(st) {
    if (g_trace.on && g_trace.slots > 0) {
      slot = g_trace.next;
      g_trace.next = (g_trace.next + 1) % g_trace.slots;
      g_trace.names.clear();
    }
  }
  void stage(const char* name) {
    if (slot < 0 || n >= kMaxStages) return;
    cudaEventRecord(g_trace.ev[(size_t)slot * (kMaxStages + 1) + n], s);
    g_trace.names.push_back(name);
    ++n;
  }
  ~StageRecorder() {
    if (slot < 0) return;
    cudaEventRecord(g_trace.ev[(size_t)slot * (kMaxStages + 1) + n], s);
    g_trace.used[slot] = n;
  }
};

#define TB_TRY(expr)                              \
  do {                                            \
    cudaError_t e_ = (expr);                      \
    if (e_ != cudaSuccess) return cuda_fail(e_, #expr); \
  } while (0)

}  // namespace
}  // namespace tb

using namespace tb;

extern "C" {

size_t tb_packed_weights_bytes(const tb_block_cfg* cfg) {
  if (check_cfg(cfg) != TB_OK) return 0;
  return packed_layout(cfg).total;
}

tb_status tb_pack_weights(const tb_block_cfg* cfg, const tb_block_weights* w, void* packed, size_t packed_bytes,
                          void* stream) {
  tb_status st = check_cfg(cfg);
  if (st != TB_OK) return st;
  if (!w || !packed) return fail(TB_ERR_INVALID_ARG, "weights and packed must be non-NULL");
  const void* ptrs[9] = {w->g_attn, w->wq, w->wk, w->wv, w->wo, w->g_mlp, w->w1, w->w3, w->w2};
  for (const void* p : ptrs)
    if (!p) return fail(TB_ERR_INVALID_ARG, "a weight pointer is NULL");
  if ((uintptr_t)packed & 255u) return fail(TB_ERR_INVALID_ARG, "packed must be 256-byte aligned");
  if (packed_bytes < packed_layout(cfg).total)
    return fail(TB_ERR_INVALID_ARG, "packed buffer too small: %zu < %zu", packed_bytes, packed_layout(cfg).total);
  const Packed P = packed_views(cfg, packed);
  TB_TRY(launch_pack(cfg->dtype, dims_of(cfg), *w, packed, P, cfg->rope_base, (cudaStream_t)stream));
  return TB_OK;
}

size_t tb_workspace_bytes(const tb_block_cfg* cfg, int32_t B, int32_t T, int32_t mode) {
  if (check_cfg(cfg) != TB_OK || B < 0 || T < 0 || (mode != 0 && mode != 1)) return 0;
  return carve(cfg, B, T, mode, nullptr).total;
}

tb_status tb_block_prefill(const tb_block_cfg* cfg, const void* packed, const void* x, void* y, int32_t y_dtype,
                           int32_t B, int32_t T, const tb_kvcache* kv, void* ws, size_t ws_bytes, void* stream) {
  tb_status st = check_cfg(cfg);
  if (st != TB_OK) return st;
  if (B < 0 || T < 0) return fail(TB_ERR_INVALID_ARG, "B and T must be non-negative");
  if (y_dtype != TB_F32 && !(y_dtype == TB_BF16 && cfg->dtype == TB_BF16))
    return fail(TB_ERR_INVALID_ARG, "y_dtype must be TB_F32, or TB_BF16 for a bf16 block");
  if (kv) {
    st = check_kv(cfg, kv, B);
    if (st != TB_OK) return st;
    if (T > kv->T_max) return fail(TB_ERR_INVALID_ARG, "T (%d) exceeds kv->T_max (%d)", T, kv->T_max);
  }
  if (B == 0 || T == 0) return TB_OK;
  if (T > cfg->max_pos) return fail(TB_ERR_INVALID_ARG, "T (%d) exceeds cfg->max_pos (%d)", T, cfg->max_pos);
  if ((long long)B * T > (1LL << 30)) return fail(TB_ERR_UNSUPPORTED, "B·T above 2^30 tokens");
  if (!packed || !x || !y || !ws) return fail(TB_ERR_INVALID_ARG, "packed, x, y and ws must be non-NULL");
  if (!aligned16(x) || !aligned16(y) || ((uintptr_t)packed & 255u) || ((uintptr_t)ws & 255u))
    return fail(TB_ERR_INVALID_ARG, "x, y must be 16-byte aligned; packed, ws 256-byte aligned");
  if (x == y) return fail(TB_ERR_INVALID_ARG, "y may not alias x");
  const Work W = carve(cfg, B, T, 0, ws);
  if (ws_bytes < W.total) return fail(TB_ERR_INVALID_ARG, "workspace too small: %zu < %zu", ws_bytes, W.total);
  int* err = device_error_word();
  if (!err) return fail(TB_ERR_CUDA, "cannot resolve the device error word");

  cudaStream_t s = (cudaStream_t)stream;
  const Dims D = dims_of(cfg);
  const Packed P = packed_views(cfg, packed);
  const int M = B * T;
  const int dt = cfg->dtype;
  const int nqkv = (cfg->H + 2 * cfg->Hkv) * cfg->dh;
  // attention reads K/V from a contiguous cache in place, else from the
  // workspace; a paged cache receives the rows as a second store, an int8
  // cache their codes
  const bool i8_cache = kv && kv->dtype == TB_I8;
  const bool contiguous_cache = kv && !kv->block_table && !i8_cache;
  void* kbuf = contiguous_cache ? kv->k : W.k;
  void* vbuf = contiguous_cache ? kv->v : W.v;
  const int kv_stride = contiguous_cache ? kv->T_max : T;

  StageRecorder rec(s);
  // The tile GEMM path (bf16, more tokens than the few-token GEMM takes) forms
  // RMSNorm-1's statistics inside the QKV GEMM; the other paths run the
  // row-statistics kernel first.
  const bool tile_stats = dt == TB_BF16 && !W.few;
  // (an int8 cache, paged or not, gets its codes from the quantiser, never the rows)
  QKVArgs qa{W.r, P.rope, W.q, kbuf, vbuf, T, kv_stride, nullptr, i8_cache ? PagedKV() : paged_of(kv, err)};
  if (tile_stats) {
    TB_TRY(cudaMemsetAsync(W.stat_done, 0, (size_t)(M + kStatRows - 1) / kStatRows * sizeof(int), s));
    qa.ts = TileStats{x, cfg->d, cfg->eps, W.r, W.stat_done, kv ? kv->lens : nullptr, T, stat_poll_ns()};
  } else {
    rec.stage("rms");
    TB_TRY(launch_row_stats(dt, x, M, cfg->d, cfg->eps, W.r, T, kv ? kv->lens : nullptr, nullptr, nullptr, 0,
                            nullptr, err, s));
  }
  const WoArgs wa{x, W.h, W.hb, RowSum{W.ssq_part, W.ssq_stride, 0}};
  W13Args ga{RowSum{W.ssq_part, W.ssq_stride, 0}, W.a};       // ssq.n: set by the Wo launch
  const W2Args ya{W.h, y, y_dtype};
  if (dt == TB_F32) {
    rec.stage("qkv");
    TB_TRY(gemm_simt_qkv(dt, x, P.wqkv, M, nqkv, cfg->d, D, qa, s));
    rec.stage("attn");
    TB_TRY(attn_prefill_simt(dt, W.q, kbuf, vbuf, W.o, B, T, cfg->H, cfg->Hkv, cfg->dh, kv_stride, cfg->window, s));
    rec.stage("wo");
    TB_TRY(gemm_simt_wo(dt, W.o, P.wo, M, cfg->d, cfg->H * cfg->dh, D, wa, s, &ga.ssq.n));
    rec.stage("w13");
    TB_TRY(gemm_simt_w13(dt, W.hb, P.w13, M, 2 * cfg->f, cfg->d, D, ga, s));
    rec.stage("w2");
    TB_TRY(gemm_simt_w2(dt, W.a, P.w2, M, cfg->d, cfg->f, D, ya, s));
  } else {
    rec.stage("qkv");
    TB_TRY(mm_qkv(W, x, P.wqkv, M, nqkv, cfg->d, D, qa, s));
    if (i8_cache) {
      rec.stage("quant");
      TB_TRY(launch_quantize_kv(*kv, W.k, W.v, T, nullptr, s));
    }
    rec.stage("attn");
    TB_TRY(attn_prefill_tc(W.q, kbuf, vbuf, W.o, B, T, cfg->H, cfg->Hkv, cfg->dh, kv_stride, cfg->window, s));
    rec.stage("wo");
    TB_TRY(mm_wo(W, W.o, P.wo, M, cfg->d, cfg->H * cfg->dh, D, wa, s, &ga.ssq.n));
    rec.stage("w13");
    TB_TRY(mm_w13(W, W.hb, P.w13, M, 2 * cfg->f, cfg->d, D, ga, s));
    rec.stage("w2");
    TB_TRY(mm_w2(W, W.a, P.w2, M, cfg->d, cfg->f, D, ya, s));
  }
  return TB_OK;
}

tb_status tb_block_decode(const tb_block_cfg* cfg, const void* packed, const void* x, void* y, int32_t y_dtype,
                          const tb_kvcache* kv, void* ws, size_t ws_bytes, void* stream) {
  tb_status st = check_cfg(cfg);
  if (st != TB_OK) return st;
  if (!kv) return fail(TB_ERR_INVALID_ARG, "decode needs a kv cache");
  if (kv->B < 0) return fail(TB_ERR_INVALID_ARG, "kv->B must be non-negative");
  st = check_kv(cfg, kv, kv->B);
  if (st != TB_OK) return st;
  if (y_dtype != TB_F32 && !(y_dtype == TB_BF16 && cfg->dtype == TB_BF16))
    return fail(TB_ERR_INVALID_ARG, "y_dtype must be TB_F32, or TB_BF16 for a bf16 block");
  if (kv->T_max > cfg->max_pos)
    return fail(TB_ERR_INVALID_ARG, "kv->T_max (%d) exceeds cfg->max_pos (%d)", kv->T_max, cfg->max_pos);
  if (kv->T_max > kDecodeMaxRows)
    return fail(TB_ERR_UNSUPPORTED, "kv->T_max (%d) above the %d rows the decode merge supports", kv->T_max,
                kDecodeMaxRows);
  const int B = kv->B;
  if (B == 0) return TB_OK;
  if (cfg->dtype == TB_BF16 && B > kDecodeMaxBatch)
    return fail(TB_ERR_UNSUPPORTED, "decode of %d sequences: the bf16 decode attention takes at most %d per call", B,
                kDecodeMaxBatch);
  if (!packed || !x || !y || !ws) return fail(TB_ERR_INVALID_ARG, "packed, x, y and ws must be non-NULL");
  if (!aligned16(x) || !aligned16(y) || ((uintptr_t)packed & 255u) || ((uintptr_t)ws & 255u))
    return fail(TB_ERR_INVALID_ARG, "x, y must be 16-byte aligned; packed, ws 256-byte aligned");
  if (x == y) return fail(TB_ERR_INVALID_ARG, "y may not alias x");
  const Work W = carve(cfg, B, kv->T_max, 1, ws);
  if (ws_bytes < W.total) return fail(TB_ERR_INVALID_ARG, "workspace too small: %zu < %zu", ws_bytes, W.total);
  int* err = device_error_word();
  if (!err) return fail(TB_ERR_CUDA, "cannot resolve the device error word");

  cudaStream_t s = (cudaStream_t)stream;
  const Dims D = dims_of(cfg);
  const Packed P = packed_views(cfg, packed);
  const int dt = cfg->dtype;
  const int nqkv = (cfg->H + 2 * cfg->Hkv) * cfg->dh;

  StageRecorder rec(s);
  // Few tokens on the bf16 path: RMSNorm-1's statistics, the positions and
  // the step's counters are formed in the few-token QKV GEMM's epilogue, and
  // the cache lengths advance in the Wo one; otherwise the row-statistics
  // kernel does all of it first.
  const bool fused_stats = dt == TB_BF16 && W.few;
  if (!fused_stats) {
    rec.stage("rms");
    TB_TRY(launch_row_stats(dt, x, B, cfg->d, cfg->eps, W.r, 1, nullptr, kv->lens, W.pos, kv->T_max, W.counter,
                            err, s));
  }
  const PagedKV pg = paged_of(kv, err);
  // an int8 cache (paged or not) gets the new rows through the workspace and the quantiser
  const bool i8 = kv->dtype == TB_I8;
  void* knew = i8 ? W.k : (pg.bt ? nullptr : kv->k);
  void* vnew = i8 ? W.v : (pg.bt ? nullptr : kv->v);
  QKVArgs qa{W.r, P.rope, W.q, knew, vnew, 1, i8 ? 1 : kv->T_max, W.pos, i8 ? PagedKV() : pg, i8};
  WoArgs wa{x, W.h, W.hb, RowSum{W.ssq_part, W.ssq_stride, 0}};
  if (fused_stats) {
    qa.st = QKVStats{x, cfg->d, cfg->eps, kv->lens, W.pos, kv->T_max, W.counter, err};
    wa.pos = W.pos;
    wa.lens = kv->lens;
  }
  W13Args ga{RowSum{W.ssq_part, W.ssq_stride, 0}, W.a};       // ssq.n: set by the Wo launch
  const W2Args ya{W.h, y, y_dtype};
  if (dt == TB_F32) {
    rec.stage("qkv");
    TB_TRY(gemm_simt_qkv(dt, x, P.wqkv, B, nqkv, cfg->d, D, qa, s));
    rec.stage("attn");
    TB_TRY(attn_decode(dt, W.q, kv->k, kv->v, W.pos, B, cfg->H, cfg->Hkv, cfg->dh, kv->T_max, W.part,
                       W.nchunk_max, W.chunk, W.counter, cfg->window, pg, W.o, s));
    rec.stage("wo");
    TB_TRY(gemm_simt_wo(dt, W.o, P.wo, B, cfg->d, cfg->H * cfg->dh, D, wa, s, &ga.ssq.n));
    rec.stage("w13");
    TB_TRY(gemm_simt_w13(dt, W.hb, P.w13, B, 2 * cfg->f, cfg->d, D, ga, s));
    rec.stage("w2");
    TB_TRY(gemm_simt_w2(dt, W.a, P.w2, B, cfg->d, cfg->f, D, ya, s));
  } else {
    rec.stage("qkv");
    TB_TRY(mm_qkv(W, x, P.wqkv, B, nqkv, cfg->d, D, qa, s));
    // The attention kernels end by pulling Wo's weights into L2, so that the
    // Wo GEMM that follows reads them from there: the last items of the
    // attention leave HBM idle, the GEMM's first loads would wait on it.
    L2Prefetch wo_pf;
    if (!((uintptr_t)P.wo & 15u)) wo_pf = L2Prefetch{P.wo, (unsigned long long)cfg->d * cfg->H * cfg->dh * 2ull};
    if (i8) {
      rec.stage("quant");
      TB_TRY(launch_quantize_kv(*kv, W.k, W.v, 1, W.pos, s));
      rec.stage("attn");
      TB_TRY(attn_decode_i8(W.q, kv->k, kv->v, kv->k_scale, kv->v_scale, W.pos, B, cfg->H, cfg->Hkv, kv->T_max,
                            W.part, W.nchunk_max, W.chunk, W.counter, cfg->window, pg, W.o, s, wo_pf));
    } else {
      rec.stage("attn");
      TB_TRY(attn_decode(dt, W.q, kv->k, kv->v, W.pos, B, cfg->H, cfg->Hkv, cfg->dh, kv->T_max, W.part,
                         W.nchunk_max, W.chunk, W.counter, cfg->window, pg, W.o, s, wo_pf));
    }
    rec.stage("wo");
    TB_TRY(mm_wo(W, W.o, P.wo, B, cfg->d, cfg->H * cfg->dh, D, wa, s, &ga.ssq.n));
    rec.stage("w13");
    TB_TRY(mm_w13(W, W.hb, P.w13, B, 2 * cfg->f, cfg->d, D, ga, s));
    rec.stage("w2");
    TB_TRY(mm_w2(W, W.a, P.w2, B, cfg->d, cfg->f, D, ya, s));
  }
  return TB_OK;
}

tb_status tb_kvcache_append(const tb_kvcache* kv, const void* k_new, const void* v_new, int32_t n, void* stream) {
  if (!kv) return fail(TB_ERR_INVALID_ARG, "kv is NULL");
  if (n < 0) return fail(TB_ERR_INVALID_ARG, "n must be non-negative");
  if (kv->dtype != TB_F32 && kv->dtype != TB_BF16 && kv->dtype != TB_I8)
    return fail(TB_ERR_INVALID_ARG, "unknown kv dtype");
  if (kv->B < 0 || kv->Hkv <= 0 || kv->dh <= 0 || kv->T_max <= 0)
    return fail(TB_ERR_INVALID_ARG, "kv shape must be positive (B may be 0)");
  if (kv->dtype == TB_I8) {
    const tb_status st = check_i8(kv);
    if (st != TB_OK) return st;
  } else if ((kv->dh * (int)esize(kv->dtype)) % 16) {
    return fail(TB_ERR_UNSUPPORTED, "dh·sizeof must be a multiple of 16");
  }
  if (n == 0 || kv->B == 0) return TB_OK;
  if (n > kv->T_max) return fail(TB_ERR_CACHE_FULL, "n (%d) exceeds T_max (%d)", n, kv->T_max);
  if (!kv->k || !kv->v || !kv->lens || !k_new || !v_new)
    return fail(TB_ERR_INVALID_ARG, "cache and new-row pointers must be non-NULL");
  if (!aligned16(kv->k) || !aligned16(kv->v) || !aligned16(k_new) || !aligned16(v_new))
    return fail(TB_ERR_INVALID_ARG, "cache and new-row pointers must be 16-byte aligned");
  if (kv->block_table &&
      (kv->page_size <= 0 || kv->T_max % kv->page_size || kv->num_pages <= 0 || ((uintptr_t)kv->block_table & 3u)))
    return fail(TB_ERR_INVALID_ARG, "paged cache: page_size must divide T_max, num_pages be positive, "
                                    "block_table 4-byte aligned");
  int* err = device_error_word();
  if (!err) return fail(TB_ERR_CUDA, "cannot resolve the device error word");
  TB_TRY(launch_kv_append(kv->dtype, *kv, k_new, v_new, n, err, (cudaStream_t)stream));
  return TB_OK;
}

tb_status tb_get_device_error(void* stream, int32_t* err_out, int32_t clear) {
  if (!err_out) return fail(TB_ERR_INVALID_ARG, "err_out is NULL");
  TB_TRY(cudaStreamSynchronize((cudaStream_t)stream));
  int* err = device_error_word();
  if (!err) return fail(TB_ERR_CUDA, "cannot resolve the device error word");
  int v = 0;
  TB_TRY(cudaMemcpy(&v, err, sizeof(int), cudaMemcpyDeviceToHost));
  *err_out = v;
  if (clear) TB_TRY(cudaMemset(err, 0, sizeof(int)));
  return TB_OK;
}

const char* tb_status_string(tb_status s) {
  switch (s) {
    case TB_OK: return "ok";
    case TB_ERR_INVALID_ARG: return "invalid argument";
    case TB_ERR_UNSUPPORTED: return "unsupported shape";
    case TB_ERR_CUDA: return "CUDA error";
    case TB_ERR_CACHE_FULL: return "KV cache full";
    case TB_ERR_TIMEOUT: return "timeout";
  }
  return "unknown status";
}

const char* tb_last_error_message(void) { return g_msg; }

// Trace hooks (not part of the public header).  tbx_trace_enable(slots)
// creates `slots` × 9 events on the current device and turns tracing on;
// slots = 0 turns it off.  tbx_trace_read(slot, ms, n) synchronises the slot's
// last event and writes up to n stage durations; it returns the number of
// stages recorded in that slot (0 if none), or -1 on a CUDA error.
TB_API int32_t tbx_trace_enable(int32_t slots) {
  for (cudaEvent_t e : g_trace.ev) cudaEventDestroy(e);
  g_trace = Trace{};
  if (slots <= 0) return 0;
  g_trace.ev.resize((size_t)slots * (kMaxStages + 1));
  for (auto& e : g_trace.ev)
    if (cudaEventCreate(&e) != cudaSuccess) return -1;
  g_trace.used.assign(slots, 0);
  g_trace.slots = slots;
  g_trace.on = true;
  return 0;
}

TB_API int32_t tbx_trace_read(int32_t slot, float* ms, int32_t n) {
  if (slot < 0 || slot >= g_trace.slots) return 0;
  const int used = g_trace.used[slot];
  cudaEvent_t* ev = &g_trace.ev[(size_t)slot * (kMaxStages + 1)];
  if (used == 0) return 0;
  if (cudaEventSynchronize(ev[used]) != cudaSuccess) return -1;
  for (int i = 0; i < used && i < n; ++i)
    if (cudaEventElapsedTime(&ms[i], ev[i], ev[i + 1]) != cudaSuccess) return -1;
  return used;
}

TB_API const char* tbx_trace_stage_name(int32_t i) {
  return (i >= 0 && i < (int)g_trace.names.size()) ? g_trace.names[i] : "";
}

// Host-side selection rules (not part of the public header), for tests that
// need no GPU: the few-token GEMM's K-range count for `tiles` weight tiles of
// `kblocks` 64-wide K blocks over `slots` resident CTAs, and the decode work
// item's key count for a GPU of `sms` SMs.
TB_API int32_t tbx_skinny_split_count(int32_t tiles, int32_t kblocks, int32_t slots) {
  return skinny_split_count(tiles, kblocks, slots);
}
TB_API int32_t tbx_decode_chunk_keys(int32_t dtype, int32_t B, int32_t Hkv, int32_t T_max, int32_t sms) {
  if (B <= 0 || Hkv <= 0 || T_max <= 0 || sms <= 0) return -1;
  return decode_chunk_keys_sms(dtype, B, Hkv, T_max, sms);
}

// Test hook (not part of the public header): how long a QKV tile epilogue
// polls for its row group's RMSNorm-1 statistics before it forms its rows'
// scales itself (default 200 us: far longer than the statistics warps of a
// resident grid take); 0 makes nearly every epilogue form its own, which must
// give the same bytes.  Returns the previous value.
TB_API uint64_t tbx_set_stat_poll_ns(uint64_t ns) { return g_stat_poll_ns.exchange(ns); }

// Test hook (not part of the public header): C[M, N] = A[M, K]·B[N, K]ᵀ in
// fp32 through the bf16 tcgen05 main loop, N-tile width bn (128 or 256); mt = 2
// takes 256-row tiles on CTA pairs (bn 256, M ≥ 128).
TB_API tb_status tbx_gemm_bf16(const void* A, const void* B, float* Cp, int32_t M, int32_t N, int32_t K, int32_t bn,
                               int32_t mt, void* stream) {
  if (!A || !B || !Cp || M < 0 || N <= 0 || K <= 0 || K % 64 || N % 4 || (bn != 128 && bn != 256) ||
      (mt != 1 && mt != 2) || (mt == 2 && (bn != 256 || M < 128)))
    return fail(TB_ERR_INVALID_ARG, "tbx_gemm_bf16: bad arguments");
  TB_TRY(gemm_tc_f32out(A, B, Cp, M, N, K, bn, mt, (cudaStream_t)stream));
  return TB_OK;
}

}  // extern "C"
