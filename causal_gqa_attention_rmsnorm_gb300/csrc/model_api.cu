// C ABI around the block: the embedding gather, the LM head with its chunked
// loss, and an L-layer stack of blocks.  Declarations and contracts are in
// tb.h.  ("Transformer block" page, tirogla.com, "How it works", steps 1 and
// 4; "The Transformer", GenerativeAIDocs, §5 "A tensor's journey".)
#include <stdint.h>

#include <algorithm>

#include "common.cuh"

namespace tb {
namespace {

constexpr int kDefaultRowChunk = 4096;

size_t esize(int dtype) { return dtype == TB_F32 ? 4 : 2; }
size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

tb_status check_head(const tb_head_cfg* c) {
  if (!c) return report(TB_ERR_INVALID_ARG, "head cfg is NULL");
  if (c->d <= 0 || c->V <= 0) return report(TB_ERR_INVALID_ARG, "d and V must be positive");
  if (c->dtype != TB_F32 && c->dtype != TB_BF16) return report(TB_ERR_INVALID_ARG, "unknown dtype %d", c->dtype);
  if (!(c->eps >= 0.f)) return report(TB_ERR_INVALID_ARG, "eps must be non-negative");
  if (c->V % 4) return report(TB_ERR_UNSUPPORTED, "V (%d) must be a multiple of 4", c->V);
  if ((c->d * (int)esize(c->dtype)) % 16) return report(TB_ERR_UNSUPPORTED, "d·sizeof must be a multiple of 16");
  if (c->dtype == TB_BF16 && c->d % 64) return report(TB_ERR_UNSUPPORTED, "bf16 head needs d a multiple of 64");
  return TB_OK;
}

// Workspace of the head: row scales, one chunk of logits, and for the fused
// loss the (max, Σ exp) pairs and target logits of one chunk.
struct HeadWork {
  float* r;
  float* chunk;
  float2* lse;
  float* tgt;
  int n_parts;
  size_t total;
};
HeadWork carve_head(const tb_head_cfg* c, int rc, void* base) {
  char* p = (char*)base;
  size_t off = 0;
  auto take = [&](size_t bytes) -> void* {
    void* r = p ? (void*)(p + off) : nullptr;
    off = align_up(off + bytes, 256);
    return r;
  };
  HeadWork w{};
  w.r = (float*)take((size_t)rc * 4);
  w.chunk = (float*)take((size_t)rc * c->V * 4);
  w.n_parts = (c->V + lse_tile_cols() - 1) / lse_tile_cols();
  if (c->dtype == TB_BF16) {
    w.lse = (float2*)take((size_t)rc * w.n_parts * sizeof(float2));
    w.tgt = (float*)take((size_t)rc * 4);
  }
  w.total = off;
  return w;
}

int row_chunk_of(int32_t row_chunk) { return row_chunk > 0 ? row_chunk : kDefaultRowChunk; }

size_t act_bytes(const tb_block_cfg* c, int B, int T) { return align_up((size_t)B * T * c->d * esize(c->dtype), 256); }

}  // namespace
}  // namespace tb

using namespace tb;

extern "C" {

tb_status tb_embed(const void* table, int32_t V, int32_t d, int32_t dtype, const int32_t* ids, int64_t n, void* x,
                   void* stream) {
  if (V <= 0 || d <= 0 || n < 0) return report(TB_ERR_INVALID_ARG, "V, d must be positive and n non-negative");
  if (dtype != TB_F32 && dtype != TB_BF16) return report(TB_ERR_INVALID_ARG, "unknown dtype %d", dtype);
  if ((d * (int)esize(dtype)) % 16) return report(TB_ERR_UNSUPPORTED, "d·sizeof must be a multiple of 16");
  if (n == 0) return TB_OK;
  if (!table || !ids || !x) return report(TB_ERR_INVALID_ARG, "table, ids and x must be non-NULL");
  if (!aligned16(table) || !aligned16(x) || ((uintptr_t)ids & 3u))
    return report(TB_ERR_INVALID_ARG, "table and x must be 16-byte aligned, ids 4-byte");
  int* err = device_error_word();
  if (!err) return report(TB_ERR_CUDA, "cannot resolve the device error word");
  const cudaError_t e = launch_embed(dtype, table, V, d, ids, n, x, err, (cudaStream_t)stream);
  return e == cudaSuccess ? TB_OK : report(TB_ERR_CUDA, "tb_embed: %s", cudaGetErrorString(e));
}

size_t tb_lm_head_packed_bytes(const tb_head_cfg* cfg) {
  if (check_head(cfg) != TB_OK) return 0;
  return align_up((size_t)cfg->V * cfg->d * esize(cfg->dtype), 1024);
}

tb_status tb_pack_lm_head(const tb_head_cfg* cfg, const void* g_final, const void* w_u, int32_t tied, void* packed,
                          size_t packed_bytes, void* stream) {
  tb_status st = check_head(cfg);
  if (st != TB_OK) return st;
  if (!g_final || !w_u || !packed) return report(TB_ERR_INVALID_ARG, "g_final, w_u and packed must be non-NULL");
  if (packed_bytes < tb_lm_head_packed_bytes(cfg)) return report(TB_ERR_INVALID_ARG, "packed buffer too small");
  if ((uintptr_t)packed & 255u) return report(TB_ERR_INVALID_ARG, "packed must be 256-byte aligned");
  const cudaError_t e =
      tied ? launch_scale_cols(cfg->dtype, w_u, g_final, cfg->V, cfg->d, packed, (cudaStream_t)stream)
           : launch_pack_transpose(cfg->dtype, w_u, cfg->d, cfg->V, g_final, packed, (cudaStream_t)stream);
  return e == cudaSuccess ? TB_OK : report(TB_ERR_CUDA, "tb_pack_lm_head: %s", cudaGetErrorString(e));
}

size_t tb_lm_head_workspace_bytes(const tb_head_cfg* cfg, int32_t row_chunk) {
  if (check_head(cfg) != TB_OK || row_chunk < 0) return 0;
  return carve_head(cfg, row_chunk_of(row_chunk), nullptr).total;
}

tb_status tb_lm_head(const tb_head_cfg* cfg, const void* packed, const void* x, int32_t M, float* logits,
                     const int32_t* targets, float* nll, int32_t row_chunk, void* ws, size_t ws_bytes, void* stream) {
  tb_status st = check_head(cfg);
  if (st != TB_OK) return st;
  if (M < 0 || row_chunk < 0) return report(TB_ERR_INVALID_ARG, "M and row_chunk must be non-negative");
  if ((targets == nullptr) != (nll == nullptr)) return report(TB_ERR_INVALID_ARG, "targets and nll go together");
  if (M == 0 || (!logits && !nll)) return TB_OK;
  if (!packed || !x || !ws) return report(TB_ERR_INVALID_ARG, "packed, x and ws must be non-NULL");
  if (!aligned16(x) || (logits && !aligned16(logits)) || ((uintptr_t)packed & 255u) || ((uintptr_t)ws & 255u))
    return report(TB_ERR_INVALID_ARG, "x, logits 16-byte aligned; packed, ws 256-byte aligned");
  const int rc = row_chunk_of(row_chunk);
  const HeadWork W = carve_head(cfg, rc, ws);
  if (ws_bytes < W.total) return report(TB_ERR_INVALID_ARG, "workspace too small: %zu < %zu", ws_bytes, W.total);
  int* err = device_error_word();
  if (!err) return report(TB_ERR_CUDA, "cannot resolve the device error word");
  cudaStream_t s = (cudaStream_t)stream;
  const size_t row_bytes = (size_t)cfg->d * esize(cfg->dtype);
  for (int r0 = 0; r0 < M; r0 += rc) {
    const int rows = std::min(rc, M - r0);
    const void* xa = (const char*)x + (size_t)r0 * row_bytes;
    float* out = logits ? logits + (size_t)r0 * cfg->V : W.chunk;
    cudaError_t e = launch_row_stats(cfg->dtype, xa, rows, cfg->d, cfg->eps, W.r, 1, nullptr, nullptr, nullptr, 0,
                                     nullptr, err, s);
    // the loss alone, on the tile GEMM: folded into the GEMM's epilogue, no logits in memory
    if (e == cudaSuccess && !logits && cfg->dtype == TB_BF16 && rows > skinny_max_tokens()) {
      e = gemm_tc_lse(xa, packed, rows, cfg->V, cfg->d, LseArgs{W.r, targets + r0, W.lse, W.tgt, W.n_parts}, s);
      if (e == cudaSuccess)
        e = launch_lse_merge(W.lse, W.n_parts, W.tgt, targets + r0, cfg->V, rows, nll + r0, err, s);
      if (e != cudaSuccess) return report(TB_ERR_CUDA, "tb_lm_head: %s", cudaGetErrorString(e));
      continue;
    }
    const LogitsArgs la{W.r, out, cfg->V};
    if (e == cudaSuccess) {
      if (cfg->dtype == TB_F32)
        e = gemm_simt_logits(cfg->dtype, xa, packed, rows, cfg->V, cfg->d, la, s);
      else if (rows <= skinny_max_tokens())
        e = gemm_skinny_logits(xa, packed, rows, cfg->V, cfg->d, la, s);
      else
        e = gemm_tc_logits(xa, packed, rows, cfg->V, cfg->d, la, s);
    }
    if (e == cudaSuccess && nll) e = launch_lse_nll(out, cfg->V, rows, cfg->V, targets + r0, nll + r0, err, s);
    if (e != cudaSuccess) return report(TB_ERR_CUDA, "tb_lm_head: %s", cudaGetErrorString(e));
  }
  return TB_OK;
}

size_t tb_stack_workspace_bytes(const tb_block_cfg* cfg, int32_t B, int32_t T, int32_t mode) {
  const size_t blk = tb_workspace_bytes(cfg, B, T, mode);
  if (!blk) return 0;
  return align_up(blk, 256) + 2 * act_bytes(cfg, B, mode == 0 ? T : 1);
}

tb_status tb_stack_prefill(const tb_block_cfg* cfg, int32_t L, const void* const* packed, const void* x, void* y,
                           int32_t y_dtype, int32_t B, int32_t T, const tb_kvcache* kvs, void* ws, size_t ws_bytes,
                           void* stream) {
  if (L < 1 || !packed) return report(TB_ERR_INVALID_ARG, "L must be positive and packed non-NULL");
  const size_t need = tb_stack_workspace_bytes(cfg, B, T, 0);
  if (!need) return report(TB_ERR_INVALID_ARG, "invalid block configuration");
  if (!ws || ws_bytes < need) return report(TB_ERR_INVALID_ARG, "workspace too small: %zu < %zu", ws_bytes, need);
  const size_t blk = align_up(tb_workspace_bytes(cfg, B, T, 0), 256);
  char* act[2] = {(char*)ws + blk, (char*)ws + blk + act_bytes(cfg, B, T)};
  const void* cur = x;
  for (int l = 0; l < L; ++l) {
    const bool last = l == L - 1;
    void* out = last ? y : act[l & 1];
    const tb_status st = tb_block_prefill(cfg, packed[l], cur, out, last ? y_dtype : cfg->dtype, B, T,
                                          kvs ? &kvs[l] : nullptr, ws, blk, stream);
    if (st != TB_OK) return st;
    cur = out;
  }
  return TB_OK;
}

tb_status tb_stack_decode(const tb_block_cfg* cfg, int32_t L, const void* const* packed, const void* x, void* y,
                          int32_t y_dtype, const tb_kvcache* kvs, void* ws, size_t ws_bytes, void* stream) {
  if (L < 1 || !packed || !kvs) return report(TB_ERR_INVALID_ARG, "L must be positive; packed and kvs non-NULL");
  const int B = kvs[0].B, T_max = kvs[0].T_max;
  for (int l = 1; l < L; ++l)
    if (kvs[l].B != B || kvs[l].T_max != T_max)
      return report(TB_ERR_INVALID_ARG, "every layer's cache must have the same B and T_max");
  const size_t need = tb_stack_workspace_bytes(cfg, B, T_max, 1);
  if (!need) return report(TB_ERR_INVALID_ARG, "invalid block configuration");
  if (!ws || ws_bytes < need) return report(TB_ERR_INVALID_ARG, "workspace too small: %zu < %zu", ws_bytes, need);
  const size_t blk = align_up(tb_workspace_bytes(cfg, B, T_max, 1), 256);
  char* act[2] = {(char*)ws + blk, (char*)ws + blk + act_bytes(cfg, B, 1)};
  const void* cur = x;
  for (int l = 0; l < L; ++l) {
    const bool last = l == L - 1;
    void* out = last ? y : act[l & 1];
    const tb_status st =
        tb_block_decode(cfg, packed[l], cur, out, last ? y_dtype : cfg->dtype, &kvs[l], ws, blk, stream);
    if (st != TB_OK) return st;
    cur = out;
  }
  return TB_OK;
}

}  // extern "C"
