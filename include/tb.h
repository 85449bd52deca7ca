/*
 * tb.h — C ABI of the GB300 (sm_103a) Llama-layout pre-norm decoder block.
 *
 * One block forward pass, as the "Transformer block" page (tirogla.com,
 * section "How it works": dataflow diagram and steps 2-3) defines it:
 *
 *   h = x + Wo · concat_h softmax(q_h·k_{h/G}ᵀ/√dh + causal) · v_{h/G}
 *       with q, k, v = RMSNorm(x)·Wq, ·Wk, ·Wv and RoPE on q and k
 *   y = h + W2 · (SiLU(hn·W1) ⊙ hn·W3),   hn = RMSNorm(h)
 *
 * in two modes: full-sequence prefill, and one decode step over a KV cache of
 * post-RoPE keys and values [B, Hkv, T_max, dh] (same page, KV-cache paragraph;
 * "Transformers", engineering.msaqlain.com, section 5.2).  Notation follows the
 * pages: B batch, T sequence, d width, H query heads, Hkv KV heads (G = H/Hkv
 * query heads share one KV head), dh = d/H head width, f MLP width.
 *
 * Conventions for every entry point:
 *  - Pointers marked "device" are CUDA device pointers on the current device;
 *    "host" pointers are ordinary host memory.  The caller owns every buffer;
 *    the library allocates no device memory.
 *  - Every call is asynchronous on `stream` (a cudaStream_t, NULL = legacy
 *    default stream) except tb_get_device_error, which synchronises it.
 *  - Arguments are checked on the host before anything is launched.  A bad
 *    argument returns TB_ERR_INVALID_ARG (or TB_ERR_UNSUPPORTED for a valid
 *    but unimplemented shape) and launches nothing; tb_last_error_message()
 *    then says which argument.
 *  - Conditions only the device can see (a sequence whose cache is full) set
 *    a bit in a per-device error word, skip the affected rows and never trap;
 *    tb_get_device_error reads it.  No kernel waits without a time limit: a
 *    wait that runs out sets TB_DEVERR_TIMEOUT and the kernel returns.
 *  - Row-major layouts throughout; weights are [in, out] (y = x·W), as in the
 *    "Transformer block" page's Rust block.
 */
#ifndef TB_H_
#define TB_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TB_API __attribute__((visibility("default")))
#else
#define TB_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TB_OK = 0,
  TB_ERR_INVALID_ARG = 1,   /* a null/misaligned pointer, inconsistent shape, too small a buffer */
  TB_ERR_UNSUPPORTED = 2,   /* a valid shape the library has no kernel for */
  TB_ERR_CUDA = 3,          /* a CUDA runtime or driver call failed */
  TB_ERR_CACHE_FULL = 4,    /* host-visible cache overflow (append of n rows past T_max) */
  TB_ERR_TIMEOUT = 5        /* reserved for a host-side wait that ran out */
} tb_status;

/* TB_I8 is a KV-cache storage type only (tb_kvcache.dtype): int8 codes with a
 * per-row fp32 scale. */
typedef enum { TB_F32 = 0, TB_BF16 = 1, TB_I8 = 2 } tb_dtype;

/* Bits of the device error word (tb_get_device_error). */
#define TB_DEVERR_CACHE_FULL 1  /* a decode/append row found lens[b] + n > T_max; that row was skipped */
#define TB_DEVERR_TIMEOUT    2  /* a kernel's bounded wait ran out; its output is not valid */
#define TB_DEVERR_BAD_PAGE   4  /* a paged cache's block table held a page id outside [0, num_pages) */
#define TB_DEVERR_BAD_TOKEN  8  /* an embedding or loss token id outside [0, V); its row is zero / NaN */

/* Block hyper-parameters.
 *  d, H, Hkv, dh, f : widths in the pages' notation; H·dh must equal d, H a
 *                     multiple of Hkv, dh even (RoPE rotates pairs).
 *  max_pos          : number of positions the packed RoPE table covers
 *                     (prefill T and every decode position must be below it).
 *  rope_base        : RoPE base; pair i of a head turns by t·base^(-2i/dh)
 *                     at 0-based position t ("Transformer block" page, RoPE).
 *  eps              : RMSNorm eps, added to the mean square inside the root.
 *  dtype            : tb_dtype of x, the weights, the gains and the KV cache.
 *                     TB_BF16 computes with bf16 tensor-core operands, fp32
 *                     accumulation, fp32 softmax and norms; TB_F32 computes in
 *                     fp32 throughout.
 *  window           : sliding-window width W.  0: full causal attention (key j
 *                     visible to query i iff j <= i).  W > 0: key j visible iff
 *                     i - W < j <= i, the query's W most recent positions, its
 *                     own included ("09 The Transformer" §5, sliding-window
 *                     attention: with W = 4096 token 10000 attends to tokens
 *                     5905..10000).  Negative values are TB_ERR_INVALID_ARG.
 *                     The cache stays indexed by position; a decode step reads
 *                     only its W most recent rows. */
typedef struct {
  int32_t d, H, Hkv, dh, f;
  int32_t max_pos;
  float rope_base;
  float eps;
  int32_t dtype;
  int32_t window;
} tb_block_cfg;

/* Unpacked weights, device pointers of cfg.dtype, [in, out] row-major:
 *  g_attn [d], wq [d, H·dh], wk [d, Hkv·dh], wv [d, Hkv·dh], wo [H·dh, d],
 *  g_mlp [d], w1 [d, f] (gate), w3 [d, f] (up), w2 [f, d].
 * Head h of q is column block [h·dh, (h+1)·dh) of x·Wq (likewise k, v). */
typedef struct {
  const void *g_attn, *wq, *wk, *wv, *wo, *g_mlp, *w1, *w3, *w2;
} tb_block_weights;

/* KV cache of post-RoPE keys and values, in one of four layouts.
 *  Contiguous (block_table == NULL, dtype == cfg.dtype):
 *    k, v  : device, cfg.dtype, [B, Hkv, T_max, dh] each, row-major.
 *  Paged (block_table != NULL), the cache allocated per sequence in fixed-size
 *  blocks ("Transformer block" page, implementation notes: paged KV cache):
 *    k, v        : device, cfg.dtype, page pools [num_pages, Hkv, page_size, dh].
 *    block_table : device int32 [B, T_max / page_size]; row t of sequence b
 *                  lives in page block_table[b·(T_max/page_size) + t/page_size]
 *                  at offset t % page_size.  Entries are caller-owned page ids
 *                  in [0, num_pages); a kernel that meets one outside that
 *                  range writes nothing through it and sets TB_DEVERR_BAD_PAGE.
 *    page_size   : a multiple of 16 that divides T_max.
 *  int8 (dtype == TB_I8, block_table == NULL), the cache quantised to int8
 *  ("The Transformer Architecture", thegeniusblogs, pitfalls: KV-cache OOM):
 *    k, v              : device int8 codes [B, Hkv, T_max, dh], row-major.
 *    k_scale, v_scale  : device fp32 [B, Hkv, T_max], one scale per row.
 *    Row x (one token of one KV head) is stored as s = max|x| / 127 and codes
 *    q = round-half-even(x / s) clamped to [-127, 127], s and x / s evaluated
 *    in fp32 (a zero row: s = 0, q = 0); it reads back as q·s.  Only a bf16
 *    block with dh = 128 and T_max a multiple of 32 takes an int8 cache.
 *  Paged int8 (dtype == TB_I8, block_table != NULL): the int8 layout in page
 *  pools, k, v codes [num_pages, Hkv, page_size, dh] and k_scale, v_scale
 *  [num_pages, Hkv, page_size], with the paged layout's block table and
 *  page_size a multiple of 32.
 *    Prefill attends over the unquantised rows and stores their codes; a
 *    decode step stores the new token's codes first, then attends over the
 *    dequantised rows, its own included.
 *  lens  : device int32 [B], the number of valid rows of each sequence.
 * Rows at or beyond lens[b] are never read.  k_scale and v_scale are ignored
 * unless dtype == TB_I8. */
typedef struct {
  void *k, *v;
  int32_t *lens;
  int32_t B, Hkv, T_max, dh;
  int32_t dtype;
  const int32_t *block_table;
  int32_t page_size, num_pages;
  float *k_scale, *v_scale;
} tb_kvcache;

/* Bytes the packed weight blob of tb_pack_weights needs. */
TB_API size_t tb_packed_weights_bytes(const tb_block_cfg *cfg);

/* Pack a weight set once for the kernels: the RMSNorm gains are folded into
 * the rows of the input dimension (RMSNorm(x)·W = r·(x·(diag(g)·W)), r the
 * per-token inverse RMS, so the norm becomes a per-row scale in the GEMM
 * epilogue), the matrices are stored transposed ([out, in], reduction axis
 * contiguous) with Wq|Wk|Wv fused and W1/W3 interleaved column by column
 * (the fused GEMMs of the "Transformer block" page's implementation notes),
 * and a [max_pos, dh/2] cos/sin table is built in fp64 and stored in fp32
 * (the same notes suggest precomputing it).
 *  w      : unpacked weights (device).
 *  packed : device, at least tb_packed_weights_bytes(cfg) bytes, 256-B aligned.
 * The packed blob depends only on cfg and w; it is read-only afterwards. */
TB_API tb_status tb_pack_weights(const tb_block_cfg *cfg, const tb_block_weights *w,
                          void *packed, size_t packed_bytes, void *stream);

/* Workspace bytes a call needs: mode 0 = prefill of B×T tokens (with K/V kept
 * in the workspace when no cache is passed, which is the larger case), mode 1
 * = decode of B sequences whose cache holds up to T positions (T = T_max). */
TB_API size_t tb_workspace_bytes(const tb_block_cfg *cfg, int32_t B, int32_t T, int32_t mode);

/* Full-sequence prefill of B sequences of T tokens.
 *  packed  : device blob from tb_pack_weights for this cfg.
 *  x       : device [B, T, d] cfg.dtype.
 *  y       : device [B, T, d] y_dtype (TB_F32, or TB_BF16 when cfg.dtype is
 *            TB_BF16).  y may not alias x.
 *  kv      : NULL, or a cache with kv->B == B, T ≤ kv->T_max: its rows [0, T)
 *            receive the post-RoPE K and V of every position and lens[b] is
 *            set to T.
 *  ws      : device workspace of ws_bytes ≥ tb_workspace_bytes(cfg, B, T, 0).
 * B == 0 or T == 0 is an empty call that returns TB_OK. */
TB_API tb_status tb_block_prefill(const tb_block_cfg *cfg, const void *packed, const void *x, void *y,
                           int32_t y_dtype, int32_t B, int32_t T, const tb_kvcache *kv,
                           void *ws, size_t ws_bytes, void *stream);

/* One decode step of kv->B sequences.  Token b sits at position p = lens[b]:
 * its k and v are rotated at p and written to cache row p, its query attends
 * over rows 0..p, and lens[b] becomes p + 1.
 *  x  : device [B, 1, d] cfg.dtype;  y : device [B, 1, d] y_dtype.
 *  kv : required; kv->T_max ≤ cfg->max_pos.
 *  ws : device workspace of ws_bytes ≥ tb_workspace_bytes(cfg, B, kv->T_max, 1).
 * A sequence with lens[b] ≥ T_max sets TB_DEVERR_CACHE_FULL, keeps its cache
 * and length unchanged, and gets an unspecified y row.  A bf16 block decodes
 * at most 2048 sequences per call (TB_ERR_UNSUPPORTED above that). */
TB_API tb_status tb_block_decode(const tb_block_cfg *cfg, const void *packed, const void *x, void *y,
                          int32_t y_dtype, const tb_kvcache *kv, void *ws, size_t ws_bytes,
                          void *stream);

/* tb_block_decode for callers that cannot allocate device memory.  The pages
 * have no counterpart to this entry point; it exists for callers that must
 * not call cudaMalloc or a framework allocator on their hot path (allocation
 * can synchronise the device and take unbounded time), plugins whose host
 * framework hands out no device memory, and runtimes without a device
 * allocator.  It runs exactly tb_block_decode with the workspace taken from a
 * file-scope device array of 64 MiB (enough for 32 sequences, a 16384-row
 * cache, d = 4096, f = 14336) that every GPU loading the library holds until
 * the process exits; the call allocates nothing.
 *  Arguments and behaviour are those of tb_block_decode minus ws/ws_bytes.
 *  A step whose tb_workspace_bytes(cfg, kv->B, kv->T_max, 1) exceeds 64 MiB
 *  returns TB_ERR_INVALID_ARG and launches nothing.
 *  The first call on each device looks up the array's device address
 *  (cudaGetSymbolAddress) with that device current; make that first call
 *  before any stream capture.  The address is kept for the life of the
 *  process, so a device reset (cudaDeviceReset) after the first call on that
 *  device is not supported: the module is reloaded and the array may move.
 *  All calls share the one array and its contents persist between calls (the
 *  step zeroes what it accumulates into), so calls that may overlap on the
 *  GPU — on different streams, or from different threads — race; serialise
 *  them, e.g. on one stream. */
TB_API tb_status tb_block_decode_noalloc(const tb_block_cfg *cfg, const void *packed, const void *x, void *y,
                                         int32_t y_dtype, const tb_kvcache *kv, void *stream);

/* Append n post-RoPE rows per sequence: k_new, v_new are device
 * [B, Hkv, n, dh] of kv->dtype (bf16 for an int8 cache, whose rows are
 * quantised as they are stored); rows go to [lens[b], lens[b]+n) and lens[b]
 * grows by n.  A sequence with lens[b] + n > T_max sets TB_DEVERR_CACHE_FULL
 * and is left unchanged.  n == 0 is a no-op. */
TB_API tb_status tb_kvcache_append(const tb_kvcache *kv, const void *k_new, const void *v_new, int32_t n,
                            void *stream);

/* Synchronise `stream` and read the current device's error word (TB_DEVERR_*
 * bits, 0 = none) into *err_out; `clear` != 0 resets it to 0. */
TB_API tb_status tb_get_device_error(void *stream, int32_t *err_out, int32_t clear);

/* Short text for a status code (static storage). */
TB_API const char *tb_status_string(tb_status s);

/* Detail of the last non-OK status returned on the calling thread. */
TB_API const char *tb_last_error_message(void);

/* ---- Around the block: embedding, an L-layer stack, final norm and LM head ----
 * "Transformer block" page (tirogla.com), "How it works": (1) token ids index an
 * embedding table [V, d]; the blocks run in order; (4) after the last block a
 * final RMSNorm, then logits = h·W_U with W_U [d, V], possibly tied to the
 * embedding table.  "The Transformer" (GenerativeAIDocs) §5, "Step 18 is a
 * memory trap": full [B, T, V] fp32 logits are large, so the head works in row
 * chunks and can return the per-token loss without materialising them. */

/* x[t] = table[ids[t]] for t < n.  table: device [V, d] of dtype; ids: device
 * int32 [n]; x: device [n, d] of dtype (16-byte aligned, d·sizeof a multiple of
 * 16).  An id outside [0, V) gives a zero row and sets TB_DEVERR_BAD_TOKEN. */
TB_API tb_status tb_embed(const void *table, int32_t V, int32_t d, int32_t dtype, const int32_t *ids, int64_t n,
                          void *x, void *stream);

/* LM head hyper-parameters: width d, vocabulary V (a multiple of 4), the final
 * RMSNorm's eps, and dtype (of x, the weights and the gain).  The bf16 path
 * needs d a multiple of 64. */
typedef struct {
  int32_t d, V;
  float eps;
  int32_t dtype;
} tb_head_cfg;

/* Packed head: W_U transposed to [V, d] with the final norm's gain g_final [d]
 * folded into its columns.  w_u: device [d, V] ([in, out], like the block's
 * weights), or with tied != 0 the embedding table [V, d] (W_U = tableᵀ). */
TB_API size_t tb_lm_head_packed_bytes(const tb_head_cfg *cfg);
TB_API tb_status tb_pack_lm_head(const tb_head_cfg *cfg, const void *g_final, const void *w_u, int32_t tied,
                                 void *packed, size_t packed_bytes, void *stream);

/* Workspace of tb_lm_head for chunks of row_chunk rows (0: 4096). */
TB_API size_t tb_lm_head_workspace_bytes(const tb_head_cfg *cfg, int32_t row_chunk);

/* Head over M rows x [M, d] (device, cfg dtype): per row r = RMSNorm scale,
 * logits = (x·r)·packedᵀ in fp32.  logits (device [M, V], or NULL) receives
 * them; with targets (device int32 [M]) and nll (device fp32 [M]) non-NULL,
 * nll[m] = logsumexp(logits[m]) - logits[m, targets[m]].  Rows are processed
 * row_chunk at a time.  With logits NULL a bf16 head folds the loss into its
 * GEMM's epilogue (a running max and Σ exp per row and 256-column tile, merged
 * per row) and never forms the logits; chunks of at most 64 rows and the fp32
 * head form one chunk of logits in ws.  A target outside [0, V) gives NaN and
 * sets TB_DEVERR_BAD_TOKEN. */
TB_API tb_status tb_lm_head(const tb_head_cfg *cfg, const void *packed, const void *x, int32_t M, float *logits,
                            const int32_t *targets, float *nll, int32_t row_chunk, void *ws, size_t ws_bytes,
                            void *stream);

/* An L-layer stack of blocks of one configuration.  packed: host array of L
 * device pointers (each a tb_pack_weights blob).  Prefill: x [B, T, d] in
 * cfg.dtype -> y [B, T, d] in y_dtype; kvs: NULL or a host array of L caches
 * (layer l's cache receives layer l's keys and values).  Decode: x [B, 1, d],
 * kvs required (all at the same lens).  Between layers the residual stream is
 * stored in cfg.dtype (each block's input type).  The workspace holds one
 * block's workspace and two activation buffers. */
TB_API size_t tb_stack_workspace_bytes(const tb_block_cfg *cfg, int32_t B, int32_t T, int32_t mode);
TB_API tb_status tb_stack_prefill(const tb_block_cfg *cfg, int32_t L, const void *const *packed, const void *x,
                                  void *y, int32_t y_dtype, int32_t B, int32_t T, const tb_kvcache *kvs, void *ws,
                                  size_t ws_bytes, void *stream);
TB_API tb_status tb_stack_decode(const tb_block_cfg *cfg, int32_t L, const void *const *packed, const void *x,
                                 void *y, int32_t y_dtype, const tb_kvcache *kvs, void *ws, size_t ws_bytes,
                                 void *stream);

#ifdef __cplusplus
}
#endif
#endif /* TB_H_ */
