"""fp64 CPU oracle of one Llama-layout pre-norm decoder block (prefill and decode).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this module.  It shares no code with
the CUDA path and imports nothing from it.

The block is an exact definition, so this file writes the definition out, in
fp64, one step after another, with numpy's matmul as the only library
primitive.  It follows:

* "Transformer block" (tirogla.com), section "How it works": the dataflow
  diagram and steps 2-3 (RMSNorm, q/k/v projections, RoPE on q and k, causal
  softmax(q·kᵀ/√dh)·v per head, Wo and the residual add, RMSNorm, SwiGLU
  W2·(SiLU(x·W1) ⊙ x·W3) and the second residual add), the GQA paragraph
  (query head h reads KV head h / (H/Hkv)) and the KV-cache paragraph (the
  cache stores post-RoPE k and v; a decode step attends one new query over it).
* "Transformers" (engineering.msaqlain.com), sections 1.3 (scaled dot-product
  attention), 5.1 (causal mask keeps j ≤ i), 5.2 (KV cache) and 7 (the block
  end to end: h = x + MHA(RMSNorm(x)), y = h + FFN(RMSNorm(h))).
* "09 The Transformer" (infra.pidoku.co.in), the Go block: RMSNorm with eps
  inside the root, RoPE on adjacent pairs, SiLU(z) = z / (1 + e^-z).

Readings where the pages are silent or disagree (each is listed in the design
notes): weights are [in, out] (y = x·W); head h of q occupies columns
[h·dh, (h+1)·dh); RoPE rotates adjacent pairs (2i, 2i+1) by t·base^(-2i/dh) with
0-based positions; eps is added to the mean square inside the square root and
the gain multiplies after normalising.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Dict, Optional, Sequence

import numpy as np

F64 = np.float64


@dataclass(frozen=True)
class Cfg:
    """Block hyper-parameters in the pages' notation (B and T travel with x)."""
    d: int
    H: int
    Hkv: int
    dh: int
    f: int
    rope_base: float
    eps: float
    window: int = 0            # sliding-window width W; 0 is full causal attention

    def __post_init__(self):
        if self.H % self.Hkv:
            raise ValueError("H must be a multiple of Hkv")
        if self.window < 0:
            raise ValueError("window must be non-negative")
        if self.dh % 2:
            raise ValueError("RoPE rotates pairs: dh must be even")

    @property
    def G(self) -> int:
        return self.H // self.Hkv


def rms_norm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: x / sqrt(mean(x²) + eps) ⊙ g.

    Transformer block page, Rust ``rms_norm``; the Go block's ``rmsnorm`` uses
    the same form with eps 1e-6.
    """
    x = np.asarray(x, F64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(g, F64)


def rope_angles(positions: Sequence[int], dh: int, base: float) -> np.ndarray:
    """Angle t·base^(-2i/dh) for every position t and pair i < dh/2, shape [T, dh/2].

    Transformer block page, Rust ``rope``: pair i of a head turns by
    pos·10000^(-2i/dh) (the base is a parameter here).
    """
    i = np.arange(dh // 2, dtype=F64)
    inv_freq = np.power(F64(base), -2.0 * i / dh)
    return np.outer(np.asarray(positions, F64), inv_freq)


def rope(u: np.ndarray, positions: Sequence[int], base: float) -> np.ndarray:
    """Rotate adjacent pairs (2i, 2i+1) of every head of u [T, heads, dh].

    (a, b) -> (a·cos φ - b·sin φ, a·sin φ + b·cos φ) with φ = t·base^(-2i/dh)
    (Transformer block page, "interleaved RoPE"; "Transformers" section 3.2
    gives the 2×2 rotation matrix).
    """
    u = np.asarray(u, F64)
    phi = rope_angles(positions, u.shape[-1], base)[:, None, :]   # [T, 1, dh/2]
    c, s = np.cos(phi), np.sin(phi)
    a, b = u[..., 0::2], u[..., 1::2]
    out = np.empty_like(u)
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = a * s + b * c
    return out


def silu(z: np.ndarray) -> np.ndarray:
    """SiLU(z) = z / (1 + e^-z) (Transformer block page, Rust ``silu``)."""
    z = np.asarray(z, F64)
    return z / (1.0 + np.exp(-z))


def softmax_rows(s: np.ndarray) -> np.ndarray:
    """Row softmax with the row maximum subtracted first ("Transformers" 1.3;
    the Transformer block page's pitfall list warns against skipping the max)."""
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def visible_keys(q_pos: Sequence[int], S: int, window: int = 0) -> np.ndarray:
    """Mask [Tq, S]: key position j is visible to the query at position i.

    Causal: j ≤ i ("Transformers" 5.1).  With a sliding window W > 0 the
    query also drops every key older than its W most recent positions, its own
    included: j > i - W ("09 The Transformer" §5, sliding-window attention:
    with W = 4096, token 10000 attends to tokens 5905..10000).
    """
    j = np.arange(S)[None, :]
    i = np.asarray(q_pos)[:, None]
    mask = j <= i
    if window > 0:
        mask = mask & (j > i - window)
    return mask


def causal_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                     q_pos: Sequence[int], window: int = 0) -> np.ndarray:
    """Causal GQA scaled dot-product attention.

    q [Tq, H, dh] at positions q_pos; k, v [S, Hkv, dh] at positions 0..S-1.
    Query head h reads KV head h // (H/Hkv).  Query i sees the keys
    ``visible_keys`` allows (j ≤ q_pos[i], and within the window when
    window > 0); the others score -inf before the softmax.
    Returns o [Tq, H, dh].
    """
    q, k, v = (np.asarray(a, F64) for a in (q, k, v))
    Tq, H, dh = q.shape
    S, Hkv, _ = k.shape
    G = H // Hkv
    visible = visible_keys(q_pos, S, window)                     # [Tq, S]
    o = np.empty((Tq, H, dh), F64)
    for h in range(H):
        kv = h // G
        s = (q[:, h, :] @ k[:, kv, :].T) / math.sqrt(dh)       # [Tq, S]
        s = np.where(visible, s, -np.inf)
        p = softmax_rows(s)
        o[:, h, :] = p @ v[:, kv, :]
    return o


def qkv_heads(xn: np.ndarray, w: Dict[str, np.ndarray], cfg: Cfg, positions: Sequence[int]):
    """q, k, v of normalised tokens xn [T, d]: project, split heads, RoPE on q and k.

    Head h of q is column block [h·dh, (h+1)·dh) of xn·Wq; v is not rotated.
    Returns q [T, H, dh], k [T, Hkv, dh] (post-RoPE), v [T, Hkv, dh].
    """
    T = xn.shape[0]
    q = (xn @ w["wq"]).reshape(T, cfg.H, cfg.dh)
    k = (xn @ w["wk"]).reshape(T, cfg.Hkv, cfg.dh)
    v = (xn @ w["wv"]).reshape(T, cfg.Hkv, cfg.dh)
    return rope(q, positions, cfg.rope_base), rope(k, positions, cfg.rope_base), v


def mlp_branch(h: np.ndarray, w: Dict[str, np.ndarray], cfg: Cfg) -> np.ndarray:
    """y = h + W2·(SiLU(hn·W1) ⊙ hn·W3) with hn = RMSNorm(h) (second residual)."""
    hn = rms_norm(h, w["g_mlp"], cfg.eps)
    a = silu(hn @ w["w1"]) * (hn @ w["w3"])
    return h + a @ w["w2"]


def _f64_weights(w) -> Dict[str, np.ndarray]:
    return {n: np.asarray(a, F64) for n, a in w.items()}


def block_prefill_seq(x: np.ndarray, w, cfg: Cfg, rows: Optional[Sequence[int]] = None):
    """Full-sequence prefill of one sequence x [T, d].

    Returns dict(y [R, d], k [Hkv, S, dh], v [Hkv, S, dh]) where R are the
    requested rows (all T by default) and S = 1 + max(rows): causality means a
    row needs only the keys at or before it, so any subset of rows is exact
    (a sliding window only removes keys).
    """
    w = _f64_weights(w)
    x = np.asarray(x, F64)
    T = x.shape[0]
    rows = np.arange(T) if rows is None else np.asarray(sorted(set(int(r) for r in rows)))
    S = int(rows.max()) + 1
    xn = rms_norm(x[:S], w["g_attn"], cfg.eps)
    q, k, v = qkv_heads(xn, w, cfg, range(S))
    o = causal_attention(q[rows], k, v, rows, cfg.window).reshape(len(rows), cfg.H * cfg.dh)
    h = x[rows] + o @ w["wo"]
    y = mlp_branch(h, w, cfg)
    return {"y": y, "rows": rows, "k": k.transpose(1, 0, 2), "v": v.transpose(1, 0, 2)}


def block_prefill(x: np.ndarray, w, cfg: Cfg) -> Dict[str, np.ndarray]:
    """Prefill of a batch x [B, T, d]: y [B, T, d] and post-RoPE K/V [B, Hkv, T, dh]."""
    outs = [block_prefill_seq(x[b], w, cfg) for b in range(x.shape[0])]
    return {n: np.stack([o[n] for o in outs]) for n in ("y", "k", "v")}


def block_decode_seq(x: np.ndarray, w, cfg: Cfg, k_cache: np.ndarray, v_cache: np.ndarray,
                     pos: int) -> Dict[str, np.ndarray]:
    """One decode step of one sequence.

    x [d] is the new token at position ``pos``; k_cache, v_cache [Hkv, >=pos, dh]
    hold the post-RoPE keys and values of positions 0..pos-1.  The new token's
    k, v are rotated at ``pos`` and appended, and its query attends over the
    pos+1 keys (Transformer block page, KV-cache paragraph), the last
    cfg.window of them when a sliding window is set.  Returns
    dict(y [d], k [Hkv, dh], v [Hkv, dh]) with k, v the appended rows.
    """
    w = _f64_weights(w)
    x = np.asarray(x, F64)[None, :]
    xn = rms_norm(x, w["g_attn"], cfg.eps)
    q, k_new, v_new = qkv_heads(xn, w, cfg, [pos])
    k_all = np.concatenate([np.asarray(k_cache, F64)[:, :pos].transpose(1, 0, 2), k_new], axis=0)
    v_all = np.concatenate([np.asarray(v_cache, F64)[:, :pos].transpose(1, 0, 2), v_new], axis=0)
    o = causal_attention(q, k_all, v_all, [pos], cfg.window).reshape(1, cfg.H * cfg.dh)
    h = x + o @ w["wo"]
    y = mlp_branch(h, w, cfg)
    return {"y": y[0], "k": k_new[0], "v": v_new[0]}


def quantize_rows(x: np.ndarray):
    """Symmetric int8 quantisation of each row (last axis) with its own scale.

    "The Transformer Architecture" (thegeniusblogs), pitfalls, KV-cache OOM:
    the cache itself can be quantised to int8.  Here every cached row (one
    token of one KV head, dh values) gets the scale s = max|x| / 127 and codes
    q = round(x / s) in [-127, 127] (ties to even); a zero row has s = 0 and
    q = 0.  The pages fix no precision for this step, so the scale is an fp32
    number (the cache stores it as one) and the division and the rounding are
    done on the fp32 row: the decision of every code is an fp32 one.
    Returns (q int8 [..., dh], s [...] as float64 holding the fp32 values).
    """
    x32 = np.asarray(x, F64).astype(np.float32)
    s = np.max(np.abs(x32), axis=-1) / np.float32(127.0)
    safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    q = np.clip(np.rint(x32 / safe[..., None]), -127, 127)
    q = np.where(s[..., None] > 0, q, 0.0)
    return q.astype(np.int8), s.astype(F64)


def dequantize_rows(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """x̂ = q · s, row by row."""
    return np.asarray(q, F64) * np.asarray(s, F64)[..., None]


def block_decode_seq_int8(x: np.ndarray, w, cfg: Cfg, k_q: np.ndarray, k_s: np.ndarray, v_q: np.ndarray,
                          v_s: np.ndarray, pos: int) -> Dict[str, np.ndarray]:
    """One decode step over an int8 cache: rows 0..pos-1 of K and V stored as
    codes [Hkv, >=pos, dh] with scales [Hkv, >=pos].  The new token's k and v
    are quantised like every cached row before the query attends over all pos+1
    dequantised rows.  Returns dict(y, k_q, k_s, v_q, v_s) with the new row's
    codes and scales."""
    w = _f64_weights(w)
    x = np.asarray(x, F64)[None, :]
    xn = rms_norm(x, w["g_attn"], cfg.eps)
    q, k_new, v_new = qkv_heads(xn, w, cfg, [pos])
    kq, ks = quantize_rows(k_new[0])
    vq, vs = quantize_rows(v_new[0])
    k_all = np.concatenate([dequantize_rows(k_q[:, :pos], k_s[:, :pos]), dequantize_rows(kq, ks)[:, None, :]], axis=1)
    v_all = np.concatenate([dequantize_rows(v_q[:, :pos], v_s[:, :pos]), dequantize_rows(vq, vs)[:, None, :]], axis=1)
    o = causal_attention(q, k_all.transpose(1, 0, 2), v_all.transpose(1, 0, 2), [pos], cfg.window)
    h = x + o.reshape(1, cfg.H * cfg.dh) @ w["wo"]
    y = mlp_branch(h, w, cfg)
    return {"y": y[0], "k_q": kq, "k_s": ks, "v_q": vq, "v_s": vs}


def gather_paged(pool: np.ndarray, block_table: Sequence[int], page_size: int, n: int) -> np.ndarray:
    """Rows 0..n-1 of one sequence of a paged cache, as a contiguous [Hkv, n, dh].

    A paged cache allocates each sequence's cache in fixed-size blocks
    ("Transformer block" page, implementation notes: "paged KV cache" instead
    of one contiguous T_max buffer per request; "The Transformer
    Architecture", pitfalls, KV-cache OOM: paged attention fragments the cache
    into pages).  Here the pages sit in one pool [num_pages, Hkv, page_size, dh]
    and row t of the sequence lives in page block_table[t // page_size] at
    offset t % page_size.
    """
    pool = np.asarray(pool)
    Hkv, dh = pool.shape[1], pool.shape[3]
    out = np.empty((Hkv, n, dh), pool.dtype)
    for t in range(n):
        out[:, t, :] = pool[int(block_table[t // page_size]), :, t % page_size, :]
    return out


def block_decode(x: np.ndarray, w, cfg: Cfg, k_cache: np.ndarray, v_cache: np.ndarray,
                 lens: Sequence[int], batches: Optional[Sequence[int]] = None) -> Dict[str, np.ndarray]:
    """Decode step for x [B, 1, d] over caches [B, Hkv, T_max, dh] of lengths lens.

    Returns y [n, d], k [n, Hkv, dh], v [n, Hkv, dh] for the requested
    sequences (all by default)."""
    batches = range(x.shape[0]) if batches is None else batches
    outs = [block_decode_seq(x[b, 0], w, cfg, k_cache[b], v_cache[b], int(lens[b])) for b in batches]
    return {n: np.stack([o[n] for o in outs]) for n in ("y", "k", "v")}
