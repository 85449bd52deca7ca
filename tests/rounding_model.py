"""A CPU model of the bf16 path's rounding points (test infrastructure).

The block's bf16 path feeds the tensor cores bf16 operands and accumulates in
fp32.  Relative to the fp64 oracle on bf16-rounded inputs it therefore rounds,
to bf16: the gain-folded weights g⊙Wqkv and g⊙W1/W3, the post-RoPE q, k, v,
the softmax numerators P, the attention output o, the residual stream h fed
to W1/W3, and the SwiGLU output a ("Transformer block", tirogla.com,
implementation notes: softmax and norms in fp32, GEMMs in bf16 with fp32
accumulation).  This model repeats the block in fp32 with exactly those
roundings (plain torch CPU ops, no CUDA) so that a test can tell rounding
noise from a kernel error.

Two summation orders of the same model are provided:

* order "a": every GEMM as one fp32 matmul, the softmax over a row's whole
  key range with its true maximum;
* order "b": every GEMM summed sequentially over 64-wide K blocks, and the
  attention as the flash-style online softmax the "Transformers" page
  (engineering.msaqlain.com, section 6) describes: 128-key tiles in base 2,
  P rounded against the running maximum in use, which is raised only when a
  tile's maximum exceeds it by more than 2^8 (prefill), or per 256-key chunk
  merged by log-sum-exp (decode).

The bf16 roundings amplify fp32 summation noise: an fp32 value within noise of
a bf16 rounding boundary rounds the other way, and a flipped SwiGLU output
(|a| up to ~20 at d = 4096, a bf16 step of 0.06 there) moves y through W2.
The distance between orders "a" and "b" is this model's own noise floor; an
implementation with the same rounding points and some other valid order lands
within a small multiple of it, while an arithmetic mistake adds an error of
its own (``rounding_consistency``).

It shares no code with the CUDA library and is not an oracle: the oracle in
``oracle/`` is the definition; this is a model of one implementation's
rounding.  ``plant`` introduces a named mistake, so that the CPU tests can show
which errors the consistency check catches.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np
import torch

import workloads

ORDERS = ("a", "b", "c")
# Orders "b" and "c": (GEMM K-block width, K blocks summed last to first,
# prefill key tile, decode key chunk).  "c" is a third valid order the CPU
# tests use to show that the consistency check accepts another order.
ORDER_STEPS = {"b": (64, False, 128, 256), "c": (32, True, 64, 512)}
RESCALE_LOG2 = 8.0    # order "b": the running maximum moves only when exceeded by more than 2^8

# Mistakes the CPU tests plant to show what the consistency check detects.
PLANTS = ("r2_partial_row", "k_rope_pos_plus_1", "diag_key_dropped", "w2_block_dropped", "h_in_bf16",
          "wrong_kv_head")


def _bf(t: torch.Tensor) -> torch.Tensor:
    return t.to(torch.bfloat16).float()


def _mm(a: torch.Tensor, w: torch.Tensor, order: str, drop_block: Optional[int] = None) -> torch.Tensor:
    """fp32 a·w; orders "b" and "c" accumulate K blocks one after another."""
    if order == "a" and drop_block is None:
        return a @ w
    kb, rev = ORDER_STEPS[order][:2] if order != "a" else (64, False)
    starts = list(range(0, a.shape[1], kb))
    acc = torch.zeros(a.shape[0], w.shape[1])
    for i in (reversed(range(len(starts))) if rev else range(len(starts))):
        if i == drop_block:
            continue
        k = starts[i]
        acc = acc + a[:, k:k + kb] @ w[k:k + kb]
    return acc


def _rope(u: torch.Tensor, pos: torch.Tensor, dh: int, base: float) -> torch.Tensor:
    """Adjacent pairs (2i, 2i+1) rotated by pos·base^(-2i/dh); the angles in fp64,
    cos and sin stored fp32 (a table), the rotation in fp32.  u [n, heads, dh]."""
    i = torch.arange(dh // 2, dtype=torch.float64)
    ang = torch.outer(pos.to(torch.float64), base ** (-2 * i / dh))
    c, sn = torch.cos(ang).float()[:, None], torch.sin(ang).float()[:, None]
    a, b = u[..., 0::2], u[..., 1::2]
    out = torch.empty_like(u)
    out[..., 0::2] = a * c - b * sn
    out[..., 1::2] = a * sn + b * c
    return out


def _attend_whole(q, k, v, q_pos, dh):
    """One head: softmax over each row's visible keys with the row's true maximum;
    P rounded to bf16, l summed from the unrounded weights.  q [R, dh] at q_pos,
    k, v [S, dh] at positions 0..S-1."""
    S = (q @ k.T) / math.sqrt(dh)
    keep = torch.arange(k.shape[0])[None, :] <= q_pos[:, None]
    S = S.masked_fill(~keep, float("-inf"))
    P = torch.exp(S - S.max(-1, keepdim=True).values)
    return (_bf(P) @ v) / P.sum(-1, keepdim=True)


def _attend_tiles(q, k, v, q_pos, dh, tile):
    """One head, online softmax in base 2 over key tiles of ``tile`` keys: a row
    starts with its first tile's maximum and keeps the maximum in use until a
    tile exceeds it by more than 2^RESCALE_LOG2, rescaling O and l then; P =
    2^(s·log2e/√dh − m) is rounded to bf16 for the P·V product.  Every row sees
    key 0, so every row starts at the first tile."""
    scale_log2 = math.log2(math.e) / math.sqrt(dh)
    S_all = q @ k.T
    l = torch.zeros(q.shape[0])
    O = torch.zeros(q.shape[0], v.shape[1])
    for j0 in range(0, k.shape[0], tile):
        if not bool((q_pos >= j0).any()):
            break
        cols = torch.arange(j0, min(j0 + tile, k.shape[0]))
        s = S_all[:, cols].masked_fill(cols[None, :] > q_pos[:, None], float("-inf"))
        mx = s.max(-1).values * scale_log2
        if j0 == 0:
            m = mx
        else:
            m_new = torch.maximum(m, mx)
            need = m_new > m + RESCALE_LOG2
            fac = torch.where(need, torch.exp2(m - m_new), torch.ones_like(m))
            O = O * fac[:, None]
            l = l * fac
            m = torch.where(need, m_new, m)
        p = torch.exp2(s * scale_log2 - m[:, None])
        l = l + p.sum(-1)
        O = O + _bf(p) @ v[cols]
    return O / l[:, None]


def _attend_chunks(q, k, v, dh, chunk):
    """One head, one query over all keys: per-chunk maxima and partial sums,
    merged by log-sum-exp (the split-K reformulation of the same softmax)."""
    scale_log2 = math.log2(math.e) / math.sqrt(dh)
    s = (q @ k.T)[0] * scale_log2
    parts = []
    for c0 in range(0, k.shape[0], chunk):
        sc = s[c0:c0 + chunk]
        mc = sc.max()
        p = torch.exp2(sc - mc)
        parts.append((mc, p.sum(), _bf(p)[None, :] @ v[c0:c0 + chunk]))
    M = max(float(pm) for pm, _, _ in parts)
    num = sum(torch.exp2(pm - M) * o for pm, _, o in parts)
    den = sum(torch.exp2(pm - M) * pl for pm, pl, _ in parts)
    return num / den


def _block_rows(inp, s: workloads.BlockShape, x: torch.Tensor, pos: torch.Tensor, kv_rows, order: str,
                plant: Optional[str], decode: bool = False, with_kv: bool = False):
    """The block for tokens x [n, d] at positions pos.  kv_rows(k_new, v_new)
    returns the keys and values [S, Hkv, dh] they attend over and each query's
    key-position limit; returns y [n, d] (fp32), and with with_kv also the
    new rows' k and v [n, Hkv, dh] as stored (bf16 values)."""
    if plant is not None and plant not in PLANTS:
        raise ValueError(plant)
    w = {nm: inp[nm].float() for nm in workloads.WEIGHT_NAMES}
    H, Hkv, dh = s.H, s.Hkv, s.dh
    n = x.shape[0]
    r = 1.0 / torch.sqrt((x * x).mean(-1, keepdim=True) + s.eps)
    wqkv = torch.cat([w["wq"], w["wk"], w["wv"]], 1)
    acc = r * _mm(x, _bf(w["g_attn"][:, None] * wqkv), order)
    q = _bf(_rope(acc[:, :H * dh].reshape(n, H, dh), pos, dh, s.rope_base))
    kpos = pos + 1 if plant == "k_rope_pos_plus_1" else pos
    k_new = _bf(_rope(acc[:, H * dh:(H + Hkv) * dh].reshape(n, Hkv, dh), kpos, dh, s.rope_base))
    v_new = _bf(acc[:, (H + Hkv) * dh:].reshape(n, Hkv, dh))
    k, v, lim = kv_rows(k_new, v_new)
    if plant == "diag_key_dropped":
        lim = torch.where(lim > 0, lim - 1, lim)
    G = H // Hkv
    o = torch.empty(n, H, dh)
    for h in range(H):
        kvh = h // G
        if plant == "wrong_kv_head" and h == H - 1:
            kvh = (kvh + 1) % Hkv if Hkv > 1 else kvh
        qh, kh, vh = q[:, h], k[:, kvh], v[:, kvh]
        if order == "a":
            o[:, h] = _attend_whole(qh, kh, vh, lim, dh)
        elif decode:
            o[:, h] = _attend_chunks(qh, kh, vh, dh, ORDER_STEPS[order][3])
        else:
            o[:, h] = _attend_tiles(qh, kh, vh, lim, dh, ORDER_STEPS[order][2])
    hh = x + _mm(_bf(o.reshape(n, H * dh)), w["wo"], order)
    if plant == "h_in_bf16":
        hh = _bf(hh)
    hs = hh[:, :s.d - 16] if plant == "r2_partial_row" else hh      # last 16 columns left out of Σh²
    r2 = 1.0 / torch.sqrt((hs * hs).sum(-1, keepdim=True) / s.d + s.eps)
    hb = _bf(hh)
    g = r2 * _mm(hb, _bf(w["g_mlp"][:, None] * w["w1"]), order)
    u = r2 * _mm(hb, _bf(w["g_mlp"][:, None] * w["w3"]), order)
    a = _bf(g / (1.0 + torch.exp(-g)) * u)
    drop = s.f // 64 // 2 if plant == "w2_block_dropped" else None
    y = hh + _mm(a, w["w2"], order, drop_block=drop)
    return (y, k_new, v_new) if with_kv else y


def emulate_prefill_seq(inp, s: workloads.BlockShape, b: int = 0, order: str = "a",
                        plant: Optional[str] = None) -> torch.Tensor:
    """fp32 prefill of sequence b of inp["x"] with the bf16 path's rounding
    points, in summation order ``order``; y [T, d].  By causality the rows of a
    prefix of x are the first rows of the whole sequence's result."""
    x = inp["x"][b].float()
    T = x.shape[0]
    pos = torch.arange(T)
    return _block_rows(inp, s, x, pos, lambda kn, vn: (kn, vn, pos), order, plant)


def emulate_decode_seq(inp, s: workloads.BlockShape, b: int, k_cache: torch.Tensor, v_cache: torch.Tensor,
                       order: str = "a", plant: Optional[str] = None) -> torch.Tensor:
    """One decode step of sequence b: x = inp["x"][b, 0] at position
    pos = k_cache.shape[1], attending over the cached post-RoPE rows
    k_cache, v_cache [Hkv, pos, dh] (stored values) and its own k, v; y [d]."""
    x = inp["x"][b, :1].float()
    P = k_cache.shape[1]
    kc = k_cache.float().permute(1, 0, 2)
    vc = v_cache.float().permute(1, 0, 2)

    def kv_rows(kn, vn):
        return torch.cat([kc, kn]), torch.cat([vc, vn]), torch.tensor([P])

    return _block_rows(inp, s, x, torch.tensor([P]), kv_rows, order, plant, decode=True)[0]


def emulate_stack_prefill_seq(ids, table: torch.Tensor, layers, s: workloads.BlockShape, g_final: torch.Tensor,
                              order: str = "a"):
    """One sequence through an L-layer stack with the bf16 path's rounding
    points, and the tied LM head: each block's input stored in bf16, the
    head's input (the last block's output) in bf16, the final norm's gain
    folded into the bf16 head weights, the logits (x·W_U')·r in fp32.
    ids [T]; table [V, d] (the embedding, also W_Uᵀ); layers: per-layer dicts
    of weights.  Returns dict(logits [T, V], k, v: per layer [Hkv, T, dh])."""
    x = table[torch.as_tensor(ids, dtype=torch.long)].float()
    pos = torch.arange(x.shape[0])
    ks, vs = [], []
    for lw in layers:
        x = _bf(x)
        y, k, v = _block_rows(lw, s, x, pos, lambda kn, vn: (kn, vn, pos), order, None, with_kv=True)
        ks.append(k.permute(1, 0, 2))
        vs.append(v.permute(1, 0, 2))
        x = y
    h = _bf(x)
    r = 1.0 / torch.sqrt((h * h).mean(-1, keepdim=True) + s.eps)
    wu = _bf(table.float() * g_final.float()[None, :])          # [V, d]
    return {"logits": r * _mm(h, wu.T.contiguous(), order), "k": ks, "v": vs}


def emulate_stack_decode_seq(token: int, table: torch.Tensor, layers, s: workloads.BlockShape,
                             g_final: torch.Tensor, k_caches, v_caches, order: str = "a"):
    """One decode step of one sequence through the stack (the token at
    position pos = k_caches[l].shape[1]), each layer over its cached rows
    [Hkv, pos, dh]; the head as in emulate_stack_prefill_seq.  Returns
    dict(logits [V], k: per layer the appended row [Hkv, dh])."""
    x = table[token].float()[None, :]
    P = k_caches[0].shape[1]
    ks = []
    for lw, kc, vc in zip(layers, k_caches, v_caches):
        x = _bf(x)
        kcp, vcp = kc.float().permute(1, 0, 2), vc.float().permute(1, 0, 2)
        x, k, _ = _block_rows(lw, s, x, torch.tensor([P]),
                              lambda kn, vn: (torch.cat([kcp, kn]), torch.cat([vcp, vn]), torch.tensor([P])), order,
                              None, decode=True, with_kv=True)
        ks.append(k[0])
    h = _bf(x)
    r = 1.0 / torch.sqrt((h * h).mean(-1, keepdim=True) + s.eps)
    wu = _bf(table.float() * g_final.float()[None, :])
    return {"logits": (r * _mm(h, wu.T.contiguous(), order))[0], "k": ks}


def _err(got, ref):
    d = np.asarray(got, np.float64) - np.asarray(ref, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.max(np.abs(d))), float(np.linalg.norm(d) / np.linalg.norm(ref))


# The consistency bars.  A result with the model's rounding points and another
# valid summation order stays within NOISE_FACTOR of the model's own order-to-
# order distance, and its error against the oracle within ERROR_FACTOR of the
# model's.
NOISE_FACTOR = 1.5
ERROR_FACTOR = 1.25


def rounding_consistency(got, emu_a, emu_b, ref) -> dict:
    """Compare a result ``got`` with the model in orders a and b and the
    oracle ``ref`` (arrays of the same rows).  Returns the distances and
    whether ``got`` is consistent with rounding noise:
      |got − emu_a| ≤ NOISE_FACTOR·|emu_b − emu_a|   (max-abs and relative L2)
      |got − ref|   ≤ ERROR_FACTOR·|emu_a − ref|      (max-abs and relative L2)."""
    noise = _err(emu_b, emu_a)
    dev = _err(got, emu_a)
    model = _err(emu_a, ref)
    err = _err(got, ref)
    ok_noise = dev[0] <= NOISE_FACTOR * noise[0] and dev[1] <= NOISE_FACTOR * noise[1]
    ok_err = err[0] <= ERROR_FACTOR * model[0] and err[1] <= ERROR_FACTOR * model[1]
    return {"noise": noise, "dev": dev, "model": model, "err": err, "ok_noise": ok_noise, "ok_err": ok_err,
            "ok": ok_noise and ok_err}
