"""fp64 CPU oracle of the steps either side of the block: token embedding, an
L-layer stack of blocks, the final norm and the LM head.

TEST INFRASTRUCTURE, like the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU baseline of ``bench.py`` may import it.

It follows "Transformer block" (tirogla.com), "How it works", steps 1 and 4:
token ids [B, T] index an embedding table [V, d] (position enters only through
RoPE inside attention); after the last block a final RMSNorm, then logits =
h·W_U with W_U [d, V], which may be tied to the embedding table (W_U = Eᵀ).
The Go listing on "09 The Transformer" (infra.pidoku.co.in) §4 "Tiny example"
runs the same forward pass: embed, every block in order, then the head on the
final norm.  "The Transformer" (GenerativeAIDocs) §5 "A tensor's journey",
"Step 18 is a memory trap", and the pitfalls after it: the loss is computed in
chunks of tokens so that the full [B, T, V] fp32 logits never exist;
``token_nll`` is the per-token loss such a chunked head returns.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import numpy as np

from .block import Cfg, F64, block_decode_seq, block_prefill_seq, rms_norm


def embed(table: np.ndarray, ids: Sequence[int]) -> np.ndarray:
    """x[t] = table[ids[t]]: [len(ids), d]."""
    table = np.asarray(table, F64)
    return table[np.asarray(ids, dtype=np.int64)]


def lm_head(h: np.ndarray, g_final: np.ndarray, w_u: np.ndarray, eps: float) -> np.ndarray:
    """logits = RMSNorm(h; g_final, eps)·W_U: [T, V] for h [T, d], W_U [d, V]."""
    return rms_norm(h, g_final, eps) @ np.asarray(w_u, F64)


def token_nll(logits: np.ndarray, targets: Sequence[int]) -> np.ndarray:
    """-log softmax(logits[t])[targets[t]] = logsumexp(logits[t]) - logits[t, targets[t]],
    with the row maximum subtracted before the exponentials."""
    z = np.asarray(logits, F64)
    m = np.max(z, axis=-1, keepdims=True)
    lse = m[:, 0] + np.log(np.sum(np.exp(z - m), axis=-1))
    return lse - z[np.arange(z.shape[0]), np.asarray(targets, dtype=np.int64)]


def stack_prefill_seq(ids: Sequence[int], table: np.ndarray, layers: List[Dict[str, np.ndarray]], cfg: Cfg,
                      g_final: np.ndarray, w_u: np.ndarray, round_between=None) -> Dict[str, object]:
    """Prefill of one sequence through the whole stack.

    Returns dict(h [T, d] after the last block, logits [T, V], k / v: the
    post-RoPE cache of every layer, [L][Hkv, T, dh]).  ``round_between``, if
    given, is applied to the residual stream between blocks (the input of block
    l+1 is stored in the block's storage type); None keeps fp64 throughout.
    """
    x = embed(table, ids)
    ks, vs = [], []
    for lw in layers:
        if round_between is not None:
            x = round_between(x)
        out = block_prefill_seq(x, lw, cfg)
        ks.append(out["k"])
        vs.append(out["v"])
        x = out["y"]
    return {"h": x, "logits": lm_head(x, g_final, w_u, cfg.eps), "k": ks, "v": vs}


def stack_decode_seq(token: int, table: np.ndarray, layers: List[Dict[str, np.ndarray]], cfg: Cfg,
                     g_final: np.ndarray, w_u: np.ndarray, k_caches: Sequence[np.ndarray],
                     v_caches: Sequence[np.ndarray], pos: int, round_between=None) -> Dict[str, object]:
    """One decode step of one sequence through the stack: the token at position
    pos, layer l attending over its cache rows 0..pos-1 plus the new row.
    Returns dict(h [d], logits [V], k / v: the appended rows per layer)."""
    x = embed(table, [token])[0]
    ks, vs = [], []
    for lw, kc, vc in zip(layers, k_caches, v_caches):
        if round_between is not None:
            x = round_between(x)
        out = block_decode_seq(x, lw, cfg, kc, vc, pos)
        ks.append(out["k"])
        vs.append(out["v"])
        x = out["y"]
    return {"h": x, "logits": lm_head(x[None, :], g_final, w_u, cfg.eps)[0], "k": ks, "v": vs}
