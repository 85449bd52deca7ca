"""Work accounting for the decoder block: parameters, FLOPs and bytes.

Conventions (each one is pinned by ``tests/test_accounting.py`` against the
numbers the pages print):

* One multiply-add is 2 FLOPs, so a weight matrix costs 2 FLOPs per parameter
  per token ("Transformer block" page, "How it works", FLOPs paragraph;
  "The Transformer" GenerativeAIDocs section 4).  The "Transformer
  Architecture" page counts a multiply-add as one FLOP; that convention is not
  used.
* Attention costs 2·T·d for q·kᵀ and 2·T·d for the weighted sum of v per token
  when the full T×T matrix is counted; a causal kernel that skips masked work
  does about half ("Transformer block" page, FLOPs paragraph).  Here the causal
  count is exact: query i meets i+1 keys.
* KV-cache bytes per token are 2·L·Hkv·dh·bytes ("Transformer block" page,
  KV-cache paragraph; "09 The Transformer", "Counting everything").
"""
from __future__ import annotations

from typing import Iterable


def block_matrix_params(d: int, H: int, Hkv: int, dh: int, f: int) -> int:
    """Parameters of the block's weight matrices: Wq, Wk, Wv, Wo, W1, W3, W2."""
    return d * (H + 2 * Hkv) * dh + H * dh * d + 3 * d * f


def block_params(d: int, H: int, Hkv: int, dh: int, f: int) -> int:
    """All parameters of one block, the two RMSNorm gain vectors included."""
    return block_matrix_params(d, H, Hkv, dh, f) + 2 * d


def gemm_flops(d: int, H: int, Hkv: int, dh: int, f: int, tokens: int) -> int:
    """FLOPs of the block's projections for ``tokens`` tokens: 2 per parameter."""
    return 2 * block_matrix_params(d, H, Hkv, dh, f) * tokens


def gemm_flops_each(d: int, H: int, Hkv: int, dh: int, f: int, tokens: int) -> dict:
    """FLOPs of each GEMM of the block (QKV, Wo, W1/W3, W2)."""
    return {
        "qkv": 2 * tokens * d * (H + 2 * Hkv) * dh,
        "wo": 2 * tokens * H * dh * d,
        "w13": 2 * tokens * d * 2 * f,
        "w2": 2 * tokens * f * d,
    }


def visible_pairs(T: int, window: int = 0) -> int:
    """(query, key) pairs a causal prefill of T tokens attends: query i meets
    i+1 keys, or min(i+1, W) with a sliding window W > 0 ("09 The Transformer"
    §5, sliding-window attention)."""
    if window <= 0 or window >= T:
        return T * (T + 1) // 2
    return window * (window + 1) // 2 + (T - window) * window


def causal_attn_flops(B: int, H: int, dh: int, T: int, window: int = 0) -> int:
    """Exact causal attention FLOPs of a prefill: 4·dh per (query head, visible
    pair)."""
    return 4 * B * H * dh * visible_pairs(T, window)


def causal_attn_flops_tiles(B: int, H: int, dh: int, T: int, tile: int = 128) -> int:
    """Causal attention FLOPs counted per tile: every (query tile, key tile)
    pair on or below the diagonal counted in full, tile x tile pairs (a
    kernel's work with the diagonal tiles unmasked)."""
    nt = (T + tile - 1) // tile
    return 4 * B * H * dh * tile * tile * nt * (nt + 1) // 2


def full_attn_flops(B: int, H: int, dh: int, T: int) -> int:
    """Attention FLOPs counting the whole T×T square (the pages' 4·T·d per token)."""
    return 4 * B * H * dh * T * T


def decode_attn_flops(H: int, dh: int, keys: Iterable[int]) -> int:
    """Decode attention FLOPs: each query head meets every attended key once."""
    return 4 * H * dh * sum(int(k) for k in keys)


def kv_bytes_per_token(L: int, Hkv: int, dh: int, bytes_per_value: int) -> int:
    """KV-cache bytes per token: K and V, every layer, Hkv heads of dh values."""
    return 2 * L * Hkv * dh * bytes_per_value


def attended_keys(lens: Iterable[int], window: int = 0) -> int:
    """Keys one decode step attends over all sequences: lens[b] cached rows plus
    the appended one, at most W of them with a sliding window W > 0 (the pages:
    the KV cache a sliding window needs is capped at W)."""
    return sum(min(int(n) + 1, window) if window > 0 else int(n) + 1 for n in lens)


def decode_kv_bytes(lens: Iterable[int], Hkv: int, dh: int, bytes_per_value: int, window: int = 0,
                    scale_bytes: int = 0) -> int:
    """KV bytes one decode step must read: the attended rows of K and V, and
    for a quantised cache each row's scale (scale_bytes per row of K and of V)."""
    return attended_keys(lens, window) * (kv_bytes_per_token(1, Hkv, dh, bytes_per_value) + 2 * Hkv * scale_bytes)


def weight_bytes(d: int, H: int, Hkv: int, dh: int, f: int, bytes_per_value: int) -> int:
    """Bytes of the block's weight matrices (what a decode step must stream)."""
    return block_matrix_params(d, H, Hkv, dh, f) * bytes_per_value


def model_params(L: int, d: int, H: int, Hkv: int, dh: int, f: int, V: int, tied: bool = False) -> int:
    """Parameters of an L-layer model: the blocks, the embedding table [V, d],
    the final norm's gain [d] and the LM head [d, V] (none when tied to the
    embedding)."""
    return L * block_params(d, H, Hkv, dh, f) + V * d + d + (0 if tied else V * d)


def lm_head_flops(tokens: int, d: int, V: int) -> int:
    """FLOPs of the LM head for ``tokens`` rows: 2·d·V per row."""
    return 2 * tokens * d * V


def logits_bytes(tokens: int, V: int, bytes_per_value: int = 4) -> int:
    """Bytes of materialised logits [tokens, V] ("The Transformer" §5, step 18)."""
    return tokens * V * bytes_per_value


def forward_flops_per_token(N: int, L: int, T: int, d: int) -> int:
    """The pages' rule 2N + 4·L·T·d forward FLOPs per token (full square)."""
    return 2 * N + 4 * L * T * d
