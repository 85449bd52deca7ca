"""A CPU model of the bf16 path's rounding points (test infrastructure).

The block's bf16 path feeds the tensor cores bf16 operands and accumulates in
fp32.  Relative to the fp64 oracle on bf16-rounded inputs it therefore rounds,
to bf16: the gain-folded weights g⊙Wqkv and g⊙W1/W3, the post-RoPE q, k, v,
the softmax numerators P, the attention output o, the residual stream h fed
to W1/W3, and the SwiGLU output a.  This model repeats the block in fp32 with
exactly those roundings (plain torch CPU ops, no CUDA) so that a test can
tell rounding noise from a kernel error: the GPU's deviation from the oracle
must look like this model's deviation.

It shares no code with the CUDA library and is not an oracle: the oracle in
``oracle/`` is the definition; this is a model of one implementation's
rounding.
"""
from __future__ import annotations

import math

import torch

import workloads


def _bf(t: torch.Tensor) -> torch.Tensor:
    return t.to(torch.bfloat16).float()


def emulate_prefill_seq(inp, s: workloads.BlockShape, b: int = 0) -> torch.Tensor:
    """fp32 prefill of sequence b with the bf16 path's rounding points; y [T, d]."""
    w = {n: inp[n].float() for n in workloads.WEIGHT_NAMES}
    x = inp["x"][b].float()
    T = x.shape[0]
    H, Hkv, dh = s.H, s.Hkv, s.dh
    r = 1.0 / torch.sqrt((x * x).mean(-1, keepdim=True) + s.eps)
    wqkv = torch.cat([w["wq"], w["wk"], w["wv"]], 1)
    acc = r * (x @ _bf(w["g_attn"][:, None] * wqkv))
    i = torch.arange(dh // 2, dtype=torch.float64)
    ang = torch.outer(torch.arange(T, dtype=torch.float64), s.rope_base ** (-2 * i / dh))
    c, sn = torch.cos(ang).float()[:, None], torch.sin(ang).float()[:, None]

    def rope(u):
        a, bb = u[..., 0::2], u[..., 1::2]
        out = torch.empty_like(u)
        out[..., 0::2] = a * c - bb * sn
        out[..., 1::2] = a * sn + bb * c
        return out

    q = _bf(rope(acc[:, :H * dh].reshape(T, H, dh)))
    k = _bf(rope(acc[:, H * dh:(H + Hkv) * dh].reshape(T, Hkv, dh)))
    v = _bf(acc[:, (H + Hkv) * dh:].reshape(T, Hkv, dh))
    G = H // Hkv
    keep = torch.ones(T, T, dtype=torch.bool).tril()
    o = torch.empty(T, H, dh)
    for h in range(H):
        S = (q[:, h] @ k[:, h // G].T) / math.sqrt(dh)
        S = S.masked_fill(~keep, float("-inf"))
        P = torch.exp(S - S.max(-1, keepdim=True).values)
        o[:, h] = (_bf(P) @ v[:, h // G]) / P.sum(-1, keepdim=True)
    hh = x + _bf(o.reshape(T, H * dh)) @ w["wo"]
    r2 = 1.0 / torch.sqrt((hh * hh).mean(-1, keepdim=True) + s.eps)
    hb = _bf(hh)
    g = r2 * (hb @ _bf(w["g_mlp"][:, None] * w["w1"]))
    u = r2 * (hb @ _bf(w["g_mlp"][:, None] * w["w3"]))
    a = _bf(g / (1.0 + torch.exp(-g)) * u)
    return hh + a @ w["w2"]
