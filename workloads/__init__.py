"""Seeded synthetic workloads for the pre-norm decoder block.

This module defines the workload shapes and draws their random inputs.  It
holds none of the block's arithmetic: it only decides sizes, seeds, value
distributions and storage rounding, so that the fp64 oracle and the CUDA path
are fed the very same bytes.

Shapes and distributions follow the workload list of the decoder-block pages
(Transformer block, tirogla.com, "How it works" notation: B batch, T sequence,
d width, H query heads, Hkv KV heads, dh head width, f MLP width) and the model
table of "The Transformer" (GenerativeAIDocs, section 8) for the Llama-shaped
cases.  Weights are stored [in, out] row-major (y = x·W), as in the Rust block
of the Transformer block page.

Draw order (fixed): x, g_attn, wq, wk, wv, wo, g_mlp, w1, w3, w2.  Every tensor
is drawn in fp32 from N(0, 1) with a CPU ``torch.Generator`` seeded once,
scaled, then rounded to the storage dtype (round-to-nearest-even for bf16).
Decode caches are drawn per sequence from a generator seeded with
``cache_seed(seed, b)`` so that one sequence can be regenerated alone.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional, Sequence

import torch


@dataclasses.dataclass(frozen=True)
class BlockShape:
    name: str
    mode: str          # "prefill" or "decode"
    dtype: str         # "f32" or "bf16" storage; accumulation is always fp32
    B: int
    T: int             # prefill sequence length; for decode, the cache capacity T_max
    d: int
    H: int
    Hkv: int
    dh: int
    f: int
    rope_base: float
    eps: float
    gains: str         # "ones" or "normal" (N(1, 0.1))
    lens_lo: int = 0   # decode only: cached lengths uniform in [lens_lo, lens_hi]
    lens_hi: int = 0
    window: int = 0    # sliding-window width W (0: full causal attention)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def tokens(self) -> int:
        return self.B * (self.T if self.mode == "prefill" else 1)

    def with_(self, **kw) -> "BlockShape":
        return dataclasses.replace(self, **kw)


# The five workloads.  Readings where the source is silent are noted inline.
CONFIGS: Dict[str, BlockShape] = {
    # fp32, gains 1, tiny: the case the oracle finishes instantly.
    "tiny_fp32": BlockShape("tiny_fp32", "prefill", "f32", B=1, T=16, d=64, H=4, Hkv=2,
                            dh=16, f=176, rope_base=1e4, eps=1e-6, gains="ones"),
    # GPT-2-small-width MHA block with a SwiGLU MLP of f = 8d/3.
    "mha_768": BlockShape("mha_768", "prefill", "bf16", B=8, T=1024, d=768, H=12, Hkv=12,
                          dh=64, f=2048, rope_base=1e4, eps=1e-6, gains="normal"),
    # Llama-2-7B-shaped block; the prefill also emits its post-RoPE K/V cache.
    "llama2_7b": BlockShape("llama2_7b", "prefill", "bf16", B=1, T=4096, d=4096, H=32, Hkv=32,
                            dh=128, f=11008, rope_base=1e4, eps=1e-6, gains="normal"),
    # Llama-3-8B-shaped GQA block, long-context prefill.
    "gqa_8k": BlockShape("gqa_8k", "prefill", "bf16", B=4, T=8192, d=4096, H=32, Hkv=8,
                         dh=128, f=14336, rope_base=5e5, eps=1e-5, gains="normal"),
    # One decode step of the GQA block over a 16384-slot cache.  The cached
    # lengths are drawn in [1024, 16383] so that the appended token fits; RoPE
    # base, eps and gains follow the gqa_8k block of the same shape.
    "gqa_decode": BlockShape("gqa_decode", "decode", "bf16", B=32, T=16384, d=4096, H=32,
                             Hkv=8, dh=128, f=14336, rope_base=5e5, eps=1e-5, gains="normal",
                             lens_lo=1024, lens_hi=16383),
}

WEIGHT_NAMES = ("g_attn", "wq", "wk", "wv", "wo", "g_mlp", "w1", "w3", "w2")
WEIGHT_STD = 0.02
GAIN_STD = 0.1


def weight_shapes(s: BlockShape) -> Dict[str, tuple]:
    """[in, out] shapes of every weight, gains [d]."""
    return {
        "g_attn": (s.d,),
        "wq": (s.d, s.H * s.dh),
        "wk": (s.d, s.Hkv * s.dh),
        "wv": (s.d, s.Hkv * s.dh),
        "wo": (s.H * s.dh, s.d),
        "g_mlp": (s.d,),
        "w1": (s.d, s.f),
        "w3": (s.d, s.f),
        "w2": (s.f, s.d),
    }


def _draw(gen: torch.Generator, shape, scale: float, mean: float, dtype: torch.dtype) -> torch.Tensor:
    t = torch.randn(shape, generator=gen, dtype=torch.float32)
    if scale != 1.0:
        t.mul_(scale)
    if mean != 0.0:
        t.add_(mean)
    return t.to(dtype)


def make_block_inputs(s: BlockShape, seed: int = 0, x_tokens: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """Draw x and all weights on the CPU in the storage dtype.

    x has shape [B, T, d] for prefill and [B, 1, d] for decode.  ``x_tokens``
    overrides the token count of x (used by tests that shorten a workload).
    """
    gen = torch.Generator().manual_seed(seed)
    dt = s.torch_dtype
    tq = x_tokens if x_tokens is not None else (s.T if s.mode == "prefill" else 1)
    out = {"x": _draw(gen, (s.B, tq, s.d), 1.0, 0.0, dt)}
    for name, shape in weight_shapes(s).items():
        if name.startswith("g_"):
            if s.gains == "ones":
                out[name] = torch.ones(shape, dtype=dt)
            else:
                out[name] = _draw(gen, shape, GAIN_STD, 1.0, dt)
        else:
            out[name] = _draw(gen, shape, WEIGHT_STD, 0.0, dt)
    return out


def cache_seed(seed: int, b: int) -> int:
    return (seed * 1_000_003 + 7919 * (b + 1)) & 0x7FFF_FFFF


def make_lens(s: BlockShape, seed: int = 0) -> torch.Tensor:
    """Per-sequence cached lengths, uniform integers in [lens_lo, lens_hi]."""
    gen = torch.Generator().manual_seed(seed ^ 0x5EED)
    return torch.randint(s.lens_lo, s.lens_hi + 1, (s.B,), generator=gen, dtype=torch.int32)


def make_cache_rows(s: BlockShape, seed: int, b: int, n: int):
    """The first n cached post-RoPE K and V rows of sequence b: two [Hkv, n, dh]
    tensors of N(0, 1) values in the storage dtype."""
    gen = torch.Generator().manual_seed(cache_seed(seed, b))
    k = _draw(gen, (s.Hkv, n, s.dh), 1.0, 0.0, s.torch_dtype)
    v = _draw(gen, (s.Hkv, n, s.dh), 1.0, 0.0, s.torch_dtype)
    return k, v


def make_decode_cache(s: BlockShape, seed: int, lens: torch.Tensor, fill: float = float("nan"),
                      device="cpu", batches: Optional[Sequence[int]] = None):
    """A [B, Hkv, T_max, dh] K and V cache whose rows < lens[b] hold N(0, 1)
    values and whose other rows hold ``fill`` (NaN in tests, to expose reads
    past the cached length)."""
    shape = (s.B, s.Hkv, s.T, s.dh)
    k = torch.full(shape, fill, dtype=s.torch_dtype, device=device)
    v = torch.full(shape, fill, dtype=s.torch_dtype, device=device)
    for b in (range(s.B) if batches is None else batches):
        n = int(lens[b])
        kb, vb = make_cache_rows(s, seed, b, n)
        k[b, :, :n].copy_(kb)
        v[b, :, :n].copy_(vb)
    return k, v


def to_f64(t: torch.Tensor):
    """The exact fp64 value of a stored tensor, as a numpy array."""
    return t.to(torch.float64).numpy()
