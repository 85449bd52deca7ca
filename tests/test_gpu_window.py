"""Sliding-window attention ("09 The Transformer" §5): key j is visible to
query i iff i - W < j <= i.  Prefill and decode through the C ABI against the
fp64 oracle with the same window, in both query-tile pairings of the
tensor-core kernel (two heads of a KV group; two query blocks of one head),
for windows below, at and across the 128-key tile, and on the fp32 path."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import assert_close, errors, oracle_cfg, oracle_weights
from test_gpu_decode import _decode_case, _oracle_step
from test_gpu_prefill import run_prefill

pytestmark = pytest.mark.gpu

GQA = workloads.BlockShape("win_gqa", "prefill", "bf16", B=2, T=300, d=256, H=4, Hkv=2, dh=64, f=512,
                           rope_base=1e4, eps=1e-6, gains="normal")
MHA = workloads.BlockShape("win_mha", "prefill", "bf16", B=1, T=333, d=512, H=4, Hkv=4, dh=128, f=1024,
                           rope_base=5e5, eps=1e-5, gains="normal")
F32 = workloads.CONFIGS["tiny_fp32"].with_(name="win_f32", B=2, T=37)
# GQA with groups of four heads at dh 128: the CTA-pair attention kernel
PAIR = workloads.BlockShape("win_pair", "prefill", "bf16", B=2, T=333, d=1024, H=8, Hkv=2, dh=128, f=1024,
                            rope_base=5e5, eps=1e-5, gains="normal")


def _prefill_vs_oracle(s, seed=3):
    inp = workloads.make_block_inputs(s, seed=seed)
    y, kv = run_prefill(s, inp, with_cache=True)
    w, cfg = oracle_weights(inp), oracle_cfg(s)
    x64 = workloads.to_f64(inp["x"])
    for b in range(s.B):
        ref = oracle.block_prefill_seq(x64[b], w, cfg)
        assert_close(y[b].cpu().double().numpy(), ref["y"], s.dtype, f"y b={b} W={s.window}")
    return y


@pytest.mark.parametrize("W", [1, 37, 127, 128, 129, 200, 300, 1000])
def test_prefill_window_gqa_head_pairs(W):
    _prefill_vs_oracle(GQA.with_(window=W))


@pytest.mark.parametrize("W", [1, 50, 128, 256])
def test_prefill_window_mha_block_pairs(W):
    _prefill_vs_oracle(MHA.with_(window=W))


@pytest.mark.parametrize("W", [1, 37, 64, 65, 127, 128, 129, 200, 1000])
def test_prefill_window_gqa_cta_pairs(W):
    _prefill_vs_oracle(PAIR.with_(window=W))


@pytest.mark.parametrize("W", [1, 5, 36, 37])
def test_prefill_window_fp32(W):
    _prefill_vs_oracle(F32.with_(window=W))


def test_window_at_least_T_is_full_attention():
    s = GQA.with_(T=200)
    y_full = _prefill_vs_oracle(s)
    y_win = _prefill_vs_oracle(s.with_(window=200))
    assert torch.equal(y_full, y_win)


@pytest.mark.parametrize("W", [1, 100, 300])
@pytest.mark.parametrize("base", ["bf16", "f32"])
def test_decode_window(W, base):
    s = (workloads.BlockShape("win_dec", "decode", "bf16", B=5, T=0, d=1024, H=8, Hkv=2, dh=128, f=1024,
                              rope_base=5e5, eps=1e-5, gains="normal") if base == "bf16"
         else workloads.CONFIGS["tiny_fp32"].with_(name="win_dec_f32", B=5)).with_(window=W)
    T_max = 700
    lens = [0, 1, W - 1 if W > 1 else 2, W + 3, 699]
    s, inp, kv, y, err = _decode_case(s, 17, lens, T_max)
    assert err == 0
    for b, pos in enumerate(lens):
        ref = _oracle_step(s, inp, kv, b, pos)
        assert_close(y[b, 0].cpu().double().numpy(), ref["y"], s.dtype, f"y b={b} W={W}")
        assert_close(kv.k[b, :, pos].cpu().double().numpy(), ref["k"], s.dtype, f"k row b={b}")


def test_decode_window_continues_prefill():
    """Prefill T-1 tokens with a window, decode token T-1: equals row T-1 of
    the windowed oracle prefill of all T tokens."""
    import causal_gqa_attention_rmsnorm_gb300 as tb
    from helpers import block_config, to_device
    s = GQA.with_(T=280, window=150)
    inp = workloads.make_block_inputs(s, seed=9)
    cfg = block_config(s, max_pos=512)
    dev = to_device(inp)
    packed = tb.tb_pack_weights(cfg, dev)
    kv = tb.KVCache.empty(s.B, s.Hkv, 512, s.dh, dtype=torch.bfloat16, fill=float("nan"))
    tb.tb_block_prefill(cfg, packed, dev["x"][:, :s.T - 1].contiguous(), kv=kv)
    y = tb.tb_block_decode(cfg, packed, dev["x"][:, s.T - 1:].contiguous(), kv)
    assert tb.tb_get_device_error(clear=True) == 0
    w, ocfg = oracle_weights(inp), oracle_cfg(s)
    for b in range(s.B):
        ref = oracle.block_prefill_seq(workloads.to_f64(inp["x"][b]), w, ocfg, rows=[s.T - 1])
        assert_close(y[b, 0].cpu().double().numpy(), ref["y"][0], s.dtype, f"y b={b}")
