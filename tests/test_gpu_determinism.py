"""Bit-for-bit reproducibility: the same call on the same inputs gives the same
bytes.  The one cross-CTA reduction of the block, the second norm's row sums
Σh², is stored as per-tile partials that its consumer adds in index order, so
no output depends on which CTA finished first."""
import pytest
import torch

import workloads
from helpers import block_config, to_device

pytestmark = pytest.mark.gpu


def _prefill_twice(s, seed):
    import causal_gqa_attention_rmsnorm_gb300 as tb
    inp = workloads.make_block_inputs(s, seed=seed)
    cfg = block_config(s, max_pos=max(s.T, 16))
    dev = to_device(inp)
    packed = tb.tb_pack_weights(cfg, dev)
    ys = [tb.tb_block_prefill(cfg, packed, dev["x"]) for _ in range(3)]
    assert tb.tb_get_device_error(clear=True) == 0
    return ys


@pytest.mark.parametrize("name,shape", [
    # tile GEMM (more than 64 tokens)
    ("tile", workloads.BlockShape("det_tile", "prefill", "bf16", B=2, T=300, d=1024, H=8, Hkv=2, dh=128, f=2048,
                                  rope_base=1e4, eps=1e-6, gains="normal")),
    # 8192 tokens at d = 4096: the Wo, W1/W3 and W2 GEMMs on CTA pairs, attention on CTA pairs
    ("pair", workloads.BlockShape("det_pair", "prefill", "bf16", B=1, T=8192, d=4096, H=32, Hkv=8, dh=128,
                                  f=4096, rope_base=5e5, eps=1e-5, gains="normal")),
    # few-token GEMM (K split over the CTAs of a cluster, reduced in distributed shared memory)
    ("skinny", workloads.BlockShape("det_few", "prefill", "bf16", B=3, T=7, d=2048, H=16, Hkv=4, dh=128, f=1024,
                                    rope_base=1e4, eps=1e-6, gains="normal")),
    # fp32 SIMT GEMM
    ("fp32", workloads.BlockShape("det_f32", "prefill", "f32", B=2, T=100, d=256, H=4, Hkv=2, dh=64, f=512,
                                  rope_base=1e4, eps=1e-6, gains="normal")),
])
def test_prefill_is_bit_reproducible(name, shape):
    ys = _prefill_twice(shape, seed=4)
    for y in ys[1:]:
        assert torch.equal(y, ys[0]), name


@pytest.mark.parametrize("name,shape", [
    # CTA-pair QKV GEMM (8192 tokens at d = 4096)
    ("pair", workloads.BlockShape("det_stats_pair", "prefill", "bf16", B=1, T=8192, d=4096, H=32, Hkv=8, dh=128,
                                  f=4096, rope_base=5e5, eps=1e-5, gains="normal")),
    # single-CTA QKV GEMM, several row groups of the statistics warps
    ("single", workloads.BlockShape("det_stats_one", "prefill", "bf16", B=2, T=3000, d=1024, H=8, Hkv=2, dh=128,
                                    f=2048, rope_base=1e4, eps=1e-6, gains="normal")),
])
def test_prefill_statistics_fallback_is_bit_identical(name, shape):
    """A QKV tile epilogue whose row group's RMSNorm-1 statistics are not ready
    in time forms its rows' scales itself, with the statistics warp's function:
    the output must be the same bytes.  A zero poll limit sends nearly every
    early tile that way."""
    from causal_gqa_attention_rmsnorm_gb300 import binding
    ys = _prefill_twice(shape, seed=5)
    prev = binding.tbx_set_stat_poll_ns(0)
    try:
        yf = _prefill_twice(shape, seed=5)
    finally:
        binding.tbx_set_stat_poll_ns(prev)
    for y in yf:
        assert torch.equal(y, ys[0]), name


@pytest.mark.parametrize("cache", ["bf16", "int8"])
def test_decode_is_bit_reproducible(cache):
    import causal_gqa_attention_rmsnorm_gb300 as tb
    s = workloads.BlockShape("det_dec", "decode", "bf16", B=5, T=512, d=1024, H=8, Hkv=2, dh=128, f=1024,
                             rope_base=5e5, eps=1e-5, gains="normal")
    lens = torch.tensor([0, 3, 100, 300, 511], dtype=torch.int32)
    inp = workloads.make_block_inputs(s, seed=9)
    cfg = block_config(s, max_pos=s.T)
    dev = to_device(inp)
    packed = tb.tb_pack_weights(cfg, dev)
    kc, vc = workloads.make_decode_cache(s, 9, lens, fill=0.0, device="cuda")
    ys = []
    for _ in range(3):
        if cache == "bf16":
            kv = tb.KVCache(kc.clone(), vc.clone(), lens.cuda())
        else:
            kv = tb.KVCache.empty_int8(s.B, s.Hkv, s.T, s.dh)
            tb.tb_kvcache_append(kv, kc, vc)
            kv.lens.copy_(lens)
        ys.append(tb.tb_block_decode(cfg, packed, dev["x"], kv))
    assert tb.tb_get_device_error(clear=True) == 0
    for y in ys[1:]:
        assert torch.equal(y, ys[0])
