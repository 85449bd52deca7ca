"""Paged KV cache ("Transformer block" page, implementation notes: allocate the
cache per sequence in fixed-size blocks).  A paged cache must give exactly the
results of the contiguous layout it stores (same kernels, same arithmetic
order: K/V rows and outputs bit for bit), and match the fp64 oracle on the rows
its block table gathers."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import assert_close, block_config, oracle_cfg, oracle_weights, to_device

pytestmark = pytest.mark.gpu

BF16 = workloads.BlockShape("pg_bf16", "decode", "bf16", B=4, T=0, d=1024, H=8, Hkv=2, dh=128, f=1024,
                            rope_base=5e5, eps=1e-5, gains="normal")
F32 = workloads.CONFIGS["tiny_fp32"].with_(name="pg_f32", mode="decode", B=4)


def _tables(B, T_max, ps, seed):
    """A shuffled pool with spare pages: block table [B, T_max / ps]."""
    per = T_max // ps
    num_pages = B * per + 5
    perm = np.random.default_rng(seed).permutation(num_pages)[:B * per]
    return torch.tensor(perm.reshape(B, per), dtype=torch.int32), num_pages


def _to_paged(kc, vc, lens, bt, ps, num_pages, fill=float("nan")):
    import causal_gqa_attention_rmsnorm_gb300 as tb
    B, Hkv, T_max, dh = kc.shape
    kv = tb.KVCache.empty_paged(B, Hkv, T_max, dh, ps, num_pages, bt, dtype=kc.dtype, fill=fill)
    btc = bt.cpu().numpy()
    for b in range(B):
        for p in range(T_max // ps):
            kv.k[btc[b, p]] = kc[b, :, p * ps:(p + 1) * ps]
            kv.v[btc[b, p]] = vc[b, :, p * ps:(p + 1) * ps]
    kv.lens.copy_(lens)
    return kv


def _gather(kv, b, n):
    return (oracle.gather_paged(kv.k.float().cpu().numpy(), kv.block_table[b].cpu().numpy(), kv.k.shape[2], n),
            oracle.gather_paged(kv.v.float().cpu().numpy(), kv.block_table[b].cpu().numpy(), kv.k.shape[2], n))


@pytest.mark.parametrize("ps", [16, 64, 256])
@pytest.mark.parametrize("base", ["bf16", "f32"])
@pytest.mark.parametrize("W", [0, 100])
def test_paged_decode_equals_contiguous_and_oracle(ps, base, W):
    import causal_gqa_attention_rmsnorm_gb300 as tb
    s = (BF16 if base == "bf16" else F32).with_(window=W)
    T_max = 768
    lens = torch.tensor([0, 17, 300, 767][:s.B], dtype=torch.int32)
    inp = workloads.make_block_inputs(s.with_(T=T_max), seed=7)
    kc, vc = workloads.make_decode_cache(s.with_(T=T_max), 7, lens, fill=float("nan"), device="cuda")
    cfg = block_config(s, max_pos=T_max)
    dev = to_device(inp)
    packed = tb.tb_pack_weights(cfg, dev)
    bt, num_pages = _tables(s.B, T_max, ps, seed=ps + W)
    paged = _to_paged(kc, vc, lens.cuda(), bt.cuda(), ps, num_pages)
    contig = tb.KVCache(kc.clone(), vc.clone(), lens.cuda())
    y_c = tb.tb_block_decode(cfg, packed, dev["x"], contig)
    y_p = tb.tb_block_decode(cfg, packed, dev["x"], paged)
    assert tb.tb_get_device_error(clear=True) == 0
    assert torch.equal(y_p, y_c)
    assert torch.equal(paged.lens, contig.lens)
    w, ocfg = oracle_weights(inp), oracle_cfg(s)
    for b, pos in enumerate(lens.tolist()):
        kg, vg = _gather(paged, b, pos + 1)
        np.testing.assert_array_equal(kg, contig.k[b, :, :pos + 1].float().cpu().numpy())
        np.testing.assert_array_equal(vg, contig.v[b, :, :pos + 1].float().cpu().numpy())
        ref = oracle.block_decode_seq(workloads.to_f64(inp["x"][b, 0]), w, ocfg, kg[:, :pos], vg[:, :pos], pos)
        assert_close(y_p[b, 0].cpu().double().numpy(), ref["y"], s.dtype, f"y b={b}")
        assert_close(kg[:, pos], ref["k"], s.dtype, f"appended k b={b}")


@pytest.mark.parametrize("ps", [16, 128])
def test_paged_prefill_fills_the_pages(ps):
    import causal_gqa_attention_rmsnorm_gb300 as tb
    s = workloads.BlockShape("pg_pre", "prefill", "bf16", B=2, T=200, d=512, H=8, Hkv=2, dh=64, f=1024,
                             rope_base=1e4, eps=1e-6, gains="normal")
    T_max = 256
    inp = workloads.make_block_inputs(s, seed=2)
    cfg = block_config(s, max_pos=T_max)
    dev = to_device(inp)
    packed = tb.tb_pack_weights(cfg, dev)
    contig = tb.KVCache.empty(s.B, s.Hkv, T_max, s.dh, dtype=torch.bfloat16, fill=float("nan"))
    bt, num_pages = _tables(s.B, T_max, ps, seed=ps)
    paged = tb.KVCache.empty_paged(s.B, s.Hkv, T_max, s.dh, ps, num_pages, bt.cuda(), fill=float("nan"))
    y_c = tb.tb_block_prefill(cfg, packed, dev["x"], kv=contig)
    y_p = tb.tb_block_prefill(cfg, packed, dev["x"], kv=paged)
    assert tb.tb_get_device_error(clear=True) == 0
    assert torch.equal(y_p, y_c)
    assert paged.lens.tolist() == [s.T] * s.B
    for b in range(s.B):
        kg, vg = _gather(paged, b, s.T)
        np.testing.assert_array_equal(kg, contig.k[b, :, :s.T].float().cpu().numpy())
        np.testing.assert_array_equal(vg, contig.v[b, :, :s.T].float().cpu().numpy())
    # a decode step continues the paged prefill exactly as it continues the contiguous one
    x1 = dev["x"][:, :1].contiguous()
    assert torch.equal(tb.tb_block_decode(cfg, packed, x1, paged), tb.tb_block_decode(cfg, packed, x1, contig))


def test_paged_append_matches_contiguous():
    import causal_gqa_attention_rmsnorm_gb300 as tb
    B, Hkv, T_max, dh, ps, n = 3, 2, 128, 64, 32, 40
    bt, num_pages = _tables(B, T_max, ps, seed=4)
    contig = tb.KVCache.empty(B, Hkv, T_max, dh, fill=0.0)
    paged = tb.KVCache.empty_paged(B, Hkv, T_max, dh, ps, num_pages, bt.cuda(), fill=0.0)
    g = torch.Generator().manual_seed(0)
    for _ in range(2):
        kn = torch.randn(B, Hkv, n, dh, generator=g).to(torch.bfloat16).cuda()
        vn = torch.randn(B, Hkv, n, dh, generator=g).to(torch.bfloat16).cuda()
        tb.tb_kvcache_append(contig, kn, vn)
        tb.tb_kvcache_append(paged, kn, vn)
    assert tb.tb_get_device_error(clear=True) == 0
    assert paged.lens.tolist() == contig.lens.tolist() == [2 * n] * B
    for b in range(B):
        kg, vg = _gather(paged, b, 2 * n)
        np.testing.assert_array_equal(kg, contig.k[b, :, :2 * n].float().cpu().numpy())
        np.testing.assert_array_equal(vg, contig.v[b, :, :2 * n].float().cpu().numpy())


def test_bad_page_id_is_flagged():
    """A block-table entry outside the pool is never dereferenced: the step
    sets TB_DEVERR_BAD_PAGE (its output is not valid) and the context stays
    usable."""
    import causal_gqa_attention_rmsnorm_gb300 as tb
    s = BF16
    T_max, ps = 256, 64
    lens = torch.tensor([10, 100, 200, 70], dtype=torch.int32)
    inp = workloads.make_block_inputs(s.with_(T=T_max), seed=1)
    kc, vc = workloads.make_decode_cache(s.with_(T=T_max), 1, lens, fill=0.0, device="cuda")
    cfg = block_config(s, max_pos=T_max)
    dev = to_device(inp)
    packed = tb.tb_pack_weights(cfg, dev)
    bt, num_pages = _tables(s.B, T_max, ps, seed=3)
    bt[2, 1] = num_pages + 1000                 # sequence 2's second page: out of range
    paged = _to_paged(kc, vc, lens.cuda(), torch.where(bt >= num_pages, 0, bt).cuda(), ps, num_pages, fill=0.0)
    paged.block_table.copy_(bt.cuda())
    tb.tb_block_decode(cfg, packed, dev["x"], paged)
    assert tb.tb_get_device_error(clear=True) & tb.TB_DEVERR_BAD_PAGE
    # the context is intact: a valid table decodes normally afterwards
    paged.block_table.copy_(torch.where(bt >= num_pages, 0, bt).cuda())
    paged.lens.copy_(lens.cuda())
    tb.tb_block_decode(cfg, packed, dev["x"], paged)
    assert tb.tb_get_device_error(clear=True) == 0
