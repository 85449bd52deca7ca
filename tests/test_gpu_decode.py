"""Decode parity: one step over a KV cache, through the C ABI, against the fp64
oracle on the same cache contents; cache appends, lengths, and the device
error word for sequences whose cache is full."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import (BF16_MAX_ABS_TOL, BF16_REL_L2_TOL, assert_close, block_config, errors, oracle_cfg,
                     oracle_weights, to_device)
from rounding_model import ERROR_FACTOR, emulate_decode_seq, rounding_consistency

pytestmark = pytest.mark.gpu


def _decode_case(s, seed, lens, T_max, batches_with_data=None, y_dtype=None):
    """Random cache rows < lens[b] (NaN beyond), one decode step on the GPU and
    the oracle's step for each sequence in `batches_with_data`."""
    import causal_gqa_attention_rmsnorm_gb300 as tb
    s = s.with_(T=T_max)
    inp = workloads.make_block_inputs(s.with_(mode="decode"), seed=seed)
    lens_t = torch.tensor(lens, dtype=torch.int32)
    kc, vc = workloads.make_decode_cache(s, seed, lens_t, fill=float("nan"), device="cuda",
                                         batches=batches_with_data)
    kv = tb.KVCache(kc, vc, lens_t.cuda())
    cfg = block_config(s, max_pos=T_max)
    dev = to_device(inp)
    packed = tb.tb_pack_weights(cfg, dev)
    y = tb.tb_block_decode(cfg, packed, dev["x"], kv, y_dtype=tb.TB_F32 if y_dtype is None else y_dtype)
    err = tb.tb_get_device_error(clear=True)
    return s, inp, kv, y, err


def _oracle_step(s, inp, kv, b, pos):
    k = kv.k[b, :, :pos].cpu().double().numpy()
    v = kv.v[b, :, :pos].cpu().double().numpy()
    return oracle.block_decode_seq(workloads.to_f64(inp["x"][b, 0]), oracle_weights(inp), oracle_cfg(s), k, v, pos)


SMALL = {
    "fp32_gqa": workloads.CONFIGS["tiny_fp32"].with_(name="fp32_gqa", B=3),
    "bf16_gqa_dh64": workloads.BlockShape("bf16_gqa_dh64", "decode", "bf16", B=3, T=0, d=256, H=4, Hkv=2,
                                          dh=64, f=512, rope_base=1e4, eps=1e-6, gains="normal"),
    "bf16_gqa4_dh128": workloads.BlockShape("bf16_gqa4_dh128", "decode", "bf16", B=4, T=0, d=1024, H=8, Hkv=2,
                                            dh=128, f=1024, rope_base=5e5, eps=1e-5, gains="normal"),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_decode_small(name):
    base = SMALL[name]
    T_max = 700
    lens = [0, 1, 699, 300][:base.B] if base.B >= 3 else [5, 600]
    lens = (lens + [257] * base.B)[:base.B]
    s, inp, kv, y, err = _decode_case(base, 11, lens, T_max)
    assert err == 0
    assert kv.lens.cpu().tolist() == [n + 1 for n in lens]
    for b, pos in enumerate(lens):
        ref = _oracle_step(s, inp, kv, b, pos)
        assert_close(y[b, 0].cpu().double().numpy(), ref["y"], s.dtype, f"y b={b}")
        assert_close(kv.k[b, :, pos].cpu().double().numpy(), ref["k"], s.dtype, f"k row b={b}")
        assert_close(kv.v[b, :, pos].cpu().double().numpy(), ref["v"], s.dtype, f"v row b={b}")
    # the step wrote exactly one row per sequence
    for b, pos in enumerate(lens):
        if pos + 1 < T_max:
            assert torch.isnan(kv.k[b, :, pos + 1:].float()).all()


# Few-token GEMMs: token counts padded to 16, 32, 48 and 64 (65 takes the tile
# GEMM), output widths that end in a partial 128-row weight tile (960, 320),
# and weight matrices long enough in K to be split unevenly over CTAs.
FEW_TOKENS = {
    "ragged_n": workloads.BlockShape("few_ragged_n", "decode", "bf16", B=1, T=0, d=320, H=5, Hkv=5, dh=64,
                                     f=192, rope_base=1e4, eps=1e-6, gains="normal"),
    "split_k": workloads.BlockShape("few_split_k", "decode", "bf16", B=1, T=0, d=1024, H=8, Hkv=8, dh=128,
                                    f=2752, rope_base=5e5, eps=1e-5, gains="normal"),
}


@pytest.mark.parametrize("B", [1, 17, 40, 64, 65])
@pytest.mark.parametrize("name", list(FEW_TOKENS))
def test_decode_token_counts(name, B):
    T_max = 64
    lens = np.random.default_rng(100 + B).integers(0, T_max - 1, size=B).tolist()
    s, inp, kv, y, err = _decode_case(FEW_TOKENS[name].with_(B=B), 21 + B, lens, T_max)
    assert err == 0
    assert kv.lens.cpu().tolist() == [n + 1 for n in lens]
    for b, pos in enumerate(lens):
        ref = _oracle_step(s, inp, kv, b, pos)
        assert_close(y[b, 0].cpu().double().numpy(), ref["y"], s.dtype, f"y b={b}")
        assert_close(kv.k[b, :, pos].cpu().double().numpy(), ref["k"], s.dtype, f"k row b={b}")
        assert_close(kv.v[b, :, pos].cpu().double().numpy(), ref["v"], s.dtype, f"v row b={b}")


def test_decode_continues_a_prefill():
    """Prefill T-1 tokens into the cache, decode token T-1: equals row T-1 of
    the oracle prefill of all T tokens (decode with a cache is the same
    computation as the last row of prefill)."""
    import causal_gqa_attention_rmsnorm_gb300 as tb
    s = workloads.BlockShape("chain", "prefill", "bf16", B=2, T=150, d=512, H=8, Hkv=2, dh=64, f=1024,
                             rope_base=1e4, eps=1e-6, gains="normal")
    inp = workloads.make_block_inputs(s, seed=5)
    cfg = block_config(s, max_pos=256)
    dev = to_device(inp)
    packed = tb.tb_pack_weights(cfg, dev)
    kv = tb.KVCache.empty(s.B, s.Hkv, 256, s.dh, dtype=torch.bfloat16, fill=float("nan"))
    tb.tb_block_prefill(cfg, packed, dev["x"][:, :s.T - 3].contiguous(), kv=kv)
    ys = [tb.tb_block_decode(cfg, packed, dev["x"][:, t:t + 1].contiguous(), kv) for t in range(s.T - 3, s.T)]
    assert tb.tb_get_device_error(clear=True) == 0
    assert kv.lens.cpu().tolist() == [s.T] * s.B
    ref = oracle.block_prefill(workloads.to_f64(inp["x"]), oracle_weights(inp), oracle_cfg(s))
    for i, t in enumerate(range(s.T - 3, s.T)):
        assert_close(ys[i][:, 0].cpu().double().numpy(), ref["y"][:, t], "bf16", f"decode step t={t}")
    assert_close(kv.k[:, :, :s.T].cpu().double().numpy(), ref["k"], "bf16", "k cache")


def test_decode_full_cache_sets_error_and_skips_row():
    base = SMALL["bf16_gqa_dh64"]
    T_max = 64
    lens = [10, T_max, 63]
    s, inp, kv, y, err = _decode_case(base, 7, lens, T_max)
    import causal_gqa_attention_rmsnorm_gb300 as tb
    assert err & tb.TB_DEVERR_CACHE_FULL
    assert kv.lens.cpu().tolist() == [11, T_max, 64]
    for b in (0, 2):
        ref = _oracle_step(s, inp, kv, b, lens[b])
        assert_close(y[b, 0].cpu().double().numpy(), ref["y"], "bf16", f"y b={b}")
    assert tb.tb_get_device_error() == 0   # cleared


def test_kvcache_append():
    import causal_gqa_attention_rmsnorm_gb300 as tb
    B, Hkv, T_max, dh = 3, 2, 40, 64
    kv = tb.KVCache.empty(B, Hkv, T_max, dh, fill=0.0)
    kv.lens.copy_(torch.tensor([0, 5, 37], dtype=torch.int32))
    g = torch.Generator().manual_seed(0)
    kn = torch.randn(B, Hkv, 3, dh, generator=g).to(torch.bfloat16).cuda()
    vn = torch.randn(B, Hkv, 3, dh, generator=g).to(torch.bfloat16).cuda()
    tb.tb_kvcache_append(kv, kn, vn)
    assert tb.tb_get_device_error(clear=True) == 0
    assert kv.lens.cpu().tolist() == [3, 8, 40]
    for b, L in enumerate([0, 5, 37]):
        assert torch.equal(kv.k[b, :, L:L + 3], kn[b]) and torch.equal(kv.v[b, :, L:L + 3], vn[b])
    # a second append overflows sequence 2 only
    tb.tb_kvcache_append(kv, kn, vn)
    assert tb.tb_get_device_error(clear=True) & tb.TB_DEVERR_CACHE_FULL
    assert kv.lens.cpu().tolist() == [6, 11, 40]


_FULL = {}
FULL_SAMPLED = [0, 3, 7, 12, 18, 21, 26, 31]


def _full_decode_report():
    """The full decode workload (B = 32, T_max = 16384, GQA 32/8, dh 128) in
    the benchmark's launch configuration, run once per session.  Only the
    sampled sequences hold cache data; every other cache row is NaN, so a read
    past a sequence's own rows or across sequences shows up as NaN in a
    checked row.  Keeps, per sampled sequence, the GPU's y, the oracle's y and
    the rounding model's y in orders "a" and "b" (over the same seeded cache
    rows), and the error reports of y and of the appended k row."""
    if not _FULL:
        s = workloads.CONFIGS["gqa_decode"]
        lens = workloads.make_lens(s, seed=0)
        s, inp, kv, y, err = _decode_case(s, 0, lens.tolist(), s.T, batches_with_data=FULL_SAMPLED)
        assert err == 0
        assert kv.lens.cpu().tolist() == [int(n) + 1 for n in lens]
        for b in FULL_SAMPLED:
            pos = int(lens[b])
            ref = _oracle_step(s, inp, kv, b, pos)
            kc, vc = workloads.make_cache_rows(s, 0, b, pos)
            got = y[b, 0].cpu().double().numpy()
            _FULL[b] = dict(got=got, ref=ref["y"],
                            emu_a=emulate_decode_seq(inp, s, b, kc, vc, order="a").double().numpy(),
                            emu_b=emulate_decode_seq(inp, s, b, kc, vc, order="b").double().numpy(),
                            ey=errors(got, ref["y"]),
                            ek=errors(kv.k[b, :, pos].cpu().double().numpy(), ref["k"]))
    return _FULL


def _stack(rep, key):
    return np.stack([r[key] for r in rep.values()])


def test_decode_gqa_full_workload_error_is_bf16_rounding():
    """On the sampled sequences of the full decode workload the GPU is as close
    to the rounding model (tests/rounding_model.py, order "a") as the model's
    second order is, within 1.5x, and its error against the oracle is within
    1.25x of the model's (max-abs and relative L2 over all sampled rows)."""
    rep = _full_decode_report()
    c = rounding_consistency(_stack(rep, "got"), _stack(rep, "emu_a"), _stack(rep, "emu_b"), _stack(rep, "ref"))
    print(f"gqa_decode sampled rows: order noise {c['noise']}, GPU to model {c['dev']}, "
          f"model error {c['model']}, GPU error {c['err']}")
    assert c["ok"], c


def test_decode_gqa_full_workload_sampled_sequences():
    """Relative-L2 bar 1e-2 per sampled sequence, max-abs within 1.25x the
    rounding model's max-abs error over the sampled rows (measured in the same
    run); the appended k rows meet both bf16 bars."""
    rep = _full_decode_report()
    bound = ERROR_FACTOR * errors(_stack(rep, "emu_a"), _stack(rep, "ref"))["max_abs"]
    for b, r in rep.items():
        ey, ek = r["ey"], r["ek"]
        assert ey["finite"] and ey["rel_l2"] <= BF16_REL_L2_TOL and ey["max_abs"] <= bound, (b, ey, bound)
        assert ek["finite"] and ek["rel_l2"] <= BF16_REL_L2_TOL and ek["max_abs"] <= BF16_MAX_ABS_TOL, (b, ek)


@pytest.mark.xfail(strict=True, reason="bf16 operand rounding alone exceeds 3e-2 max-abs at d = 4096 "
                                       "(see test_rounding_floor.py)")
def test_decode_gqa_full_workload_max_abs_bar():
    for b, r in _full_decode_report().items():
        assert r["ey"]["max_abs"] <= BF16_MAX_ABS_TOL, (b, r["ey"])


@pytest.mark.parametrize("cache", ["bf16", "int8"])
def test_decode_at_the_batch_limit(cache):
    """2048 sequences, the most one decode call takes: sampled sequences match
    the oracle (the kernels' per-sequence tables still fit in shared memory)."""
    import causal_gqa_attention_rmsnorm_gb300 as tb
    s = workloads.BlockShape("max_b", "decode", "bf16", B=2048, T=0, d=256, H=2, Hkv=1, dh=128, f=256,
                             rope_base=1e4, eps=1e-6, gains="normal")
    T_max = 64
    lens = np.random.default_rng(3).integers(0, T_max - 1, size=s.B).tolist()
    sampled = [0, 1, 777, 2047]
    if cache == "bf16":
        s, inp, kv, y, err = _decode_case(s, 13, lens, T_max, batches_with_data=sampled)
        assert err == 0
        for b in sampled:
            ref = _oracle_step(s, inp, kv, b, lens[b])
            assert_close(y[b, 0].cpu().double().numpy(), ref["y"], "bf16", f"y b={b}")
    else:
        s = s.with_(T=T_max)
        inp = workloads.make_block_inputs(s, seed=13)
        # the sampled sequences hold the oracle's codes of N(0, 1) rows, the others zero codes and scales
        shape = (s.B, s.Hkv, T_max, s.dh)
        kq, vq = np.zeros(shape, np.int8), np.zeros(shape, np.int8)
        ks, vs = np.zeros(shape[:3], np.float32), np.zeros(shape[:3], np.float32)
        for b in sampled:
            kb, vb = workloads.make_cache_rows(s, 13, b, lens[b])
            kq[b, :, :lens[b]], ks[b, :, :lens[b]] = oracle.quantize_rows(workloads.to_f64(kb))
            vq[b, :, :lens[b]], vs[b, :, :lens[b]] = oracle.quantize_rows(workloads.to_f64(vb))
        kv = tb.KVCache(torch.from_numpy(kq).cuda(), torch.from_numpy(vq).cuda(),
                        torch.tensor(lens, dtype=torch.int32).cuda(), None, torch.from_numpy(ks).cuda(),
                        torch.from_numpy(vs).cuda())
        cfg = block_config(s, max_pos=T_max)
        dev = to_device(inp)
        packed = tb.tb_pack_weights(cfg, dev)
        y = tb.tb_block_decode(cfg, packed, dev["x"], kv)
        assert tb.tb_get_device_error(clear=True) == 0
        for b in sampled:
            ref = oracle.block_decode_seq_int8(workloads.to_f64(inp["x"][b, 0]), oracle_weights(inp), oracle_cfg(s),
                                               kq[b], ks[b].astype(np.float64), vq[b], vs[b].astype(np.float64),
                                               lens[b])
            assert_close(y[b, 0].cpu().double().numpy(), ref["y"], "bf16", f"y b={b}")
    assert kv.lens.cpu().tolist() == [n + 1 for n in lens]
