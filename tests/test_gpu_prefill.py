"""Prefill parity: the CUDA path through the C ABI against the fp64 oracle on
the same seeded inputs (bf16 cases: the oracle sees the bf16-rounded values).

Small cases span several tiles and a ragged tail; the full workloads run in
the launch configuration the benchmark times, with every row checked where
the oracle is quick and sampled rows (computed exactly, by causality, from
all keys before them) where it is not."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import (BF16_MAX_ABS_TOL, BF16_REL_L2_TOL, assert_close, block_config, errors, oracle_cfg,
                     oracle_weights, to_device)
from rounding_model import ERROR_FACTOR, emulate_prefill_seq, rounding_consistency

pytestmark = pytest.mark.gpu

SMALL = {
    # fp32 storage, GQA 4/2, the tiny workload itself
    "tiny_fp32": workloads.CONFIGS["tiny_fp32"],
    # fp32, MQA, ragged T, two sequences
    "fp32_mqa_ragged": workloads.CONFIGS["tiny_fp32"].with_(name="fp32_mqa_ragged", B=2, T=37, Hkv=1,
                                                           rope_base=500.0),
    # bf16, GQA 4/2, dh 64, two sequences, T not a multiple of 128
    "bf16_gqa_dh64": workloads.BlockShape("bf16_gqa_dh64", "prefill", "bf16", B=2, T=200, d=256, H=4, Hkv=2,
                                          dh=64, f=512, rope_base=1e4, eps=1e-6, gains="normal"),
    # bf16, MQA 4/1, dh 128, ragged
    "bf16_mqa_dh128": workloads.BlockShape("bf16_mqa_dh128", "prefill", "bf16", B=1, T=333, d=512, H=4, Hkv=1,
                                           dh=128, f=1024, rope_base=5e5, eps=1e-5, gains="normal"),
    # bf16, MHA (odd group size 1): query blocks run in pairs; 3 blocks leave the last pair half empty
    "bf16_mha_odd_blocks": workloads.BlockShape("bf16_mha_odd_blocks", "prefill", "bf16", B=2, T=333, d=256, H=4,
                                                Hkv=4, dh=64, f=512, rope_base=1e4, eps=1e-6, gains="normal"),
    # bf16, MHA, dh 128, 5 query blocks (pairs 0-1, 2-3, 4-empty), ragged
    "bf16_mha_dh128": workloads.BlockShape("bf16_mha_dh128", "prefill", "bf16", B=1, T=520, d=512, H=4, Hkv=4,
                                           dh=128, f=1024, rope_base=5e5, eps=1e-5, gains="normal"),
    # bf16, 46 tokens in all: the few-token (K-split) GEMMs in a prefill
    "bf16_few_tokens": workloads.BlockShape("bf16_few_tokens", "prefill", "bf16", B=2, T=23, d=512, H=8, Hkv=2,
                                            dh=64, f=1024, rope_base=1e4, eps=1e-6, gains="normal"),
    # bf16, GQA 8/2, dh 128: the CTA-pair attention with two KV groups of four heads, several query
    # blocks and a ragged last one, two sequences
    "bf16_gqa4_dh128": workloads.BlockShape("bf16_gqa4_dh128", "prefill", "bf16", B=2, T=520, d=1024, H=8,
                                            Hkv=2, dh=128, f=1024, rope_base=5e5, eps=1e-5, gains="normal"),
    # bf16, GQA 8/1 (largest group), one token per sequence
    "bf16_t1": workloads.BlockShape("bf16_t1", "prefill", "bf16", B=3, T=1, d=1024, H=8, Hkv=1, dh=128,
                                    f=1536, rope_base=1e4, eps=1e-6, gains="normal"),
    # bf16, 67 tokens in all: the smallest tile-GEMM prefill; the QKV GEMM's
    # statistics warps cover one partial row group, most CTAs own no row
    "bf16_tile_min": workloads.BlockShape("bf16_tile_min", "prefill", "bf16", B=1, T=67, d=512, H=8, Hkv=2,
                                          dh=64, f=1024, rope_base=1e4, eps=1e-6, gains="normal"),
    # bf16, 2 × 1100 tokens: row groups of 2048 rows, the second one partial,
    # sequence boundaries inside a group
    "bf16_two_groups": workloads.BlockShape("bf16_two_groups", "prefill", "bf16", B=2, T=1100, d=256, H=4,
                                            Hkv=1, dh=64, f=512, rope_base=1e4, eps=1e-6, gains="normal"),
}


def run_prefill(s, inp, with_cache=False, y_dtype=None, T_max=None):
    import causal_gqa_attention_rmsnorm_gb300 as tb
    T = inp["x"].shape[1]
    cfg = block_config(s, max_pos=max(T, T_max or 0, 1))
    dev = to_device(inp)
    packed = tb.tb_pack_weights(cfg, dev)
    kv = None
    if with_cache:
        kv = tb.KVCache.empty(s.B, s.Hkv, T_max or T, s.dh, dtype=s.torch_dtype, fill=float("nan"))
    y = tb.tb_block_prefill(cfg, packed, dev["x"], y_dtype=tb.TB_F32 if y_dtype is None else y_dtype, kv=kv)
    assert tb.tb_get_device_error(clear=True) == 0
    return y, kv


@pytest.mark.parametrize("name", list(SMALL))
def test_prefill_small(name):
    s = SMALL[name]
    inp = workloads.make_block_inputs(s, seed=0)
    y, kv = run_prefill(s, inp, with_cache=True, T_max=s.T + 5)
    ref = oracle.block_prefill(workloads.to_f64(inp["x"]), oracle_weights(inp), oracle_cfg(s))
    assert_close(y.cpu().double().numpy(), ref["y"], s.dtype, "y")
    # the emitted cache holds the post-RoPE keys and values of every position
    assert_close(kv.k[:, :, :s.T].cpu().double().numpy(), ref["k"], s.dtype, "k cache")
    assert_close(kv.v[:, :, :s.T].cpu().double().numpy(), ref["v"], s.dtype, "v cache")
    assert kv.lens.cpu().tolist() == [s.T] * s.B
    # rows past T are untouched
    assert torch.isnan(kv.k[:, :, s.T:].float()).all()


def test_prefill_without_cache_equals_with_cache():
    s = SMALL["bf16_gqa_dh64"]
    inp = workloads.make_block_inputs(s, seed=3)
    y0, _ = run_prefill(s, inp, with_cache=False)
    y1, _ = run_prefill(s, inp, with_cache=True, T_max=256)
    torch.testing.assert_close(y0, y1, rtol=0, atol=1e-5)


def test_prefill_bf16_output():
    import causal_gqa_attention_rmsnorm_gb300 as tb
    s = SMALL["bf16_gqa_dh64"]
    inp = workloads.make_block_inputs(s, seed=1)
    y, _ = run_prefill(s, inp, y_dtype=tb.TB_BF16)
    assert y.dtype == torch.bfloat16
    ref = oracle.block_prefill(workloads.to_f64(inp["x"]), oracle_weights(inp), oracle_cfg(s))
    assert_close(y.cpu().double().numpy(), ref["y"], "bf16", "y (bf16)")


def test_prefill_causality_on_gpu():
    """A prefix of the sequence gives the same rows as the whole sequence."""
    s = SMALL["bf16_mqa_dh128"]
    inp = workloads.make_block_inputs(s, seed=2)
    full, _ = run_prefill(s, inp)
    short = dict(inp, x=inp["x"][:, :130].contiguous())
    part, _ = run_prefill(s.with_(T=130), short)
    torch.testing.assert_close(part, full[:, :130], rtol=0, atol=1e-5)


def test_empty_prefill_is_a_noop():
    import causal_gqa_attention_rmsnorm_gb300 as tb
    s = SMALL["bf16_gqa_dh64"]
    inp = workloads.make_block_inputs(s.with_(B=1, T=4), seed=0)
    cfg = block_config(s, 16)
    dev = to_device(inp)
    packed = tb.tb_pack_weights(cfg, dev)
    x = torch.empty((0, 4, s.d), dtype=torch.bfloat16, device="cuda")
    y = tb.tb_block_prefill(cfg, packed, x)
    assert y.shape == (0, 4, s.d)


def _full_rows_case(name, sample=None, seed=0):
    """Prefill of a whole workload on the GPU and the oracle's rows of every
    sequence (all rows, or ``sample(b, T)``); returns the shape, the inputs,
    y, one error report per checked sequence, and sequence 0's GPU and oracle
    rows as fp64 arrays."""
    s = workloads.CONFIGS[name]
    inp = workloads.make_block_inputs(s, seed=seed)
    y, kv = run_prefill(s, inp, with_cache=True)
    w = oracle_weights(inp)
    cfg = oracle_cfg(s)
    x64 = workloads.to_f64(inp["x"])
    report, seq0 = [], None
    for b in range(s.B):
        rows = None if sample is None else sample(b, s.T)
        if rows is not None and len(rows) == 0:
            continue
        ref = oracle.block_prefill_seq(x64[b], w, cfg, rows=rows)
        got = y[b].cpu().double().numpy()[ref["rows"]]
        report.append(errors(got, ref["y"]))
        if b == 0:
            seq0 = (got, ref["y"])
        S = ref["k"].shape[1]
        assert_close(kv.k[b, :, :S].cpu().double().numpy(), ref["k"], s.dtype, f"k cache b={b}")
        assert_close(kv.v[b, :, :S].cpu().double().numpy(), ref["v"], s.dtype, f"v cache b={b}")
    return s, inp, y, report, seq0


def test_prefill_mha_768_all_rows():
    s, inp, y, rep, _ = _full_rows_case("mha_768")
    for e in rep:
        assert e["finite"] and e["rel_l2"] <= BF16_REL_L2_TOL and e["max_abs"] <= BF16_MAX_ABS_TOL, e


def _gqa_rows(b, T):
    """gqa_8k rows checked against the oracle: every row of sequence 0; of the
    others the first 64, the last 64 and 256 seeded-random rows (each computed
    over the sequence's full K/V; the emitted cache is compared whole)."""
    if b == 0:
        return None
    rng = np.random.default_rng(100 + b)
    return np.unique(np.r_[np.arange(64), np.arange(T - 64, T), rng.choice(T, 256, replace=False)])


_D4096 = {}
ANCHOR_ROWS = 1024


def _d4096_run(name):
    """Run a d = 4096 workload once per session: its error reports, sequence
    0's GPU rows and oracle rows (all T), and the rounding model of sequence 0
    in order "a" (all T rows)."""
    if name not in _D4096:
        sample = _gqa_rows if name == "gqa_8k" else None
        s, inp, y, rep, (got0, ref0) = _full_rows_case(name, sample=sample)
        assert torch.isfinite(y).all()
        del y
        emu0 = emulate_prefill_seq(inp, s, b=0, order="a").double().numpy()
        model = errors(emu0, ref0)
        for b, e in enumerate(rep):
            print(f"{name} seq {b}: rel_l2 {e['rel_l2']:.2e} max_abs {e['max_abs']:.2e}")
        print(f"{name} rounding model, seq 0: rel_l2 {model['rel_l2']:.2e} max_abs {model['max_abs']:.2e}")
        _D4096[name] = dict(s=s, inp=inp, rep=rep, got0=got0, ref0=ref0, emu0=emu0, model=model)
    return _D4096[name]


@pytest.mark.parametrize("name", ["llama2_7b", "gqa_8k"])
def test_prefill_d4096_error_is_bf16_rounding(name):
    """The GPU's deviation at d = 4096 is the bf16 rounding the path is built
    with, and nothing else.  On the first 1024 rows of sequence 0 the GPU is as
    close to the rounding model (tests/rounding_model.py, order "a") as the
    model's second summation order is (within 1.5x, max-abs and relative L2);
    over all rows of sequence 0 its error against the oracle is within 1.25x of
    the model's."""
    r = _d4096_run(name)
    R = ANCHOR_ROWS
    pre = dict(r["inp"], x=r["inp"]["x"][:1, :R])
    emu_b = emulate_prefill_seq(pre, r["s"], b=0, order="b").double().numpy()
    c = rounding_consistency(r["got0"][:R], r["emu0"][:R], emu_b, r["ref0"][:R])
    print(f"{name} first {R} rows: order noise {c['noise']}, GPU to model {c['dev']}, "
          f"model error {c['model']}, GPU error {c['err']}")
    assert c["ok_noise"], c
    gpu, model = errors(r["got0"], r["ref0"]), r["model"]
    assert gpu["max_abs"] <= ERROR_FACTOR * model["max_abs"], (gpu, model)
    assert gpu["rel_l2"] <= ERROR_FACTOR * model["rel_l2"], (gpu, model)


@pytest.mark.parametrize("name", ["llama2_7b", "gqa_8k"])
def test_prefill_d4096_rel_l2_and_rounding_bound(name):
    """Relative-L2 bar 1e-2 on every checked sequence, and max-abs within
    1.25x the rounding model's max-abs error on all rows of sequence 0 (a
    bound measured in the same run, over at least as many outputs as any
    other checked sequence has)."""
    r = _d4096_run(name)
    bound = ERROR_FACTOR * r["model"]["max_abs"]
    for e in r["rep"]:
        assert e["finite"] and e["rel_l2"] <= BF16_REL_L2_TOL, e
        assert e["max_abs"] <= bound, (e, bound)


@pytest.mark.xfail(strict=True, reason="bf16 operand rounding alone exceeds 3e-2 max-abs at d = 4096 "
                                       "(see test_rounding_floor.py)")
@pytest.mark.parametrize("name", ["llama2_7b", "gqa_8k"])
def test_prefill_d4096_max_abs_bar(name):
    for e in _d4096_run(name)["rep"]:
        assert e["max_abs"] <= BF16_MAX_ABS_TOL, e
