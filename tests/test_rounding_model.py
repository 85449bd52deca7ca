"""The bf16 rounding model and its consistency check, on the CPU.

The GPU parity tests at d = 4096 hold the CUDA path to the model of its bf16
rounding points (tests/rounding_model.py): the GPU must sit as close to the
model as another summation order of the model does, and its error against the
fp64 oracle must be the model's.  These tests show, without a GPU, what that
check accepts and what it catches: a third valid order passes; planted
arithmetic mistakes fail, including one whose error (max-abs ≈ 0.1, relative
L2 ≈ 6e-3) passes the plain relative-L2 bar of 1e-2.
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import BF16_REL_L2_TOL, errors, oracle_cfg, oracle_weights
import rounding_model as rm

T = 256


@pytest.fixture(scope="module")
def gqa():
    s = workloads.CONFIGS["gqa_8k"]
    inp = workloads.make_block_inputs(s.with_(B=1), seed=0, x_tokens=T)
    ref = oracle.block_prefill_seq(workloads.to_f64(inp["x"][0]), oracle_weights(inp), oracle_cfg(s))["y"]
    a = rm.emulate_prefill_seq(inp, s, order="a").double().numpy()
    b = rm.emulate_prefill_seq(inp, s, order="b").double().numpy()
    return s, inp, ref, a, b


def test_orders_differ_by_less_than_the_rounding(gqa):
    """Two summation orders of the model differ (the bf16 roundings amplify
    fp32 order noise), by clearly less than the model's error against the
    oracle; both meet the relative-L2 bar and both miss the 3e-2 max-abs bar."""
    s, inp, ref, a, b = gqa
    noise, ea, eb = errors(b, a), errors(a, ref), errors(b, ref)
    assert noise["max_abs"] > 0
    assert noise["rel_l2"] < 0.6 * ea["rel_l2"]
    for e in (ea, eb):
        assert e["rel_l2"] < BF16_REL_L2_TOL and e["max_abs"] > 3e-2


def test_a_third_order_is_consistent(gqa):
    s, inp, ref, a, b = gqa
    c = rm.emulate_prefill_seq(inp, s, order="c").double().numpy()
    r = rm.rounding_consistency(c, a, b, ref)
    assert r["ok"], r


@pytest.mark.parametrize("plant", [p for p in rm.PLANTS if p != "h_in_bf16"])
def test_planted_mistake_is_caught(gqa, plant):
    s, inp, ref, a, b = gqa
    got = rm.emulate_prefill_seq(inp, s, order="c", plant=plant).double().numpy()
    r = rm.rounding_consistency(got, a, b, ref)
    assert not r["ok"], r


def test_subtle_mistake_passes_the_plain_bars_but_not_the_check(gqa):
    """The second norm's Σh² missing its last 16 columns (r2 off by ~0.2%):
    the result still meets relative L2 ≤ 1e-2 against the oracle, and its
    max-abs error stays at about 0.1, inside the range a fixed d = 4096
    bound would have to allow; the consistency check rejects it."""
    s, inp, ref, a, b = gqa
    got = rm.emulate_prefill_seq(inp, s, order="c", plant="r2_partial_row").double().numpy()
    e = errors(got, ref)
    assert e["rel_l2"] <= BF16_REL_L2_TOL and e["max_abs"] < 0.15
    r = rm.rounding_consistency(got, a, b, ref)
    assert not r["ok_noise"] and not r["ok_err"], r


def test_bf16_residual_stream_is_inside_the_noise(gqa):
    """A limit of the check: rounding h itself to bf16 before the residual
    add adds less error than the order noise, so the check cannot tell it
    apart; the kernels keep h in fp32, which the reading of the rounding
    points fixes, not this test."""
    s, inp, ref, a, b = gqa
    got = rm.emulate_prefill_seq(inp, s, order="c", plant="h_in_bf16").double().numpy()
    assert rm.rounding_consistency(got, a, b, ref)["ok"]


def test_decode_model_matches_oracle_step():
    """One decode step of the model (both orders) over a seeded cache is within
    the relative-L2 bar of the oracle's step, and the orders differ by less
    than the model's error."""
    s = workloads.CONFIGS["gqa_decode"].with_(B=2, T=2048)
    inp = workloads.make_block_inputs(s, seed=3)
    pos = 1500
    k, v = workloads.make_cache_rows(s, 3, 1, pos)
    ref = oracle.block_decode_seq(workloads.to_f64(inp["x"][1, 0]), oracle_weights(inp), oracle_cfg(s),
                                  workloads.to_f64(k), workloads.to_f64(v), pos)["y"]
    ya = rm.emulate_decode_seq(inp, s, 1, k, v, order="a").double().numpy()
    yb = rm.emulate_decode_seq(inp, s, 1, k, v, order="b").double().numpy()
    ea, eb, noise = errors(ya, ref), errors(yb, ref), errors(yb, ya)
    assert ea["rel_l2"] < BF16_REL_L2_TOL and eb["rel_l2"] < BF16_REL_L2_TOL
    assert 0 < noise["rel_l2"] < ea["rel_l2"]


def test_model_prefix_is_the_prefix_of_the_whole():
    """Causality holds in the model too (both orders): the rows of a prefix are
    the first rows of the whole sequence, so the GPU tests may model a prefix."""
    s = workloads.BlockShape("m", "prefill", "bf16", B=1, T=300, d=256, H=4, Hkv=2, dh=64, f=512,
                             rope_base=1e4, eps=1e-6, gains="normal")
    inp = workloads.make_block_inputs(s, seed=4)
    pre = dict(inp, x=inp["x"][:, :130])
    for order in ("a", "b"):
        full = rm.emulate_prefill_seq(inp, s, order=order).numpy()
        part = rm.emulate_prefill_seq(pre, s, order=order).numpy()
        np.testing.assert_allclose(part, full[:130], rtol=0, atol=1e-5)
