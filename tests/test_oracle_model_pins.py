"""Pins of the model-level oracle (embedding, stack, final norm, LM head,
per-token loss) to facts fixed outside it, with planted mistakes each pin set
must catch.  "Transformer block" (tirogla.com), "How it works", steps 1 and 4;
"The Transformer" (GenerativeAIDocs) §5 "A tensor's journey"."""
import math

import numpy as np
import pytest

import oracle
import oracle.block as ob
import oracle.model as om

RNG = np.random.default_rng(77)


def _cfg(window=0):
    return ob.Cfg(d=24, H=4, Hkv=2, dh=6, f=40, rope_base=1e4, eps=1e-6, window=window)


def _layer(cfg, rng, std=0.25):
    return {
        "g_attn": 1 + 0.1 * rng.standard_normal(cfg.d), "g_mlp": 1 + 0.1 * rng.standard_normal(cfg.d),
        "wq": std * rng.standard_normal((cfg.d, cfg.H * cfg.dh)),
        "wk": std * rng.standard_normal((cfg.d, cfg.Hkv * cfg.dh)),
        "wv": std * rng.standard_normal((cfg.d, cfg.Hkv * cfg.dh)),
        "wo": std * rng.standard_normal((cfg.H * cfg.dh, cfg.d)),
        "w1": std * rng.standard_normal((cfg.d, cfg.f)), "w3": std * rng.standard_normal((cfg.d, cfg.f)),
        "w2": std * rng.standard_normal((cfg.f, cfg.d)),
    }


def _model(cfg, L, V, rng):
    return (rng.standard_normal((V, cfg.d)), [_layer(cfg, rng) for _ in range(L)],
            1 + 0.1 * rng.standard_normal(cfg.d), 0.3 * rng.standard_normal((cfg.d, V)))


def check_embed_gather():
    table = RNG.standard_normal((11, 5))
    ids = [3, 0, 10, 3, 7]
    x = om.embed(table, ids)
    for t, i in enumerate(ids):
        np.testing.assert_array_equal(x[t], table[i])


def check_nll_closed_forms():
    V = 37
    # uniform logits: every token costs ln V
    np.testing.assert_allclose(om.token_nll(np.zeros((3, V)), [0, 5, 36]), math.log(V), rtol=1e-15)
    # library cross-check of logsumexp, and shift invariance at huge logits
    from scipy.special import logsumexp
    z = 3 * RNG.standard_normal((4, V))
    t = [1, 2, 30, 0]
    want = logsumexp(z, axis=1) - z[np.arange(4), t]
    np.testing.assert_allclose(om.token_nll(z, t), want, rtol=1e-13)
    np.testing.assert_allclose(om.token_nll(z + 3000.0, t), want, rtol=1e-9)
    # a target 20 above the rest costs log(1 + (V-1)·e^-20) (to the rounding of lse ≈ 20)
    z = np.zeros((1, V)); z[0, 4] = 20.0
    assert abs(om.token_nll(z, [4])[0] - math.log1p((V - 1) * math.exp(-20.0))) < 1e-13


def check_head_final_norm():
    # the final RMSNorm makes the logits independent of the residual's scale (eps = 0)
    d, V = 16, 9
    h = RNG.standard_normal((5, d)); g = 1 + 0.1 * RNG.standard_normal(d); w = RNG.standard_normal((d, V))
    np.testing.assert_allclose(om.lm_head(7.5 * h, g, w, 0.0), om.lm_head(h, g, w, 0.0), rtol=1e-12)
    # closed form on a constant residual row c·1: RMSNorm gives g, logits = g·W_U
    np.testing.assert_allclose(om.lm_head(np.full((1, d), -2.0), g, w, 0.0)[0], -(g @ w), rtol=1e-12)


def check_stack_zero_layers_and_tied_head():
    cfg = _cfg()
    table, _, g, _ = _model(cfg, 0, 13, RNG)
    ids = [4, 4, 12, 0]
    out = om.stack_prefill_seq(ids, table, [], cfg, g, table.T)
    # no blocks: the head sees the embeddings; a tied head scores token v by RMSNorm(x)·E[v]
    xn = ob.rms_norm(table[ids], g, cfg.eps)
    np.testing.assert_allclose(out["logits"], xn @ table.T, rtol=1e-13)
    for t in range(len(ids)):
        for v in (0, 5, 12):
            assert abs(out["logits"][t, v] - float(xn[t] @ table[v])) < 1e-12


def check_stack_decode_continues_prefill():
    for W in (0, 3):
        cfg = _cfg(W)
        table, layers, g, wu = _model(cfg, 3, 17, RNG)
        ids = list(RNG.integers(0, 17, size=9))
        full = om.stack_prefill_seq(ids, table, layers, cfg, g, wu)
        pre = om.stack_prefill_seq(ids[:-1], table, layers, cfg, g, wu)
        dec = om.stack_decode_seq(ids[-1], table, layers, cfg, g, wu, pre["k"], pre["v"], len(ids) - 1)
        np.testing.assert_allclose(dec["logits"], full["logits"][-1], rtol=1e-10, atol=1e-12)
        for l in range(3):
            np.testing.assert_allclose(dec["k"][l], full["k"][l][:, -1], rtol=1e-12, atol=1e-13)


def check_stack_is_blocks_in_order():
    # swapping two different layers changes the output: the layers run in the given order
    cfg = _cfg()
    table, layers, g, wu = _model(cfg, 2, 11, RNG)
    ids = [1, 2, 3, 4, 5]
    a = om.stack_prefill_seq(ids, table, layers, cfg, g, wu)["logits"]
    b = om.stack_prefill_seq(ids, table, layers[::-1], cfg, g, wu)["logits"]
    assert np.max(np.abs(a - b)) > 1e-3
    # and each layer is one block applied to the previous one's output
    x = om.embed(table, ids)
    for lw in layers:
        x = ob.block_prefill_seq(x, lw, cfg)["y"]
    np.testing.assert_allclose(a, om.lm_head(x, g, wu, cfg.eps), rtol=1e-13)


CHECKS = [check_embed_gather, check_nll_closed_forms, check_head_final_norm,
          check_stack_zero_layers_and_tied_head, check_stack_decode_continues_prefill, check_stack_is_blocks_in_order]


def _run(check):
    global RNG
    RNG = np.random.default_rng(abs(hash(check.__name__)) % (2 ** 32))
    check()


@pytest.mark.parametrize("check", CHECKS, ids=lambda c: c.__name__)
def test_model_oracle_pin(check):
    _run(check)


def mut_no_final_norm(monkeypatch):
    monkeypatch.setattr(om, "lm_head", lambda h, g, w, eps: np.asarray(h, float) * np.asarray(g, float) @ w)


def mut_nll_no_max(monkeypatch):
    def nll(z, t):
        z = np.asarray(z, float)
        return np.log(np.sum(np.exp(z), axis=-1)) - z[np.arange(z.shape[0]), np.asarray(t)]
    monkeypatch.setattr(om, "token_nll", nll)


def mut_embed_shift(monkeypatch):
    monkeypatch.setattr(om, "embed", lambda table, ids: np.asarray(table, float)[(np.asarray(ids) + 1) % len(table)])


MUTANTS = [mut_no_final_norm, mut_nll_no_max, mut_embed_shift]


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda m: m.__name__)
def test_planted_mistake_is_caught(mutant, monkeypatch):
    mutant(monkeypatch)
    caught = False
    for check in CHECKS:
        try:
            with np.errstate(all="ignore"):
                _run(check)
        except (AssertionError, FloatingPointError, ValueError):
            caught = True
    assert caught
