"""Pins of the fp64 oracle to facts fixed outside itself.

Each ``check_*`` asserts a closed form, an invariant, a library cross-check or a
brute-force result.  The tests at the bottom plant plausible mistakes in the
oracle (the pitfalls the "Transformer block" page lists, plus sign, index and
scale slips) and require that at least one check catches each of them.
"""
import math
import zlib

import numpy as np
import pytest
import torch

import oracle
import oracle.block as ob

RNG = np.random.default_rng(1234)


def _cfg(d=32, H=4, Hkv=2, dh=8, f=48, base=1e4, eps=1e-6):
    return ob.Cfg(d, H, Hkv, dh, f, base, eps)


def _weights(cfg, rng, std=0.3, gains=True):
    w = {
        "g_attn": 1 + 0.1 * rng.standard_normal(cfg.d) if gains else np.ones(cfg.d),
        "wq": std * rng.standard_normal((cfg.d, cfg.H * cfg.dh)),
        "wk": std * rng.standard_normal((cfg.d, cfg.Hkv * cfg.dh)),
        "wv": std * rng.standard_normal((cfg.d, cfg.Hkv * cfg.dh)),
        "wo": std * rng.standard_normal((cfg.H * cfg.dh, cfg.d)),
        "g_mlp": 1 + 0.1 * rng.standard_normal(cfg.d) if gains else np.ones(cfg.d),
        "w1": std * rng.standard_normal((cfg.d, cfg.f)),
        "w3": std * rng.standard_normal((cfg.d, cfg.f)),
        "w2": std * rng.standard_normal((cfg.f, cfg.d)),
    }
    return w


# ----------------------------------------------------------------------------
# RoPE: "Transformers" 3.2 and the Transformer block page (interleaved pairs,
# angle t·base^(-2i/dh)).
# ----------------------------------------------------------------------------

def check_rope_closed_form():
    # dh = 4, base 100, position 1: pair 0 turns by 1 rad, pair 1 by 100^(-1/2) = 0.1 rad.
    u = np.array([[[1.0, 0.0, 0.0, 1.0]]])          # [T=1, heads=1, dh=4]
    got = ob.rope(u, [1], 100.0)[0, 0]
    want = [math.cos(1.0), math.sin(1.0), -math.sin(0.1), math.cos(0.1)]
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-15)
    # position 3: angles 3 and 0.3
    got = ob.rope(np.array([[[2.0, -1.0, 0.5, 0.25]]]), [3], 100.0)[0, 0]
    c3, s3, c03, s03 = math.cos(3), math.sin(3), math.cos(0.3), math.sin(0.3)
    want = [2 * c3 + s3, 2 * s3 - c3, 0.5 * c03 - 0.25 * s03, 0.5 * s03 + 0.25 * c03]
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-15)


def check_rope_invariants():
    T, heads, dh = 9, 3, 16
    u = RNG.standard_normal((T, heads, dh))
    pos = np.arange(T) * 37
    r = ob.rope(u, pos, 1e4)
    # position 0 is the identity
    np.testing.assert_array_equal(ob.rope(u[:1], [0], 1e4), u[:1])
    # rotations keep every pair's norm
    np.testing.assert_allclose(r[..., 0::2] ** 2 + r[..., 1::2] ** 2,
                               u[..., 0::2] ** 2 + u[..., 1::2] ** 2, rtol=1e-12)
    # <R_m q, R_n k> depends only on n - m
    q, k = RNG.standard_normal(dh), RNG.standard_normal(dh)
    for m, n, s in [(0, 5, 11), (7, 2, 100), (1000, 1003, 4321)]:
        a = ob.rope(q[None, None], [m], 1e4)[0, 0] @ ob.rope(k[None, None], [n], 1e4)[0, 0]
        b = ob.rope(q[None, None], [m + s], 1e4)[0, 0] @ ob.rope(k[None, None], [n + s], 1e4)[0, 0]
        c = q @ ob.rope(k[None, None], [n - m], 1e4)[0, 0]
        assert abs(a - b) < 1e-10 and abs(a - c) < 1e-10


# ----------------------------------------------------------------------------
# RMSNorm: Transformer block page (Rust rms_norm), Go rmsnorm.
# ----------------------------------------------------------------------------

def check_rmsnorm():
    d, eps = 16, 1e-6
    # a constant vector c·1 maps to c / sqrt(c² + eps) · g
    g = 1 + 0.1 * RNG.standard_normal(d)
    for c in (0.01, -0.003, 2.5):
        got = ob.rms_norm(np.full((1, d), c), g, eps)[0]
        np.testing.assert_allclose(got, c / math.sqrt(c * c + eps) * g, rtol=1e-13)
    # with unit gains the mean square of the output is ms / (ms + eps)
    x = 0.01 * RNG.standard_normal((5, d))
    y = ob.rms_norm(x, np.ones(d), eps)
    ms = np.mean(x * x, axis=1)
    np.testing.assert_allclose(np.mean(y * y, axis=1), ms / (ms + eps), rtol=1e-12)
    # with eps = 0 the map is invariant to a positive scale of its input
    np.testing.assert_allclose(ob.rms_norm(7.0 * x, g, 0.0), ob.rms_norm(x, g, 0.0), rtol=1e-12)


# ----------------------------------------------------------------------------
# SiLU: SiLU(z) = z·σ(z); SiLU(0) = 0 and SiLU(z) - SiLU(-z) = z.
# ----------------------------------------------------------------------------

def check_silu():
    z = np.linspace(-20, 20, 81)
    assert ob.silu(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(ob.silu(z) - ob.silu(-z), z, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(ob.silu(np.array([1.0])), [1.0 / (1.0 + math.exp(-1.0))], rtol=1e-15)


# ----------------------------------------------------------------------------
# Softmax and attention: "Transformers" 1.3 and 5.1.
# ----------------------------------------------------------------------------

def check_softmax():
    s = RNG.standard_normal((6, 9)) * 5
    s[2, 5:] = -np.inf
    p = ob.softmax_rows(s)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    assert (p >= 0).all() and (p[2, 5:] == 0).all()
    # scores far beyond exp's range still give a finite, shift-invariant result
    np.testing.assert_allclose(ob.softmax_rows(s + 5000.0), p, rtol=1e-12, atol=1e-300)


def _sdpa_reference(q, k, v):
    """torch's fp64 CPU scaled_dot_product_attention with the causal flag;
    GQA by repeating each KV head for its H/Hkv query heads."""
    G = q.shape[1] // k.shape[1]
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]
    kt = torch.from_numpy(k).permute(1, 0, 2)[None].repeat_interleave(G, dim=1)
    vt = torch.from_numpy(v).permute(1, 0, 2)[None].repeat_interleave(G, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True)
    return o[0].permute(1, 0, 2).numpy()


def check_attention_vs_library():
    for (T, H, Hkv, dh, scale) in [(7, 4, 2, 8, 1.0), (33, 6, 3, 16, 1.0), (20, 4, 1, 8, 60.0)]:
        q = RNG.standard_normal((T, H, dh)) * scale
        k = RNG.standard_normal((T, Hkv, dh)) * scale
        v = RNG.standard_normal((T, Hkv, dh))
        got = ob.causal_attention(q, k, v, np.arange(T))
        assert np.isfinite(got).all()
        np.testing.assert_allclose(got, _sdpa_reference(q, k, v), rtol=1e-10, atol=1e-12)


def check_attention_closed_forms():
    H, Hkv, dh = 4, 2, 6
    # one token: the output is its own value vector
    q = RNG.standard_normal((1, H, dh)); k = RNG.standard_normal((1, Hkv, dh))
    v = RNG.standard_normal((1, Hkv, dh))
    o = ob.causal_attention(q, k, v, [0])
    for h in range(H):
        np.testing.assert_allclose(o[0, h], v[0, h // (H // Hkv)], rtol=1e-15)
    # zero queries give uniform weights: o_i is the mean of v_0..v_i
    T = 9
    k = RNG.standard_normal((T, Hkv, dh)); v = RNG.standard_normal((T, Hkv, dh))
    o = ob.causal_attention(np.zeros((T, H, dh)), k, v, np.arange(T))
    run_mean = np.cumsum(v, axis=0) / np.arange(1, T + 1)[:, None, None]
    for h in range(H):
        np.testing.assert_allclose(o[:, h], run_mean[:, h // (H // Hkv)], rtol=1e-13, atol=1e-15)
    # one-hot values expose the weights: row i sums to 1 and is 0 past the diagonal
    T = 6
    q = RNG.standard_normal((T, 2, T)); k = RNG.standard_normal((T, 1, T))
    v = np.eye(T)[:, None, :]
    p = ob.causal_attention(q, k, v, np.arange(T))[:, 0]
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-14)
    assert (p >= 0).all() and np.all(np.triu(p, 1) == 0) and (np.diag(p) > 0).all()


def check_attention_brute_force():
    # tiny case with scalar loops: query head h uses KV head h // (H/Hkv),
    # key j is visible to query i iff j <= i
    T, H, Hkv, dh = 4, 2, 1, 3
    q = RNG.standard_normal((T, H, dh)); k = RNG.standard_normal((T, Hkv, dh))
    v = RNG.standard_normal((T, Hkv, dh))
    got = ob.causal_attention(q, k, v, list(range(T)))
    for i in range(T):
        for h in range(H):
            g = h // (H // Hkv)
            w = [math.exp(sum(q[i, h, e] * k[j, g, e] for e in range(dh)) / math.sqrt(dh))
                 for j in range(i + 1)]
            for e in range(dh):
                want = sum(w[j] * v[j, g, e] for j in range(i + 1)) / sum(w)
                assert abs(got[i, h, e] - want) < 1e-12


# ----------------------------------------------------------------------------
# Sliding window: "09 The Transformer" §5, sliding-window attention.
# ----------------------------------------------------------------------------

def _golden_rows(name):
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", name)
    rows = []
    with open(path) as fh:
        for line in fh:
            if line.strip() and not line.startswith("#"):
                rows.append([int(x) for x in line.split()])
    return rows


def check_window_worked_example():
    # the pages' example: with W = 4096 token 10000 sees exactly tokens 5905..10000
    for W, i, first, last in _golden_rows("window_example.tsv"):
        idx = np.nonzero(ob.visible_keys([i], i + 1, W)[0])[0]
        assert idx[0] == first and idx[-1] == last and len(idx) == last - first + 1, (W, i, idx[[0, -1]])


def check_window_reductions():
    T, H, Hkv, dh = 12, 4, 2, 6
    G = H // Hkv
    q = RNG.standard_normal((T, H, dh)); k = RNG.standard_normal((T, Hkv, dh))
    v = RNG.standard_normal((T, Hkv, dh))
    full = ob.causal_attention(q, k, v, np.arange(T))
    # a window at least as long as the sequence is full causal attention
    for W in (T, T + 3):
        np.testing.assert_array_equal(ob.causal_attention(q, k, v, np.arange(T), W), full)
    # W = 1: every query sees only itself
    o1 = ob.causal_attention(q, k, v, np.arange(T), 1)
    for h in range(H):
        np.testing.assert_allclose(o1[:, h], v[:, h // G], rtol=1e-15)
    # zero queries: o_i is the mean of v over the last min(i + 1, W) positions
    W = 4
    o = ob.causal_attention(np.zeros((T, H, dh)), k, v, np.arange(T), W)
    for i in range(T):
        lo = max(0, i - W + 1)
        for h in range(H):
            np.testing.assert_allclose(o[i, h], v[lo:i + 1, h // G].mean(axis=0), rtol=1e-13, atol=1e-15)


def check_window_brute_force():
    # scalar loops: key j visible to query i iff i - W < j <= i
    T, H, Hkv, dh, W = 7, 2, 1, 3, 3
    q = RNG.standard_normal((T, H, dh)); k = RNG.standard_normal((T, Hkv, dh))
    v = RNG.standard_normal((T, Hkv, dh))
    got = ob.causal_attention(q, k, v, list(range(T)), W)
    for i in range(T):
        js = range(max(0, i - W + 1), i + 1)
        for h in range(H):
            g = h // (H // Hkv)
            w = [math.exp(sum(q[i, h, e] * k[j, g, e] for e in range(dh)) / math.sqrt(dh)) for j in js]
            for e in range(dh):
                want = sum(wj * v[j, g, e] for wj, j in zip(w, js)) / sum(w)
                assert abs(got[i, h, e] - want) < 1e-12


def check_window_decode_matches_prefill():
    # decoding token T-1 over the windowed cache equals row T-1 of the windowed prefill
    base = _cfg()
    for W in (1, 3, 8):
        cfg = ob.Cfg(base.d, base.H, base.Hkv, base.dh, base.f, base.rope_base, base.eps, W)
        w = _weights(cfg, RNG)
        T = 11
        x = RNG.standard_normal((T, cfg.d))
        pre = ob.block_prefill_seq(x, w, cfg)
        dec = ob.block_decode_seq(x[T - 1], w, cfg, pre["k"], pre["v"], T - 1)
        np.testing.assert_allclose(dec["y"], pre["y"][T - 1], rtol=1e-12, atol=1e-12)
        # and differs from full attention's row
        full = ob.block_prefill_seq(x, w, _cfg())
        assert np.max(np.abs(pre["y"][T - 1] - full["y"][T - 1])) > 1e-6


# ----------------------------------------------------------------------------
# Paged cache layout: "Transformer block" page, implementation notes.
# ----------------------------------------------------------------------------

def check_paged_gather():
    # scatter a contiguous cache into a shuffled pool by direct indexing, then
    # the gather must give it back exactly, including a partial last page
    Hkv, dh, ps, n, num_pages = 3, 5, 4, 14, 9
    cache = RNG.standard_normal((Hkv, n, dh))
    table = RNG.permutation(num_pages)[: (n + ps - 1) // ps]
    pool = np.full((num_pages, Hkv, ps, dh), np.nan)
    for t in range(n):
        pool[table[t // ps], :, t % ps, :] = cache[:, t, :]
    np.testing.assert_array_equal(ob.gather_paged(pool, table, ps, n), cache)
    # row 6 sits in the second page of the table at offset 2
    np.testing.assert_array_equal(ob.gather_paged(pool, table, ps, n)[:, 6], pool[table[1], :, 2])


# ----------------------------------------------------------------------------
# int8 cache rows: "The Transformer Architecture", pitfalls (quantise the cache).
# ----------------------------------------------------------------------------

def check_int8_rows():
    # rows of very different magnitudes, each with its own scale
    x = RNG.standard_normal((6, 32)) * np.array([1e-3, 0.1, 1, 10, 300, 1])[:, None]
    x[5] = 0.0
    q, s = ob.quantize_rows(x)
    assert q.dtype == np.int8 and s.shape == (6,)
    # the scale is the fp32 number max|x|/127 (two fp32 roundings from the exact quotient)
    np.testing.assert_allclose(s[:5], np.max(np.abs(x[:5]), axis=1) / 127, rtol=2.5e-7)
    # the largest element of a row maps to ±127; every element is within s/2
    for r in range(5):
        assert abs(int(q[r, np.argmax(np.abs(x[r]))])) == 127
        assert np.all(np.abs(ob.dequantize_rows(q, s)[r] - x[r]) <= s[r] / 2 * (1 + 1e-4))
    assert s[5] == 0 and not q[5].any()
    # rows built from codes and a scale come back exactly
    codes = RNG.integers(-127, 128, size=(3, 16)); codes[:, 0] = 127
    q2, s2 = ob.quantize_rows(codes * 0.25)
    np.testing.assert_array_equal(q2, codes)
    np.testing.assert_array_equal(s2, 0.25)
    # halfway values go to the even code: x/s = 0.5, 1.5, 2.5, -0.5, -1.5 with s = 0.25
    q3, s3 = ob.quantize_rows(np.array([31.75, 0.125, 0.375, 0.625, -0.125, -0.375]))
    assert s3 == 0.25
    np.testing.assert_array_equal(q3, [127, 0, 2, 2, 0, -2])


def check_int8_decode_close_to_exact():
    cfg = _cfg()
    w = _weights(cfg, RNG)
    T = 12
    x = RNG.standard_normal((T, cfg.d))
    pre = ob.block_prefill_seq(x, w, cfg)
    kq, ks = ob.quantize_rows(pre["k"][:, :T - 1])
    vq, vs = ob.quantize_rows(pre["v"][:, :T - 1])
    dec = ob.block_decode_seq_int8(x[T - 1], w, cfg, kq, ks, vq, vs, T - 1)
    exact = pre["y"][T - 1]
    rel = np.linalg.norm(dec["y"] - exact) / np.linalg.norm(exact)
    assert 0 < rel < 1e-2, rel
    # the appended row is the quantised exact k
    kq_new, ks_new = ob.quantize_rows(pre["k"][:, T - 1])
    np.testing.assert_array_equal(dec["k_q"], kq_new)


# ----------------------------------------------------------------------------
# Block-level: residual wiring, GQA sharing, causality, decode vs prefill.
# ----------------------------------------------------------------------------

def check_block_zero_branches():
    cfg = _cfg()
    w = _weights(cfg, RNG)
    x = RNG.standard_normal((10, cfg.d))
    w0 = dict(w, wo=np.zeros_like(w["wo"]), w2=np.zeros_like(w["w2"]))
    np.testing.assert_array_equal(ob.block_prefill_seq(x, w0, cfg)["y"], x)


def check_block_uniform_attention_closed_form():
    # MHA with d = H·dh, Wq = 0 (uniform attention), Wv = Wo = I and W2 = 0:
    # y_t = x_t + mean_{j<=t} RMSNorm(x_j)
    cfg = ob.Cfg(d=24, H=3, Hkv=3, dh=8, f=16, rope_base=1e4, eps=1e-6)
    w = _weights(cfg, RNG)
    w.update(wq=np.zeros((24, 24)), wv=np.eye(24), wo=np.eye(24), w2=np.zeros((16, 24)))
    x = RNG.standard_normal((11, 24))
    xn = ob.rms_norm(x, w["g_attn"], cfg.eps)
    want = x + np.cumsum(xn, axis=0) / np.arange(1, 12)[:, None]
    np.testing.assert_allclose(ob.block_prefill_seq(x, w, cfg)["y"], want, rtol=1e-12, atol=1e-13)


def check_gqa_equals_duplicated_mha():
    cfg = _cfg(d=32, H=4, Hkv=2, dh=8)
    w = _weights(cfg, RNG)
    G = cfg.G
    mha = ob.Cfg(cfg.d, cfg.H, cfg.H, cfg.dh, cfg.f, cfg.rope_base, cfg.eps)
    dup = lambda m: np.concatenate([m[:, (h // G) * cfg.dh:(h // G + 1) * cfg.dh]
                                    for h in range(cfg.H)], axis=1)
    wm = dict(w, wk=dup(w["wk"]), wv=dup(w["wv"]))
    x = RNG.standard_normal((13, cfg.d))
    np.testing.assert_allclose(ob.block_prefill_seq(x, w, cfg)["y"],
                               ob.block_prefill_seq(x, wm, mha)["y"], rtol=1e-12, atol=1e-13)


def check_causality_prefix():
    cfg = _cfg()
    w = _weights(cfg, RNG)
    x = RNG.standard_normal((12, cfg.d))
    full = ob.block_prefill_seq(x, w, cfg)
    for Tp in (1, 5, 11):
        part = ob.block_prefill_seq(x[:Tp], w, cfg)
        np.testing.assert_allclose(part["y"], full["y"][:Tp], rtol=1e-12, atol=1e-13)
    sub = ob.block_prefill_seq(x, w, cfg, rows=[0, 4, 7])
    np.testing.assert_allclose(sub["y"], full["y"][[0, 4, 7]], rtol=1e-12, atol=1e-13)


def check_decode_matches_prefill():
    cfg = _cfg(base=500.0)
    w = _weights(cfg, RNG)
    T = 10
    x = RNG.standard_normal((T, cfg.d))
    full = ob.block_prefill_seq(x, w, cfg)
    # one step over a cache the prefill of the first T-1 tokens emitted
    pre = ob.block_prefill_seq(x[:T - 1], w, cfg)
    cache_k = np.concatenate([pre["k"], np.full((cfg.Hkv, 5, cfg.dh), np.nan)], axis=1)
    cache_v = np.concatenate([pre["v"], np.full((cfg.Hkv, 5, cfg.dh), np.nan)], axis=1)
    dec = ob.block_decode_seq(x[T - 1], w, cfg, cache_k, cache_v, T - 1)
    np.testing.assert_allclose(dec["y"], full["y"][T - 1], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dec["k"], full["k"][:, T - 1], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dec["v"], full["v"][:, T - 1], rtol=1e-12, atol=1e-13)
    # a chain of decode steps from a 3-token prefill reproduces rows 3..T-1
    pre = ob.block_prefill_seq(x[:3], w, cfg)
    ck, cv = list(pre["k"].transpose(1, 0, 2)), list(pre["v"].transpose(1, 0, 2))
    for t in range(3, T):
        dec = ob.block_decode_seq(x[t], w, cfg, np.stack(ck, 1), np.stack(cv, 1), t)
        np.testing.assert_allclose(dec["y"], full["y"][t], rtol=1e-12, atol=1e-13)
        ck.append(dec["k"]); cv.append(dec["v"])


def check_swiglu_closed_form():
    # one token, d = 2, f = 1: W1 reads component 0, W3 reads component 1, W2
    # writes component 0, eps = 0.  SiLU acts on the W1 (gate) product only.
    cfg = ob.Cfg(d=2, H=1, Hkv=1, dh=2, f=1, rope_base=1e4, eps=0.0)
    w = {"g_mlp": np.ones(2), "w1": np.array([[1.0], [0.0]]), "w3": np.array([[0.0], [1.0]]),
         "w2": np.array([[1.0, 0.0]])}
    h = np.array([[3.0, 4.0]])                        # mean square 12.5
    a0, a1 = 3.0 / math.sqrt(12.5), 4.0 / math.sqrt(12.5)
    want = np.array([[3.0 + a0 / (1.0 + math.exp(-a0)) * a1, 4.0]])
    np.testing.assert_allclose(ob.mlp_branch(h, w, cfg), want, rtol=1e-15)


CHECKS = [check_rope_closed_form, check_swiglu_closed_form, check_rope_invariants, check_rmsnorm, check_silu, check_softmax,
          check_attention_vs_library, check_attention_closed_forms, check_attention_brute_force,
          check_block_zero_branches, check_block_uniform_attention_closed_form,
          check_gqa_equals_duplicated_mha, check_causality_prefix, check_decode_matches_prefill,
          check_window_worked_example, check_window_reductions, check_window_brute_force,
          check_window_decode_matches_prefill, check_paged_gather, check_int8_rows,
          check_int8_decode_close_to_exact]


def _run(check):
    """Run a check with its own seeded random stream, so that its inputs do
    not depend on which checks ran before it."""
    global RNG
    RNG = np.random.default_rng(zlib.crc32(check.__name__.encode()))
    check()


@pytest.mark.parametrize("check", CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    _run(check)


def test_batched_entry_points_match_per_sequence():
    cfg = _cfg()
    w = _weights(cfg, RNG)
    x = RNG.standard_normal((3, 7, cfg.d))
    out = oracle.block_prefill(x, w, cfg)
    for b in range(3):
        np.testing.assert_array_equal(out["y"][b], ob.block_prefill_seq(x[b], w, cfg)["y"])
    assert out["k"].shape == (3, cfg.Hkv, 7, cfg.dh)


# ----------------------------------------------------------------------------
# Planted mistakes.  Each mutant replaces one oracle function on the CPU; the
# pins above must reject it.
# ----------------------------------------------------------------------------

def _orig(name):
    return getattr(ob, name)


def mut_diagonal(monkeypatch):
    # mask built with j < i
    def attn(q, k, v, q_pos, window=0):
        q, k, v = (np.asarray(a, float) for a in (q, k, v))
        G = q.shape[1] // k.shape[1]
        vis = np.arange(k.shape[0])[None, :] < np.asarray(q_pos)[:, None]
        if window > 0:
            vis = vis & (np.arange(k.shape[0])[None, :] > np.asarray(q_pos)[:, None] - window)
        o = np.empty_like(q)
        for h in range(q.shape[1]):
            s = np.where(vis, q[:, h] @ k[:, h // G].T / math.sqrt(q.shape[2]), -np.inf)
            with np.errstate(invalid="ignore"):
                o[:, h] = ob.softmax_rows(s) @ v[:, h // G]
        return o
    monkeypatch.setattr(ob, "causal_attention", attn)


def mut_rope_on_v(monkeypatch):
    orig = _orig("qkv_heads")
    def qkv(xn, w, cfg, positions):
        q, k, v = orig(xn, w, cfg, positions)
        return q, k, ob.rope(v, positions, cfg.rope_base)
    monkeypatch.setattr(ob, "qkv_heads", qkv)


def mut_cache_pre_rope(monkeypatch):
    orig = _orig("block_prefill_seq")
    def prefill(x, w, cfg, rows=None):
        out = orig(x, w, cfg, rows)
        S = out["k"].shape[1]
        xn = ob.rms_norm(np.asarray(x, float)[:S], w["g_attn"], cfg.eps)
        out["k"] = (xn @ w["wk"]).reshape(S, cfg.Hkv, cfg.dh).transpose(1, 0, 2)
        return out
    monkeypatch.setattr(ob, "block_prefill_seq", prefill)


def mut_no_max(monkeypatch):
    def sm(s):
        with np.errstate(over="ignore", invalid="ignore"):
            e = np.exp(s)
            return e / np.sum(e, axis=-1, keepdims=True)
    monkeypatch.setattr(ob, "softmax_rows", sm)


def mut_rope_halves(monkeypatch):
    def rope(u, positions, base):
        u = np.asarray(u, float)
        half = u.shape[-1] // 2
        phi = ob.rope_angles(positions, u.shape[-1], base)[:, None, :]
        a, b = u[..., :half], u[..., half:]
        return np.concatenate([a * np.cos(phi) - b * np.sin(phi), a * np.sin(phi) + b * np.cos(phi)], -1)
    monkeypatch.setattr(ob, "rope", rope)


def mut_rope_freq(monkeypatch):
    def angles(positions, dh, base):
        i = np.arange(dh // 2, dtype=float)
        return np.outer(np.asarray(positions, float), np.power(float(base), -i / dh))
    monkeypatch.setattr(ob, "rope_angles", angles)


def mut_rope_sign(monkeypatch):
    orig = _orig("rope")
    monkeypatch.setattr(ob, "rope", lambda u, positions, base: orig(u, -np.asarray(positions), base))


def mut_eps_outside(monkeypatch):
    def rn(x, g, eps):
        x = np.asarray(x, float)
        return x / (np.sqrt(np.mean(x * x, axis=-1, keepdims=True)) + eps) * g
    monkeypatch.setattr(ob, "rms_norm", rn)


def mut_gqa_modulo(monkeypatch):
    def attn(q, k, v, q_pos, window=0):
        q, k, v = (np.asarray(a, float) for a in (q, k, v))
        Hkv = k.shape[1]
        vis = ob.visible_keys(q_pos, k.shape[0], window)
        o = np.empty_like(q)
        for h in range(q.shape[1]):
            s = np.where(vis, q[:, h] @ k[:, h % Hkv].T / math.sqrt(q.shape[2]), -np.inf)
            o[:, h] = ob.softmax_rows(s) @ v[:, h % Hkv]
        return o
    monkeypatch.setattr(ob, "causal_attention", attn)


def mut_scale_dh(monkeypatch):
    orig = _orig("causal_attention")
    def attn(q, k, v, q_pos, window=0):
        return orig(np.asarray(q) / math.sqrt(np.asarray(q).shape[-1]), k, v, q_pos, window)
    monkeypatch.setattr(ob, "causal_attention", attn)


def mut_no_residual(monkeypatch):
    def mlp(h, w, cfg):
        hn = ob.rms_norm(h, w["g_mlp"], cfg.eps)
        return (ob.silu(hn @ w["w1"]) * (hn @ w["w3"])) @ w["w2"]
    monkeypatch.setattr(ob, "mlp_branch", mlp)


def mut_silu_sign(monkeypatch):
    monkeypatch.setattr(ob, "silu", lambda z: np.asarray(z, float) / (1.0 + np.exp(np.asarray(z, float))))


def mut_gate_up_swapped(monkeypatch):
    def mlp(h, w, cfg):
        hn = ob.rms_norm(h, w["g_mlp"], cfg.eps)
        return h + (ob.silu(hn @ w["w3"]) * (hn @ w["w1"])) @ w["w2"]
    monkeypatch.setattr(ob, "mlp_branch", mlp)


def mut_window_one_more(monkeypatch):
    # window keeps j >= i - W (W + 1 keys)
    def vis(q_pos, S, window=0):
        j = np.arange(S)[None, :]; i = np.asarray(q_pos)[:, None]
        m = j <= i
        return m & (j >= i - window) if window > 0 else m
    monkeypatch.setattr(ob, "visible_keys", vis)


def mut_window_decode_ignored(monkeypatch):
    # decode attends over the whole cache whatever the window
    orig = _orig("block_decode_seq")
    def dec(x, w, cfg, k_cache, v_cache, pos):
        full = ob.Cfg(cfg.d, cfg.H, cfg.Hkv, cfg.dh, cfg.f, cfg.rope_base, cfg.eps, 0)
        return orig(x, w, full, k_cache, v_cache, pos)
    monkeypatch.setattr(ob, "block_decode_seq", dec)


def mut_paged_offset(monkeypatch):
    # offset counted from the wrong end of the page
    def gather(pool, block_table, page_size, n):
        pool = np.asarray(pool)
        out = np.empty((pool.shape[1], n, pool.shape[3]), pool.dtype)
        for t in range(n):
            out[:, t, :] = pool[int(block_table[t // page_size]), :, page_size - 1 - t % page_size, :]
        return out
    monkeypatch.setattr(ob, "gather_paged", gather)


def mut_int8_floor(monkeypatch):
    def quant(x):
        x = np.asarray(x, float)
        s = np.max(np.abs(x), axis=-1) / 127.0
        safe = np.where(s > 0, s, 1.0)
        return np.clip(np.floor(x / safe[..., None]), -127, 127).astype(np.int8), s
    monkeypatch.setattr(ob, "quantize_rows", quant)


def mut_int8_scale_128(monkeypatch):
    def quant(x):
        x = np.asarray(x, float)
        s = np.max(np.abs(x), axis=-1) / 128.0
        safe = np.where(s > 0, s, 1.0)
        return np.clip(np.rint(x / safe[..., None]), -127, 127).astype(np.int8), s
    monkeypatch.setattr(ob, "quantize_rows", quant)


def mut_int8_one_scale(monkeypatch):
    def quant(x):
        x = np.asarray(x, float)
        s = np.full(x.shape[:-1], np.max(np.abs(x)) / 127.0)
        safe = np.where(s > 0, s, 1.0)
        return np.clip(np.rint(x / safe[..., None]), -127, 127).astype(np.int8), s
    monkeypatch.setattr(ob, "quantize_rows", quant)


def mut_int8_half_away(monkeypatch):
    # round half away from zero instead of to even
    def quant(x):
        x = np.asarray(x, np.float64)
        s = np.max(np.abs(x), axis=-1) / 127.0
        safe = np.where(s > 0, s, 1.0)
        y = x / safe[..., None]
        return np.clip(np.sign(y) * np.floor(np.abs(y) + 0.5), -127, 127).astype(np.int8), s
    monkeypatch.setattr(ob, "quantize_rows", quant)


MUTANTS = [mut_int8_half_away, mut_int8_floor, mut_int8_scale_128, mut_int8_one_scale, mut_paged_offset, mut_window_one_more, mut_window_decode_ignored, mut_diagonal, mut_rope_on_v, mut_cache_pre_rope, mut_no_max, mut_rope_halves,
           mut_rope_freq, mut_rope_sign, mut_eps_outside, mut_gqa_modulo, mut_scale_dh,
           mut_no_residual, mut_silu_sign, mut_gate_up_swapped]


def _caught(check):
    try:
        with np.errstate(all="ignore"):
            _run(check)
    except (AssertionError, FloatingPointError, ValueError):
        return True
    return False


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda m: m.__name__)
def test_planted_mistake_is_caught(mutant, monkeypatch):
    mutant(monkeypatch)
    caught = [c.__name__ for c in CHECKS if _caught(c)]
    assert caught, f"{mutant.__name__} passes every pin"
