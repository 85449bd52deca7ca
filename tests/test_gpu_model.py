"""Around the block, through the C ABI against the fp64 oracle: the embedding
gather, the LM head (logits and the chunked per-token loss, tied and untied),
and an L-layer stack in prefill and decode ("Transformer block" page, "How it
works", steps 1 and 4; "The Transformer" §5, "A tensor's journey")."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import block_config, errors, oracle_cfg, oracle_weights, to_device
from rounding_model import ERROR_FACTOR, emulate_stack_decode_seq, emulate_stack_prefill_seq

pytestmark = pytest.mark.gpu


def _bf16_round(a):
    return torch.as_tensor(np.asarray(a)).to(torch.bfloat16).double().numpy()


def _close_normwise(got, ref, tol, what):
    e = errors(got, ref)
    assert e["finite"] and e["normwise"] <= tol and e["rel_l2"] <= tol, (what, e)


def test_embed_gather_and_bad_ids():
    import causal_gqa_attention_rmsnorm_gb300 as tb
    g = torch.Generator().manual_seed(0)
    table = torch.randn(1000, 256, generator=g).to(torch.bfloat16).cuda()
    ids = torch.randint(0, 1000, (3, 37), generator=g, dtype=torch.int32).cuda()
    x = tb.tb_embed(table, ids)
    assert tb.tb_get_device_error(clear=True) == 0
    assert torch.equal(x, table[ids.long()])
    bad = ids.clone()
    bad[1, 5] = 1000
    bad[2, 0] = -3
    x = tb.tb_embed(table, bad)
    assert tb.tb_get_device_error(clear=True) & tb.TB_DEVERR_BAD_TOKEN
    assert (x[1, 5] == 0).all() and (x[2, 0] == 0).all() and torch.equal(x[0], table[ids[0].long()])


def _head_case(dtype, M, V=1000, d=256, tied=False, seed=1):
    import causal_gqa_attention_rmsnorm_gb300 as tb
    g = torch.Generator().manual_seed(seed)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    x = torch.randn(M, d, generator=g).to(tdt)
    gain = (1 + 0.1 * torch.randn(d, generator=g)).to(tdt)
    w = (0.02 * torch.randn(V, d, generator=g) if tied else 0.02 * torch.randn(d, V, generator=g)).to(tdt)
    targets = torch.randint(0, V, (M,), generator=g, dtype=torch.int32)
    cfg = tb.HeadConfig(d, V, 1e-5, tb.TB_F32 if dtype == "f32" else tb.TB_BF16)
    packed = tb.tb_pack_lm_head(cfg, gain.cuda(), w.cuda(), tied=tied)
    w_u = w.double().numpy().T if tied else w.double().numpy()
    ref = oracle.lm_head(x.double().numpy(), gain.double().numpy(), w_u, 1e-5)
    return cfg, packed, x.cuda(), targets, ref


@pytest.mark.parametrize("M", [3, 64, 200])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("tied", [False, True])
def test_lm_head_logits_and_loss(M, dtype, tied):
    import causal_gqa_attention_rmsnorm_gb300 as tb
    cfg, packed, x, targets, ref = _head_case(dtype, M, tied=tied)
    logits, nll = tb.tb_lm_head(cfg, packed, x, targets=targets.cuda())
    assert tb.tb_get_device_error(clear=True) == 0
    tol = 1e-4 if dtype == "f32" else 1e-2
    _close_normwise(logits.cpu().double().numpy(), ref, tol, "logits")
    want = oracle.token_nll(ref, targets.numpy())
    np.testing.assert_allclose(nll.cpu().double().numpy(), want, atol=1e-4 if dtype == "f32" else 3e-2)


def test_lm_head_chunked_loss_without_logits():
    """Row chunks of 50 with no logits buffer: the same losses as one pass that
    materialises the logits (the loss never needs the full [M, V] logits)."""
    import causal_gqa_attention_rmsnorm_gb300 as tb
    cfg, packed, x, targets, ref = _head_case("bf16", 230, V=4096)
    t = targets.cuda()
    logits, nll_full = tb.tb_lm_head(cfg, packed, x, targets=t, row_chunk=256)
    none, nll_chunk = tb.tb_lm_head(cfg, packed, x, want_logits=False, targets=t, row_chunk=50)
    assert none is None and tb.tb_get_device_error(clear=True) == 0
    torch.testing.assert_close(nll_chunk, nll_full, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(nll_chunk.cpu().double().numpy(), oracle.token_nll(ref, targets.numpy()), atol=3e-2)
    bad = t.clone()
    bad[7] = 4096
    _, nll_bad = tb.tb_lm_head(cfg, packed, x, want_logits=False, targets=bad, row_chunk=50)
    assert tb.tb_get_device_error(clear=True) & tb.TB_DEVERR_BAD_TOKEN
    assert torch.isnan(nll_bad[7]) and torch.isfinite(nll_bad[:7]).all()


@pytest.mark.parametrize("V,row_chunk", [(4096, 0), (1000, 100), (520, 130)])
def test_lm_head_loss_inside_the_gemm(V, row_chunk):
    """No logits buffer and row chunks above 64 rows: the bf16 head folds the
    loss into its GEMM's epilogue (a running max and Σ exp per row and tile)
    and never forms the logits.  Same losses as the materialised logits, and
    the oracle's; a bad target gives NaN and the error bit; chunk ends that
    fall to few rows (the last chunk) take the logits path."""
    import causal_gqa_attention_rmsnorm_gb300 as tb
    M = 333
    cfg, packed, x, targets, ref = _head_case("bf16", M, V=V, tied=V == 1000)
    t = targets.cuda()
    logits, nll_full = tb.tb_lm_head(cfg, packed, x, targets=t, row_chunk=512)
    none, nll_fused = tb.tb_lm_head(cfg, packed, x, want_logits=False, targets=t, row_chunk=row_chunk)
    assert none is None and tb.tb_get_device_error(clear=True) == 0
    torch.testing.assert_close(nll_fused, nll_full, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(nll_fused.cpu().double().numpy(), oracle.token_nll(ref, targets.numpy()), atol=3e-2)
    # the target that sits in the last, partial column tile, and out-of-range targets
    t2 = t.clone()
    t2[0] = V - 1
    t2[5] = V
    t2[9] = -1
    _, nll_bad = tb.tb_lm_head(cfg, packed, x, want_logits=False, targets=t2, row_chunk=row_chunk)
    assert tb.tb_get_device_error(clear=True) & tb.TB_DEVERR_BAD_TOKEN
    assert torch.isnan(nll_bad[5]) and torch.isnan(nll_bad[9])
    z = logits[0].double()
    want0 = (torch.logsumexp(z, 0) - z[V - 1]).item()
    assert abs(nll_bad[0].item() - want0) < 1e-3
    keep = torch.ones(M, dtype=torch.bool)
    keep[[0, 5, 9]] = False
    torch.testing.assert_close(nll_bad[keep.cuda()], nll_full[keep.cuda()], rtol=1e-5, atol=1e-5)


STACK = workloads.BlockShape("stack", "prefill", "bf16", B=2, T=90, d=256, H=4, Hkv=2, dh=64, f=512,
                             rope_base=1e4, eps=1e-6, gains="normal")


def _stack_model(s, L, V, seed=5):
    import causal_gqa_attention_rmsnorm_gb300 as tb
    layers = [workloads.make_block_inputs(s, seed=seed + l) for l in range(L)]
    cfg = block_config(s, max_pos=128)
    packed = [tb.tb_pack_weights(cfg, to_device(lw)) for lw in layers]
    g = torch.Generator().manual_seed(seed)
    table = torch.randn(V, s.d, generator=g).to(torch.bfloat16)
    gain = (1 + 0.1 * torch.randn(s.d, generator=g)).to(torch.bfloat16)
    hcfg = tb.HeadConfig(s.d, V, s.eps, tb.TB_BF16)
    head = tb.tb_pack_lm_head(hcfg, gain.cuda(), table.cuda(), tied=True)
    ids = torch.randint(0, V, (s.B, s.T), generator=g, dtype=torch.int32)
    return cfg, packed, layers, table, gain, hcfg, head, ids


def _within_model(got, model, ref, what):
    """The GPU's error against the oracle is at most 1.25x the error of the
    bf16 rounding model (tests/rounding_model.py) on the same outputs, in the
    normwise and relative-L2 measures: the stack adds no error of its own to
    the rounding its path is built with (the block's d = 4096 tests hold the
    same ratio)."""
    e, em = errors(got, ref), errors(model, ref)
    assert e["finite"], what
    for k in ("normwise", "rel_l2"):
        assert e[k] <= ERROR_FACTOR * em[k], (what, k, e[k], em[k])


def test_stack_prefill_and_decode_against_the_oracle():
    """Three blocks with the residual stream stored in bf16 between them, and
    the tied LM head on the last block's bf16 output.  The oracle takes the
    same bf16 rounding of each block's input; the bound is 1.25x the rounding
    model's own error on the same outputs (about 6e-4 normwise and 2e-3
    relative L2 for the logits, 3e-3 normwise for the caches at this shape)."""
    import causal_gqa_attention_rmsnorm_gb300 as tb
    s, L, V = STACK, 3, 520
    cfg, packed, layers, table, gain, hcfg, head, ids = _stack_model(s, L, V)
    ocfg = oracle_cfg(s)
    ow = [oracle_weights(lw) for lw in layers]
    tab64, g64 = table.double().numpy(), gain.double().numpy()
    # prefill of the first T-1 tokens into per-layer caches, then one decode step
    kvs = [tb.KVCache.empty(s.B, s.Hkv, 128, s.dh, fill=float("nan")) for _ in range(L)]
    x = tb.tb_embed(table.cuda(), ids[:, :s.T - 1].contiguous().cuda())
    h = tb.tb_stack_prefill(cfg, packed, x, kvs=kvs, y_dtype=tb.TB_BF16)
    logits, _ = tb.tb_lm_head(hcfg, head, h.reshape(-1, s.d))
    x1 = tb.tb_embed(table.cuda(), ids[:, s.T - 1:].contiguous().cuda())
    h1 = tb.tb_stack_decode(cfg, packed, x1, kvs, y_dtype=tb.TB_BF16)
    logits1, _ = tb.tb_lm_head(hcfg, head, h1.reshape(-1, s.d))
    assert tb.tb_get_device_error(clear=True) == 0
    logits = logits.reshape(s.B, s.T - 1, V)
    for b in range(s.B):
        ref = oracle.stack_prefill_seq(ids[b].tolist(), tab64, ow, ocfg, g64, tab64.T, round_between=_bf16_round)
        pre = ids[b, :s.T - 1].tolist()
        model = emulate_stack_prefill_seq(pre, table, layers, s, gain)
        model1 = emulate_stack_decode_seq(int(ids[b, s.T - 1]), table, layers, s, gain, model["k"], model["v"])
        _within_model(logits[b].cpu().double().numpy(), model["logits"].double().numpy(), ref["logits"][:s.T - 1],
                      f"prefill logits b={b}")
        _within_model(logits1[b].cpu().double().numpy(), model1["logits"].double().numpy(), ref["logits"][s.T - 1],
                      f"decode logits b={b}")
        for l in range(L):
            mk = torch.cat([model["k"][l], model1["k"][l][:, None]], 1).double().numpy()
            _within_model(kvs[l].k[b, :, :s.T].cpu().double().numpy(), mk, ref["k"][l], f"k cache l={l} b={b}")


def test_stack_of_one_is_the_block():
    import causal_gqa_attention_rmsnorm_gb300 as tb
    s = STACK
    cfg, packed, layers, table, gain, hcfg, head, ids = _stack_model(s, 1, 64)
    x = to_device(layers[0])["x"]
    y_stack = tb.tb_stack_prefill(cfg, packed, x)
    y_block = tb.tb_block_prefill(cfg, packed[0], x)
    # the same kernels on the same inputs: the same bytes
    assert torch.equal(y_stack, y_block)


def test_stack_over_int8_caches_is_the_blocks_layer_by_layer():
    """The stack entry points with an int8 cache per layer run the same kernels
    as the block calls one layer after another: the same bytes in the outputs
    and in every layer's codes and scales."""
    import causal_gqa_attention_rmsnorm_gb300 as tb
    s = STACK.with_(name="stack_i8", d=512, dh=128)
    L = 2
    cfg, packed, layers, table, gain, hcfg, head, ids = _stack_model(s, L, 64)
    x = tb.tb_embed(table.cuda(), ids[:, :s.T - 1].contiguous().cuda())
    x1 = tb.tb_embed(table.cuda(), ids[:, s.T - 1:].contiguous().cuda())
    kv_s = [tb.KVCache.empty_int8(s.B, s.Hkv, 128, s.dh) for _ in range(L)]
    h = tb.tb_stack_prefill(cfg, packed, x, kvs=kv_s, y_dtype=tb.TB_BF16)
    h1 = tb.tb_stack_decode(cfg, packed, x1, kv_s, y_dtype=tb.TB_BF16)
    kv_b = [tb.KVCache.empty_int8(s.B, s.Hkv, 128, s.dh) for _ in range(L)]
    g, g1 = x, x1
    for l in range(L):
        g = tb.tb_block_prefill(cfg, packed[l], g, kv=kv_b[l], y_dtype=tb.TB_BF16)
    for l in range(L):
        g1 = tb.tb_block_decode(cfg, packed[l], g1, kv_b[l], y_dtype=tb.TB_BF16)
    assert tb.tb_get_device_error(clear=True) == 0
    assert torch.equal(h, g) and torch.equal(h1, g1)
    for l in range(L):
        for a, b in ((kv_s[l].k, kv_b[l].k), (kv_s[l].v, kv_b[l].v), (kv_s[l].k_scale, kv_b[l].k_scale),
                     (kv_s[l].v_scale, kv_b[l].v_scale), (kv_s[l].lens, kv_b[l].lens)):
            assert torch.equal(a, b), l
