"""int8 KV cache ("The Transformer Architecture", thegeniusblogs, pitfalls:
the KV cache can be quantised to int8).  Every cached row is stored as int8
codes with one fp32 scale, s = max|x|/127, codes round-half-even(x/s).

  * The quantiser is checked bit for bit: rows appended through the C ABI get
    exactly the oracle's codes and scales (both decide in fp32).
  * A decode step over an int8 cache is checked against the oracle's decode
    over the same codes and scales, at the bf16 tolerances.  The new token's
    own row is quantised by each side from its own k and v, which differ by
    bf16 rounding, so its codes may differ by one (never more).
  * Prefill with an int8 cache attends over the unquantised rows and stores
    their codes: its output equals the bf16-cache prefill's, and the stored
    rows are within half a step of the rows that cache holds.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import assert_close, block_config, dequantized, errors, oracle_cfg, oracle_weights, to_device

pytestmark = pytest.mark.gpu

BASE = workloads.BlockShape("i8", "decode", "bf16", B=4, T=0, d=1024, H=8, Hkv=2, dh=128, f=1024,
                            rope_base=5e5, eps=1e-5, gains="normal")


def _int8_cache(s, seed, lens, T_max, batches=None):
    """Rows < lens[b]: the oracle's codes and scales of the N(0, 1) bf16 rows
    make_cache_rows draws; every other row: random codes with NaN scales, so a
    read past a sequence's rows shows up as NaN.  Returns the cache and host
    copies (kq, ks, vq, vs)."""
    import causal_gqa_attention_rmsnorm_gb300 as tb
    g = np.random.default_rng(seed + 1000)
    shape = (s.B, s.Hkv, T_max, s.dh)
    kq = g.integers(-127, 128, size=shape, dtype=np.int8)
    vq = g.integers(-127, 128, size=shape, dtype=np.int8)
    ks = np.full(shape[:3], np.nan, np.float32)
    vs = np.full(shape[:3], np.nan, np.float32)
    for b in (range(s.B) if batches is None else batches):
        n = int(lens[b])
        kb, vb = workloads.make_cache_rows(s, seed, b, n)
        kq[b, :, :n], ks[b, :, :n] = oracle.quantize_rows(workloads.to_f64(kb))
        vq[b, :, :n], vs[b, :, :n] = oracle.quantize_rows(workloads.to_f64(vb))
    kv = tb.KVCache(torch.from_numpy(kq).cuda(), torch.from_numpy(vq).cuda(),
                    torch.tensor(lens, dtype=torch.int32).cuda(), None,
                    torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda())
    return kv, (kq, ks, vq, vs)


def _oracle_i8(s, inp, host, b, pos):
    kq, ks, vq, vs = host
    return oracle.block_decode_seq_int8(workloads.to_f64(inp["x"][b, 0]), oracle_weights(inp), oracle_cfg(s),
                                        kq[b], ks[b].astype(np.float64), vq[b], vs[b].astype(np.float64), pos)


def _check_new_row(kv, b, pos, ref, what):
    """The appended row: codes within one step of the oracle's, scale within
    bf16 rounding of it."""
    for name, codes, scales in (("k", kv.k, kv.k_scale), ("v", kv.v, kv.v_scale)):
        got = codes[b, :, pos].cpu().numpy().astype(np.int64)
        want = ref[f"{name}_q"].astype(np.int64)
        assert np.abs(got - want).max() <= 1, f"{what} {name} codes"
        assert (got != want).mean() <= 0.25, f"{what} {name} codes: {(got != want).mean()}"
        sg = scales[b, :, pos].cpu().double().numpy()
        np.testing.assert_allclose(sg, ref[f"{name}_s"], rtol=2 ** -7, err_msg=f"{what} {name} scale")


def test_append_quantises_exactly_like_the_oracle():
    import causal_gqa_attention_rmsnorm_gb300 as tb
    B, Hkv, T_max, dh, n = 4, 2, 64, 128, 37
    lens0 = [0, 5, 27, 40]                      # the last sequence would pass T_max
    g = torch.Generator().manual_seed(3)
    mags = torch.tensor([1e-37, 1e-3, 0.1, 1.0, 10.0, 300.0])
    rows = []
    for _ in range(2):
        x = torch.randn(B, Hkv, n, dh, generator=g)
        x *= mags[torch.randint(0, len(mags), (B, Hkv, n, 1), generator=g)]
        x[0, 0, 3] = 0.0                        # a zero row
        x[1, 1, 0] = 0.0
        x[1, 1, 0, :6] = torch.tensor([31.75, 0.125, 0.375, 0.625, -0.125, -0.375])   # halfway codes
        rows.append(x.to(torch.bfloat16))
    kn, vn = rows
    kv = tb.KVCache(torch.full((B, Hkv, T_max, dh), 77, dtype=torch.int8, device="cuda"),
                    torch.full((B, Hkv, T_max, dh), 77, dtype=torch.int8, device="cuda"),
                    torch.tensor(lens0, dtype=torch.int32, device="cuda"), None,
                    torch.full((B, Hkv, T_max), -1.0, device="cuda"), torch.full((B, Hkv, T_max), -1.0, device="cuda"))
    tb.tb_kvcache_append(kv, kn.cuda(), vn.cuda())
    assert tb.tb_get_device_error(clear=True) == tb.TB_DEVERR_CACHE_FULL
    assert kv.lens.tolist() == [37, 42, 64, 40]
    for name, src, codes, scales in (("k", kn, kv.k, kv.k_scale), ("v", vn, kv.v, kv.v_scale)):
        codes, scales = codes.cpu().numpy(), scales.cpu().numpy()
        for b, L in enumerate(lens0):
            if L + n > T_max:
                assert (codes[b] == 77).all() and (scales[b] == -1).all(), f"{name} b={b} was written"
                continue
            q, s = oracle.quantize_rows(workloads.to_f64(src[b]))
            np.testing.assert_array_equal(codes[b, :, L:L + n], q, err_msg=f"{name} codes b={b}")
            np.testing.assert_array_equal(scales[b, :, L:L + n], s.astype(np.float32), err_msg=f"{name} s b={b}")
            assert (codes[b, :, :L] == 77).all() and (codes[b, :, L + n:] == 77).all()
            assert (scales[b, :, :L] == -1).all() and (scales[b, :, L + n:] == -1).all()
    # halfway values went to the even code, the zero row to scale 0 and codes 0
    assert kv.k[1, 1, 5, :6].tolist() == [127, 0, 2, 2, 0, -2]
    assert kv.k_scale[0, 0, 3].item() == 0 and not kv.k[0, 0, 3].any()


@pytest.mark.parametrize("Hkv", [8, 4, 2, 1])
@pytest.mark.parametrize("W", [0, 100])
def test_int8_decode_matches_oracle(Hkv, W):
    import causal_gqa_attention_rmsnorm_gb300 as tb
    T_max = 800
    lens = [0, 1, 15, 16, 17, 255, 256, 257, 500, 783]
    s = BASE.with_(B=len(lens), Hkv=Hkv, window=W, T=T_max)
    inp = workloads.make_block_inputs(s, seed=31 + Hkv)
    kv, host = _int8_cache(s, 31 + Hkv, lens, T_max)
    cfg = block_config(s, max_pos=T_max)
    dev = to_device(inp)
    packed = tb.tb_pack_weights(cfg, dev)
    y = tb.tb_block_decode(cfg, packed, dev["x"], kv)
    assert tb.tb_get_device_error(clear=True) == 0
    assert kv.lens.cpu().tolist() == [n + 1 for n in lens]
    w, ocfg = oracle_weights(inp), oracle_cfg(s)
    for b, pos in enumerate(lens):
        yb = y[b, 0].cpu().double().numpy()
        ref = _oracle_i8(s, inp, host, b, pos)
        assert_close(yb, ref["y"], "bf16", f"y b={b}")
        _check_new_row(kv, b, pos, ref, f"b={b}")
        # the cost of the quantisation itself: against the unquantised rows the
        # step stays within the bf16 bar
        kb, vb = workloads.make_cache_rows(s, 31 + Hkv, b, pos)
        exact = oracle.block_decode_seq(workloads.to_f64(inp["x"][b, 0]), w, ocfg, workloads.to_f64(kb),
                                        workloads.to_f64(vb), pos)
        assert errors(yb, exact["y"])["rel_l2"] <= 1e-2, f"b={b}: {errors(yb, exact['y'])}"
    # the step wrote one row per sequence and nothing else
    kq = kv.k.cpu().numpy()
    for b, pos in enumerate(lens):
        np.testing.assert_array_equal(np.delete(kq[b], pos, axis=1), np.delete(host[0][b], pos, axis=1))


def test_int8_decode_full_cache_sets_error_and_skips_row():
    """A sequence whose cache is full is skipped (error bit set, its rows and
    length untouched); the others step normally."""
    import causal_gqa_attention_rmsnorm_gb300 as tb
    T_max = 64
    lens = [10, T_max, 63]
    s = BASE.with_(B=3, T=T_max)
    inp = workloads.make_block_inputs(s, seed=5)
    kv, host = _int8_cache(s, 5, lens[:1] + [T_max - 1] + lens[2:], T_max)
    kv.lens.copy_(torch.tensor(lens, dtype=torch.int32))
    cfg = block_config(s, max_pos=T_max)
    dev = to_device(inp)
    packed = tb.tb_pack_weights(cfg, dev)
    y = tb.tb_block_decode(cfg, packed, dev["x"], kv)
    assert tb.tb_get_device_error(clear=True) & tb.TB_DEVERR_CACHE_FULL
    assert kv.lens.cpu().tolist() == [11, T_max, 64]
    np.testing.assert_array_equal(kv.k[1].cpu().numpy(), host[0][1])
    np.testing.assert_array_equal(kv.k_scale[1].cpu().numpy(), host[1][1])
    for b in (0, 2):
        ref = _oracle_i8(s, inp, host, b, lens[b])
        assert_close(y[b, 0].cpu().double().numpy(), ref["y"], "bf16", f"y b={b}")
        _check_new_row(kv, b, lens[b], ref, f"b={b}")


def test_int8_decode_noalloc_equals_decode():
    import causal_gqa_attention_rmsnorm_gb300 as tb
    lens = [3, 300, 700]
    s = BASE.with_(B=3, T=768)
    inp = workloads.make_block_inputs(s, seed=8)
    cfg = block_config(s, max_pos=768)
    dev = to_device(inp)
    packed = tb.tb_pack_weights(cfg, dev)
    a, _ = _int8_cache(s, 8, lens, 768)
    b, _ = _int8_cache(s, 8, lens, 768)
    ya = tb.tb_block_decode(cfg, packed, dev["x"], a)
    yb = tb.tb_block_decode_noalloc(cfg, packed, dev["x"], b)
    assert tb.tb_get_device_error(clear=True) == 0
    assert torch.equal(yb, ya)
    assert torch.equal(a.k, b.k) and torch.equal(a.v, b.v)


def test_int8_prefill_then_decode_follows_oracle():
    """Prefill T tokens into an int8 cache, then decode three more: the prefill
    output equals the bf16-cache prefill's, the stored rows are within half a
    step (plus bf16 rounding) of the rows that cache holds and within one code
    of the oracle's, and each decode step matches the oracle's int8 decode
    continuing its own quantised prefill."""
    import causal_gqa_attention_rmsnorm_gb300 as tb
    T, T_max, extra = 200, 256, 3
    s = BASE.with_(mode="prefill", B=2, T=T + extra, window=0)
    inp = workloads.make_block_inputs(s, seed=12)
    cfg = block_config(s, max_pos=T_max)
    dev = to_device(inp)
    packed = tb.tb_pack_weights(cfg, dev)
    x0 = dev["x"][:, :T].contiguous()
    ref_kv = tb.KVCache.empty(s.B, s.Hkv, T_max, s.dh, dtype=torch.bfloat16, fill=float("nan"))
    kv = tb.KVCache.empty_int8(s.B, s.Hkv, T_max, s.dh)
    kv.k_scale.fill_(float("nan"))
    kv.v_scale.fill_(float("nan"))
    y_ref = tb.tb_block_prefill(cfg, packed, x0, kv=ref_kv)
    y = tb.tb_block_prefill(cfg, packed, x0, kv=kv)
    assert tb.tb_get_device_error(clear=True) == 0
    assert torch.equal(y, y_ref)
    assert kv.lens.tolist() == [T] * s.B
    kd, vd = dequantized(kv)
    for got, exact, sc in ((kd, ref_kv.k, kv.k_scale), (vd, ref_kv.v, kv.v_scale)):
        err = (got[:, :, :T] - exact[:, :, :T].float()).abs()
        bound = sc[:, :, :T, None] * (0.5 + 2 ** -7) + exact[:, :, :T].float().abs() * 2 ** -8
        assert bool((err <= bound).all())
        assert torch.isnan(sc[:, :, T:]).all()      # rows past T untouched
    ys = [tb.tb_block_decode(cfg, packed, dev["x"][:, T + i:T + i + 1].contiguous(), kv) for i in range(extra)]
    assert tb.tb_get_device_error(clear=True) == 0
    w, ocfg = oracle_weights(inp), oracle_cfg(s)
    for b in range(s.B):
        xb = workloads.to_f64(inp["x"][b])
        pre = oracle.block_prefill_seq(xb[:T], w, ocfg)
        kq, ks = oracle.quantize_rows(pre["k"])
        vq, vs = oracle.quantize_rows(pre["v"])
        for name, codes, want in (("k", kv.k, kq), ("v", kv.v, vq)):
            got = codes[b, :, :T].cpu().numpy().astype(np.int64)
            assert np.abs(got - want).max() <= 1, name
            assert (got != want).mean() <= 0.25, name
        # the oracle continues from its own codes
        pad = lambda a: np.concatenate([a, np.zeros(a.shape[:1] + (extra,) + a.shape[2:], a.dtype)], 1)
        kq, ks, vq, vs = pad(kq), pad(ks), pad(vq), pad(vs)
        for i in range(extra):
            ref = oracle.block_decode_seq_int8(xb[T + i], w, ocfg, kq, ks, vq, vs, T + i)
            kq[:, T + i], ks[:, T + i], vq[:, T + i], vs[:, T + i] = ref["k_q"], ref["k_s"], ref["v_q"], ref["v_s"]
            assert_close(ys[i][b, 0].cpu().double().numpy(), ref["y"], "bf16", f"step {i} b={b}")


def test_int8_decode_full_workload_sampled_sequences():
    """The full decode workload (B = 32, T_max = 16384, GQA 32/8, dh 128) over
    an int8 cache in the benchmark's launch configuration: sampled sequences
    against the oracle (every other sequence's rows have NaN scales).  The
    max-abs bound is 1.25x the error of the bf16 rounding model
    (tests/rounding_model.py) over the same dequantised rows: the int8 path
    keeps the block's bf16 GEMM operands and rounds q and P no coarser."""
    import causal_gqa_attention_rmsnorm_gb300 as tb
    from rounding_model import ERROR_FACTOR, emulate_decode_seq
    s = workloads.CONFIGS["gqa_decode"]
    lens = workloads.make_lens(s, seed=0).tolist()
    sampled = [0, 7, 21, 31]
    inp = workloads.make_block_inputs(s.with_(mode="decode"), seed=0)
    kv, host = _int8_cache(s, 0, lens, s.T, batches=sampled)
    cfg = block_config(s, max_pos=s.T)
    dev = to_device(inp)
    packed = tb.tb_pack_weights(cfg, dev)
    y = tb.tb_block_decode(cfg, packed, dev["x"], kv)
    assert tb.tb_get_device_error(clear=True) == 0
    kq, ks, vq, vs = host
    got, refs, model = [], [], []
    for b in sampled:
        n = lens[b]
        ref = _oracle_i8(s, inp, host, b, n)
        kd = torch.from_numpy(oracle.dequantize_rows(kq[b, :, :n], ks[b, :, :n].astype(np.float64))).float()
        vd = torch.from_numpy(oracle.dequantize_rows(vq[b, :, :n], vs[b, :, :n].astype(np.float64))).float()
        got.append(y[b, 0].cpu().double().numpy())
        refs.append(ref["y"])
        model.append(emulate_decode_seq(inp, s, b, kd, vd, order="a").double().numpy())
        _check_new_row(kv, b, n, ref, f"b={b}")
    bound = ERROR_FACTOR * errors(np.stack(model), np.stack(refs))["max_abs"]
    for b, g, r in zip(sampled, got, refs):
        e = errors(g, r)
        assert e["finite"] and e["rel_l2"] <= 1e-2 and e["max_abs"] <= bound, (b, e, bound)


# ---- paged int8 caches: the int8 layout in page pools ------------------------

def _paged_copy(kv, ps, seed):
    """The rows of a contiguous int8 cache in shuffled page pools (a few spare
    pages, zero codes and NaN scales outside the table)."""
    import causal_gqa_attention_rmsnorm_gb300 as tb
    B, Hkv, T_max, dh = kv.k.shape
    per = T_max // ps
    num_pages = B * per + 3
    perm = np.random.default_rng(seed).permutation(num_pages)[:B * per].reshape(B, per)
    codes = lambda: torch.zeros((num_pages, Hkv, ps, dh), dtype=torch.int8, device="cuda")
    scales = lambda: torch.full((num_pages, Hkv, ps), float("nan"), dtype=torch.float32, device="cuda")
    pk, pv, pks, pvs = codes(), codes(), scales(), scales()
    for b in range(B):
        for p in range(per):
            sl = slice(p * ps, (p + 1) * ps)
            pk[perm[b, p]], pv[perm[b, p]] = kv.k[b, :, sl], kv.v[b, :, sl]
            pks[perm[b, p]], pvs[perm[b, p]] = kv.k_scale[b, :, sl], kv.v_scale[b, :, sl]
    return tb.KVCache(pk, pv, kv.lens.clone(), torch.tensor(perm, dtype=torch.int32, device="cuda"), pks, pvs)


def _assert_same_rows(paged, contig, n_of):
    """Every sequence's first n_of[b] rows, gathered through the block table,
    equal the contiguous cache's: codes and scales bit for bit."""
    bt = paged.block_table.cpu().numpy()
    ps = paged.k.shape[2]
    for b, n in enumerate(n_of):
        for name, pc, cc in (("k", paged.k, contig.k), ("v", paged.v, contig.v),
                             ("k_scale", paged.k_scale, contig.k_scale), ("v_scale", paged.v_scale, contig.v_scale)):
            pool, want = pc.cpu().numpy(), cc[b, :, :n].cpu().numpy()
            if pool.ndim == 3:                   # scale pools: one value per row
                pool, want = pool[..., None], want[..., None]
            got = oracle.gather_paged(pool, bt[b], ps, n)
            np.testing.assert_array_equal(got, want, err_msg=f"{name} b={b}")


@pytest.mark.parametrize("ps", [32, 128])
@pytest.mark.parametrize("W", [0, 100])
def test_paged_int8_decode_equals_contiguous(ps, W):
    """Same kernels, same arithmetic: a decode step over the paged pools gives
    the contiguous int8 cache's output and appended rows bit for bit."""
    import causal_gqa_attention_rmsnorm_gb300 as tb
    T_max = 512
    lens = [0, 31, 32, 300, 510]
    s = BASE.with_(B=len(lens), window=W, T=T_max)
    inp = workloads.make_block_inputs(s, seed=41)
    contig, _ = _int8_cache(s, 41, lens, T_max)
    paged = _paged_copy(contig, ps, seed=ps + W)
    cfg = block_config(s, max_pos=T_max)
    dev = to_device(inp)
    packed = tb.tb_pack_weights(cfg, dev)
    for x in (dev["x"], workloads.make_block_inputs(s, seed=42)["x"].cuda()):     # two steps
        y_c = tb.tb_block_decode(cfg, packed, x, contig)
        y_p = tb.tb_block_decode(cfg, packed, x, paged)
        assert tb.tb_get_device_error(clear=True) == 0
        assert torch.equal(y_p, y_c)
        assert torch.equal(paged.lens, contig.lens)
    _assert_same_rows(paged, contig, [n + 2 for n in lens])


def test_paged_int8_prefill_and_append_equal_contiguous():
    """Prefill into paged int8 pools, then append rows: the pools hold the
    contiguous int8 cache's codes and scales, and the outputs are equal."""
    import causal_gqa_attention_rmsnorm_gb300 as tb
    T, T_max, ps = 200, 256, 64
    s = BASE.with_(mode="prefill", B=2, T=T, window=0)
    inp = workloads.make_block_inputs(s, seed=13)
    cfg = block_config(s, max_pos=T_max)
    dev = to_device(inp)
    packed = tb.tb_pack_weights(cfg, dev)
    contig = tb.KVCache.empty_int8(s.B, s.Hkv, T_max, s.dh)
    paged = _paged_copy(contig, ps, seed=5)
    y_c = tb.tb_block_prefill(cfg, packed, dev["x"], kv=contig)
    y_p = tb.tb_block_prefill(cfg, packed, dev["x"], kv=paged)
    assert tb.tb_get_device_error(clear=True) == 0
    assert torch.equal(y_p, y_c)
    g = torch.Generator().manual_seed(6)
    kn = torch.randn(s.B, s.Hkv, 40, s.dh, generator=g).to(torch.bfloat16).cuda()
    vn = torch.randn(s.B, s.Hkv, 40, s.dh, generator=g).to(torch.bfloat16).cuda()
    tb.tb_kvcache_append(contig, kn, vn)
    tb.tb_kvcache_append(paged, kn, vn)
    assert tb.tb_get_device_error(clear=True) == 0
    assert paged.lens.tolist() == contig.lens.tolist() == [T + 40] * s.B
    _assert_same_rows(paged, contig, [T + 40] * s.B)


def test_paged_int8_bad_page_is_flagged():
    """A block-table entry outside the pool is never dereferenced by the
    quantiser or the attention: the step sets TB_DEVERR_BAD_PAGE and the
    context stays usable."""
    import causal_gqa_attention_rmsnorm_gb300 as tb
    T_max, ps = 256, 64
    lens = [10, 100, 200, 70]
    s = BASE.with_(T=T_max)
    inp = workloads.make_block_inputs(s, seed=2)
    contig, _ = _int8_cache(s, 2, lens, T_max)
    paged = _paged_copy(contig, ps, seed=3)
    good = paged.block_table.clone()
    bad = good.clone()
    bad[2, 1] = 10 ** 6                          # sequence 2's second page: outside the pool
    bad[1, 1] = -1                               # sequence 1's new row lands in a bad page
    paged.block_table.copy_(bad)
    cfg = block_config(s, max_pos=T_max)
    dev = to_device(inp)
    packed = tb.tb_pack_weights(cfg, dev)
    tb.tb_block_decode(cfg, packed, dev["x"], paged)
    assert tb.tb_get_device_error(clear=True) & tb.TB_DEVERR_BAD_PAGE
    paged.block_table.copy_(good)
    paged.lens.copy_(torch.tensor(lens, dtype=torch.int32))
    y_p = tb.tb_block_decode(cfg, packed, dev["x"], paged)
    assert tb.tb_get_device_error(clear=True) == 0
    assert torch.isfinite(y_p).all()
