"""The work-accounting formulas against the counts the pages print.

Every row of ``golden/page_counts.tsv`` is a number printed on one of the
pages, with its citation; the formulas must reproduce it within the page's
rounding.
"""
import json
import os

import pytest

from causal_gqa_attention_rmsnorm_gb300 import accounting as acc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_counts.tsv")


def _rows():
    with open(GOLDEN) as fh:
        for line in fh:
            if not line.strip() or line.startswith("#"):
                continue
            rid, qty, args, printed, tol, cite = line.rstrip("\n").split("\t")
            yield pytest.param(qty, json.loads(args), float(printed), float(tol), id=rid)


def _model(a):
    return acc.model_params(a["L"], a["d"], a["H"], a["Hkv"], a["dh"], a["f"], a["V"], a.get("tied", False))


def _evaluate(qty, a):
    if qty == "12Ld2":
        # an MHA block with f = 8d/3 has exactly 12·d² matrix parameters
        d = a["d"]
        return a["L"] * acc.block_matrix_params(d, 1, 1, d, 8 * d / 3)
    if qty == "attn_params":
        return acc.block_matrix_params(a["d"], a["H"], a["Hkv"], a["dh"], 0)
    if qty == "mlp_params":
        return acc.block_matrix_params(a["d"], 0, 0, 0, a["f"])
    if qty == "model":
        return _model(a)
    if qty == "gemm_flops_per_token":
        return acc.gemm_flops(a["d"], a["H"], a["Hkv"], a["dh"], a["f"], 1)
    if qty == "full_attn_flops_per_token":
        # 4·T·d per token: one head of width d over T keys
        return acc.full_attn_flops(1, 1, a["d"], a["T"]) / a["T"]
    if qty == "attn_share":
        d, T = a["d"], a["T"]
        att = acc.full_attn_flops(1, 1, d, T) / T
        return att / (att + acc.gemm_flops(d, 1, 1, d, 8 * d / 3, 1))
    if qty == "kv_bytes":
        return acc.kv_bytes_per_token(a["L"], a["Hkv"], a["dh"], a["bytes"]) * a["n"]
    if qty == "gemm_flops_one":
        return 2 * a["k"] * a["n"]
    if qty == "weight_bytes_one":
        return a["k"] * a["n"] * a["bytes"]
    if qty == "embed_params":
        return a["V"] * a["d"]
    if qty == "logits_bytes":
        return acc.logits_bytes(a["tokens"], a["V"])
    if qty == "stack_matrix_params":
        return a["L"] * acc.block_matrix_params(a["d"], a["H"], a["Hkv"], a["dh"], a["f"])
    if qty == "gpt2_total":
        d = a["d"]
        return a["L"] * acc.block_matrix_params(d, 1, 1, d, 8 * d / 3) + a["V"] * d + a["P"] * d
    raise KeyError(qty)


@pytest.mark.parametrize("qty,args,printed,tol", list(_rows()))
def test_page_printed_counts(qty, args, printed, tol):
    got = _evaluate(qty, args)
    assert abs(got - printed) <= tol * abs(printed), (got, printed)


def test_mha_768_block_is_12d2_plus_norms():
    # d = 768, f = 2048 = 8d/3 exactly: 12·d² matrix parameters and 2·d gains
    assert acc.block_matrix_params(768, 12, 12, 64, 2048) == 12 * 768 ** 2 == 7_077_888
    assert acc.block_params(768, 12, 12, 64, 2048) == 7_079_424


def test_gemm_flops_split_adds_up():
    for (d, H, Hkv, dh, f) in [(768, 12, 12, 64, 2048), (4096, 32, 8, 128, 14336)]:
        each = acc.gemm_flops_each(d, H, Hkv, dh, f, 7)
        assert sum(each.values()) == acc.gemm_flops(d, H, Hkv, dh, f, 7)


def test_causal_attention_is_about_half_the_square():
    # causal kernels do about half of the attention term
    full = acc.full_attn_flops(4, 32, 128, 8192)
    causal = acc.causal_attn_flops(4, 32, 128, 8192)
    assert causal == 4 * 4 * 32 * 128 * 8192 * 8193 // 2
    assert abs(causal / full - 0.5) < 1e-3


def test_tile_granular_attention_count():
    # one tile: the whole tile square; T a multiple of the tile: nt(nt+1)/2 squares,
    # just above the exact pair count by the upper halves of the diagonal tiles
    assert acc.causal_attn_flops_tiles(1, 1, 1, 128) == 4 * 128 * 128
    T, nt = 8192, 64
    tiles = acc.causal_attn_flops_tiles(4, 32, 128, T)
    exact = acc.causal_attn_flops(4, 32, 128, T)
    assert tiles - exact == 4 * 4 * 32 * 128 * nt * (128 * 127 // 2)


def test_decode_kv_bytes():
    # GQA decode reads lens+1 rows of K and V per KV head
    assert acc.decode_kv_bytes([3, 0], Hkv=8, dh=128, bytes_per_value=2) == (4 + 1) * 2 * 8 * 128 * 2
    assert acc.kv_bytes_per_token(1, 8, 128, 2) == 4096


def test_window_pairs_and_keys():
    # the pages' example: with W = 4096 token 10000 meets 4096 keys, without a window 10001
    assert acc.attended_keys([10000], 4096) == 4096 and acc.attended_keys([10000]) == 10001
    # brute force over queries, for windows inside and beyond the sequence
    for T in (1, 5, 37):
        for W in (0, 1, 2, 7, 37, 50):
            want = sum(min(i + 1, W) if W > 0 else i + 1 for i in range(T))
            assert acc.visible_pairs(T, W) == want
    # the KV read of a windowed decode is capped at W rows per sequence
    lens = [3, 0, 9000, 4095]
    assert acc.decode_kv_bytes(lens, 8, 128, 2, window=4096) == (4 + 1 + 4096 + 4096) * 4096
    assert acc.decode_kv_bytes(lens, 8, 128, 2, window=100000) == acc.decode_kv_bytes(lens, 8, 128, 2)


def test_int8_kv_bytes():
    # an int8 row of dh codes plus its fp32 scale, for K and V of every KV head
    assert acc.decode_kv_bytes([3, 0], 8, 128, 1, scale_bytes=4) == (4 + 1) * 2 * 8 * (128 + 4)
    # a little over half the bf16 read
    r = acc.decode_kv_bytes([9000], 8, 128, 1, scale_bytes=4) / acc.decode_kv_bytes([9000], 8, 128, 2)
    assert r == (128 + 4) / 256
