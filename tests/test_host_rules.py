"""Host-side selection rules of the library, checked without a GPU through
its test hooks: the few-token GEMM's K-split count (its cluster size) and the
decode work-item size.  Each hook takes the SM count, so the GB300's 152 SMs
can be given here."""
import itertools
import os
import random

import pytest

from causal_gqa_attention_rmsnorm_gb300 import binding

SMS = 152
MAX_CLUSTER = 8        # a portable thread-block cluster


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(binding.LIB_PATH):
        pytest.skip("libtb.so not built")
    return binding.lib()


@pytest.mark.parametrize("name,N,K,expect", [
    ("qkv", (32 + 2 * 8) * 128, 4096, 4),
    ("wo", 4096, 4096, 8),
    ("w13", 2 * 14336, 4096, 1),
    ("w2", 4096, 14336, 8),
])
def test_split_counts_of_the_decode_gemms(lib, name, N, K, expect):
    """The counts for two CTAs per SM at 152 SMs."""
    assert lib.tbx_skinny_split_count(N // 128, K // 64, 2 * SMS) == expect


@pytest.mark.parametrize("name,N,K,two,three", [
    ("qkv", (32 + 2 * 8) * 128, 4096, 4, 8),
    ("wo", 4096, 4096, 8, 8),
    ("w13", 2 * 14336, 4096, 1, 2),
    ("w2", 4096, 14336, 8, 8),
])
def test_decode_gemms_take_three_ctas_per_sm_for_a_larger_split(lib, name, N, K, two, three):
    """The launcher runs three CTAs per SM when that allows a larger split in
    one wave: the decode QKV and W1/W3 GEMMs; Wo and W2 keep two."""
    assert lib.tbx_skinny_split_count(N // 128, K // 64, 2 * SMS) == two
    assert lib.tbx_skinny_split_count(N // 128, K // 64, 3 * SMS) == three


def test_split_count_rule(lib):
    """Against the stated rule: the largest power of two that one wave of the
    resident CTAs allows, at most a portable cluster, at least four K blocks
    per CTA, and never fewer than one."""
    rng = random.Random(0)
    cases = [(t, kb, s) for t, kb, s in itertools.product([1, 3, 16, 32, 48, 224, 1002], [1, 4, 7, 64, 224, 448],
                                                           [2, 304, 160])]
    cases += [(rng.randint(1, 1100), rng.randint(1, 600), rng.randint(1, 400)) for _ in range(300)]
    for tiles, kblocks, slots in cases:
        sp = lib.tbx_skinny_split_count(tiles, kblocks, slots)
        assert 1 <= sp <= MAX_CLUSTER
        lim = min(slots // tiles, MAX_CLUSTER, kblocks // 4)
        assert sp & (sp - 1) == 0                     # a power of two
        assert sp == 1 or sp <= lim
        assert 2 * sp > lim or 2 * sp > MAX_CLUSTER   # the largest one
        if sp > 1:
            assert tiles * sp <= slots          # one wave
            assert kblocks // sp >= 4


def test_split_count_rejects_empty_shapes(lib):
    assert lib.tbx_skinny_split_count(0, 64, 304) == -1
    assert lib.tbx_skinny_split_count(32, 0, 304) == -1
    assert lib.tbx_skinny_split_count(32, 64, 0) == -1


@pytest.mark.parametrize("B,expect", [(32, 256), (16, 256), (4, 256), (2, 128), (1, 64)])
def test_decode_item_size_for_the_decode_workload(lib, B, expect):
    """gqa_decode's shape (Hkv 8, T_max 16384): full-size items unless a full
    cache would leave warps of the 152 × 8 without an item."""
    assert lib.tbx_decode_chunk_keys(binding.TB_BF16, B, 8, 16384, SMS) == expect


def test_decode_item_size_rules(lib):
    warps = SMS * 8
    for dtype in (binding.TB_BF16, binding.TB_I8):
        for B in (1, 2, 3, 5, 8, 17, 64, 2048):
            for Hkv in (1, 2, 8):
                for T in (32, 1000, 4096, 16384, 131072, 262144):
                    c = lib.tbx_decode_chunk_keys(dtype, B, Hkv, T, SMS)
                    assert c in (64, 128, 256)                   # multiples of the int8 kernel's 32-key stage
                    chunks = -(-T // c)
                    assert chunks <= 1024                        # the merge's chunk limit
                    if c < 256:                                  # halved only for want of items
                        assert B * Hkv * (-(-T // (2 * c))) < warps
                        assert -(-T // c) <= 1024
    for B in (1, 32):
        assert lib.tbx_decode_chunk_keys(binding.TB_F32, B, 8, 16384, SMS) == 256


def test_decode_item_size_rejects_empty_shapes(lib):
    assert lib.tbx_decode_chunk_keys(binding.TB_BF16, 0, 8, 16384, SMS) == -1
    assert lib.tbx_decode_chunk_keys(binding.TB_BF16, 1, 8, 16384, 0) == -1
