"""Host-side selection rules of the library, checked without a GPU through
its test hooks: the few-token GEMM's K-split count and the decode work-item
size.  Each hook takes the SM count, so the GB300's 152 SMs can be given here."""
import itertools
import random

import pytest

from causal_gqa_attention_rmsnorm_gb300 import binding

SMS = 152
MAX_ITEMS = 1024       # the few-token GEMM's partial buffer holds this many items


@pytest.fixture(scope="module")
def lib():
    return binding.lib()


def fill(tiles, sp, slots):
    items = tiles * sp
    waves = -(-items // slots)
    return items / (waves * slots)


@pytest.mark.parametrize("name,N,K,expect", [
    ("qkv", (32 + 2 * 8) * 128, 4096, 6),
    ("wo", 4096, 4096, 9),
    ("w13", 2 * 14336, 4096, 4),
    ("w2", 4096, 14336, 19),
])
def test_split_counts_of_the_decode_gemms(lib, name, N, K, expect):
    """The counts the decode step of the GQA block uses at 152 SMs."""
    assert lib.tbx_skinny_split_count(N // 128, K // 64, 2 * SMS) == expect


def test_split_count_fills_its_last_wave_best(lib):
    """Against the stated rule: among the allowed counts (at least four K
    blocks per item, at most MAX_ITEMS items) the result fills its last wave
    as well as the best one, up to the rule's tie margin of 1e-3."""
    rng = random.Random(0)
    cases = [(t, kb, s) for t, kb, s in itertools.product([1, 3, 16, 32, 48, 224, 1002], [4, 7, 64, 224, 448],
                                                           [2, 304, 160])]
    cases += [(rng.randint(1, 1100), rng.randint(1, 600), rng.randint(1, 400)) for _ in range(300)]
    for tiles, kblocks, slots in cases:
        sp = lib.tbx_skinny_split_count(tiles, kblocks, slots)
        spmax = min(kblocks // 4, MAX_ITEMS // tiles)
        if spmax < 1:
            assert sp == 1
            continue
        assert 1 <= sp <= spmax
        best = max(fill(tiles, s, slots) for s in range(1, spmax + 1))
        assert fill(tiles, sp, slots) >= best - 1e-3 - 1e-12


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
