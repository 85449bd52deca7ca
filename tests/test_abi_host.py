"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point include/tb.h declares, and rejects bad arguments before it
launches anything."""
import ctypes
import os
import re

import pytest

import causal_gqa_attention_rmsnorm_gb300 as tb
from causal_gqa_attention_rmsnorm_gb300 import binding

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "tb.h")


def declared_entry_points():
    src = open(HEADER).read()
    return re.findall(r"TB_API\s+[\w\s\*]+?\b(tb_\w+)\s*\(", src)


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(binding.LIB_PATH):
        pytest.skip("libtb.so not built")
    return binding.lib()


def test_header_declares_the_entry_points():
    names = declared_entry_points()
    assert set(names) == set(binding.EXPORTED), names
    for n in ("tb_block_prefill", "tb_block_decode", "tb_kvcache_append"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_entry_points():
        assert hasattr(lib, n), n


def cfg(**kw):
    base = dict(d=256, H=4, Hkv=2, dh=64, f=512, max_pos=1024, rope_base=1e4, eps=1e-6, dtype=tb.TB_BF16)
    base.update(kw)
    return binding.tb_block_cfg(*[base[k] for k in ("d", "H", "Hkv", "dh", "f", "max_pos", "rope_base", "eps",
                                                    "dtype")])


FAKE = 0x7F0000000000  # never dereferenced: every call below fails validation first


@pytest.mark.parametrize("bad,status", [
    (dict(H=3), 1),               # H not a multiple of Hkv
    (dict(dh=32), 1),             # dh != d / H
    (dict(max_pos=0), 1),
    (dict(rope_base=0.0), 1),
    (dict(eps=-1.0), 1),
    (dict(dtype=7), 1),
    (dict(d=48, H=3, Hkv=3, dh=16, f=96), 2),   # bf16 needs d, f multiples of 64
    (dict(d=120, H=4, Hkv=4, dh=30, f=128, dtype=tb.TB_F32), 2),   # no attention kernel for dh 30
    (dict(H=4, Hkv=1, d=256, dh=64, f=512), 0),  # MQA is valid
])
def test_cfg_validation(lib, bad, status):
    c = cfg(**bad)
    n = lib.tb_packed_weights_bytes(ctypes.byref(c))
    if status == 0:
        assert n > 0
    else:
        assert n == 0
        st = lib.tb_block_prefill(ctypes.byref(c), FAKE, FAKE, FAKE + 4096, 0, 1, 1, None, FAKE, 1 << 30, None)
        assert st == status, lib.tb_last_error_message()


def test_prefill_argument_checks(lib):
    c = cfg()
    ws = lib.tb_workspace_bytes(ctypes.byref(c), 2, 64, 0)
    assert ws > 0
    call = lambda **k: lib.tb_block_prefill(ctypes.byref(c), k.get("packed", FAKE), k.get("x", FAKE),
                                            k.get("y", FAKE + (1 << 20)), k.get("ydt", 0), k.get("B", 2),
                                            k.get("T", 64), k.get("kv", None), k.get("ws", FAKE),
                                            k.get("wsb", ws), None)
    assert call(B=-1) == 1
    assert call(B=0) == 0 and call(T=0) == 0          # empty calls launch nothing
    assert call(T=2048) == 1                           # T beyond max_pos
    assert call(x=None) == 1
    assert call(x=FAKE + 8) == 1                       # misaligned
    assert call(wsb=ws - 1) == 1                       # workspace too small
    assert call(ydt=5) == 1
    assert call(y=FAKE) == 1                           # y aliases x
    kv = binding.tb_kvcache(FAKE, FAKE, FAKE, 3, 2, 128, 64, 1)
    assert call(kv=ctypes.byref(kv)) == 1              # kv->B != B
    kv = binding.tb_kvcache(FAKE, FAKE, FAKE, 2, 2, 32, 64, 1)
    assert call(kv=ctypes.byref(kv)) == 1              # T > T_max
    kv = binding.tb_kvcache(FAKE, FAKE, FAKE, 2, 2, 128, 64, 0)
    assert call(kv=ctypes.byref(kv)) == 1              # cache dtype differs
    assert b"dtype" in lib.tb_last_error_message()


def test_fp32_block_rejects_bf16_output(lib):
    c = cfg(dtype=tb.TB_F32)
    assert lib.tb_block_prefill(ctypes.byref(c), FAKE, FAKE, FAKE + 4096, 1, 1, 1, None, FAKE, 1 << 30, None) == 1


def test_decode_argument_checks(lib):
    c = cfg()
    assert lib.tb_block_decode(ctypes.byref(c), FAKE, FAKE, FAKE + 4096, 0, None, FAKE, 1 << 30, None) == 1
    kv = binding.tb_kvcache(FAKE, FAKE, FAKE, 2, 2, 4096, 64, 1)     # T_max > max_pos
    assert lib.tb_block_decode(ctypes.byref(c), FAKE, FAKE, FAKE + 4096, 0, ctypes.byref(kv), FAKE, 1 << 30,
                               None) == 1
    kv = binding.tb_kvcache(FAKE, FAKE, FAKE, 2049, 2, 512, 64, 1)    # above the decode batch limit
    assert lib.tb_block_decode(ctypes.byref(c), FAKE, FAKE, FAKE + 4096, 0, ctypes.byref(kv), FAKE, 1 << 40,
                               None) == 2
    kv = binding.tb_kvcache(FAKE, FAKE, FAKE, 0, 2, 512, 64, 1)       # no sequences: no-op
    assert lib.tb_block_decode(ctypes.byref(c), FAKE, FAKE, FAKE + 4096, 0, ctypes.byref(kv), FAKE, 0, None) == 0


def test_noalloc_decode_rejects_steps_beyond_its_scratch(lib):
    # 64 sequences of a 16384-row cache at d = 4096 need more than the 64 MiB scratch
    c = cfg(d=4096, H=32, Hkv=8, dh=128, f=14336, max_pos=16384)
    assert lib.tb_workspace_bytes(ctypes.byref(c), 64, 16384, 1) > 64 << 20
    kv = binding.tb_kvcache(FAKE, FAKE, FAKE, 64, 8, 16384, 128, 1)
    st = lib.tb_block_decode_noalloc(ctypes.byref(c), FAKE, FAKE, FAKE + 4096, 0, ctypes.byref(kv), None)
    assert st == 1 and b"static scratch" in lib.tb_last_error_message()
    # a step that fits is not rejected for its size (its bad pointers are, later)
    assert lib.tb_workspace_bytes(ctypes.byref(c), 32, 16384, 1) <= 64 << 20
    st = lib.tb_block_decode_noalloc(ctypes.byref(c), FAKE, None, FAKE + 4096, 0, ctypes.byref(kv), None)
    assert st == 1


def test_append_argument_checks(lib):
    kv = binding.tb_kvcache(FAKE, FAKE, FAKE, 2, 2, 16, 64, 1)
    assert lib.tb_kvcache_append(ctypes.byref(kv), FAKE, FAKE, -1, None) == 1
    assert lib.tb_kvcache_append(ctypes.byref(kv), FAKE, FAKE, 0, None) == 0
    assert lib.tb_kvcache_append(ctypes.byref(kv), FAKE, FAKE, 17, None) == 4     # more rows than T_max
    assert lib.tb_kvcache_append(ctypes.byref(kv), None, FAKE, 3, None) == 1


def test_int8_cache_checks(lib):
    """An int8 cache takes a bf16 block with dh 128, T_max a multiple of 32, both
    scale arrays and, paged, a page size that is a multiple of 32; anything else
    is refused before a launch."""
    c = cfg(d=512, H=4, Hkv=2, dh=128)
    decode = lambda kv, cc=c: lib.tb_block_decode(ctypes.byref(cc), FAKE, FAKE, FAKE + 4096, 0, ctypes.byref(kv),
                                                  FAKE, 1 << 30, None)
    i8 = lambda **k: binding.tb_kvcache(FAKE, FAKE, FAKE, 2, 2, k.get("T_max", 256), k.get("dh", 128), tb.TB_I8,
                                        k.get("bt", None), k.get("ps", 0), k.get("np", 0), k.get("ks", FAKE),
                                        k.get("vs", FAKE))
    assert decode(i8(ks=None)) == 1 and b"k_scale" in lib.tb_last_error_message()
    assert decode(i8(vs=FAKE + 4)) == 1                       # misaligned scales
    assert decode(i8(T_max=240)) == 2                         # T_max not a multiple of 32
    assert decode(i8(bt=FAKE, ps=16, np=8)) == 2              # paged: page_size not a multiple of 32
    assert b"page_size" in lib.tb_last_error_message()
    assert lib.tb_kvcache_append(ctypes.byref(i8(bt=FAKE, ps=48, np=8, T_max=96)), FAKE, FAKE, 3, None) == 2
    assert decode(i8(), cfg(d=512, H=4, Hkv=2, dh=128, dtype=tb.TB_F32)) == 2   # fp32 block
    assert decode(i8(dh=64), cfg()) == 2                      # dh 64
    # append: bf16 rows into the int8 layout, same rules
    assert lib.tb_kvcache_append(ctypes.byref(i8(T_max=240)), FAKE, FAKE, 3, None) == 2
    assert lib.tb_kvcache_append(ctypes.byref(i8(ks=None)), FAKE, FAKE, 3, None) == 1
    assert lib.tb_kvcache_append(ctypes.byref(i8()), FAKE, FAKE, 300, None) == 4    # more rows than T_max


def test_workspace_grows_with_tokens(lib):
    c = cfg()
    a = lib.tb_workspace_bytes(ctypes.byref(c), 1, 128, 0)
    b = lib.tb_workspace_bytes(ctypes.byref(c), 2, 128, 0)
    assert 0 < a < b
    assert lib.tb_workspace_bytes(ctypes.byref(c), 1, 128, 7) == 0


def test_status_strings(lib):
    assert tb.tb_status_string(0) == "ok"
    assert tb.tb_status_string(4) == "KV cache full"


def test_model_level_entry_points_validate_first(lib):
    """The embedding, LM head and stack entry points reject bad arguments on the
    host, before any launch."""
    P = ctypes.POINTER
    # embedding: unknown dtype, and d·sizeof not a multiple of 16
    assert lib.tb_embed(FAKE, 10, 64, 7, FAKE, 5, FAKE, None) == 1
    assert lib.tb_embed(FAKE, 10, 12, tb.TB_BF16, FAKE, 5, FAKE, None) == 2
    # head: V not a multiple of 4, bf16 d not a multiple of 64, targets without nll
    bad_v = binding.tb_head_cfg(256, 1001, 1e-5, tb.TB_BF16)
    assert lib.tb_lm_head_packed_bytes(ctypes.byref(bad_v)) == 0
    bad_d = binding.tb_head_cfg(96, 1000, 1e-5, tb.TB_BF16)
    assert lib.tb_lm_head_workspace_bytes(ctypes.byref(bad_d), 16) == 0
    good = binding.tb_head_cfg(256, 1000, 1e-5, tb.TB_BF16)
    assert lib.tb_lm_head_packed_bytes(ctypes.byref(good)) >= 256 * 1000 * 2
    assert lib.tb_lm_head(ctypes.byref(good), FAKE, FAKE, 4, None, FAKE, None, 0, FAKE, 1 << 30, None) == 1
    # nothing requested: a no-op
    assert lib.tb_lm_head(ctypes.byref(good), FAKE, FAKE, 4, None, None, None, 0, FAKE, 1 << 30, None) == 0
    # stack: L = 0, and a workspace smaller than the stack needs
    c = cfg()
    arr = (ctypes.c_void_p * 2)(FAKE, FAKE)
    assert lib.tb_stack_prefill(ctypes.byref(c), 0, arr, FAKE, FAKE + 4096, 0, 2, 16, None, FAKE, 1 << 30, None) == 1
    need = lib.tb_stack_workspace_bytes(ctypes.byref(c), 2, 16, 0)
    assert need > lib.tb_workspace_bytes(ctypes.byref(c), 2, 16, 0)
    assert lib.tb_stack_prefill(ctypes.byref(c), 2, arr, FAKE, FAKE + 4096, 0, 2, 16, None, FAKE, need - 1, None) == 1
