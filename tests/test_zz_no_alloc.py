"""The no-allocation decode entry point against the workspace one.

tb_block_decode_noalloc is for callers that cannot allocate device memory
(no cudaMalloc or framework allocator allowed on their hot path, or none
available): it runs the decode step with the library's own fixed device
scratch instead of a caller workspace.  Here two identical caches take two
decode steps in a row, one through tb_block_decode with a caller workspace
and one through tb_block_decode_noalloc, called through the C ABI.  Both run
the same kernels on the same inputs, and every kernel of the step is
bit-reproducible, so outputs, caches and lengths must be identical after each
step: a wrong scratch offset, or state left over in the shared scratch from an
earlier call, would show as a difference.  This file is collected last so
that a failure here never hides another test.
"""
import pytest
import torch

import workloads
from helpers import block_config, to_device

pytestmark = pytest.mark.gpu


def test_noalloc_decode_matches_workspace_decode_two_steps():
    import causal_gqa_attention_rmsnorm_gb300 as tb
    s = workloads.BlockShape("noalloc", "decode", "bf16", B=4, T=600, d=1024, H=8, Hkv=2, dh=128, f=2048,
                             rope_base=1e4, eps=1e-6, gains="normal")
    lens = torch.tensor([5, 130, 598, 257], dtype=torch.int32)
    inp = workloads.make_block_inputs(s, seed=21)
    x2 = workloads.make_block_inputs(s, seed=22)["x"]          # the second step's tokens
    kc, vc = workloads.make_decode_cache(s, 21, lens, fill=float("nan"), device="cuda")
    kv_ws = tb.KVCache(kc.clone(), vc.clone(), lens.cuda())
    kv_na = tb.KVCache(kc.clone(), vc.clone(), lens.cuda())
    cfg = block_config(s, max_pos=s.T)
    dev = to_device(inp)
    packed = tb.tb_pack_weights(cfg, dev)
    for step, x in enumerate((dev["x"], x2.cuda())):
        y_ws = tb.tb_block_decode(cfg, packed, x, kv_ws)
        y_na = tb.tb_block_decode_noalloc(cfg, packed, x, kv_na)
        assert tb.tb_get_device_error(clear=True) == 0
        assert torch.isfinite(y_na).all(), step
        assert torch.equal(y_na, y_ws), step
        assert torch.equal(kv_na.lens, kv_ws.lens), step
        # bit patterns, so that the NaN rows no step has written compare too
        assert torch.equal(kv_na.k.view(torch.int16), kv_ws.k.view(torch.int16)), step
        assert torch.equal(kv_na.v.view(torch.int16), kv_ws.v.view(torch.int16)), step
    assert kv_na.lens.cpu().tolist() == [int(n) + 2 for n in lens]
