"""The no-allocation decode entry point against the workspace one.

tb_block_decode_noalloc is for callers that cannot allocate device memory
(no cudaMalloc or framework allocator allowed on their hot path, or none
available): it runs the decode step with the library's own fixed device
scratch instead of a caller workspace.  Here two identical caches take two
decode steps in a row, one through tb_block_decode with a caller workspace
and one through tb_block_decode_noalloc, called through the C ABI; outputs,
caches and lengths must agree within the bf16 tolerance of the other tests.
This file is collected last so that a failure here never hides another test.
"""
import pytest
import torch

import workloads
from helpers import BF16_MAX_ABS_TOL, BF16_REL_L2_TOL, block_config, errors, to_device

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
    for x in (dev["x"], x2.cuda()):
        y_ws = tb.tb_block_decode(cfg, packed, x, kv_ws)
        y_na = tb.tb_block_decode_noalloc(cfg, packed, x, kv_na)
        assert tb.tb_get_device_error(clear=True) == 0
        e = errors(y_na.cpu().double().numpy(), y_ws.cpu().double().numpy())
        assert e["finite"] and e["rel_l2"] <= BF16_REL_L2_TOL and e["max_abs"] <= BF16_MAX_ABS_TOL, e
    assert torch.equal(kv_na.lens, kv_ws.lens)
    assert kv_na.lens.cpu().tolist() == [int(n) + 2 for n in lens]
    n = int(lens.max()) + 2
    e = errors(kv_na.k[:, :, :n].float().nan_to_num(7.0).cpu().numpy(),
               kv_ws.k[:, :, :n].float().nan_to_num(7.0).cpu().numpy())
    assert e["max_abs"] <= BF16_MAX_ABS_TOL, e
