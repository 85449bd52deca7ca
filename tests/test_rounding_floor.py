"""Why the 3e-2 max-abs bar is out of reach at d = 4096 with bf16 operands.

A CPU fp32 model of the bf16 path's rounding points (tests/rounding_model.py,
no CUDA) is compared with the fp64 oracle on a slice of the gqa_8k workload.
The rounding alone already exceeds 3e-2 max-abs while staying far inside the
1e-2 relative-L2 bar; the GPU parity tests therefore hold d = 4096 workloads
to the relative-L2 bar plus a max-abs bound measured from this model in the
same run (after showing that the GPU's deviation is the model's), and keep
the 3e-2 bar as a strict expected failure.
"""
import numpy as np

import oracle
import workloads
from helpers import errors, oracle_cfg, oracle_weights
from rounding_model import emulate_prefill_seq


def test_bf16_rounding_floor_at_d4096():
    s = workloads.CONFIGS["gqa_8k"]
    T = 512
    inp = workloads.make_block_inputs(s.with_(B=1), seed=0, x_tokens=T)
    ref = oracle.block_prefill_seq(workloads.to_f64(inp["x"][0]), oracle_weights(inp), oracle_cfg(s))["y"]
    e = errors(emulate_prefill_seq(inp, s).double().numpy(), ref)
    assert e["rel_l2"] < 1e-2                      # the relative bar holds with margin
    assert e["max_abs"] > 3e-2                     # rounding alone misses the max-abs bar
