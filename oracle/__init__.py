"""fp64 CPU oracle of the Llama-layout pre-norm decoder block.

TEST INFRASTRUCTURE, not part of the product.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
it.  It shares no code with the CUDA library and never imports it.

Every function is pinned by ``tests/test_oracle_pins.py`` against what the
pages and the mathematics fix (closed forms, invariants, a library
cross-check, brute force on tiny inputs); none is "parity unpinned".
"""
from .block import (Cfg, rms_norm, rope_angles, rope, silu, softmax_rows, visible_keys,
                    causal_attention,
                    qkv_heads, mlp_branch, block_prefill_seq, block_prefill, block_decode_seq,
                    gather_paged, quantize_rows, dequantize_rows, block_decode_seq_int8, block_decode)

from .model import embed, lm_head, token_nll, stack_prefill_seq, stack_decode_seq

__all__ = ["embed", "lm_head", "token_nll", "stack_prefill_seq", "stack_decode_seq", "Cfg", "rms_norm", "rope_angles", "rope", "silu", "softmax_rows", "visible_keys", "causal_attention",
           "qkv_heads", "mlp_branch", "block_prefill_seq", "block_prefill", "block_decode_seq",
           "gather_paged", "quantize_rows", "dequantize_rows", "block_decode_seq_int8", "block_decode"]
