"""GB300-native Llama-layout pre-norm decoder block (prefill and decode).

The compute path is the C ABI of ``libtb.so`` (include/tb.h): hand-written
sm_103a CUDA kernels.  This package holds the ctypes binding (``binding``),
the build step (``build``) and the work accounting used by the benchmark
(``accounting``).
"""
from .binding import (TB_BF16, TB_F32, TB_I8, TB_DEVERR_CACHE_FULL, TB_DEVERR_TIMEOUT, TB_DEVERR_BAD_PAGE, TB_DEVERR_BAD_TOKEN,
                      BlockConfig, HeadConfig, KVCache, TbError, tb_embed, tb_lm_head, tb_pack_lm_head,
                      tb_stack_decode, tb_stack_prefill,
                      tb_block_decode, tb_block_decode_noalloc, tb_block_prefill, tb_get_device_error, tb_kvcache_append,
                      tb_pack_weights, tb_packed_weights_bytes, tb_status_string, tb_workspace_bytes)

__all__ = ["TB_BF16", "TB_F32", "TB_I8", "TB_DEVERR_CACHE_FULL", "TB_DEVERR_TIMEOUT", "TB_DEVERR_BAD_PAGE", "TB_DEVERR_BAD_TOKEN", "BlockConfig", "HeadConfig", "KVCache", "TbError",
           "tb_embed", "tb_lm_head", "tb_pack_lm_head", "tb_stack_decode", "tb_stack_prefill",
           "tb_block_decode", "tb_block_decode_noalloc", "tb_block_prefill", "tb_get_device_error", "tb_kvcache_append", "tb_pack_weights",
           "tb_packed_weights_bytes", "tb_status_string", "tb_workspace_bytes"]
