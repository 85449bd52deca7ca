"""ctypes binding of libtb (include/tb.h): argument marshalling only.

Every function here has the name of the C entry point it calls and does no
arithmetic of the block: it checks that tensors are on the GPU with the right
dtype and layout, reads sizes off their shapes, allocates caller-owned
buffers through torch when the caller passes none, and forwards raw pointers
and the current CUDA stream.  A missing library raises; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import c_float, c_int32, c_size_t, c_void_p
from dataclasses import dataclass
from typing import Dict, Optional

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtb.so")

TB_F32, TB_BF16, TB_I8 = 0, 1, 2
TB_DEVERR_CACHE_FULL, TB_DEVERR_TIMEOUT, TB_DEVERR_BAD_PAGE, TB_DEVERR_BAD_TOKEN = 1, 2, 4, 8
STATUS = {0: "TB_OK", 1: "TB_ERR_INVALID_ARG", 2: "TB_ERR_UNSUPPORTED", 3: "TB_ERR_CUDA",
          4: "TB_ERR_CACHE_FULL", 5: "TB_ERR_TIMEOUT"}
WEIGHT_FIELDS = ("g_attn", "wq", "wk", "wv", "wo", "g_mlp", "w1", "w3", "w2")
EXPORTED = ("tb_packed_weights_bytes", "tb_pack_weights", "tb_workspace_bytes", "tb_block_prefill",
            "tb_block_decode", "tb_block_decode_noalloc", "tb_kvcache_append", "tb_get_device_error", "tb_status_string",
            "tb_last_error_message", "tb_embed", "tb_lm_head_packed_bytes", "tb_pack_lm_head",
            "tb_lm_head_workspace_bytes", "tb_lm_head", "tb_stack_workspace_bytes", "tb_stack_prefill",
            "tb_stack_decode")


class tb_block_cfg(ctypes.Structure):
    _fields_ = [("d", c_int32), ("H", c_int32), ("Hkv", c_int32), ("dh", c_int32), ("f", c_int32),
                ("max_pos", c_int32), ("rope_base", c_float), ("eps", c_float), ("dtype", c_int32),
                ("window", c_int32)]


class tb_block_weights(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in WEIGHT_FIELDS]


class tb_kvcache(ctypes.Structure):
    _fields_ = [("k", c_void_p), ("v", c_void_p), ("lens", c_void_p), ("B", c_int32), ("Hkv", c_int32),
                ("T_max", c_int32), ("dh", c_int32), ("dtype", c_int32), ("block_table", c_void_p),
                ("page_size", c_int32), ("num_pages", c_int32), ("k_scale", c_void_p), ("v_scale", c_void_p)]


class tb_head_cfg(ctypes.Structure):
    _fields_ = [("d", c_int32), ("V", c_int32), ("eps", c_float), ("dtype", c_int32)]


class TbError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {STATUS.get(status, status)}: {msg}")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libtb.so.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m causal_gqa_attention_rmsnorm_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER
        L.tb_packed_weights_bytes.argtypes = [P(tb_block_cfg)]
        L.tb_packed_weights_bytes.restype = c_size_t
        L.tb_pack_weights.argtypes = [P(tb_block_cfg), P(tb_block_weights), c_void_p, c_size_t, c_void_p]
        L.tb_workspace_bytes.argtypes = [P(tb_block_cfg), c_int32, c_int32, c_int32]
        L.tb_workspace_bytes.restype = c_size_t
        L.tb_block_prefill.argtypes = [P(tb_block_cfg), c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32,
                                       P(tb_kvcache), c_void_p, c_size_t, c_void_p]
        L.tb_block_decode.argtypes = [P(tb_block_cfg), c_void_p, c_void_p, c_void_p, c_int32, P(tb_kvcache),
                                      c_void_p, c_size_t, c_void_p]
        L.tb_block_decode_noalloc.argtypes = [P(tb_block_cfg), c_void_p, c_void_p, c_void_p, c_int32,
                                              P(tb_kvcache), c_void_p]
        L.tb_kvcache_append.argtypes = [P(tb_kvcache), c_void_p, c_void_p, c_int32, c_void_p]
        L.tb_get_device_error.argtypes = [c_void_p, P(c_int32), c_int32]
        L.tb_status_string.argtypes = [c_int32]
        L.tb_status_string.restype = ctypes.c_char_p
        L.tb_last_error_message.argtypes = []
        L.tb_last_error_message.restype = ctypes.c_char_p
        L.tbx_gemm_bf16.argtypes = [c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32, c_int32,
                                    c_void_p]
        L.tbx_trace_enable.argtypes = [c_int32]
        L.tbx_trace_enable.restype = c_int32
        L.tbx_trace_read.argtypes = [c_int32, ctypes.POINTER(c_float), c_int32]
        L.tbx_trace_read.restype = c_int32
        L.tbx_trace_stage_name.argtypes = [c_int32]
        L.tbx_trace_stage_name.restype = ctypes.c_char_p
        L.tbx_skinny_split_count.argtypes = [c_int32, c_int32, c_int32]
        L.tbx_skinny_split_count.restype = c_int32
        L.tbx_decode_chunk_keys.argtypes = [c_int32, c_int32, c_int32, c_int32, c_int32]
        L.tbx_decode_chunk_keys.restype = c_int32
        L.tbx_set_stat_poll_ns.argtypes = [ctypes.c_uint64]
        L.tbx_set_stat_poll_ns.restype = ctypes.c_uint64
        L.tb_embed.argtypes = [c_void_p, c_int32, c_int32, c_int32, c_void_p, ctypes.c_int64, c_void_p, c_void_p]
        L.tb_lm_head_packed_bytes.argtypes = [P(tb_head_cfg)]
        L.tb_lm_head_packed_bytes.restype = c_size_t
        L.tb_pack_lm_head.argtypes = [P(tb_head_cfg), c_void_p, c_void_p, c_int32, c_void_p, c_size_t, c_void_p]
        L.tb_lm_head_workspace_bytes.argtypes = [P(tb_head_cfg), c_int32]
        L.tb_lm_head_workspace_bytes.restype = c_size_t
        L.tb_lm_head.argtypes = [P(tb_head_cfg), c_void_p, c_void_p, c_int32, c_void_p, c_void_p, c_void_p, c_int32,
                                 c_void_p, c_size_t, c_void_p]
        L.tb_stack_workspace_bytes.argtypes = [P(tb_block_cfg), c_int32, c_int32, c_int32]
        L.tb_stack_workspace_bytes.restype = c_size_t
        L.tb_stack_prefill.argtypes = [P(tb_block_cfg), c_int32, P(c_void_p), c_void_p, c_void_p, c_int32, c_int32,
                                       c_int32, P(tb_kvcache), c_void_p, c_size_t, c_void_p]
        L.tb_stack_decode.argtypes = [P(tb_block_cfg), c_int32, P(c_void_p), c_void_p, c_void_p, c_int32,
                                      P(tb_kvcache), c_void_p, c_size_t, c_void_p]
        for fn in ("tb_pack_weights", "tb_block_prefill", "tb_block_decode", "tb_block_decode_noalloc",
                   "tb_kvcache_append", "tb_embed", "tb_pack_lm_head", "tb_lm_head", "tb_stack_prefill",
                   "tb_stack_decode", "tb_get_device_error", "tbx_gemm_bf16"):
            getattr(L, fn).restype = c_int32
        _lib = L
    return _lib


def _check(fn: str, status: int):
    if status != 0:
        raise TbError(fn, status, lib().tb_last_error_message().decode())


@dataclass(frozen=True)
class BlockConfig:
    """Python mirror of tb_block_cfg."""
    d: int
    H: int
    Hkv: int
    dh: int
    f: int
    max_pos: int
    rope_base: float
    eps: float
    dtype: int = TB_BF16
    window: int = 0          # sliding-window width W (0: full causal)

    def c(self) -> tb_block_cfg:
        return tb_block_cfg(self.d, self.H, self.Hkv, self.dh, self.f, self.max_pos, self.rope_base, self.eps,
                            self.dtype, self.window)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == TB_F32 else torch.bfloat16


@dataclass
class KVCache:
    """Caller-owned cache tensors.  Contiguous: k, v [B, Hkv, T_max, dh].
    Paged (block_table given): k, v page pools [num_pages, Hkv, page_size, dh]
    and block_table int32 [B, T_max / page_size].  int8 (k, v of torch.int8):
    codes [B, Hkv, T_max, dh] with fp32 row scales k_scale, v_scale
    [B, Hkv, T_max], or paged: code pools [num_pages, Hkv, page_size, dh] and
    scale pools [num_pages, Hkv, page_size].  lens int32 [B]."""
    k: torch.Tensor
    v: torch.Tensor
    lens: torch.Tensor
    block_table: Optional[torch.Tensor] = None
    k_scale: Optional[torch.Tensor] = None
    v_scale: Optional[torch.Tensor] = None

    def c(self) -> tb_kvcache:
        for t in (self.k, self.v):
            if not (t.is_cuda and t.is_contiguous()):
                raise ValueError("cache tensors must be contiguous CUDA tensors")
        if self.v.shape != self.k.shape or self.v.dtype != self.k.dtype:
            raise ValueError("k and v caches must match")
        dt = {torch.float32: TB_F32, torch.bfloat16: TB_BF16, torch.int8: TB_I8}.get(self.k.dtype)
        if dt is None:
            raise ValueError(f"cache dtype {self.k.dtype} is not float32, bfloat16 or int8")
        if self.block_table is None:
            B, Hkv, T_max, dh = self.k.shape
            bt, ps, npages = None, 0, 0
        else:
            npages, Hkv, ps, dh = self.k.shape
            bt = self.block_table
            if not (bt.is_cuda and bt.dtype == torch.int32 and bt.dim() == 2 and bt.is_contiguous()):
                raise ValueError("block_table must be a contiguous CUDA int32 tensor [B, pages per sequence]")
            B, T_max = bt.shape[0], bt.shape[1] * ps
        if not (self.lens.is_cuda and self.lens.dtype == torch.int32 and self.lens.numel() == B):
            raise ValueError("lens must be a CUDA int32 tensor of B entries")
        ks = vs = None
        if dt == TB_I8:
            for name, t in (("k_scale", self.k_scale), ("v_scale", self.v_scale)):
                if t is None:
                    raise ValueError(f"an int8 cache needs {name}")
                _need(t, name, torch.float32, (B, Hkv, T_max) if bt is None else (npages, Hkv, ps))
            ks, vs = self.k_scale.data_ptr(), self.v_scale.data_ptr()
        return tb_kvcache(self.k.data_ptr(), self.v.data_ptr(), self.lens.data_ptr(), B, Hkv, T_max, dh, dt,
                          None if bt is None else bt.data_ptr(), ps, npages, ks, vs)

    @property
    def T_max(self) -> int:
        return self.k.shape[2] if self.block_table is None else self.block_table.shape[1] * self.k.shape[2]

    @staticmethod
    def empty(B: int, Hkv: int, T_max: int, dh: int, dtype=torch.bfloat16, device="cuda", fill=None) -> "KVCache":
        mk = (lambda: torch.full((B, Hkv, T_max, dh), fill, dtype=dtype, device=device)) if fill is not None \
            else (lambda: torch.empty((B, Hkv, T_max, dh), dtype=dtype, device=device))
        return KVCache(mk(), mk(), torch.zeros(B, dtype=torch.int32, device=device))

    @staticmethod
    def empty_int8(B: int, Hkv: int, T_max: int, dh: int = 128, device="cuda") -> "KVCache":
        """Zeroed int8 codes and scales (every row reads back as 0)."""
        codes = lambda: torch.zeros((B, Hkv, T_max, dh), dtype=torch.int8, device=device)
        scales = lambda: torch.zeros((B, Hkv, T_max), dtype=torch.float32, device=device)
        return KVCache(codes(), codes(), torch.zeros(B, dtype=torch.int32, device=device), None, scales(), scales())

    @staticmethod
    def empty_paged(B: int, Hkv: int, T_max: int, dh: int, page_size: int, num_pages: int, block_table: torch.Tensor,
                    dtype=torch.bfloat16, device="cuda", fill=None) -> "KVCache":
        """Page pools of num_pages pages and the caller's block table [B, T_max / page_size]."""
        shape = (num_pages, Hkv, page_size, dh)
        mk = (lambda: torch.full(shape, fill, dtype=dtype, device=device)) if fill is not None \
            else (lambda: torch.empty(shape, dtype=dtype, device=device))
        if block_table.shape != (B, T_max // page_size):
            raise ValueError("block_table must be [B, T_max / page_size]")
        return KVCache(mk(), mk(), torch.zeros(B, dtype=torch.int32, device=device),
                       block_table.to(device=device, dtype=torch.int32).contiguous())


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def tb_status_string(status: int) -> str:
    return lib().tb_status_string(status).decode()


def tb_packed_weights_bytes(cfg: BlockConfig) -> int:
    n = lib().tb_packed_weights_bytes(ctypes.byref(cfg.c()))
    if n == 0:
        raise TbError("tb_packed_weights_bytes", 1, lib().tb_last_error_message().decode())
    return n


def tb_workspace_bytes(cfg: BlockConfig, B: int, T: int, mode: int) -> int:
    return lib().tb_workspace_bytes(ctypes.byref(cfg.c()), B, T, mode)


def tb_pack_weights(cfg: BlockConfig, weights: Dict[str, torch.Tensor], packed: Optional[torch.Tensor] = None,
                    stream=None) -> torch.Tensor:
    """Pack [in, out] weights (dict with the tb_block_weights field names)."""
    dev = weights["wq"].device
    for n in WEIGHT_FIELDS:
        _need(weights[n], n, cfg.torch_dtype)
    nbytes = tb_packed_weights_bytes(cfg)
    if packed is None:
        packed = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    w = tb_block_weights(*[weights[n].data_ptr() for n in WEIGHT_FIELDS])
    _check("tb_pack_weights", lib().tb_pack_weights(ctypes.byref(cfg.c()), ctypes.byref(w), packed.data_ptr(),
                                                    packed.numel() * packed.element_size(), _stream(stream)))
    return packed


def _workspace(cfg, B, T, mode, ws, device):
    need = tb_workspace_bytes(cfg, B, T, mode)
    if ws is None:
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    return ws, ws.numel() * ws.element_size()


def tb_block_prefill(cfg: BlockConfig, packed: torch.Tensor, x: torch.Tensor, y: Optional[torch.Tensor] = None,
                     y_dtype: int = TB_F32, kv: Optional[KVCache] = None, ws: Optional[torch.Tensor] = None,
                     stream=None) -> torch.Tensor:
    """Prefill x [B, T, d] -> y [B, T, d]; with kv, also fills the cache."""
    if x.dim() != 3:
        raise ValueError("x must be [B, T, d]")
    B, T, d = x.shape
    _need(x, "x", cfg.torch_dtype)
    ydt = torch.float32 if y_dtype == TB_F32 else torch.bfloat16
    if y is None:
        y = torch.empty((B, T, d), dtype=ydt, device=x.device)
    _need(y, "y", ydt, (B, T, d))
    ws, ws_bytes = _workspace(cfg, B, T, 0, ws, x.device)
    kvc = ctypes.byref(kv.c()) if kv is not None else None
    _check("tb_block_prefill", lib().tb_block_prefill(ctypes.byref(cfg.c()), packed.data_ptr(), x.data_ptr(),
                                                      y.data_ptr(), y_dtype, B, T, kvc, ws.data_ptr(), ws_bytes,
                                                      _stream(stream)))
    return y


def tb_block_decode(cfg: BlockConfig, packed: torch.Tensor, x: torch.Tensor, kv: KVCache,
                    y: Optional[torch.Tensor] = None, y_dtype: int = TB_F32, ws: Optional[torch.Tensor] = None,
                    stream=None) -> torch.Tensor:
    """One decode step: x [B, 1, d] at positions kv.lens -> y [B, 1, d]; appends to the cache."""
    kvs = kv.c()
    B = kvs.B
    _need(x, "x", cfg.torch_dtype, (B, 1, cfg.d))
    ydt = torch.float32 if y_dtype == TB_F32 else torch.bfloat16
    if y is None:
        y = torch.empty((B, 1, cfg.d), dtype=ydt, device=x.device)
    _need(y, "y", ydt, (B, 1, cfg.d))
    ws, ws_bytes = _workspace(cfg, B, kvs.T_max, 1, ws, x.device)
    _check("tb_block_decode", lib().tb_block_decode(ctypes.byref(cfg.c()), packed.data_ptr(), x.data_ptr(),
                                                    y.data_ptr(), y_dtype, ctypes.byref(kvs), ws.data_ptr(),
                                                    ws_bytes, _stream(stream)))
    return y


def tb_block_decode_noalloc(cfg: BlockConfig, packed: torch.Tensor, x: torch.Tensor, kv: KVCache,
                            y: Optional[torch.Tensor] = None, y_dtype: int = TB_F32, stream=None) -> torch.Tensor:
    """tb_block_decode without a workspace argument: the library uses its own
    fixed 64 MiB device scratch, for callers that cannot allocate device
    memory.  Calls that may overlap on the GPU must be serialised."""
    kvs = kv.c()
    B = kvs.B
    _need(x, "x", cfg.torch_dtype, (B, 1, cfg.d))
    ydt = torch.float32 if y_dtype == TB_F32 else torch.bfloat16
    if y is None:
        y = torch.empty((B, 1, cfg.d), dtype=ydt, device=x.device)
    _need(y, "y", ydt, (B, 1, cfg.d))
    _check("tb_block_decode_noalloc", lib().tb_block_decode_noalloc(ctypes.byref(cfg.c()), packed.data_ptr(),
                                                                    x.data_ptr(), y.data_ptr(), y_dtype,
                                                                    ctypes.byref(kvs), _stream(stream)))
    return y


def tb_kvcache_append(kv: KVCache, k_new: torch.Tensor, v_new: torch.Tensor, stream=None) -> None:
    """Append k_new, v_new [B, Hkv, n, dh] at rows lens[b].. of each sequence
    (bf16 rows for an int8 cache, quantised as they are stored)."""
    kvs = kv.c()
    n = k_new.shape[2]
    shape = (kvs.B, kvs.Hkv, n, kvs.dh)
    row_dtype = torch.bfloat16 if kv.k.dtype == torch.int8 else kv.k.dtype
    _need(k_new, "k_new", row_dtype, shape)
    _need(v_new, "v_new", row_dtype, shape)
    _check("tb_kvcache_append", lib().tb_kvcache_append(ctypes.byref(kvs), k_new.data_ptr(), v_new.data_ptr(), n,
                                                        _stream(stream)))


def tb_get_device_error(stream=None, clear: bool = False) -> int:
    """Synchronise the stream and return the device error word (TB_DEVERR_* bits)."""
    out = c_int32(0)
    _check("tb_get_device_error", lib().tb_get_device_error(_stream(stream), ctypes.byref(out), int(clear)))
    return out.value


def tbx_gemm_bf16(A: torch.Tensor, B: torch.Tensor, bn: int = 256, mt: int = 1, stream=None) -> torch.Tensor:
    """Test hook: A [M, K] · B [N, K]ᵀ in fp32 through the tcgen05 main loop
    (mt = 2: 256-row tiles on CTA pairs, M = 256 MMAs)."""
    _need(A, "A", torch.bfloat16)
    _need(B, "B", torch.bfloat16)
    M, K = A.shape
    N = B.shape[0]
    C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _check("tbx_gemm_bf16", lib().tbx_gemm_bf16(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, bn, mt,
                                                _stream(stream)))
    return C


def tbx_set_stat_poll_ns(ns: int) -> int:
    """Test hook: how long a prefill QKV tile epilogue polls for its row group's
    RMSNorm-1 statistics before forming its rows' scales itself; returns the
    previous value."""
    return int(lib().tbx_set_stat_poll_ns(int(ns)))


def tbx_trace_enable(slots: int) -> None:
    """Record per-stage CUDA events for the next calls, in a ring of `slots`
    calls (0 turns tracing off and frees the events)."""
    if lib().tbx_trace_enable(int(slots)) != 0:
        raise RuntimeError("tbx_trace_enable: cudaEventCreate failed")


def tbx_trace_read(slot: int):
    """Stage durations (ms) of one traced call: list of (name, ms)."""
    buf = (c_float * 8)()
    n = lib().tbx_trace_read(int(slot), buf, 8)
    if n < 0:
        raise RuntimeError("tbx_trace_read: CUDA error")
    return [(lib().tbx_trace_stage_name(i).decode(), float(buf[i])) for i in range(n)]


# ---- around the block: embedding, LM head, L-layer stack -------------------

@dataclass
class HeadConfig:
    """Python mirror of tb_head_cfg."""
    d: int
    V: int
    eps: float
    dtype: int = TB_BF16

    def c(self) -> tb_head_cfg:
        return tb_head_cfg(self.d, self.V, self.eps, self.dtype)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == TB_F32 else torch.bfloat16


def tb_embed(table: torch.Tensor, ids: torch.Tensor, x: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """x[t] = table[ids[t]]: table [V, d], ids int32 (any shape) -> x [*ids.shape, d]."""
    V, d = table.shape
    _need(table, "table", table.dtype)
    _need(ids, "ids", torch.int32)
    if x is None:
        x = torch.empty((*ids.shape, d), dtype=table.dtype, device=table.device)
    _need(x, "x", table.dtype, (*ids.shape, d))
    dt = TB_F32 if table.dtype == torch.float32 else TB_BF16
    _check("tb_embed", lib().tb_embed(table.data_ptr(), V, d, dt, ids.data_ptr(), ids.numel(), x.data_ptr(),
                                      _stream(stream)))
    return x


def tb_pack_lm_head(cfg: HeadConfig, g_final: torch.Tensor, w_u: torch.Tensor, tied: bool = False,
                    stream=None) -> torch.Tensor:
    """Pack the head: w_u [d, V], or with tied=True the embedding table [V, d]."""
    _need(g_final, "g_final", cfg.torch_dtype, (cfg.d,))
    _need(w_u, "w_u", cfg.torch_dtype, (cfg.V, cfg.d) if tied else (cfg.d, cfg.V))
    n = lib().tb_lm_head_packed_bytes(ctypes.byref(cfg.c()))
    if n == 0:
        raise TbError("tb_lm_head_packed_bytes", 1, lib().tb_last_error_message().decode())
    packed = torch.empty(n, dtype=torch.uint8, device=w_u.device)
    _check("tb_pack_lm_head", lib().tb_pack_lm_head(ctypes.byref(cfg.c()), g_final.data_ptr(), w_u.data_ptr(),
                                                    1 if tied else 0, packed.data_ptr(), n, _stream(stream)))
    return packed


def tb_lm_head(cfg: HeadConfig, packed: torch.Tensor, x: torch.Tensor, want_logits: bool = True,
               targets: Optional[torch.Tensor] = None, row_chunk: int = 0, ws: Optional[torch.Tensor] = None,
               stream=None):
    """Head over x [M, d]: returns (logits [M, V] fp32 or None, nll [M] fp32 or None)."""
    M = x.shape[0]
    _need(x, "x", cfg.torch_dtype, (M, cfg.d))
    logits = torch.empty((M, cfg.V), dtype=torch.float32, device=x.device) if want_logits else None
    nll = None
    if targets is not None:
        _need(targets, "targets", torch.int32, (M,))
        nll = torch.empty(M, dtype=torch.float32, device=x.device)
    need = lib().tb_lm_head_workspace_bytes(ctypes.byref(cfg.c()), row_chunk)
    if ws is None:
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    _check("tb_lm_head", lib().tb_lm_head(ctypes.byref(cfg.c()), packed.data_ptr(), x.data_ptr(), M,
                                          None if logits is None else logits.data_ptr(),
                                          None if targets is None else targets.data_ptr(),
                                          None if nll is None else nll.data_ptr(), row_chunk, ws.data_ptr(),
                                          ws.numel(), _stream(stream)))
    return logits, nll


def _packed_array(packed):
    arr = (c_void_p * len(packed))(*[p.data_ptr() for p in packed])
    return arr


def tb_stack_prefill(cfg: BlockConfig, packed, x: torch.Tensor, kvs=None, y_dtype: int = TB_F32,
                     ws: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """An L-layer prefill (L = len(packed)); kvs: None or a list of L KVCache."""
    B, T, d = x.shape
    _need(x, "x", cfg.torch_dtype, (B, T, cfg.d))
    L = len(packed)
    ydt = torch.float32 if y_dtype == TB_F32 else torch.bfloat16
    y = torch.empty((B, T, d), dtype=ydt, device=x.device)
    kv_arr = None
    if kvs is not None:
        if len(kvs) != L:
            raise ValueError("one cache per layer")
        kv_arr = (tb_kvcache * L)(*[kv.c() for kv in kvs])
    need = lib().tb_stack_workspace_bytes(ctypes.byref(cfg.c()), B, T, 0)
    if ws is None:
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    _check("tb_stack_prefill", lib().tb_stack_prefill(ctypes.byref(cfg.c()), L, _packed_array(packed), x.data_ptr(),
                                                      y.data_ptr(), y_dtype, B, T, kv_arr, ws.data_ptr(), ws.numel(),
                                                      _stream(stream)))
    return y


def tb_stack_decode(cfg: BlockConfig, packed, x: torch.Tensor, kvs, y_dtype: int = TB_F32,
                    ws: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """One decode step through the L-layer stack: x [B, 1, d]; kvs a list of L KVCache."""
    L = len(packed)
    if len(kvs) != L:
        raise ValueError("one cache per layer")
    kv_arr = (tb_kvcache * L)(*[kv.c() for kv in kvs])
    B, T_max = kv_arr[0].B, kv_arr[0].T_max
    _need(x, "x", cfg.torch_dtype, (B, 1, cfg.d))
    ydt = torch.float32 if y_dtype == TB_F32 else torch.bfloat16
    y = torch.empty((B, 1, cfg.d), dtype=ydt, device=x.device)
    need = lib().tb_stack_workspace_bytes(ctypes.byref(cfg.c()), B, T_max, 1)
    if ws is None:
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    _check("tb_stack_decode", lib().tb_stack_decode(ctypes.byref(cfg.c()), L, _packed_array(packed), x.data_ptr(),
                                                    y.data_ptr(), y_dtype, kv_arr, ws.data_ptr(), ws.numel(),
                                                    _stream(stream)))
    return y
