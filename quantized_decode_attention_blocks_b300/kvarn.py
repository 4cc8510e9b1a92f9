"""Thin ctypes binding of libkvarn (include/kvarn.h).

Argument marshalling only: every step of quantization and decode attention
runs in the CUDA kernels of libkvarn.so.  torch supplies device memory and the
current stream.  If the library is missing the import fails loudly; there is
no CPU fallback.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkvarn.so")

HEAD_DIM = 128
BLOCK_TOKENS = 128
PAGE_BYTES = 15360
PAGE_BYTES_M16 = 13824     # KVARN_PAGE_BYTES_M16: format variant "_m16"
PAGE_BYTES_G64 = 17408     # KVARN_PAGE_BYTES_G64: format variant "k4v2_g64"
PAGE_BYTES_V4 = 19456      # KVARN_PAGE_BYTES_V4: format variant "k4v4_g128"
PAGE_BYTES_K8 = 27648      # KVARN_PAGE_BYTES_K8: format variant "k8v4_g128"
FP8_PAGE_BYTES = 33792     # KVARN_FP8_PAGE_BYTES
FP16_PAGE_BYTES = 65536            # KVARN_FP16_PAGE_BYTES
NOALLOC_SCRATCH_BYTES = 16 << 20   # KVARN_NOALLOC_SCRATCH_BYTES

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_WORKSPACE = -3
ERR_LAUNCH = -4
STATUS_BAD_PAGE = 1
STATUS_BAD_LENGTH = 2
STATUS_TIMEOUT = 4


class KvarnError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} ({code})")
        self.code = code


class Config(ctypes.Structure):
    _fields_ = [("head_dim", ctypes.c_int), ("block_tokens", ctypes.c_int),
                ("group", ctypes.c_int), ("k_bits", ctypes.c_int), ("v_bits", ctypes.c_int),
                ("sinkhorn_iters", ctypes.c_int), ("num_q_heads", ctypes.c_int),
                ("num_kv_heads", ctypes.c_int), ("sinkhorn_rms", ctypes.c_int),
                ("meta_fp16", ctypes.c_int), ("per_channel", ctypes.c_int)]

    @property
    def g(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def page_bytes(self) -> int:
        """Bytes of one page record of this format (kvarn_page_bytes)."""
        if self.group == 64:
            return PAGE_BYTES_G64
        if self.k_bits == 8:
            return PAGE_BYTES_K8
        if self.v_bits == 4:
            return PAGE_BYTES_V4
        return PAGE_BYTES_M16 if self.meta_fp16 else PAGE_BYTES


# every symbol include/kvarn.h declares, with its ctypes signature
_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_int64
SIGNATURES = {
    "kvarn_config_from_string": (_I, [ctypes.c_char_p, _I, _I, ctypes.POINTER(Config)]),
    "kvarn_config_validate": (_I, [ctypes.POINTER(Config)]),
    "kvarn_page_bytes": (ctypes.c_size_t, [ctypes.POINTER(Config)]),
    "kvarn_quantize_blocks": (_I, [ctypes.POINTER(Config), _P, _P, _L, _L, _L, _I, _P, _I, _P,
                                   _I, _P, _L, _P, _P, _P, _P]),
    "kvarn_append_token": (_I, [ctypes.POINTER(Config), _P, _P, _P, _I, _P, _I, _P, _L, _P, _P,
                                _P, _P]),
    "kvarn_decode_split_plan": (_I, [ctypes.POINTER(Config), _I, _I, _I, ctypes.POINTER(_I),
                                     ctypes.POINTER(_I), ctypes.POINTER(ctypes.c_size_t)]),
    "kvarn_decode_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(Config), _I, _I]),
    "kvarn_decode_attention": (_I, [ctypes.POINTER(Config), _P, _P, _L, _P, _I, _P, _I, _I, _P,
                                    _P, ctypes.c_float, _P, _P, ctypes.c_size_t, _P, _P]),
    "kvarn_decode_attention_noalloc": (_I, [ctypes.POINTER(Config), _P, _P, _L, _P, _I, _P, _I,
                                            _I, _P, _P, ctypes.c_float, _P, _P, _P]),
    "kvarn_chunk_attention": (_I, [ctypes.POINTER(Config), _P, _I, _P, _P, _I, _I, _P, _L, _P,
                                   _I, _P, _P, ctypes.c_float, _P, _P, _P]),
    "kvarn_dequantize_pages": (_I, [_P, _L, _P, _P, _P]),
    "kvarn_dequantize_records": (_I, [_P, _P, _L, _P, _P, _P]),
    "kvarn_wait_check": (_I, [_P, _I, ctypes.c_uint32, _P]),
    "kvarn_fp16_write_blocks": (_I, [_P, _P, _L, _L, _L, _I, _I, _P, _I, _P, _I, _P, _L, _P,
                                     _P]),
    "kvarn_fp16_decode_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I]),
    "kvarn_fp16_decode_attention": (_I, [_P, _I, _I, _P, _L, _P, _I, _P, _I, _I,
                                         ctypes.c_float, _P, _P, ctypes.c_size_t, _P, _P]),
    "kvarn_fp8_write_blocks": (_I, [_P, _P, _L, _L, _L, _I, _I, _P, _I, _P, _I, _P, _L, _P,
                                    _P]),
    "kvarn_fp8_decode_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I]),
    "kvarn_fp8_decode_attention": (_I, [_P, _I, _I, _P, _L, _P, _I, _P, _I, _I,
                                        ctypes.c_float, _P, _P, ctypes.c_size_t, _P, _P]),
    "kvarn_snapkv_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(Config), _I, _I, _I]),
    "kvarn_snapkv_select": (_I, [ctypes.POINTER(Config), _P, _I, _P, _L, _L, _L, _P, _I, _I, _I,
                                 _I, ctypes.c_float, _P, _P, _P, ctypes.c_size_t, _P, _P]),
    "kvarn_snapkv_gather": (_I, [_P, _P, _L, _L, _L, _I, _I, _I, _P, _I, _P, _P, _P]),
    "kvarn_status_string": (ctypes.c_char_p, [_I]),
    "kvarn_version": (ctypes.c_char_p, []),
}

_lib = None


def lib():
    """Loads libkvarn.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libkvarn.so not built at {LIB_PATH}; run "
                              "python -m quantized_decode_attention_blocks_b300.build")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().kvarn_status_string(int(code)).decode()


def version() -> str:
    return lib().kvarn_version().decode()


def _check(rc: int, what: str):
    if rc != OK:
        raise KvarnError(rc, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _on(device):
    """Makes `device` current for the call when it is not already: the library
    launches on the current device, and the pointers belong to `device`."""
    if (device.type == "cuda" and device.index is not None
            and device.index != torch.cuda.current_device()):
        return torch.cuda.device(device)
    return contextlib.nullcontext()


# Checked on every tensor argument.  The C ABI addresses each buffer from its
# base pointer with a fixed layout, and cannot see the allocation, so a wrong
# dtype, shape or stride would make the kernels read or write outside it.  The
# CPU tests of these checks clear _REQUIRE_CUDA and replace the library.
_REQUIRE_CUDA = True


class _AtLeast:
    def __init__(self, n: int):
        self.n = int(n)

    def ok(self, x: int) -> bool:
        return x >= self.n

    def __repr__(self) -> str:
        return f">={self.n}"


def _arg(t, name: str, dtype, shape=None, device=None, contiguous: bool = True):
    """t must be a tensor of `dtype` (None: any) on `device` (None: any CUDA
    device); shape entries are an exact size, _AtLeast(n) or None (any).
    Returns t.device."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor, got {type(t).__name__}")
    if _REQUIRE_CUDA and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}; the other arguments are on {device}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None:
        fits = t.dim() == len(shape) and all(
            s is None or (s.ok(n) if isinstance(s, _AtLeast) else n == s)
            for n, s in zip(t.shape, shape))
        if not fits:
            want = "[" + "][".join("*" if s is None else repr(s) for s in shape) + "]"
            raise ValueError(f"{name} must have shape {want}, got {list(t.shape)}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.device


def _kv_pair(k, v, hkv: int):
    """Prefill inputs: fp16 [B][S][Hkv][128] with a dense last dim, sharing strides."""
    dev = _arg(k, "k", torch.float16, (None, None, hkv, HEAD_DIM), contiguous=False)
    _arg(v, "v", torch.float16, tuple(k.shape), device=dev, contiguous=False)
    if k.stride() != v.stride() or k.stride(3) != 1:
        raise ValueError("k and v must share shape/strides [B][S][Hkv][128], last dim dense")
    return dev


def _lens_table(dev, B: int, seq_lens, lens_name: str, block_table):
    _arg(seq_lens, lens_name, torch.int32, (_AtLeast(B),), device=dev)
    _arg(block_table, "block_table", torch.int32, (_AtLeast(B), None), device=dev)


def _tails(dev, cfg, B: int, tail_k, tail_v):
    shape = (_AtLeast(B), cfg.num_kv_heads, BLOCK_TOKENS, HEAD_DIM)
    _arg(tail_k, "tail_k", torch.float16, shape, device=dev)
    _arg(tail_v, "tail_v", torch.float16, tuple(tail_k.shape), device=dev)


def _status(dev, status):
    if status is not None:
        _arg(status, "status", torch.int32, (_AtLeast(1),), device=dev)


# ------------------------------------------------------------------ config --

def config_from_string(fmt: str, num_q_heads: int, num_kv_heads: int) -> Config:
    c = Config()
    _check(lib().kvarn_config_from_string(fmt.encode(), num_q_heads, num_kv_heads,
                                          ctypes.byref(c)), "kvarn_config_from_string")
    return c


def config_validate(cfg: Config) -> int:
    return lib().kvarn_config_validate(ctypes.byref(cfg))


def page_bytes(cfg: Config) -> int:
    return lib().kvarn_page_bytes(ctypes.byref(cfg))


# --------------------------------------------------------------- allocation --

def alloc_pool(cfg: Config, num_pages: int, device="cuda") -> torch.Tensor:
    return torch.zeros((num_pages, cfg.num_kv_heads, cfg.page_bytes), dtype=torch.uint8,
                       device=device)


def alloc_tails(cfg: Config, batch: int, device="cuda"):
    shape = (batch, cfg.num_kv_heads, BLOCK_TOKENS, HEAD_DIM)
    return (torch.zeros(shape, dtype=torch.float16, device=device),
            torch.zeros(shape, dtype=torch.float16, device=device))


def decode_split_plan(cfg: Config, batch: int, max_seq: int, num_sms: int = 0):
    """(pages_per_split, nsplit, workspace_bytes) of decode on a GPU with
    `num_sms` SMs (0: the current device)."""
    pps, ns, ws = _I(0), _I(0), ctypes.c_size_t(0)
    _check(lib().kvarn_decode_split_plan(ctypes.byref(cfg), batch, max_seq, num_sms,
                                         ctypes.byref(pps), ctypes.byref(ns), ctypes.byref(ws)),
           "kvarn_decode_split_plan")
    return pps.value, ns.value, ws.value


def decode_workspace_bytes(cfg: Config, batch: int, max_seq: int) -> int:
    return lib().kvarn_decode_workspace_bytes(ctypes.byref(cfg), batch, max_seq)


def alloc_decode_workspace(cfg: Config, batch: int, max_seq: int, device="cuda"):
    n = decode_workspace_bytes(cfg, batch, max_seq)
    return torch.zeros((max(n, 16),), dtype=torch.uint8, device=device)


# ---------------------------------------------------------------- the calls --

def kvarn_quantize_blocks(cfg: Config, k: torch.Tensor, v: torch.Tensor, seq_lens: torch.Tensor,
                          max_seq: int, block_table: torch.Tensor, pool: torch.Tensor,
                          tail_k: torch.Tensor, tail_v: torch.Tensor,
                          status: Optional[torch.Tensor] = None, stream=None) -> None:
    """k, v: fp16 [B][S][Hkv][128] (any strides with a dense last dim);
    seq_lens int32 [B] (each <= S); block_table int32 [B][max_blocks]; pool
    uint8 [num_pages][Hkv][15360]; tails fp16 [B][Hkv][128][128]."""
    dev = _kv_pair(k, v, cfg.num_kv_heads)
    B = k.shape[0]
    _lens_table(dev, B, seq_lens, "seq_lens", block_table)
    _arg(pool, "pool", torch.uint8, (None, cfg.num_kv_heads, cfg.page_bytes), device=dev)
    _tails(dev, cfg, B, tail_k, tail_v)
    _status(dev, status)
    with _on(dev):
        _check(lib().kvarn_quantize_blocks(
            ctypes.byref(cfg), _ptr(k), _ptr(v), k.stride(0), k.stride(1), k.stride(2), B,
            _ptr(seq_lens), int(max_seq), _ptr(block_table), block_table.shape[-1], _ptr(pool),
            pool.shape[0], _ptr(tail_k), _ptr(tail_v), _ptr(status), _stream(stream, dev)),
            "kvarn_quantize_blocks")


def kvarn_append_token(cfg: Config, k_new: torch.Tensor, v_new: torch.Tensor, pos: torch.Tensor,
                       block_table: torch.Tensor, pool: torch.Tensor, tail_k: torch.Tensor,
                       tail_v: torch.Tensor, status: Optional[torch.Tensor] = None,
                       stream=None) -> None:
    """k_new, v_new: fp16 [B][Hkv][128]; pos: int32 [B] length before the append."""
    dev = _arg(k_new, "k_new", torch.float16, (None, cfg.num_kv_heads, HEAD_DIM))
    _arg(v_new, "v_new", torch.float16, tuple(k_new.shape), device=dev)
    B = k_new.shape[0]
    _lens_table(dev, B, pos, "pos", block_table)
    _arg(pool, "pool", torch.uint8, (None, cfg.num_kv_heads, cfg.page_bytes), device=dev)
    _tails(dev, cfg, B, tail_k, tail_v)
    _status(dev, status)
    with _on(dev):
        _check(lib().kvarn_append_token(
            ctypes.byref(cfg), _ptr(k_new), _ptr(v_new), _ptr(pos), B, _ptr(block_table),
            block_table.shape[-1], _ptr(pool), pool.shape[0], _ptr(tail_k), _ptr(tail_v),
            _ptr(status), _stream(stream, dev)), "kvarn_append_token")


def _decode_args(cfg, q, pool, block_table, seq_lens, tail_k, tail_v, out, status):
    dev = _arg(q, "q", torch.float16, (None, cfg.num_q_heads, HEAD_DIM))
    _arg(out, "out", torch.float16, tuple(q.shape), device=dev)
    B = q.shape[0]
    _lens_table(dev, B, seq_lens, "seq_lens", block_table)
    _arg(pool, "pool", torch.uint8, (None, cfg.num_kv_heads, cfg.page_bytes), device=dev)
    _tails(dev, cfg, B, tail_k, tail_v)
    _status(dev, status)
    return dev


def kvarn_decode_attention(cfg: Config, q: torch.Tensor, pool: torch.Tensor,
                           block_table: torch.Tensor, seq_lens: torch.Tensor, max_seq: int,
                           tail_k: torch.Tensor, tail_v: torch.Tensor, out: torch.Tensor,
                           workspace: Optional[torch.Tensor], softmax_scale: float = None,
                           status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """q, out: fp16 [B][Hq][128]; seq_lens int32 [B] (pages + tail tokens)."""
    dev = _decode_args(cfg, q, pool, block_table, seq_lens, tail_k, tail_v, out, status)
    if workspace is not None:
        _arg(workspace, "workspace", None, device=dev)
    if softmax_scale is None:
        softmax_scale = HEAD_DIM ** -0.5
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with _on(dev):
        _check(lib().kvarn_decode_attention(
            ctypes.byref(cfg), _ptr(q), _ptr(pool), pool.shape[0], _ptr(block_table),
            block_table.shape[-1], _ptr(seq_lens), q.shape[0], int(max_seq), _ptr(tail_k),
            _ptr(tail_v), float(softmax_scale), _ptr(out), _ptr(workspace), ws_bytes,
            _ptr(status), _stream(stream, dev)), "kvarn_decode_attention")
    return out


def kvarn_chunk_attention(cfg: Config, q: torch.Tensor, start: torch.Tensor,
                          chunk_lens: torch.Tensor, max_seq: int, pool: torch.Tensor,
                          block_table: torch.Tensor, tail_k: torch.Tensor, tail_v: torch.Tensor,
                          out: torch.Tensor, softmax_scale: float = None,
                          status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Chunked prefill: q, out fp16 [B][M][Hq][128]; start, chunk_lens int32
    [B]; the cache holds start + chunk_lens tokens per sequence."""
    dev = _arg(q, "q", torch.float16, (None, None, cfg.num_q_heads, HEAD_DIM))
    _arg(out, "out", torch.float16, tuple(q.shape), device=dev)
    B = q.shape[0]
    _lens_table(dev, B, start, "start", block_table)
    _arg(chunk_lens, "chunk_lens", torch.int32, (_AtLeast(B),), device=dev)
    _arg(pool, "pool", torch.uint8, (None, cfg.num_kv_heads, cfg.page_bytes), device=dev)
    _tails(dev, cfg, B, tail_k, tail_v)
    _status(dev, status)
    if softmax_scale is None:
        softmax_scale = HEAD_DIM ** -0.5
    with _on(dev):
        _check(lib().kvarn_chunk_attention(
            ctypes.byref(cfg), _ptr(q), q.shape[1], _ptr(start), _ptr(chunk_lens), B,
            int(max_seq), _ptr(pool), pool.shape[0], _ptr(block_table), block_table.shape[-1],
            _ptr(tail_k), _ptr(tail_v), float(softmax_scale), _ptr(out), _ptr(status),
            _stream(stream, dev)), "kvarn_chunk_attention")
    return out


def kvarn_decode_attention_noalloc(cfg: Config, q: torch.Tensor, pool: torch.Tensor,
                                   block_table: torch.Tensor, seq_lens: torch.Tensor,
                                   max_seq: int, tail_k: torch.Tensor, tail_v: torch.Tensor,
                                   out: torch.Tensor, softmax_scale: float = None,
                                   status: Optional[torch.Tensor] = None,
                                   stream=None) -> torch.Tensor:
    """Decode attention for callers that cannot allocate: the split-K scratch
    is a fixed array inside the library (see include/kvarn.h)."""
    dev = _decode_args(cfg, q, pool, block_table, seq_lens, tail_k, tail_v, out, status)
    if softmax_scale is None:
        softmax_scale = HEAD_DIM ** -0.5
    with _on(dev):
        _check(lib().kvarn_decode_attention_noalloc(
            ctypes.byref(cfg), _ptr(q), _ptr(pool), pool.shape[0], _ptr(block_table),
            block_table.shape[-1], _ptr(seq_lens), q.shape[0], int(max_seq), _ptr(tail_k),
            _ptr(tail_v), float(softmax_scale), _ptr(out), _ptr(status), _stream(stream, dev)),
            "kvarn_decode_attention_noalloc")
    return out


def kvarn_dequantize_pages(records: torch.Tensor, stream=None):
    """records: uint8 [n][15360] (contiguous) -> (yk, yv) float32 [n][128][128]."""
    dev = _arg(records, "records", torch.uint8, (None, PAGE_BYTES))
    n = records.shape[0]
    yk = torch.empty((n, BLOCK_TOKENS, HEAD_DIM), dtype=torch.float32, device=dev)
    yv = torch.empty_like(yk)
    with _on(dev):
        _check(lib().kvarn_dequantize_pages(_ptr(records), n, _ptr(yk), _ptr(yv),
                                            _stream(stream, dev)), "kvarn_dequantize_pages")
    return yk, yv


def kvarn_dequantize_records(cfg: Config, records: torch.Tensor, stream=None):
    """records: uint8 [n][cfg.page_bytes] (contiguous) -> (yk, yv) float32
    [n][128][128], for any record format."""
    dev = _arg(records, "records", torch.uint8, (None, cfg.page_bytes))
    n = records.shape[0]
    yk = torch.empty((n, BLOCK_TOKENS, HEAD_DIM), dtype=torch.float32, device=dev)
    yv = torch.empty_like(yk)
    with _on(dev):
        _check(lib().kvarn_dequantize_records(ctypes.byref(cfg), _ptr(records), n, _ptr(yk),
                                              _ptr(yv), _stream(stream, dev)),
               "kvarn_dequantize_records")
    return yk, yv


# ------------------------------------------- the FP16 cache (the baseline) --

def alloc_fp16_pool(num_kv_heads: int, num_pages: int, device="cuda") -> torch.Tensor:
    """uint8 [num_pages][Hkv][65536]: K then V, [128 tokens][128] fp16 each."""
    return torch.zeros((num_pages, num_kv_heads, FP16_PAGE_BYTES), dtype=torch.uint8,
                       device=device)


def kvarn_fp16_write_blocks(k: torch.Tensor, v: torch.Tensor, seq_lens: torch.Tensor,
                            max_seq: int, block_table: torch.Tensor, pool: torch.Tensor,
                            status: Optional[torch.Tensor] = None, stream=None) -> None:
    """k, v: fp16 [B][S][Hkv][128] (any strides with a dense last dim); pool
    from alloc_fp16_pool with the same Hkv."""
    dev = _kv_pair(k, v, None)
    B, hkv = k.shape[0], k.shape[2]
    _lens_table(dev, B, seq_lens, "seq_lens", block_table)
    _arg(pool, "pool", torch.uint8, (None, hkv, FP16_PAGE_BYTES), device=dev)
    _status(dev, status)
    with _on(dev):
        _check(lib().kvarn_fp16_write_blocks(
            _ptr(k), _ptr(v), k.stride(0), k.stride(1), k.stride(2), B, hkv, _ptr(seq_lens),
            int(max_seq), _ptr(block_table), block_table.shape[-1], _ptr(pool), pool.shape[0],
            _ptr(status), _stream(stream, dev)), "kvarn_fp16_write_blocks")


def fp16_decode_workspace_bytes(num_q_heads: int, num_kv_heads: int, batch: int,
                                max_seq: int) -> int:
    return lib().kvarn_fp16_decode_workspace_bytes(num_q_heads, num_kv_heads, batch, max_seq)


def alloc_fp16_decode_workspace(num_q_heads: int, num_kv_heads: int, batch: int, max_seq: int,
                                device="cuda") -> torch.Tensor:
    n = fp16_decode_workspace_bytes(num_q_heads, num_kv_heads, batch, max_seq)
    return torch.zeros((max(n, 16),), dtype=torch.uint8, device=device)


def kvarn_fp16_decode_attention(q: torch.Tensor, num_kv_heads: int, pool: torch.Tensor,
                                block_table: torch.Tensor, seq_lens: torch.Tensor, max_seq: int,
                                out: torch.Tensor, workspace: Optional[torch.Tensor],
                                softmax_scale: float = None,
                                status: Optional[torch.Tensor] = None,
                                stream=None) -> torch.Tensor:
    """q, out: fp16 [B][Hq][128]; pool from alloc_fp16_pool."""
    dev = _arg(q, "q", torch.float16, (None, None, HEAD_DIM))
    _arg(out, "out", torch.float16, tuple(q.shape), device=dev)
    B = q.shape[0]
    _lens_table(dev, B, seq_lens, "seq_lens", block_table)
    _arg(pool, "pool", torch.uint8, (None, int(num_kv_heads), FP16_PAGE_BYTES), device=dev)
    _status(dev, status)
    if workspace is not None:
        _arg(workspace, "workspace", None, device=dev)
    if softmax_scale is None:
        softmax_scale = HEAD_DIM ** -0.5
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with _on(dev):
        _check(lib().kvarn_fp16_decode_attention(
            _ptr(q), q.shape[1], int(num_kv_heads), _ptr(pool), pool.shape[0], _ptr(block_table),
            block_table.shape[-1], _ptr(seq_lens), B, int(max_seq), float(softmax_scale),
            _ptr(out), _ptr(workspace), ws_bytes, _ptr(status), _stream(stream, dev)),
            "kvarn_fp16_decode_attention")
    return out


# ------------------------------------------------------------ FP8 cache --

def alloc_fp8_pool(num_kv_heads: int, num_pages: int, device="cuda") -> torch.Tensor:
    return torch.zeros((num_pages, num_kv_heads, FP8_PAGE_BYTES), dtype=torch.uint8,
                       device=device)


def kvarn_fp8_write_blocks(k: torch.Tensor, v: torch.Tensor, seq_lens: torch.Tensor,
                           max_seq: int, block_table: torch.Tensor, pool: torch.Tensor,
                           status: Optional[torch.Tensor] = None, stream=None) -> None:
    """k, v fp16 [B][S][Hkv][128] -> fp8 pool uint8 [num_pages][Hkv][33792]."""
    hkv = k.shape[2]
    dev = _kv_pair(k, v, hkv)
    B = k.shape[0]
    _lens_table(dev, B, seq_lens, "seq_lens", block_table)
    _arg(pool, "pool", torch.uint8, (None, hkv, FP8_PAGE_BYTES), device=dev)
    _status(dev, status)
    with _on(dev):
        _check(lib().kvarn_fp8_write_blocks(
            _ptr(k), _ptr(v), k.stride(0), k.stride(1), k.stride(2), B, hkv, _ptr(seq_lens),
            int(max_seq), _ptr(block_table), block_table.shape[-1], _ptr(pool), pool.shape[0],
            _ptr(status), _stream(stream, dev)), "kvarn_fp8_write_blocks")


def fp8_decode_workspace_bytes(num_q_heads: int, num_kv_heads: int, batch: int,
                               max_seq: int) -> int:
    return lib().kvarn_fp8_decode_workspace_bytes(num_q_heads, num_kv_heads, batch, max_seq)


def alloc_fp8_decode_workspace(num_q_heads: int, num_kv_heads: int, batch: int, max_seq: int,
                               device="cuda") -> Optional[torch.Tensor]:
    n = fp8_decode_workspace_bytes(num_q_heads, num_kv_heads, batch, max_seq)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device) if n else None


def kvarn_fp8_decode_attention(q: torch.Tensor, num_kv_heads: int, pool: torch.Tensor,
                               block_table: torch.Tensor, seq_lens: torch.Tensor, max_seq: int,
                               out: torch.Tensor, workspace: Optional[torch.Tensor],
                               softmax_scale: float = None,
                               status: Optional[torch.Tensor] = None, stream=None):
    """q, out fp16 [B][Hq][128] over the fp8 pages."""
    hq = q.shape[1]
    dev = _arg(q, "q", torch.float16, (None, hq, HEAD_DIM))
    _arg(out, "out", torch.float16, tuple(q.shape), device=dev)
    B = q.shape[0]
    _lens_table(dev, B, seq_lens, "seq_lens", block_table)
    _arg(pool, "pool", torch.uint8, (None, num_kv_heads, FP8_PAGE_BYTES), device=dev)
    _status(dev, status)
    if workspace is not None:
        _arg(workspace, "workspace", None, device=dev)
    if softmax_scale is None:
        softmax_scale = HEAD_DIM ** -0.5
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with _on(dev):
        _check(lib().kvarn_fp8_decode_attention(
            _ptr(q), hq, num_kv_heads, _ptr(pool), pool.shape[0], _ptr(block_table),
            block_table.shape[-1], _ptr(seq_lens), B, int(max_seq), float(softmax_scale),
            _ptr(out), _ptr(workspace), ws_bytes, _ptr(status), _stream(stream, dev)),
            "kvarn_fp8_decode_attention")
    return out


# ------------------------------------------------- SnapKV-style selection --

def snapkv_workspace_bytes(cfg: Config, batch: int, window: int, max_seq: int) -> int:
    return lib().kvarn_snapkv_workspace_bytes(ctypes.byref(cfg), batch, window, max_seq)


def kvarn_snapkv_select(cfg: Config, q_window: torch.Tensor, k: torch.Tensor,
                        seq_lens: torch.Tensor, max_seq: int, capacity: int,
                        votes: torch.Tensor, indices: torch.Tensor, workspace: torch.Tensor,
                        pool_kernel: int = 7, softmax_scale: float = None,
                        status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """q_window fp16 [B][W][Hq][128]; k fp16 [B][S][Hkv][128] (dense last dim);
    votes float32 [B][Hkv][max_seq]; indices int32 [B][Hkv][capacity]."""
    dev = _arg(q_window, "q_window", torch.float16, (None, None, cfg.num_q_heads, HEAD_DIM))
    B, W = q_window.shape[0], q_window.shape[1]
    _arg(k, "k", torch.float16, (B, _AtLeast(max_seq), cfg.num_kv_heads, HEAD_DIM), device=dev,
         contiguous=False)
    if k.stride(3) != 1:
        raise ValueError("k must have a dense last dimension")
    _arg(seq_lens, "seq_lens", torch.int32, (_AtLeast(B),), device=dev)
    _arg(votes, "votes", torch.float32, (B, cfg.num_kv_heads, max_seq), device=dev)
    _arg(indices, "indices", torch.int32, (B, cfg.num_kv_heads, capacity), device=dev)
    _arg(workspace, "workspace", None, device=dev)
    _status(dev, status)
    if softmax_scale is None:
        softmax_scale = HEAD_DIM ** -0.5
    ws_bytes = workspace.numel() * workspace.element_size()
    with _on(dev):
        _check(lib().kvarn_snapkv_select(
            ctypes.byref(cfg), _ptr(q_window), W, _ptr(k), k.stride(0), k.stride(1), k.stride(2),
            _ptr(seq_lens), B, int(max_seq), int(capacity), int(pool_kernel),
            float(softmax_scale), _ptr(votes), _ptr(indices), _ptr(workspace), ws_bytes,
            _ptr(status), _stream(stream, dev)), "kvarn_snapkv_select")
    return indices


def kvarn_snapkv_gather(k: torch.Tensor, v: torch.Tensor, indices: torch.Tensor,
                        k_out: torch.Tensor, v_out: torch.Tensor, stream=None) -> None:
    """k, v fp16 [B][S][Hkv][128]; indices int32 [B][Hkv][C]; k_out, v_out
    fp16 [B][C][Hkv][128]."""
    hkv = k.shape[2]
    dev = _kv_pair(k, v, hkv)
    B = k.shape[0]
    C = indices.shape[-1]
    _arg(indices, "indices", torch.int32, (B, hkv, C), device=dev)
    _arg(k_out, "k_out", torch.float16, (B, C, hkv, HEAD_DIM), device=dev)
    _arg(v_out, "v_out", torch.float16, (B, C, hkv, HEAD_DIM), device=dev)
    with _on(dev):
        _check(lib().kvarn_snapkv_gather(
            _ptr(k), _ptr(v), k.stride(0), k.stride(1), k.stride(2), B, k.shape[1], hkv,
            _ptr(indices), C,
            _ptr(k_out), _ptr(v_out), _stream(stream, dev)), "kvarn_snapkv_gather")
