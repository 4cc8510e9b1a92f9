"""Thin ctypes binding of libkvarn (include/kvarn.h).

Argument marshalling only: every step of quantization and decode attention
runs in the CUDA kernels of libkvarn.so.  torch supplies device memory and the
current stream.  If the library is missing the import fails loudly; there is
no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkvarn.so")

HEAD_DIM = 128
BLOCK_TOKENS = 128
PAGE_BYTES = 15360
FP16_PAGE_BYTES = 65536            # KVARN_FP16_PAGE_BYTES
NOALLOC_SCRATCH_BYTES = 4 << 20   # KVARN_NOALLOC_SCRATCH_BYTES

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
                ("num_kv_heads", ctypes.c_int)]

    @property
    def g(self) -> int:
        return self.num_q_heads // self.num_kv_heads


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
    "kvarn_decode_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(Config), _I, _I]),
    "kvarn_decode_attention": (_I, [ctypes.POINTER(Config), _P, _P, _L, _P, _I, _P, _I, _I, _P,
                                    _P, ctypes.c_float, _P, _P, ctypes.c_size_t, _P, _P]),
    "kvarn_decode_attention_noalloc": (_I, [ctypes.POINTER(Config), _P, _P, _L, _P, _I, _P, _I,
                                            _I, _P, _P, ctypes.c_float, _P, _P, _P]),
    "kvarn_dequantize_pages": (_I, [_P, _L, _P, _P, _P]),
    "kvarn_fp16_write_blocks": (_I, [_P, _P, _L, _L, _L, _I, _I, _P, _I, _P, _I, _P, _L, _P,
                                     _P]),
    "kvarn_fp16_decode_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I]),
    "kvarn_fp16_decode_attention": (_I, [_P, _I, _I, _P, _L, _P, _I, _P, _I, _I,
                                         ctypes.c_float, _P, _P, ctypes.c_size_t, _P, _P]),
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


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


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
    return torch.zeros((num_pages, cfg.num_kv_heads, PAGE_BYTES), dtype=torch.uint8,
                       device=device)


def alloc_tails(cfg: Config, batch: int, device="cuda"):
    shape = (batch, cfg.num_kv_heads, BLOCK_TOKENS, HEAD_DIM)
    return (torch.zeros(shape, dtype=torch.float16, device=device),
            torch.zeros(shape, dtype=torch.float16, device=device))


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
    """k, v: fp16 [B][S][Hkv][128] (any strides with a dense last dim)."""
    _dev(k, torch.float16, "k")
    _dev(v, torch.float16, "v")
    if k.shape != v.shape or k.stride() != v.stride() or k.dim() != 4 or k.stride(3) != 1:
        raise ValueError("k and v must share shape/strides [B][S][Hkv][128], last dim dense")
    B = k.shape[0]
    _check(lib().kvarn_quantize_blocks(
        ctypes.byref(cfg), _ptr(k), _ptr(v), k.stride(0), k.stride(1), k.stride(2), B,
        _ptr(seq_lens), int(max_seq), _ptr(block_table), block_table.shape[-1], _ptr(pool),
        pool.shape[0], _ptr(tail_k), _ptr(tail_v), _ptr(status), _stream(stream)),
        "kvarn_quantize_blocks")


def kvarn_append_token(cfg: Config, k_new: torch.Tensor, v_new: torch.Tensor, pos: torch.Tensor,
                       block_table: torch.Tensor, pool: torch.Tensor, tail_k: torch.Tensor,
                       tail_v: torch.Tensor, status: Optional[torch.Tensor] = None,
                       stream=None) -> None:
    """k_new, v_new: fp16 [B][Hkv][128]; pos: int32 [B] length before the append."""
    _dev(k_new, torch.float16, "k_new")
    _dev(v_new, torch.float16, "v_new")
    _check(lib().kvarn_append_token(
        ctypes.byref(cfg), _ptr(k_new), _ptr(v_new), _ptr(pos), k_new.shape[0],
        _ptr(block_table), block_table.shape[-1], _ptr(pool), pool.shape[0], _ptr(tail_k),
        _ptr(tail_v), _ptr(status), _stream(stream)), "kvarn_append_token")


def kvarn_decode_attention(cfg: Config, q: torch.Tensor, pool: torch.Tensor,
                           block_table: torch.Tensor, seq_lens: torch.Tensor, max_seq: int,
                           tail_k: torch.Tensor, tail_v: torch.Tensor, out: torch.Tensor,
                           workspace: Optional[torch.Tensor], softmax_scale: float = None,
                           status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """q, out: fp16 [B][Hq][128]."""
    _dev(q, torch.float16, "q")
    _dev(out, torch.float16, "out")
    if softmax_scale is None:
        softmax_scale = HEAD_DIM ** -0.5
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().kvarn_decode_attention(
        ctypes.byref(cfg), _ptr(q), _ptr(pool), pool.shape[0], _ptr(block_table),
        block_table.shape[-1], _ptr(seq_lens), q.shape[0], int(max_seq), _ptr(tail_k),
        _ptr(tail_v), float(softmax_scale), _ptr(out), _ptr(workspace), ws_bytes, _ptr(status),
        _stream(stream)), "kvarn_decode_attention")
    return out


def kvarn_decode_attention_noalloc(cfg: Config, q: torch.Tensor, pool: torch.Tensor,
                                   block_table: torch.Tensor, seq_lens: torch.Tensor,
                                   max_seq: int, tail_k: torch.Tensor, tail_v: torch.Tensor,
                                   out: torch.Tensor, softmax_scale: float = None,
                                   status: Optional[torch.Tensor] = None,
                                   stream=None) -> torch.Tensor:
    """Decode attention for callers that cannot allocate: the split-K scratch
    is a fixed array inside the library (see include/kvarn.h)."""
    _dev(q, torch.float16, "q")
    _dev(out, torch.float16, "out")
    if softmax_scale is None:
        softmax_scale = HEAD_DIM ** -0.5
    _check(lib().kvarn_decode_attention_noalloc(
        ctypes.byref(cfg), _ptr(q), _ptr(pool), pool.shape[0], _ptr(block_table),
        block_table.shape[-1], _ptr(seq_lens), q.shape[0], int(max_seq), _ptr(tail_k),
        _ptr(tail_v), float(softmax_scale), _ptr(out), _ptr(status), _stream(stream)),
        "kvarn_decode_attention_noalloc")
    return out


def kvarn_dequantize_pages(records: torch.Tensor, stream=None):
    """records: uint8 [n][15360] (contiguous) -> (yk, yv) float32 [n][128][128]."""
    n = records.shape[0]
    yk = torch.empty((n, BLOCK_TOKENS, HEAD_DIM), dtype=torch.float32, device=records.device)
    yv = torch.empty_like(yk)
    _check(lib().kvarn_dequantize_pages(_ptr(records), n, _ptr(yk), _ptr(yv), _stream(stream)),
           "kvarn_dequantize_pages")
    return yk, yv


# ------------------------------------------- the FP16 cache (the baseline) --

def alloc_fp16_pool(num_kv_heads: int, num_pages: int, device="cuda") -> torch.Tensor:
    """uint8 [num_pages][Hkv][65536]: K then V, [128 tokens][128] fp16 each."""
    return torch.zeros((num_pages, num_kv_heads, FP16_PAGE_BYTES), dtype=torch.uint8,
                       device=device)


def kvarn_fp16_write_blocks(k: torch.Tensor, v: torch.Tensor, seq_lens: torch.Tensor,
                            max_seq: int, block_table: torch.Tensor, pool: torch.Tensor,
                            status: Optional[torch.Tensor] = None, stream=None) -> None:
    """k, v: fp16 [B][S][Hkv][128] (any strides with a dense last dim)."""
    _dev(k, torch.float16, "k")
    _dev(v, torch.float16, "v")
    if k.shape != v.shape or k.stride() != v.stride() or k.dim() != 4 or k.stride(3) != 1:
        raise ValueError("k and v must share shape/strides [B][S][Hkv][128], last dim dense")
    _check(lib().kvarn_fp16_write_blocks(
        _ptr(k), _ptr(v), k.stride(0), k.stride(1), k.stride(2), k.shape[0], k.shape[2],
        _ptr(seq_lens), int(max_seq), _ptr(block_table), block_table.shape[-1], _ptr(pool),
        pool.shape[0], _ptr(status), _stream(stream)), "kvarn_fp16_write_blocks")


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
    _dev(q, torch.float16, "q")
    _dev(out, torch.float16, "out")
    if softmax_scale is None:
        softmax_scale = HEAD_DIM ** -0.5
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().kvarn_fp16_decode_attention(
        _ptr(q), q.shape[1], int(num_kv_heads), _ptr(pool), pool.shape[0], _ptr(block_table),
        block_table.shape[-1], _ptr(seq_lens), q.shape[0], int(max_seq), float(softmax_scale),
        _ptr(out), _ptr(workspace), ws_bytes, _ptr(status), _stream(stream)),
        "kvarn_fp16_decode_attention")
    return out
