"""Small drivers of the CUDA path (through the Python binding of the C ABI)."""
from __future__ import annotations

import numpy as np
import torch

import quantized_decode_attention_blocks_b300 as kv

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


def config(hq, hkv, iters=None, rms=False, m16=False, pc=False, g64=False, v4=False,
           k8=False):
    fmt = (("k4v2_g64" if g64 else "k8v4_g128" if k8 else "k4v4_g128" if v4 else "k4v2_g128")
           + ("_rms" if rms else "")
           + ("_m16" if m16 else "") + ("_pc" if pc else "")
           + ("" if iters is None else f"_s{iters}"))
    return kv.config_from_string(fmt, hq, hkv)


def prefill(cfg, k, v, lens, table, num_pages, max_seq=None):
    """k, v on the GPU [B][S][Hkv][128]; lens, table (cpu or gpu int32)."""
    B = k.shape[0]
    max_seq = int(lens.max()) if max_seq is None else max_seq
    pool = kv.alloc_pool(cfg, num_pages, DEV)
    tk, tv = kv.alloc_tails(cfg, B, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kv.kvarn_quantize_blocks(cfg, k, v, lens.to(DEV), max_seq, table.to(DEV), pool, tk, tv,
                             status)
    return pool, tk, tv, status


def decode(cfg, q, pool, table, lens, tk, tv, max_seq=None, status=None):
    B = q.shape[0]
    max_seq = int(lens.max()) if max_seq is None else max_seq
    out = torch.full((B, cfg.num_q_heads, 128), float("nan"), dtype=torch.float16, device=DEV)
    ws = kv.alloc_decode_workspace(cfg, B, max_seq, DEV)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kv.kvarn_decode_attention(cfg, q.to(DEV), pool, table.to(DEV), lens.to(DEV), max_seq, tk, tv,
                              out, ws, status=status)
    return out, status, ws


def host(t):
    return t.detach().cpu().numpy()


def bits16(t):
    return host(t).view(np.uint16)
