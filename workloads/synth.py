"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds no arithmetic of the method: it only draws random K, V and
query tensors with the shapes and value distributions of the workloads, and
builds block tables and sequence lengths.  Both the product side and the
oracle side read these tensors; neither side's code lives here.

Distributions (the pages print no data, so these are the stated synthetic
stand-ins for long-context LLM KV caches):
  * K = N(0,1) * s_c per channel, where s_c = exp(sigma_k * N(0,1)) is drawn
    once per (layer, KV head, channel), and `n_outliers` channels of each
    (layer, KV head) are multiplied by an outlier factor;
  * V = N(0,1), optionally times a per-(token, head) log-normal scale
    exp(sigma_v * N(0,1));
  * queries N(0,1).
Everything is drawn in fp32 and rounded to fp16.

Shapes (WORKLOADS below), each after a setting the pages name:
  * long sequences, because the KVarN page (blog.edumints.com) presents the
    method for agents and long contexts (its feature list);
  * GQA with several query heads per KV head ("KV Cache (Anahtar-Deger
    Onbellegi)", yapayzekasozluk.tr, "Sik Sorulan Sorular");
  * the Qwen2.5-1.5B KV geometry, 28 layers x 2 KV heads x 128, as in the KVTC
    page's per-token KV example (trimsalonaandekust.nl);
  * requests of mixed lengths on scattered pages, the case paged attention
    serves (same glossary, "Paged Attention (vLLM)").
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

D = 128          # head_dim
T = 128          # tokens per block / page


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    layers: int
    hkv: int
    hq: int
    batch: int
    seq: int                      # tokens per sequence (max, for mixed lengths)
    sigma_k: float                # per-channel log-normal sigma of K
    n_outliers: int
    outlier_lo: float
    outlier_hi: float
    sigma_v: float                # per-(token, head) log-normal sigma of V (0: none)
    table: str                    # "identity", "perm" or "shared_perm"
    seed: int
    min_seq: Optional[int] = None  # mixed lengths: uniform in [min_seq, seq]
    decode_steps: int = 1
    reserve_tokens: int = 0       # extra room per sequence for appended tokens

    @property
    def g(self) -> int:
        return self.hq // self.hkv


WORKLOADS = {
    # 1 layer, 1 KV head, 1 query head, 4 blocks of 128 tokens; seed 0.
    "tiny": Workload("tiny", 1, 1, 1, 1, 512, 0.5, 2, 20.0, 20.0, 0.0, "identity", 0),
    # Llama-3-8B-like layer: 8 KV heads, 32 query heads, batch 16 x 4096.
    "llama3_8b_layer": Workload("llama3_8b_layer", 1, 8, 32, 16, 4096, 1.0, 4, 10.0, 30.0,
                                0.5, "identity", 2),
    # Long context: batch 1 x 131072, pages a random permutation of 1024.
    "long_context": Workload("long_context", 1, 8, 32, 1, 131072, 1.0, 4, 10.0, 30.0, 0.5,
                             "perm", 3),
    # Qwen2.5-1.5B-like KV shape: 28 layers, 2 KV heads, 12 query heads, 64 x 8192.
    "qwen25_15b": Workload("qwen25_15b", 28, 2, 12, 64, 8192, 1.0, 4, 10.0, 30.0, 0.5,
                           "shared_perm", 4),
    # Mixed serving: 128 requests, lengths uniform in [1024, 32768], 64 decode steps.
    "mixed_serving": Workload("mixed_serving", 1, 8, 32, 128, 32768, 1.0, 4, 10.0, 30.0, 0.5,
                              "perm", 5, min_seq=1024, decode_steps=64, reserve_tokens=64),
}


def scaled(w: Workload, **kw) -> Workload:
    """Same distributions, other sizes (for parity runs the oracle can finish)."""
    return dataclasses.replace(w, **kw)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def seq_lens(w: Workload, device="cpu") -> torch.Tensor:
    """int32 [B]: every sequence at w.seq, or uniform in [min_seq, seq]."""
    if w.min_seq is None:
        return torch.full((w.batch,), w.seq, dtype=torch.int32, device=device)
    g = _gen(w.seed * 1000 + 999, "cpu")
    lens = torch.randint(w.min_seq, w.seq + 1, (w.batch,), generator=g, dtype=torch.int64)
    return lens.to(torch.int32).to(device)


def max_blocks(w: Workload) -> int:
    return (w.seq + w.reserve_tokens + T - 1) // T


def block_tables(w: Workload, device="cpu"):
    """Returns (tables, num_pages).  tables: int32 [layers][B][max_blocks].
    Unused entries are -1.  identity: sequence b, block j -> page b*max_blocks + j.
    perm: every (b, j) gets a distinct page of a random permutation of the pages
    one layer needs.  shared_perm: one pool for all layers; each layer's table
    is a slice of one random permutation of the whole pool."""
    mb = max_blocks(w)
    lens = seq_lens(w).to(torch.int64)
    need = ((lens + w.reserve_tokens + T - 1) // T).clamp(max=mb)
    tables = torch.full((w.layers, w.batch, mb), -1, dtype=torch.int32)
    g = _gen(w.seed * 1000 + 777, "cpu")
    if w.table == "identity":
        num_pages = w.batch * mb
        for b in range(w.batch):
            n = int(need[b])
            tables[:, b, :n] = torch.arange(b * mb, b * mb + n, dtype=torch.int32)
    elif w.table == "perm":
        per_layer = int(need.sum())
        num_pages = per_layer * w.layers
        for layer in range(w.layers):
            perm = torch.randperm(per_layer, generator=g).to(torch.int32) + layer * per_layer
            off = 0
            for b in range(w.batch):
                n = int(need[b])
                tables[layer, b, :n] = perm[off:off + n]
                off += n
    elif w.table == "shared_perm":
        per_layer = int(need.sum())
        num_pages = per_layer * w.layers
        perm = torch.randperm(num_pages, generator=g).to(torch.int32)
        off = 0
        for layer in range(w.layers):
            for b in range(w.batch):
                n = int(need[b])
                tables[layer, b, :n] = perm[off:off + n]
                off += n
    else:
        raise ValueError(w.table)
    return tables.to(device), num_pages


def kv(w: Workload, layer: int = 0, device="cpu", seq: Optional[int] = None):
    """fp16 K, V [B][S][Hkv][128] for one layer (S = seq or w.seq)."""
    S = w.seq if seq is None else seq
    dev = torch.device(device)
    g = _gen(w.seed * 1000 + layer, dev)
    B, H = w.batch, w.hkv
    # per-(KV head, channel) log-normal scale and outlier channels of K
    ch_scale = torch.exp(w.sigma_k * torch.randn((H, D), generator=g, device=dev))
    for h in range(H):
        if w.n_outliers:
            idx = torch.randperm(D, generator=g, device=dev)[:w.n_outliers]
            fac = w.outlier_lo + (w.outlier_hi - w.outlier_lo) * torch.rand(
                (w.n_outliers,), generator=g, device=dev)
            ch_scale[h, idx] *= fac
    k = torch.randn((B, S, H, D), generator=g, device=dev)
    k.mul_(ch_scale)
    v = torch.randn((B, S, H, D), generator=g, device=dev)
    if w.sigma_v > 0:
        v.mul_(torch.exp(w.sigma_v * torch.randn((B, S, H, 1), generator=g, device=dev)))
    return k.to(torch.float16), v.to(torch.float16)


def new_tokens(w: Workload, step: int, layer: int = 0, device="cpu"):
    """fp16 k_new, v_new [B][Hkv][128] for decode step `step` (same distributions:
    the K channel scales are the layer's own)."""
    dev = torch.device(device)
    g = _gen(w.seed * 1000 + layer, dev)
    H = w.hkv
    ch_scale = torch.exp(w.sigma_k * torch.randn((H, D), generator=g, device=dev))
    for h in range(H):
        if w.n_outliers:
            idx = torch.randperm(D, generator=g, device=dev)[:w.n_outliers]
            fac = w.outlier_lo + (w.outlier_hi - w.outlier_lo) * torch.rand(
                (w.n_outliers,), generator=g, device=dev)
            ch_scale[h, idx] *= fac
    g2 = _gen(w.seed * 100003 + layer * 1009 + step + 1, dev)
    k = torch.randn((w.batch, H, D), generator=g2, device=dev) * ch_scale
    v = torch.randn((w.batch, H, D), generator=g2, device=dev)
    if w.sigma_v > 0:
        v.mul_(torch.exp(w.sigma_v * torch.randn((w.batch, H, 1), generator=g2, device=dev)))
    return k.to(torch.float16), v.to(torch.float16)


def queries(w: Workload, step: int = 0, layer: int = 0, device="cpu"):
    """fp16 q [B][Hq][128], N(0,1)."""
    dev = torch.device(device)
    g = _gen(w.seed * 7919 + layer * 131 + step + 17, dev)
    return torch.randn((w.batch, w.hq, D), generator=g, device=dev).to(torch.float16)


def nbytes_fp16_kv(w: Workload) -> int:
    """fp16 K+V bytes of one layer at full length: 2 x B x S x Hkv x 128 x 2."""
    return 2 * w.batch * w.seq * w.hkv * D * 2


def describe(w: Workload) -> str:
    return (f"{w.name}: layers={w.layers} B={w.batch} S={w.seq} Hkv={w.hkv} Hq={w.hq} "
            f"g={w.g} table={w.table} seed={w.seed}")


__all__ = ["Workload", "WORKLOADS", "scaled", "seq_lens", "block_tables", "kv", "new_tokens",
           "queries", "max_blocks", "nbytes_fp16_kv", "describe", "D", "T"]

