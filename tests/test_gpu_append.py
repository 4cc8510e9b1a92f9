"""Decode-time append on the GPU: tail writes and the in-launch quantization of
a filled block ("KV Cache Nasil Calisir?": only the new token's K,V are added)."""
import numpy as np
import pytest
import torch

import quantized_decode_attention_blocks_b300 as kv
from oracle import kvref
from tests import parity
from tests.gpu_helpers import DEV, bits16, config, host, prefill
from workloads import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("m16,pc,g64,v4,k8", [(False, False, False, False, False),
                                              (True, False, False, False, False),
                                              (False, True, False, False, False),
                                              (False, False, True, False, False),
                                              (False, False, False, True, False),
                                              (False, False, False, False, True)])
def test_append_fills_pages_like_prefill(m16, pc, g64, v4, k8):
    # m16: format variant "_m16" (fp16 metadata, 13824-byte records); pc:
    # format variant "_pc" (per-channel groups)
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=3, seq=384, hkv=2, hq=8)
    k, v = synth.kv(w, device=DEV)
    cfg = config(w.hq, w.hkv, m16=m16, pc=pc, g64=g64, v4=v4, k8=k8)
    table = torch.arange(9, dtype=torch.int32).reshape(3, 3)
    lens = torch.tensor([384, 384, 384], dtype=torch.int32)
    ref_pool, _, _, _ = prefill(cfg, k, v, lens, table, 9)
    pool = kv.alloc_pool(cfg, 9, DEV)
    tk, tv = kv.alloc_tails(cfg, 3, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    tdev = table.to(DEV)
    for p in range(384):
        pos = torch.full((3,), p, dtype=torch.int32, device=DEV)
        pos[1] = p if p < 200 else -1          # sequence 1 goes idle after 200 tokens
        kv.kvarn_append_token(cfg, k[:, p].contiguous(), v[:, p].contiguous(), pos, tdev, pool,
                              tk, tv, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # bit-exact against the prefill kernel for every filled page
    assert torch.equal(pool[[0, 1, 2, 6, 7, 8]], ref_pool[[0, 1, 2, 6, 7, 8]])
    assert torch.equal(pool[3], ref_pool[3])
    assert not pool[4:6].any()
    # sequence 1 stopped at 200 tokens: 72 in the tail
    assert torch.equal(tk[1, :, :72], k[1, 128:200].transpose(0, 1))
    # and against the oracle (boundary rule)
    ref = kvref.quantize_blocks(host(k), host(v), host(lens), host(table), 9, 2, want_u=True,
                                meta16=m16, pc=pc, g64=g64, v4=v4, k8=k8)
    ref32 = kvref.quantize_blocks(host(k), host(v), host(lens), host(table), 9, 2) if m16 else None
    stats = {}
    for b in (0, 2):
        for j in range(3):
            for h in range(2):
                page = table[b, j]
                parity.compare_record(host(pool)[page, h], ref["pool"][page, h],
                                      ref["u_k"][b, j, h], ref["u_v"][b, j, h], stats,
                                      meta16=m16,
                                      ref32=ref32["pool"][page, h] if m16 else None, pc=pc,
                                      g64=g64, v4=v4, k8=k8)
    parity.check_flip_rate(stats)


def test_append_reports_missing_page():
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=1, seq=128, hkv=1, hq=1)
    cfg = config(1, 1)
    pool = kv.alloc_pool(cfg, 2, DEV)
    tk, tv = kv.alloc_tails(cfg, 1, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    table = torch.tensor([[7, 1]], dtype=torch.int32, device=DEV)   # 7 outside a 2-page pool
    kn = torch.ones((1, 1, 128), dtype=torch.float16, device=DEV)
    kv.kvarn_append_token(cfg, kn, kn, torch.tensor([127], dtype=torch.int32, device=DEV), table,
                          pool, tk, tv, status)
    torch.cuda.synchronize()
    assert int(status.item()) & kv.kvarn.STATUS_BAD_PAGE
    assert not pool.any()
