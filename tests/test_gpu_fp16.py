"""The FP16 paged cache (the baseline the quantized cache is measured against)
on the GPU, against the float64 oracle's plain attention over the same fp16
keys and values.

Attention: "KV Cache (Anahtar-Deger Onbellegi)" (yapayzekasozluk.tr), "KV Cache
Nasil Calisir?" and "Paged Attention (vLLM)".  The KVarN page
(blog.edumints.com) states its gains relative to such an FP16 cache.
"""
import numpy as np
import pytest
import torch

import quantized_decode_attention_blocks_b300 as kv
from oracle import kvref
from tests import parity
from tests.gpu_helpers import DEV, host
from workloads import synth

pytestmark = pytest.mark.gpu


def _run(w, lens, table, num_pages, max_seq=None, seqs=None):
    max_seq = int(lens.max()) if max_seq is None else max_seq
    S = max(int(lens.max()), 1)
    k, v = synth.kv(w, device=DEV, seq=S)
    pool = kv.alloc_fp16_pool(w.hkv, num_pages, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kv.kvarn_fp16_write_blocks(k, v, lens.to(DEV), max_seq, table.to(DEV), pool, st)
    q = synth.queries(w).to(DEV)
    out = torch.full((q.shape[0], w.hq, 128), float("nan"), dtype=torch.float16, device=DEV)
    ws = kv.alloc_fp16_decode_workspace(w.hq, w.hkv, q.shape[0], max_seq, DEV)
    kv.kvarn_fp16_decode_attention(q, w.hkv, pool, table.to(DEV), lens.to(DEV), max_seq, out,
                                   ws, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, kv.status_string(int(st.item()))
    sel = list(range(q.shape[0])) if seqs is None else seqs
    ref = kvref.attention_fp16(host(q[sel]), host(k[sel]), host(v[sel]), host(lens)[sel], w.hq,
                               w.hkv)
    parity.compare_attention(host(out[sel]), ref)
    return q, pool, out, ws, st, max_seq


@pytest.mark.parametrize("hq,hkv", [(1, 1), (8, 2), (12, 2), (8, 1), (32, 8)])
def test_group_sizes_and_ragged_lengths(hq, hkv):
    lens = torch.tensor([0, 1, 63, 64, 65, 127, 128, 129, 300, 1000, 2048], dtype=torch.int32)
    B = len(lens)
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=B, seq=2048, hkv=hkv, hq=hq)
    mb = 16
    g = torch.Generator().manual_seed(21)
    table = torch.randperm(B * mb, generator=g).to(torch.int32).reshape(B, mb)
    _run(w, lens, table, B * mb)


def test_many_splits_long_sequence_and_second_call():
    # one sequence of 20000 tokens: many splits merged through the workspace,
    # whose tickets are left at zero for the next call
    w = synth.scaled(synth.WORKLOADS["long_context"], batch=1, seq=20000, hkv=2, hq=8)
    lens = torch.tensor([20000], dtype=torch.int32)
    g = torch.Generator().manual_seed(22)
    table = torch.randperm(157, generator=g).to(torch.int32).reshape(1, 157)
    q, pool, out, ws, st, max_seq = _run(w, lens, table, 157)
    out2 = torch.empty_like(out)
    kv.kvarn_fp16_decode_attention(q, w.hkv, pool, table.to(DEV), lens.to(DEV), max_seq, out2,
                                   ws, status=st)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)


def test_llama_like_layer_full_size_sampled():
    w = synth.WORKLOADS["llama3_8b_layer"]
    lens = synth.seq_lens(w)
    tables, n = synth.block_tables(w)
    _run(w, lens, tables[0].contiguous(), n, seqs=[0, 7, 15])


def test_bad_page_reported():
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=1, seq=512, hkv=2, hq=8)
    k, v = synth.kv(w, device=DEV)
    lens = torch.tensor([512], dtype=torch.int32, device=DEV)
    pool = kv.alloc_fp16_pool(w.hkv, 4, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    good = torch.tensor([[0, 1, 2, 3]], dtype=torch.int32, device=DEV)
    kv.kvarn_fp16_write_blocks(k, v, lens, 512, good, pool, st)
    bad = torch.tensor([[0, 1, -5, 3]], dtype=torch.int32, device=DEV)
    q = synth.queries(w).to(DEV)
    out = torch.empty((1, w.hq, 128), dtype=torch.float16, device=DEV)
    ws = kv.alloc_fp16_decode_workspace(w.hq, w.hkv, 1, 512, DEV)
    kv.kvarn_fp16_decode_attention(q, w.hkv, pool, bad, lens, 512, out, ws, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & kv.kvarn.STATUS_BAD_PAGE
    assert torch.isfinite(out.float()).all()
