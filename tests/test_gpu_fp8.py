"""The FP8 paged cache (the second baseline: the glossary's INT8/FP8 KV
quantization, "KV Cache (Anahtar-Deger Onbellegi)", yapayzekasozluk.tr, "Sik
Sorulan Sorular") on the GPU, against the float64 oracle.

Codes and scales are a decision taken in fp32 on both sides, so the written
pages are compared bit for bit; decode attention (fed the GPU's own pages)
within the attention tolerance.
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


def _write(w, k, v, lens, table, num_pages, max_seq):
    pool = kv.alloc_fp8_pool(w.hkv, num_pages, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kv.kvarn_fp8_write_blocks(k, v, lens.to(DEV), max_seq, table.to(DEV), pool, st)
    return pool, st


def _check_pages(pool, ref, table, lens):
    got = host(pool)
    for b in range(len(lens)):
        n = int(lens[b])
        for j in range((n + 127) // 128):
            p = int(table[b, j])
            m = min(128, n - 128 * j)
            for part in (0, 16384):
                assert np.array_equal(got[p, :, part:part + 128 * m],
                                      ref[p, :, part:part + 128 * m]), (b, j, part)
            for off in (32768, 33280):
                assert np.array_equal(got[p, :, off:off + 4 * m], ref[p, :, off:off + 4 * m])


def _run(w, lens, table, num_pages, max_seq=None, seqs=None, check_pages=True):
    max_seq = int(lens.max()) if max_seq is None else max_seq
    S = max(int(lens.max()), 1)
    k, v = synth.kv(w, device=DEV, seq=S)
    pool, st = _write(w, k, v, lens, table, num_pages, max_seq)
    q = synth.queries(w).to(DEV)
    out = torch.full((q.shape[0], w.hq, 128), float("nan"), dtype=torch.float16, device=DEV)
    ws = kv.alloc_fp8_decode_workspace(w.hq, w.hkv, q.shape[0], max_seq, DEV)
    kv.kvarn_fp8_decode_attention(q, w.hkv, pool, table.to(DEV), lens.to(DEV), max_seq, out,
                                  ws, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, kv.status_string(int(st.item()))
    if check_pages:
        ref_pool = kvref.fp8_write_blocks(host(k), host(v), host(lens), host(table), num_pages)
        _check_pages(pool, ref_pool, host(table), host(lens))
    sel = list(range(q.shape[0])) if seqs is None else seqs
    hp = host(pool)
    ref = kvref.fp8_decode_attention(host(q[sel]), hp, host(table)[sel], host(lens)[sel],
                                     w.hq, w.hkv)
    parity.compare_attention(host(out[sel]), ref)
    return q, pool, out, ws, st, max_seq


@pytest.mark.parametrize("hq,hkv", [(1, 1), (4, 2), (6, 2), (8, 2), (14, 2), (8, 1), (32, 8)])
def test_group_sizes_and_ragged_lengths(hq, hkv):
    lens = torch.tensor([0, 1, 63, 64, 65, 127, 128, 129, 300, 1000, 2048], dtype=torch.int32)
    B = len(lens)
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=B, seq=2048, hkv=hkv, hq=hq)
    mb = 16
    g = torch.Generator().manual_seed(31)
    table = torch.randperm(B * mb, generator=g).to(torch.int32).reshape(B, mb)
    _run(w, lens, table, B * mb)


def test_special_tokens_zero_and_outliers():
    # a zero token (scale 0, codes 0), one with a single huge channel and one
    # at the fp16 extremes
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=1, seq=256, hkv=2, hq=8)
    k, v = synth.kv(w, device=DEV)
    k[0, 5] = 0
    v[0, 5] = 0
    k[0, 9, 0, 17] = 60000.0
    v[0, 12, 1] = torch.linspace(-65504, 65504, 128, device=DEV).to(torch.float16)
    lens = torch.tensor([256], dtype=torch.int32)
    table = torch.tensor([[1, 0]], dtype=torch.int32)
    pool, st = _write(w, k, v, lens, table, 2, 256)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = kvref.fp8_write_blocks(host(k), host(v), host(lens), host(table), 2)
    _check_pages(pool, ref, host(table), host(lens))


def test_many_splits_long_sequence_and_second_call():
    w = synth.scaled(synth.WORKLOADS["long_context"], batch=1, seq=20000, hkv=2, hq=8)
    lens = torch.tensor([20000], dtype=torch.int32)
    g = torch.Generator().manual_seed(32)
    table = torch.randperm(157, generator=g).to(torch.int32).reshape(1, 157)
    q, pool, out, ws, st, max_seq = _run(w, lens, table, 157, check_pages=False)
    out2 = torch.empty_like(out)
    kv.kvarn_fp8_decode_attention(q, w.hkv, pool, table.to(DEV), lens.to(DEV), max_seq, out2,
                                  ws, status=st)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)


def test_llama_like_layer_full_size_sampled():
    w = synth.WORKLOADS["llama3_8b_layer"]
    lens = synth.seq_lens(w)
    tables, n = synth.block_tables(w)
    _run(w, lens, tables[0].contiguous(), n, seqs=[0, 7, 15], check_pages=False)


def test_bad_page_reported():
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=1, seq=512, hkv=2, hq=8)
    k, v = synth.kv(w, device=DEV)
    lens = torch.tensor([512], dtype=torch.int32)
    good = torch.tensor([[0, 1, 2, 3]], dtype=torch.int32)
    pool, st = _write(w, k, v, lens, good, 4, 512)
    bad = torch.tensor([[0, 1, -5, 3]], dtype=torch.int32, device=DEV)
    q = synth.queries(w).to(DEV)
    out = torch.empty((1, w.hq, 128), dtype=torch.float16, device=DEV)
    ws = kv.alloc_fp8_decode_workspace(w.hq, w.hkv, 1, 512, DEV)
    kv.kvarn_fp8_decode_attention(q, w.hkv, pool, bad, lens.to(DEV), 512, out, ws, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & kv.kvarn.STATUS_BAD_PAGE
    assert torch.isfinite(out.float()).all()
