"""Chunked-prefill attention over the quantized cache, on the GPU, against the
float64 oracle (kvref.chunk_attention fed the GPU's own pool and tails).

"KV Cache (Anahtar-Deger Onbellegi)" (yapayzekasozluk.tr), "KV Cache Nasil
Calisir?" (each token attends to the cached tokens up to its own position) and
"Paged Attention (vLLM)"; KVarN page (blog.edumints.com), "KVarN Nasil
Calisir?", stage 2 (the rotation keeps scores).  The cache of each sequence is
its state after the chunk was appended, built here by kvarn_quantize_blocks
over start + chunk_len tokens.
"""
import numpy as np
import pytest
import torch

import quantized_decode_attention_blocks_b300 as kv
from oracle import kvref
from tests import parity
from tests.gpu_helpers import DEV, config, host, prefill
from workloads import synth

pytestmark = pytest.mark.gpu


def _case(starts, chunk_lens, M, hq, hkv, seed, perm=True, table=None, num_pages=None,
          m16=False, pc=False, g64=False, v4=False, k8=False):
    starts = np.asarray(starts, dtype=np.int64)
    cls = np.asarray(chunk_lens, dtype=np.int64)
    n = starts + cls
    B = len(starts)
    S = max(int(n.max()), 1)
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=B, seq=S, hkv=hkv, hq=hq)
    k, v = synth.kv(w, layer=seed, device=DEV)
    cfg = config(hq, hkv, m16=m16, pc=pc, g64=g64, v4=v4, k8=k8)
    mb = (S + 127) // 128
    if table is None:
        g = torch.Generator().manual_seed(seed)
        order = torch.randperm(B * mb, generator=g) if perm else torch.arange(B * mb)
        table = order.to(torch.int32).reshape(B, mb)
        num_pages = B * mb
    lens = torch.tensor(n, dtype=torch.int32)
    pool, tk, tv, st = prefill(cfg, k, v, lens, table, num_pages, max_seq=S)
    gq = torch.Generator(device=DEV).manual_seed(1000 + seed)
    q = torch.randn((B, M, hq, 128), generator=gq, device=DEV).to(torch.float16)
    out = torch.full_like(q, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kv.kvarn_chunk_attention(cfg, q, torch.tensor(starts, dtype=torch.int32, device=DEV),
                             torch.tensor(cls, dtype=torch.int32, device=DEV), S, pool,
                             table.to(DEV), tk, tv, out, status=status)
    torch.cuda.synchronize()
    return dict(cfg=cfg, q=q, out=out, status=status, st=st, pool=pool, tk=tk, tv=tv,
                table=table, starts=starts, cls=cls, hq=hq, hkv=hkv, m16=m16, pc=pc,
                fmt=dict(g64=g64, v4=v4, k8=k8))


def _check(c):
    assert int(c["st"].item()) == 0 and int(c["status"].item()) == 0, \
        kv.status_string(int(c["status"].item()))
    got = host(c["out"]).astype(np.float64)
    assert np.isfinite(got).all()
    ref = kvref.chunk_attention(host(c["q"]), c["starts"], c["cls"], host(c["pool"]),
                                host(c["table"]), host(c["tk"]), host(c["tv"]), c["hq"],
                                c["hkv"], meta16=c["m16"], pc=c["pc"], **c["fmt"])
    for b, cl in enumerate(c["cls"]):
        assert not got[b, int(cl):].any(), "rows past the chunk must be zeros"
    return parity.compare_attention(got, ref)


@pytest.mark.parametrize("hq,hkv", [(4, 1), (8, 2), (12, 2), (16, 2), (32, 8)])
def test_chunks_ragged_with_pages_and_tail(hq, hkv):
    # chunks that start mid-page, inside the first block, at zero, and end in
    # the fp16 tail; several query tiles per (sequence, KV head) for g <= 4
    _check(_case([250, 100, 0, 300], [150, 60, 60, 1], 150, hq, hkv, seed=1))


@pytest.mark.parametrize("hq,hkv", [(8, 2), (12, 2)])
def test_m16_format(hq, hkv):
    # format variant "_m16" (fp16 metadata): ragged chunks over pages and tail
    _check(_case([250, 100, 0, 300], [150, 60, 60, 1], 150, hq, hkv, seed=8, m16=True))


@pytest.mark.parametrize("hq,hkv", [(8, 2), (12, 2)])
def test_pc_format(hq, hkv):
    # format variant "_pc" (per-channel groups)
    _check(_case([250, 100, 0, 300], [150, 60, 60, 1], 150, hq, hkv, seed=9, pc=True))


def test_chunk_of_whole_pages_and_inside_the_tail():
    # start and end on page boundaries (no tail at all); a chunk that lies
    # inside one block (all keys from the fp16 tail); a one-token chunk
    _check(_case([256, 10, 511, 0], [128, 50, 1, 128], 128, 8, 2, seed=2))


def test_long_prefix_many_blocks():
    # a 2000-token prefix: 16 blocks stream through the two page buffers and
    # the lazy softmax rescale
    _check(_case([2000, 1500], [200, 64], 200, 16, 4, seed=3))


def test_single_query_rows_equal_decode():
    # a chunk of one token at position n - 1 is decode attention over n tokens
    c = _case([700, 128], [1, 1], 1, 8, 2, seed=4)
    _check(c)
    lens = torch.tensor(c["starts"] + c["cls"], dtype=torch.int32)
    ref = kvref.decode_attention(host(c["q"][:, 0]), host(c["pool"]), host(c["table"]),
                                 host(lens), host(c["tk"]), host(c["tv"]), 8, 2)
    parity.compare_attention(host(c["out"][:, 0]).astype(np.float64), ref)


def test_bad_page_is_reported_and_its_tiles_are_zero():
    B, S = 2, 600
    mb = 5
    table = torch.arange(B * mb, dtype=torch.int32).reshape(B, mb)
    c = _case([400, 300], [100, 100], 100, 8, 2, seed=5, table=table, num_pages=B * mb)
    bad = table.clone()
    bad[1, 2] = 10 ** 6
    out = torch.full_like(c["q"], float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kv.kvarn_chunk_attention(c["cfg"], c["q"], torch.tensor([400, 300], dtype=torch.int32,
                                                            device=DEV),
                             torch.tensor([100, 100], dtype=torch.int32, device=DEV), S,
                             c["pool"], bad.to(DEV), c["tk"], c["tv"], out, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & kv.kvarn.STATUS_BAD_PAGE
    got = host(out).astype(np.float64)
    assert not got[1].any() and np.isfinite(got).all()
    parity.compare_attention(got[0], host(c["out"][0]).astype(np.float64))


def test_chunk_prefill_workload_sampled():
    # the bench's chunked-prefill workload: 16 sequences of the Llama-3-8B-like
    # layer, 3584 cached tokens + a 512-token chunk; two sequences checked
    w = synth.WORKLOADS["llama3_8b_layer"]
    B, M, start = 16, 512, 3584
    S = start + M
    k, v = synth.kv(synth.scaled(w, seq=S), device=DEV)
    cfg = config(w.hq, w.hkv)
    mb = S // 128
    table = torch.arange(B * mb, dtype=torch.int32).reshape(B, mb)
    lens = torch.full((B,), S, dtype=torch.int32)
    pool, tk, tv, st = prefill(cfg, k, v, lens, table, B * mb, max_seq=S)
    gq = torch.Generator(device=DEV).manual_seed(77)
    q = torch.randn((B, M, w.hq, 128), generator=gq, device=DEV).to(torch.float16)
    out = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    starts = torch.full((B,), start, dtype=torch.int32, device=DEV)
    cls = torch.full((B,), M, dtype=torch.int32, device=DEV)
    kv.kvarn_chunk_attention(cfg, q, starts, cls, S, pool, table.to(DEV), tk, tv, out,
                             status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and int(st.item()) == 0
    for b in (3, 14):
        used = table[b]
        ref = kvref.chunk_attention(host(q[b:b + 1]), [start], [M], host(pool[used.long()]),
                                    np.arange(mb, dtype=np.int32)[None], host(tk[b:b + 1]),
                                    host(tv[b:b + 1]), w.hq, w.hkv)
        parity.compare_attention(host(out[b:b + 1]).astype(np.float64), ref)


@pytest.mark.parametrize("fmt", ["g64", "v4", "k8"])
@pytest.mark.parametrize("hq,hkv", [(8, 2), (12, 2)])
def test_large_record_formats(fmt, hq, hkv):
    # formats "k4v2_g64", "k4v4_g128" and "k8v4_g128": one page record in
    # flight (two do not fit beside the six operands); ragged chunks over
    # pages and tail
    _check(_case([250, 100, 0, 300], [150, 60, 60, 1], 150, hq, hkv, seed=10,
                 **{fmt: True}))


@pytest.mark.parametrize("fmt", ["g64", "k8"])
def test_large_record_formats_long_prefix(fmt):
    # 16 blocks through the single record buffer
    _check(_case([2000, 1500], [200, 64], 200, 16, 4, seed=11, **{fmt: True}))
