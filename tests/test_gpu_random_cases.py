"""Seeded random decode and chunk cases over the record formats, GQA groups,
ragged lengths and permuted block tables, each against the float64 oracle
(fed the GPU's own pool).  "KV Cache Nasil Calisir?" and "Paged Attention
(vLLM)" (yapayzekasozluk.tr); the KVarN page (blog.edumints.com)."""
import numpy as np
import pytest
import torch

import quantized_decode_attention_blocks_b300 as kv
from oracle import kvref
from tests import parity
from tests.gpu_helpers import DEV, config, decode, host, prefill
from workloads import synth

pytestmark = pytest.mark.gpu

VARIANTS = ["f32", "m16", "pc", "g64", "v4", "k8"]


def _case(seed):
    rng = np.random.default_rng(seed)
    variant = VARIANTS[seed % len(VARIANTS)]
    hkv = int(rng.choice([1, 2, 4]))
    g = int(rng.integers(1, 9))
    B = int(rng.integers(1, 7))
    max_seq = int(rng.integers(1, 3000))
    lens = rng.integers(0, max_seq + 1, size=B)
    lens[int(rng.integers(B))] = max_seq
    return variant, hkv, g, B, max_seq, lens


@pytest.mark.parametrize("seed", range(24))
def test_random_decode_case(seed):
    variant, hkv, g, B, max_seq, lens = _case(seed)
    fmt = {} if variant == "f32" else {variant: True}
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=B, seq=max_seq, hkv=hkv,
                     hq=g * hkv, seed=300 + seed)
    k, v = synth.kv(w, device=DEV)
    cfg = config(w.hq, w.hkv, **fmt)
    mb = max((max_seq + 127) // 128, 1)
    perm = torch.randperm(B * mb, generator=torch.Generator().manual_seed(seed))
    table = perm.to(torch.int32).reshape(B, mb)
    lt = torch.tensor(lens, dtype=torch.int32)
    pool, tk, tv, st = prefill(cfg, k, v, lt, table, B * mb, max_seq=max_seq)
    q = synth.queries(w).to(DEV)
    out, st2, _ = decode(cfg, q, pool, table, lt, tk, tv, max_seq=max_seq)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(st2.item()) == 0
    okw = {("meta16" if variant == "m16" else variant): True} if fmt else {}
    ref = kvref.decode_attention(host(q), host(pool), host(table), host(lt), host(tk), host(tv),
                                 w.hq, w.hkv, **okw)
    parity.compare_attention(host(out).astype(np.float64), ref)


@pytest.mark.parametrize("seed", range(12))
def test_random_chunk_case(seed):
    # a chunk of new tokens per sequence after a random cached prefix, the
    # chunk's tokens appended to the cache before the call
    rng = np.random.default_rng(1000 + seed)
    variant = VARIANTS[seed % len(VARIANTS)]
    fmt = {} if variant == "f32" else {variant: True}
    hkv = int(rng.choice([1, 2]))
    g = int(rng.integers(1, 9))
    B = int(rng.integers(1, 4))
    M = int(rng.integers(1, 200))
    starts = rng.integers(0, 1500, size=B)
    cls = rng.integers(0, M + 1, size=B)
    cls[int(rng.integers(B))] = M
    n = starts + cls
    S = max(int(n.max()), 1)
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=B, seq=S, hkv=hkv, hq=g * hkv,
                     seed=700 + seed)
    k, v = synth.kv(w, device=DEV)
    cfg = config(w.hq, w.hkv, **fmt)
    mb = (S + 127) // 128
    table = torch.randperm(B * mb, generator=torch.Generator().manual_seed(seed)).to(
        torch.int32).reshape(B, mb)
    lens = torch.tensor(n, dtype=torch.int32)
    pool, tk, tv, st = prefill(cfg, k, v, lens, table, B * mb, max_seq=S)
    gq = torch.Generator(device=DEV).manual_seed(2000 + seed)
    q = torch.randn((B, M, w.hq, 128), generator=gq, device=DEV).to(torch.float16)
    out = torch.full_like(q, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kv.kvarn_chunk_attention(cfg, q, torch.tensor(starts, dtype=torch.int32, device=DEV),
                             torch.tensor(cls, dtype=torch.int32, device=DEV), S, pool,
                             table.to(DEV), tk, tv, out, status=status)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(status.item()) == 0
    okw = {("meta16" if variant == "m16" else variant): True} if fmt else {}
    ref = kvref.chunk_attention(host(q), starts, cls, host(pool), host(table), host(tk),
                                host(tv), w.hq, w.hkv, **okw)
    got = host(out).astype(np.float64)
    for b, c in enumerate(cls):
        assert not got[b, int(c):].any()
    parity.compare_attention(got, ref)


@pytest.mark.parametrize("seed", range(6))
def test_random_append_case(seed):
    # sequences of random lengths each take 1..150 decode-time appends; the
    # pages they fill equal the prefill of the final lengths bit for bit, the
    # tails hold the leftover tokens
    rng = np.random.default_rng(3000 + seed)
    variant = VARIANTS[seed % len(VARIANTS)]
    fmt = {} if variant == "f32" else {variant: True}
    B, hkv = int(rng.integers(1, 5)), int(rng.choice([1, 2]))
    steps = int(rng.integers(1, 151))
    start = rng.integers(0, 400, size=B)
    S = int(start.max()) + steps
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=B, seq=S, hkv=hkv, hq=2 * hkv,
                     seed=900 + seed)
    k, v = synth.kv(w, device=DEV)
    cfg = config(w.hq, w.hkv, **fmt)
    mb = (S + 127) // 128
    table = torch.randperm(B * mb, generator=torch.Generator().manual_seed(seed)).to(
        torch.int32).reshape(B, mb)
    pool, tk, tv, st = prefill(cfg, k, v, torch.tensor(start, dtype=torch.int32), table,
                               B * mb, max_seq=S)
    tdev = table.to(DEV)
    for s in range(steps):
        pos = torch.tensor(start + s, dtype=torch.int32, device=DEV)
        kn = torch.stack([k[b, int(start[b]) + s] for b in range(B)]).contiguous()
        vn = torch.stack([v[b, int(start[b]) + s] for b in range(B)]).contiguous()
        kv.kvarn_append_token(cfg, kn, vn, pos, tdev, pool, tk, tv, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    final = torch.tensor(start + steps, dtype=torch.int32)
    ref_pool, ref_tk, ref_tv, st2 = prefill(cfg, k, v, final, table, B * mb, max_seq=S)
    torch.cuda.synchronize()
    for b in range(B):
        nfull = int(final[b]) // 128
        pages = table[b, :nfull].long()
        assert torch.equal(pool[pages], ref_pool[pages]), (variant, b)
        rem = int(final[b]) % 128
        assert torch.equal(tk[b, :, :rem], ref_tk[b, :, :rem])
        assert torch.equal(tv[b, :, :rem], ref_tv[b, :, :rem])


@pytest.mark.parametrize("seed", range(6))
def test_random_snapkv_case(seed):
    # SnapKV-style selection over random prompt lengths, windows, capacities
    # and pooling kernels, through the same checks as its own tests
    from tests.test_gpu_snapkv import _check, _run
    rng = np.random.default_rng(5000 + seed)
    hkv = int(rng.choice([1, 2, 8]))
    g = int(rng.choice([1, 2, 4, 8]))
    W = int(rng.choice([8, 16, 32, 64]))
    B = int(rng.integers(1, 5))
    lens = [int(x) for x in rng.integers(W, 3000, size=B)]
    capacity = int(rng.integers(W + 1, 1200))
    kern = int(rng.choice([1, 3, 5, 7]))
    _check(_run(lens, W, capacity, g * hkv, hkv, seed=40 + seed, kern=kern))


@pytest.mark.parametrize("seed", range(6))
def test_random_quantize_case(seed):
    # prefill of random lengths on permuted pages, random Sinkhorn iteration
    # count and statistic, every record against the oracle's
    from tests.test_gpu_quantize import _check_prefill
    rng = np.random.default_rng(7000 + seed)
    variant = VARIANTS[(seed + 3) % len(VARIANTS)]
    fmt = {} if variant == "f32" else {variant: True}
    B, hkv = int(rng.integers(1, 4)), int(rng.choice([1, 2, 4]))
    S = int(rng.integers(128, 1400))
    lens = torch.tensor(rng.integers(0, S + 1, size=B), dtype=torch.int32)
    lens[int(rng.integers(B))] = S
    iters = int(rng.integers(0, 5))
    rms = bool(rng.integers(0, 2))
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=B, seq=S, hkv=hkv, hq=hkv,
                     seed=800 + seed)
    mb = (S + 127) // 128
    table = torch.randperm(B * mb, generator=torch.Generator().manual_seed(seed)).to(
        torch.int32).reshape(B, mb)
    _check_prefill(w, lens, table, B * mb, iters=iters, rms=rms, **fmt)
