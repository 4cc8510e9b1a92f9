"""The five workloads at their full sizes, on the CUDA path, against the
float64 oracle on sampled outputs.

Every workload is quantized and decoded in full on the GPU, with the same
launch configuration the bench uses.  The oracle then recomputes what it can
finish in seconds: a seeded sample of whole tiles (every code and scale of
those records, under the boundary rule) and whole sequences of decode
attention (every head, every channel; fed the GPU's own pool so that decode is
judged apart from boundary flips).  Mixed serving additionally checks every
page that filled during its 64 append steps.

Quantization: KVarN page (blog.edumints.com), "KVarN Nasil Calisir?", all
four stages.  Decode and paging: "KV Cache (Anahtar-Deger Onbellegi)"
(yapayzekasozluk.tr), "KV Cache Nasil Calisir?" and "Paged Attention (vLLM)".
"""
import numpy as np
import pytest
import torch

import quantized_decode_attention_blocks_b300 as kv
from oracle import kvref
from tests import parity
from tests.gpu_helpers import DEV, bits16, config, host
from workloads import synth

pytestmark = pytest.mark.gpu

ITERS = 2


def _oracle_record(tile_k, tile_v):
    """Oracle record (both parts) of one (page, head) and its pre-rounding values."""
    rk = kvref.quantize_tile(tile_k, False, ITERS)
    rv = kvref.quantize_tile(tile_v, True, ITERS)
    rec = rk["rec"].copy()
    rec[9728:] = rv["rec"][9728:]
    return rec, rk["u"], rv["u"]


def _check_sampled_tiles(k, v, lens, table, pool, rng, n, stats):
    """n random full blocks (b, j, head): GPU record against the oracle."""
    lens_np = host(lens).astype(np.int64)
    nfull = lens_np // 128
    hkv = k.shape[2]
    cand = [(b, j) for b in range(len(lens_np)) for j in range(int(nfull[b]))]
    picks = rng.choice(len(cand), size=min(n, len(cand)), replace=False)
    tab = host(table)
    for i in picks:
        b, j = cand[int(i)]
        h = int(rng.integers(hkv))
        tk = bits16(k[b, 128 * j:128 * j + 128, h])
        tv = bits16(v[b, 128 * j:128 * j + 128, h])
        ref, u_k, u_v = _oracle_record(tk, tv)
        got = host(pool[int(tab[b, j]), h])
        parity.compare_record(got, ref, u_k, u_v, stats)


def _check_sampled_decode(cfg, q, out, pool, table, lens, tk, tv, seqs, **fmt):
    """Whole sequences `seqs`: the oracle reads a compact copy of just their
    pages.  `fmt`: the record format's oracle flags (m16, pc, g64, v4, k8)."""
    sel = torch.tensor(seqs, dtype=torch.long, device=DEV)
    tab = table[sel]
    used = torch.unique(tab[tab >= 0])
    remap = torch.full((pool.shape[0],), -1, dtype=torch.int32, device=DEV)
    remap[used] = torch.arange(used.numel(), dtype=torch.int32, device=DEV)
    tab_c = torch.where(tab >= 0, remap[tab.clamp(min=0).long()], tab)
    ref = kvref.decode_attention(host(q[sel]), host(pool[used]), host(tab_c), host(lens[sel]),
                                 host(tk[sel]), host(tv[sel]), cfg.num_q_heads,
                                 cfg.num_kv_heads, route=1,
                                 **{("meta16" if k == "m16" else k): v for k, v in fmt.items()})
    return parity.compare_attention(host(out[sel]), ref)


def _decode(cfg, q, pool, table, lens, max_seq, tk, tv):
    out = torch.full((q.shape[0], cfg.num_q_heads, 128), float("nan"), dtype=torch.float16,
                     device=DEV)
    ws = kv.alloc_decode_workspace(cfg, q.shape[0], max_seq, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kv.kvarn_decode_attention(cfg, q, pool, table, lens, max_seq, tk, tv, out, ws, status=st)
    return out, st


@pytest.mark.parametrize("name", ["llama3_8b_layer", "long_context"])
def test_single_layer_workload_full_size(name):
    w = synth.WORKLOADS[name]
    rng = np.random.default_rng(100 + w.seed)
    cfg = config(w.hq, w.hkv)
    k, v = synth.kv(w, device=DEV)
    lens = synth.seq_lens(w, device=DEV)
    tables, num_pages = synth.block_tables(w, device=DEV)
    table = tables[0].contiguous()
    pool = kv.alloc_pool(cfg, num_pages, DEV)
    tk, tv = kv.alloc_tails(cfg, w.batch, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kv.kvarn_quantize_blocks(cfg, k, v, lens, w.seq, table, pool, tk, tv, st)
    # one decode step: append the new token, then attend over len + 1 tokens
    kn, vn = synth.new_tokens(w, 0, device=DEV)
    kv.kvarn_append_token(cfg, kn, vn, lens, table, pool, tk, tv, st)
    lens1 = lens + 1
    q = synth.queries(w, device=DEV)
    out, st2 = _decode(cfg, q, pool, table, lens1, w.seq + 1, tk, tv)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(st2.item()) == 0
    assert torch.isfinite(out.float()).all()
    stats = {}
    _check_sampled_tiles(k, v, lens, table, pool, rng, 8, stats)
    parity.check_flip_rate(stats)
    seqs = sorted(rng.choice(w.batch, size=min(2, w.batch), replace=False).tolist())
    _check_sampled_decode(cfg, q, out, pool, table, lens1, tk, tv, seqs)


def test_qwen_like_workload_layers_full_size():
    """28 layers share one pool of pages scattered across it; the first, a
    middle and the last layer are run at full size (the others differ only in
    their seed and their slice of the pool)."""
    w = synth.WORKLOADS["qwen25_15b"]
    rng = np.random.default_rng(100 + w.seed)
    cfg = config(w.hq, w.hkv)
    tables, num_pages = synth.block_tables(w, device=DEV)
    pool = kv.alloc_pool(cfg, num_pages, DEV)
    lens = synth.seq_lens(w, device=DEV)
    stats = {}
    for layer in (0, w.layers // 2 - 1, w.layers - 1):
        table = tables[layer].contiguous()
        k, v = synth.kv(w, layer=layer, device=DEV)
        tk, tv = kv.alloc_tails(cfg, w.batch, DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        kv.kvarn_quantize_blocks(cfg, k, v, lens, w.seq, table, pool, tk, tv, st)
        q = synth.queries(w, layer=layer, device=DEV)
        out, st2 = _decode(cfg, q, pool, table, lens, w.seq, tk, tv)
        torch.cuda.synchronize()
        assert int(st.item()) == 0 and int(st2.item()) == 0
        _check_sampled_tiles(k, v, lens, table, pool, rng, 6, stats)
        seqs = sorted(rng.choice(w.batch, size=2, replace=False).tolist())
        _check_sampled_decode(cfg, q, out, pool, table, lens, tk, tv, seqs)
        del k, v
    parity.check_flip_rate(stats)


def test_mixed_serving_full_size_with_appends():
    """128 requests of mixed lengths, pages scattered; 64 decode steps, each
    appending one token per request (a filled tail block is quantized in the
    same launch) and attending over the pages plus the fp16 tail."""
    w = synth.WORKLOADS["mixed_serving"]
    rng = np.random.default_rng(100 + w.seed)
    cfg = config(w.hq, w.hkv)
    k, v = synth.kv(w, device=DEV)
    lens = synth.seq_lens(w, device=DEV)
    tables, num_pages = synth.block_tables(w, device=DEV)
    table = tables[0].contiguous()
    pool = kv.alloc_pool(cfg, num_pages, DEV)
    tk, tv = kv.alloc_tails(cfg, w.batch, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    max_seq = w.seq + w.decode_steps
    kv.kvarn_quantize_blocks(cfg, k, v, lens, w.seq, table, pool, tk, tv, st)
    # decode is checked against the oracle on 8 requests at the first step, at
    # the first step whose append fills a tail block (one of those requests
    # is among the 8: it reads its fresh page and an empty tail) and at the
    # last step
    lens_h = host(lens).astype(np.int64)
    fills = [(s, b) for s in range(1, w.decode_steps) for b in range(w.batch)
             if (lens_h[b] + s) % 128 == 127]
    s_fill, b_fill = fills[0]
    checks = {0: None, s_fill: b_fill, w.decode_steps - 1: None}
    new = []
    cur = lens.clone()
    for step in range(w.decode_steps):
        kn, vn = synth.new_tokens(w, step, device=DEV)
        new.append((kn, vn))
        kv.kvarn_append_token(cfg, kn, vn, cur, table, pool, tk, tv, st)
        cur = cur + 1
        q = synth.queries(w, step=step, device=DEV)
        out, st2 = _decode(cfg, q, pool, table, cur, max_seq, tk, tv)
        if step in checks:
            torch.cuda.synchronize()
            assert int(st.item()) == 0 and int(st2.item()) == 0
            must = checks[step]
            pool_ids = [b for b in range(w.batch) if b != must]
            seqs = rng.choice(pool_ids, size=8 if must is None else 7, replace=False).tolist()
            if must is not None:
                assert int(host(cur)[must]) % 128 == 0     # the block just filled
                seqs.append(must)
            _check_sampled_decode(cfg, q, out, pool, table, cur, tk, tv, sorted(seqs))
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(st2.item()) == 0
    stats = {}
    _check_sampled_tiles(k, v, lens, table, pool, rng, 8, stats)
    # every block that filled during the appends: prefill leftovers + new tokens
    lens0 = host(lens).astype(np.int64)
    tab = host(table)
    new_k = np.stack([bits16(kn) for kn, _ in new])     # [step][B][Hkv][128]
    new_v = np.stack([bits16(vn) for _, vn in new])
    filled = 0
    for b in range(w.batch):
        start = int(lens0[b] // 128) * 128
        n_old = int(lens0[b]) - start
        if lens0[b] + w.decode_steps < start + 128:
            continue
        j = start // 128
        old_k = bits16(k[b, start:start + n_old])        # [n_old][Hkv][128]
        old_v = bits16(v[b, start:start + n_old])
        got = host(pool[int(tab[b, j])])
        for h in range(w.hkv):
            tile_k = np.concatenate([old_k[:, h], new_k[:128 - n_old, b, h]])
            tile_v = np.concatenate([old_v[:, h], new_v[:128 - n_old, b, h]])
            ref, u_k, u_v = _oracle_record(tile_k, tile_v)
            parity.compare_record(got[h], ref, u_k, u_v, stats)
            filled += 1
    assert filled > 0
    parity.check_flip_rate(stats)


_KPART = {"m16": 8960, "pc": 9728, "g64": 10752, "v4": 9728, "k8": 17920}


@pytest.mark.parametrize("variant", ["rms", "m16", "pc", "g64", "v4", "k8"])
def test_format_variants_at_the_llama_like_size(variant):
    # every format variant the bench times, at the size and in the launch
    # configuration it is timed in: one prefill, one append, one decode;
    # sampled whole tiles and whole sequences against the oracle
    w = synth.WORKLOADS["llama3_8b_layer"]
    rng = np.random.default_rng(300 + len(variant))
    rms = variant == "rms"
    fmt = {} if rms else {("meta16" if variant == "m16" else variant): True}
    cfg = config(w.hq, w.hkv, rms=rms, **({} if rms else {variant: True}))
    k, v = synth.kv(w, device=DEV)
    lens = synth.seq_lens(w, device=DEV)
    tables, num_pages = synth.block_tables(w, device=DEV)
    table = tables[0].contiguous()
    pool = kv.alloc_pool(cfg, num_pages, DEV)
    tk, tv = kv.alloc_tails(cfg, w.batch, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kv.kvarn_quantize_blocks(cfg, k, v, lens, w.seq, table, pool, tk, tv, st)
    kn, vn = synth.new_tokens(w, 0, device=DEV)
    kv.kvarn_append_token(cfg, kn, vn, lens, table, pool, tk, tv, st)
    lens1 = lens + 1
    q = synth.queries(w, device=DEV)
    out, st2 = _decode(cfg, q, pool, table, lens1, w.seq + 1, tk, tv)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(st2.item()) == 0
    assert torch.isfinite(out.float()).all()
    # sampled tiles
    kpart = _KPART.get(variant, 9728)
    lens_np = host(lens).astype(np.int64)
    tab = host(table)
    stats = {}
    for _ in range(6):
        b = int(rng.integers(w.batch))
        j = int(rng.integers(lens_np[b] // 128))
        h = int(rng.integers(w.hkv))
        tkb = bits16(k[b, 128 * j:128 * j + 128, h])
        tvb = bits16(v[b, 128 * j:128 * j + 128, h])
        rk = kvref.quantize_tile(tkb, False, ITERS, rms=rms, **fmt)
        rv = kvref.quantize_tile(tvb, True, ITERS, rms=rms, **fmt)
        ref = rk["rec"].copy()
        ref[kpart:] = rv["rec"][kpart:]
        ref32 = None
        if variant == "m16":
            r32k = kvref.quantize_tile(tkb, False, ITERS)["rec"]
            ref32 = r32k.copy()
            ref32[9728:] = kvref.quantize_tile(tvb, True, ITERS)["rec"][9728:]
        got = host(pool[int(tab[b, j]), h])
        parity.compare_record(got, ref, rk["u"], rv["u"], stats, meta16=variant == "m16",
                              ref32=ref32, pc=variant == "pc", g64=variant == "g64",
                              v4=variant == "v4", k8=variant == "k8")
    parity.check_flip_rate(stats)
    # sampled whole sequences of decode
    seqs = sorted(rng.choice(w.batch, size=2, replace=False).tolist())
    sel = torch.tensor(seqs, dtype=torch.long, device=DEV)
    tsel = table[sel]
    used = torch.unique(tsel[tsel >= 0])
    remap = torch.full((pool.shape[0],), -1, dtype=torch.int32, device=DEV)
    remap[used] = torch.arange(used.numel(), dtype=torch.int32, device=DEV)
    tab_c = torch.where(tsel >= 0, remap[tsel.clamp(min=0).long()], tsel)
    ref = kvref.decode_attention(host(q[sel]), host(pool[used]), host(tab_c), host(lens1[sel]),
                                 host(tk[sel]), host(tv[sel]), w.hq, w.hkv, route=1, **fmt)
    parity.compare_attention(host(out[sel]), ref)


def test_end_to_end_step_matches_the_resident_step():
    """The bench's end-to-end step, whose K and V cross from pinned host memory
    on copy streams into two alternating device buffers while the previous
    layer computes, leaves every layer the output, pages and tails of the same
    step run on device-resident inputs, bit for bit: no copy overwrites a
    buffer before its quantize has read it."""
    import bench
    w = synth.scaled(synth.WORKLOADS["qwen25_15b"], layers=6, batch=4, seq=1000)
    units, per_step = bench.build_units(w, DEV, 0)
    assert per_step == 6
    for u in units:
        u.quantize()
        u.append()
        u.decode()
    torch.cuda.synchronize()
    ref_out = [u.out.clone() for u in units]
    ref_tails = [(u.tk.clone(), u.tv.clone()) for u in units]
    ref_pool = units[0].pool.clone()
    units[0].pool.zero_()
    for u in units:
        u.out.zero_()
        u.tk.zero_()
        u.tv.zero_()
    step, hostbufs = bench.make_e2e_step(units, torch.cuda.current_stream())
    for _ in range(3):   # the third step's copies wait on the second's kernels
        step()
    torch.cuda.synchronize()
    assert all(int(u.status.item()) == 0 for u in units)
    assert torch.equal(units[0].pool, ref_pool)
    for u, h, o, (tk, tv) in zip(units, hostbufs, ref_out, ref_tails):
        assert torch.equal(h["out"].to(DEV).view(torch.int16), o.view(torch.int16))
        assert torch.equal(u.tk, tk) and torch.equal(u.tv, tv)
