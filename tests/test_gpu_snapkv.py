"""SnapKV-style one-shot selection on the GPU against the float64 oracle.

"Makale Bulteni - SnapKV" (cmlonder.com): the observation window's attention
over the prompt picks each head's clustered critical positions once, at the
end of prefill.  Votes are compared element by element; the selection made
from the GPU's own votes must equal the oracle's selection from those votes
(the same pooling and tie rule on the same numbers), and must be a valid top
set for the oracle's float64 votes; the gather is bit-exact.
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


def _run(lens, W, capacity, hq, hkv, seed, S=None, kern=7):
    lens = torch.tensor(lens, dtype=torch.int32)
    B = len(lens)
    S = int(lens.max()) if S is None else S
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=B, seq=S, hkv=hkv, hq=hq)
    k, v = synth.kv(w, layer=seed, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(seed)
    qw = torch.randn((B, W, hq, 128), generator=g, device=DEV).to(torch.float16)
    cfg = config(hq, hkv)
    votes = torch.full((B, hkv, S), float("nan"), device=DEV)
    idx = torch.full((B, hkv, capacity), -7, dtype=torch.int32, device=DEV)
    ws = torch.zeros(kv.snapkv_workspace_bytes(cfg, B, W, S), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kv.kvarn_snapkv_select(cfg, qw, k, lens.to(DEV), S, capacity, votes, idx, ws,
                           pool_kernel=kern, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return dict(k=k, v=v, qw=qw, votes=host(votes), idx=host(idx), lens=host(lens), W=W,
                capacity=capacity, hq=hq, hkv=hkv, kern=kern, cfg=cfg)


def _check(c):
    ref = kvref.snapkv_votes(host(c["qw"]), host(c["k"]), c["lens"], c["hq"], c["hkv"])
    got = c["votes"].astype(np.float64)
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    rel = (err / np.maximum(np.abs(ref), 1e-30)).max()
    assert np.all(err <= 1e-4 * np.abs(ref) + 1e-7), f"votes: max rel err {rel:.3e}"
    # the selection from the GPU's votes is exactly the oracle's rule on them
    sel = kvref.snapkv_select(got, c["lens"], c["W"], c["capacity"], c["kern"])
    assert np.array_equal(c["idx"], sel)
    # and a valid top set for the float64 votes: every kept prefix position
    # scores at least the oracle's threshold, up to the votes' tolerance
    B, hkv = ref.shape[:2]
    keep = c["capacity"] - c["W"]
    for b in range(B):
        npre = int(c["lens"][b]) - c["W"]
        if npre <= keep:
            continue
        for h in range(hkv):
            pooled = kvref.snapkv_pool(ref[b, h, :npre], c["kern"])
            thr = np.sort(pooled)[::-1][keep - 1]
            kept = c["idx"][b, h, :keep]
            assert np.all(pooled[kept] >= thr * (1 - 2e-4) - 2e-7)


@pytest.mark.parametrize("hq,hkv,W", [(8, 2, 32), (12, 2, 32), (8, 8, 64), (32, 8, 16)])
def test_votes_and_selection_ragged(hq, hkv, W):
    # prompts shorter than the capacity (kept whole), one window only, one over
    # a chunk boundary (2048), several row tiles when W x g > 128
    c = _run([5000, 700, W + 3, 2100], W=W, capacity=512, hq=hq, hkv=hkv, seed=3)
    _check(c)


def test_kernel_sizes_and_exact_capacity():
    for kern in (1, 3, 9):
        c = _run([3000, 1500], W=32, capacity=400, hq=8, hkv=2, seed=4 + kern, kern=kern)
        _check(c)
    c = _run([1032], W=32, capacity=1032, hq=8, hkv=2, seed=9)   # prefix == capacity - W
    assert np.array_equal(c["idx"][0, 0], np.arange(1032))


def test_gather_then_compact_decode():
    c = _run([4000, 2600], W=32, capacity=1024, hq=8, hkv=2, seed=11)
    _check(c)
    B, C, hkv = 2, 1024, 2
    ko = torch.empty((B, C, hkv, 128), dtype=torch.float16, device=DEV)
    vo = torch.empty_like(ko)
    idx = torch.from_numpy(c["idx"]).to(DEV)
    kv.kvarn_snapkv_gather(c["k"], c["v"], idx, ko, vo)
    torch.cuda.synchronize()
    kh, vh, koh, voh = host(c["k"]), host(c["v"]), host(ko), host(vo)
    for b in range(B):
        for h in range(hkv):
            sel = c["idx"][b, h]
            assert np.array_equal(koh[b, :, h], kh[b, sel, h])
            assert np.array_equal(voh[b, :, h], vh[b, sel, h])
    # the compact cache quantized and decoded like any other
    lens = torch.full((B,), C, dtype=torch.int32)
    table = torch.arange(B * 8, dtype=torch.int32).reshape(B, 8)
    pool, tk, tv, st = prefill(c["cfg"], ko, vo, lens, table, B * 8)
    q = torch.randn((B, 8, 128), device=DEV).to(torch.float16)
    out = torch.empty_like(q)
    ws = kv.alloc_decode_workspace(c["cfg"], B, C, DEV)
    kv.kvarn_decode_attention(c["cfg"], q, pool, table.to(DEV), lens.to(DEV), C, tk, tv, out, ws,
                              status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = kvref.decode_attention(host(q), host(pool), host(table), host(lens), host(tk),
                                 host(tv), 8, 2)
    parity.compare_attention(host(out), ref)
