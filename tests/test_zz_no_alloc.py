"""The decode entry point for callers that cannot allocate GPU memory.

Some callers can only hand a kernel its inputs and outputs (plugin hosts of
inference engines), or cannot afford the device synchronisation of cudaMalloc
in their serving loop, so they cannot provide the split-K workspace that
kvarn_decode_attention takes.  kvarn_decode_attention_noalloc keeps that
scratch in a fixed array inside the library.  These tests call it through the
C ABI and hold it to the float64 oracle and to the output of
kvarn_decode_attention, call after call.
This file is collected last so that a run stopping at its first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import quantized_decode_attention_blocks_b300 as kv
from quantized_decode_attention_blocks_b300 import kvarn as K


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_noalloc_rejects_requests_beyond_its_scratch():
    # On a B300 (148 SMs) every request fits the built-in scratch: one wave of
    # split CTAs with at most 16 query heads per KV head stays under 16 MiB.
    # A device with many more SMs plans more splits; a request whose partial
    # states pass the scratch must be refused before touching the GPU.  The
    # call here only runs where it cannot launch (no device: it cannot plan
    # and says so); on a GPU whose plan fits, it is not made at all, since its
    # pointers are fake.
    cfg = kv.config_from_string("k4v2_g128", 16, 1)
    S = 1 << 22
    assert kv.decode_split_plan(cfg, 1, S, 148)[2] <= K.NOALLOC_SCRATCH_BYTES
    assert kv.decode_split_plan(cfg, 1, S, 2000)[2] > K.NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(4096)
    args = (ctypes.byref(cfg), fake, fake, 1 << 20, fake, S // 128, fake, 1, S, fake, fake,
            ctypes.c_float(128 ** -0.5), fake, None, None)
    if not torch.cuda.is_available():
        assert kv.lib().kvarn_decode_attention_noalloc(*args) == K.ERR_LAUNCH
        return
    if kv.decode_split_plan(cfg, 1, S, 0)[2] <= K.NOALLOC_SCRATCH_BYTES:
        pytest.skip("every request fits the scratch on this device")
    assert kv.lib().kvarn_decode_attention_noalloc(*args) == K.ERR_WORKSPACE


def _noalloc_twice(lens, max_seq, hkv, hq, seed, **fmt):
    """Prefills a seeded cache, then calls the no-alloc decode twice through
    the C ABI and checks both outputs against the float64 oracle (fed the
    GPU's own pool) and against kvarn_decode_attention."""
    from oracle import kvref
    from tests import parity
    from tests.gpu_helpers import DEV, config, host, prefill
    from workloads import synth
    B = len(lens)
    lens = torch.tensor(lens, dtype=torch.int32)
    w = synth.scaled(synth.WORKLOADS["long_context"], batch=B, seq=max_seq, hkv=hkv, hq=hq)
    k, v = synth.kv(w, layer=seed, device=DEV)
    cfg = config(w.hq, w.hkv, **fmt)
    mb = (max_seq + 127) // 128
    g = torch.Generator().manual_seed(seed)
    table = torch.randperm(B * mb, generator=g).to(torch.int32).reshape(B, mb)
    pool, tk, tv, st = prefill(cfg, k, v, lens, table, B * mb, max_seq=max_seq)
    q = synth.queries(w).to(DEV)
    tdev, ldev = table.to(DEV), lens.to(DEV)
    plan = kv.decode_split_plan(cfg, B, max_seq)

    ref = torch.empty((B, w.hq, 128), dtype=torch.float16, device=DEV)
    ws = kv.alloc_decode_workspace(cfg, B, max_seq, DEV)
    kv.kvarn_decode_attention(cfg, q, pool, tdev, ldev, max_seq, tk, tv, ref, ws, status=st)
    torch.cuda.synchronize()
    okw = {("meta16" if k == "m16" else k): v for k, v in fmt.items()}
    want_oracle = kvref.decode_attention(host(q), host(pool), host(table), host(lens), host(tk),
                                         host(tv), w.hq, w.hkv, **okw)
    want_cuda = ref.float().cpu().numpy().astype(np.float64)

    L = kv.lib()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        rc = L.kvarn_decode_attention_noalloc(
            ctypes.byref(cfg), _ptr(q), _ptr(pool), pool.shape[0], _ptr(tdev), mb, _ptr(ldev),
            B, max_seq, _ptr(tk), _ptr(tv), ctypes.c_float(128 ** -0.5), _ptr(out),
            _ptr(status), stream)
        assert rc == K.OK, kv.status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0 and int(st.item()) == 0
        got = out.float().cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all(), f"call {call}: non-finite output"
        parity.compare_attention(got, want_oracle)
        err = np.abs(got - want_cuda)
        assert np.all(err <= 2e-3 + 1e-3 * np.abs(want_cuda)), f"call {call}: max err {err.max()}"
    return plan


@pytest.mark.gpu
def test_noalloc_matches_oracle_twice_with_ticket_merge():
    # long sequences: decode splits every sequence more than four ways, so the
    # scratch holds partial softmax states and the arrival tickets
    plan = _noalloc_twice([20000, 13000, 300], 20000, hkv=2, hq=8, seed=7)
    assert plan[1] > 4 and plan[2] > 0


@pytest.mark.gpu
def test_noalloc_matches_oracle_twice_with_cluster_merge():
    # 16 sequences x 8 KV heads of 1536 tokens: 2 to 4 splits per (sequence,
    # KV head), merged inside a thread-block cluster (no tickets are read)
    plan = _noalloc_twice([1536] * 12 + [1400, 1290, 700, 5], 1536, hkv=8, hq=32, seed=11)
    assert 2 <= plan[1] <= 4


@pytest.mark.gpu
@pytest.mark.parametrize("variant", ["m16", "pc", "g64", "v4", "k8"])
def test_noalloc_format_variants(variant):
    # every record format through the built-in scratch (ticket merge)
    plan = _noalloc_twice([9000, 4000, 130], 9000, hkv=2, hq=8, seed=13, **{variant: True})
    assert plan[1] > 4
