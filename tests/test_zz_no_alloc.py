"""The decode entry point for callers that cannot allocate GPU memory.

Some callers can only hand a kernel its inputs and outputs (plugin hosts of
inference engines), or cannot afford the device synchronisation of cudaMalloc
in their serving loop, so they cannot provide the split-K workspace that
kvarn_decode_attention takes.  kvarn_decode_attention_noalloc keeps that
scratch in a fixed array inside the library.  These tests call it through the
C ABI and hold it to the output of kvarn_decode_attention, call after call.
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
    # one sequence of 131072 tokens with 16 query heads per KV head is split
    # into so many parts that its partial states need more than the built-in
    # scratch; the call must say so before touching the GPU (the pointers are
    # never used)
    cfg = kv.config_from_string("k4v2_g128", 16, 1)
    need = kv.decode_workspace_bytes(cfg, 1, 131072)
    assert need > K.NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(4096)
    rc = kv.lib().kvarn_decode_attention_noalloc(
        ctypes.byref(cfg), fake, fake, 1 << 20, fake, 1024, fake, 1, 131072, fake, fake,
        ctypes.c_float(128 ** -0.5), fake, None, None)
    assert rc == K.ERR_WORKSPACE


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    from tests.gpu_helpers import DEV, config, prefill
    from workloads import synth
    # long sequences so that decode splits every sequence many ways and the
    # scratch (partial softmax states and tickets) is really used
    lens = torch.tensor([20000, 13000, 300], dtype=torch.int32)
    w = synth.scaled(synth.WORKLOADS["long_context"], batch=3, seq=20000, hkv=2, hq=8)
    k, v = synth.kv(w, device=DEV)
    cfg = config(w.hq, w.hkv)
    mb = 157
    g = torch.Generator().manual_seed(7)
    table = torch.randperm(3 * mb, generator=g).to(torch.int32).reshape(3, mb)
    pool, tk, tv, st = prefill(cfg, k, v, lens, table, 3 * mb, max_seq=20000)
    q = synth.queries(w).to(DEV)
    tdev, ldev = table.to(DEV), lens.to(DEV)
    assert kv.decode_workspace_bytes(cfg, 3, 20000) > 0

    ref = torch.empty((3, w.hq, 128), dtype=torch.float16, device=DEV)
    ws = kv.alloc_decode_workspace(cfg, 3, 20000, DEV)
    kv.kvarn_decode_attention(cfg, q, pool, tdev, ldev, 20000, tk, tv, ref, ws, status=st)

    L = kv.lib()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        rc = L.kvarn_decode_attention_noalloc(
            ctypes.byref(cfg), _ptr(q), _ptr(pool), pool.shape[0], _ptr(tdev), mb, _ptr(ldev),
            3, 20000, _ptr(tk), _ptr(tv), ctypes.c_float(128 ** -0.5), _ptr(out), _ptr(status),
            stream)
        assert rc == K.OK, kv.status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0 and int(st.item()) == 0
        got = out.float().cpu().numpy().astype(np.float64)
        want = ref.float().cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all(), f"call {call}: non-finite output"
        err = np.abs(got - want)
        assert np.all(err <= 2e-3 + 1e-3 * np.abs(want)), f"call {call}: max err {err.max()}"
