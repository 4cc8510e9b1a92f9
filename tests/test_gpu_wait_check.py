"""The bounded waits of the library's kernels, run out on purpose without any
fault: kvarn_wait_check waits on a barrier that nothing arrives at, reports
KVARN_STATUS_TIMEOUT, and the context stays usable for the next calls."""
import ctypes

import numpy as np
import pytest
import torch

import quantized_decode_attention_blocks_b300 as kv
from quantized_decode_attention_blocks_b300 import kvarn as K
from oracle import kvref
from tests import parity
from tests.gpu_helpers import DEV, config, decode, host, prefill
from workloads import synth

pytestmark = pytest.mark.gpu


def _check(status, arrive, limit_us):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    rc = kv.lib().kvarn_wait_check(ctypes.c_void_p(status.data_ptr()), arrive, limit_us, stream)
    e1.record()
    torch.cuda.synchronize()
    assert rc == K.OK
    return e0.elapsed_time(e1) * 1e3   # microseconds


def test_a_wait_with_its_arrival_does_not_time_out():
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    _check(status, 1, 2000)
    assert int(status.item()) == 0


def test_a_wait_without_arrival_times_out_and_the_context_stays_usable():
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    us = _check(status, 0, 3000)
    assert int(status.item()) == K.STATUS_TIMEOUT
    assert us >= 3000          # it waited its limit, then gave up
    # the next calls run normally: a small prefill and decode at parity
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=2, seq=300, hkv=2, hq=8)
    k, v = synth.kv(w, device=DEV)
    cfg = config(w.hq, w.hkv)
    lens = torch.tensor([300, 129], dtype=torch.int32)
    table = torch.tensor([[0, 1, 2], [3, 4, 5]], dtype=torch.int32)
    pool, tk, tv, st = prefill(cfg, k, v, lens, table, 6)
    q = synth.queries(w).to(DEV)
    out, st2, _ = decode(cfg, q, pool, table, lens, tk, tv)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(st2.item()) == 0
    ref = kvref.decode_attention(host(q), host(pool), host(table), host(lens), host(tk), host(tv),
                                 w.hq, w.hkv)
    parity.compare_attention(host(out).astype(np.float64), ref)
