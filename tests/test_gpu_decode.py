"""Decode attention on the GPU against the float64 oracle.

The oracle reads the GPU's own pool (rotated route), so decode is judged apart
from boundary flips of quantization.  "KV Cache (Anahtar-Deger Onbellegi)"
(yapayzekasozluk.tr), "KV Cache Nasil Calisir?" and "Paged Attention (vLLM)";
KVarN page (blog.edumints.com), "KVarN Nasil Calisir?", stage 2.
"""
import numpy as np
import pytest
import torch

from oracle import kvref
from tests import parity
from tests.gpu_helpers import DEV, config, decode, host, prefill
from workloads import synth

pytestmark = pytest.mark.gpu


def _run(w, lens, table, num_pages, q=None, max_seq=None, m16=False, pc=False, g64=False,
         v4=False, k8=False):
    max_seq = int(lens.max()) if max_seq is None else max_seq
    S = max(int(lens.max()), 1)
    k, v = synth.kv(w, device=DEV, seq=S)
    cfg = config(w.hq, w.hkv, m16=m16, pc=pc, g64=g64, v4=v4, k8=k8)
    pool, tk, tv, st = prefill(cfg, k, v, lens, table, num_pages, max_seq=max_seq)
    if q is None:
        q = synth.queries(w)
    out, st2, ws = decode(cfg, q, pool, table, lens, tk, tv, max_seq=max_seq)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(st2.item()) == 0
    ref = kvref.decode_attention(host(q), host(pool), host(table), host(lens), host(tk),
                                 host(tv), w.hq, w.hkv, route=1, meta16=m16, pc=pc, g64=g64,
                                 v4=v4, k8=k8)
    res = parity.compare_attention(host(out), ref)
    res.update(got=host(out).astype(np.float64), ref=ref)
    return res, (cfg, q, pool, table, lens, tk, tv, out, ws, max_seq)


@pytest.mark.parametrize("hq,hkv", [(1, 1), (4, 2), (6, 2), (8, 2), (10, 2), (12, 2), (14, 2),
                                    (8, 1), (16, 1), (32, 8), (24, 8), (40, 8), (56, 8)])
def test_group_sizes_and_ragged_lengths(hq, hkv):
    # every GQA group the tensor-core kernel pads (g = 2, 3, 5, 6, 7 to 4 or 8
    # query heads) next to the exact fits (1, 4, 8) and the CUDA-core g = 16
    lens = torch.tensor([0, 1, 127, 128, 129, 300, 1000, 2048], dtype=torch.int32)
    B = len(lens)
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=B, seq=2048, hkv=hkv, hq=hq)
    mb = 16
    g = torch.Generator().manual_seed(11)
    table = torch.randperm(B * mb, generator=g).to(torch.int32).reshape(B, mb)
    _run(w, lens, table, B * mb)


@pytest.mark.parametrize("hq,hkv", [(1, 1), (4, 2), (6, 2), (8, 2), (12, 2), (32, 8)])
def test_m16_format_group_sizes(hq, hkv):
    # format variant "_m16" (fp16 metadata): both head-tile counts of the
    # tensor-core kernel (g = 1..4: one, g = 6: two), over ragged lengths on
    # permuted pages
    lens = torch.tensor([0, 1, 127, 128, 129, 300, 1000, 2048], dtype=torch.int32)
    B = len(lens)
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=B, seq=2048, hkv=hkv, hq=hq)
    mb = 16
    g = torch.Generator().manual_seed(61)
    table = torch.randperm(B * mb, generator=g).to(torch.int32).reshape(B, mb)
    _run(w, lens, table, B * mb, m16=True)


def test_m16_format_cuda_core_kernel_and_many_splits():
    # g = 16 runs on the CUDA-core kernel; one long sequence takes the
    # workspace merge
    w = synth.scaled(synth.WORKLOADS["long_context"], batch=2, seq=9000, hkv=1, hq=16)
    lens = torch.tensor([9000, 333], dtype=torch.int32)
    table = torch.arange(2 * 71, dtype=torch.int32).reshape(2, 71)
    _run(w, lens, table, 2 * 71, m16=True)
    w = synth.scaled(synth.WORKLOADS["long_context"], batch=1, seq=20000, hkv=2, hq=8)
    lens = torch.tensor([20000], dtype=torch.int32)
    table = torch.arange(157, dtype=torch.int32).reshape(1, 157)
    _run(w, lens, table, 157, m16=True)


@pytest.mark.parametrize("hq,hkv", [(1, 1), (4, 2), (6, 2), (8, 2), (12, 2), (32, 8), (16, 1)])
def test_pc_format_group_sizes(hq, hkv):
    # format variant "_pc" (per-channel groups): one and two head tiles of the
    # tensor-core kernel and the CUDA-core kernel (g = 16), ragged lengths
    lens = torch.tensor([0, 1, 127, 128, 129, 300, 1000, 2048], dtype=torch.int32)
    B = len(lens)
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=B, seq=2048, hkv=hkv, hq=hq)
    mb = 16
    g = torch.Generator().manual_seed(63)
    table = torch.randperm(B * mb, generator=g).to(torch.int32).reshape(B, mb)
    _run(w, lens, table, B * mb, pc=True)


@pytest.mark.parametrize("hq,hkv", [(1, 1), (4, 2), (6, 2), (8, 2), (12, 2), (32, 8), (16, 1)])
def test_g64_format_group_sizes(hq, hkv):
    # format variant "k4v2_g64" (two groups per token): one and two head tiles
    # of the tensor-core kernel and the CUDA-core kernel (g = 16)
    lens = torch.tensor([0, 1, 127, 128, 129, 300, 1000, 2048], dtype=torch.int32)
    B = len(lens)
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=B, seq=2048, hkv=hkv, hq=hq)
    mb = 16
    g = torch.Generator().manual_seed(64)
    table = torch.randperm(B * mb, generator=g).to(torch.int32).reshape(B, mb)
    _run(w, lens, table, B * mb, g64=True)


@pytest.mark.parametrize("hq,hkv", [(1, 1), (4, 2), (6, 2), (8, 2), (12, 2), (32, 8), (16, 1)])
def test_v4_format_group_sizes(hq, hkv):
    # format variant "k4v4_g128" (4-bit values): one and two head tiles of the
    # tensor-core kernel and the CUDA-core kernel (g = 16)
    lens = torch.tensor([0, 1, 127, 128, 129, 300, 1000, 2048], dtype=torch.int32)
    B = len(lens)
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=B, seq=2048, hkv=hkv, hq=hq)
    mb = 16
    g = torch.Generator().manual_seed(65)
    table = torch.randperm(B * mb, generator=g).to(torch.int32).reshape(B, mb)
    _run(w, lens, table, B * mb, v4=True)


@pytest.mark.parametrize("hq,hkv", [(1, 1), (4, 2), (6, 2), (8, 2), (12, 2), (32, 8), (16, 1)])
def test_k8_format_group_sizes(hq, hkv):
    # format variant "k8v4_g128" (8-bit keys): one and two head tiles of the
    # tensor-core kernel and the CUDA-core kernel (g = 16)
    lens = torch.tensor([0, 1, 127, 128, 129, 300, 1000, 2048], dtype=torch.int32)
    B = len(lens)
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=B, seq=2048, hkv=hkv, hq=hq)
    mb = 16
    g = torch.Generator().manual_seed(66)
    table = torch.randperm(B * mb, generator=g).to(torch.int32).reshape(B, mb)
    _run(w, lens, table, B * mb, k8=True)


def test_k8_format_many_splits():
    w = synth.scaled(synth.WORKLOADS["long_context"], batch=1, seq=20000, hkv=2, hq=8)
    lens = torch.tensor([20000], dtype=torch.int32)
    table = torch.arange(157, dtype=torch.int32).reshape(1, 157)
    _run(w, lens, table, 157, k8=True)


def test_v4_format_many_splits():
    w = synth.scaled(synth.WORKLOADS["long_context"], batch=1, seq=20000, hkv=2, hq=8)
    lens = torch.tensor([20000], dtype=torch.int32)
    table = torch.arange(157, dtype=torch.int32).reshape(1, 157)
    _run(w, lens, table, 157, v4=True)


def test_g64_format_many_splits():
    w = synth.scaled(synth.WORKLOADS["long_context"], batch=1, seq=20000, hkv=2, hq=8)
    lens = torch.tensor([20000], dtype=torch.int32)
    table = torch.arange(157, dtype=torch.int32).reshape(1, 157)
    _run(w, lens, table, 157, g64=True)


def test_pc_format_many_splits():
    w = synth.scaled(synth.WORKLOADS["long_context"], batch=1, seq=20000, hkv=2, hq=8)
    lens = torch.tensor([20000], dtype=torch.int32)
    table = torch.arange(157, dtype=torch.int32).reshape(1, 157)
    _run(w, lens, table, 157, pc=True)


@pytest.mark.parametrize("variant", ["f32", "m16", "pc", "g64", "v4", "k8"])
def test_no_bias_common_to_all_channels(variant):
    # Every (sequence, head) of a Llama-3-8B layer at 1024 tokens: whole pages,
    # no fp16 tail.  An error shared by all 128 rotated channels lands on
    # output channel 0 alone (the first row of H is constant), where it would
    # hide inside the per-element tolerance; its mean over the 512 heads must
    # vanish down to the fp16 rounding of the output (~2e-5 for this mean).
    # A truncated inner sum in the tensor-core value sum left about -5e-4.
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=16, seq=1024, hkv=8, hq=32)
    lens = torch.full((16,), 1024, dtype=torch.int32)
    table = torch.arange(16 * 8, dtype=torch.int32).reshape(16, 8)
    res, _ = _run(w, lens, table, 16 * 8, **({} if variant == "f32" else {variant: True}))
    e0 = res["got"][:, :, 0] - res["ref"][:, :, 0]
    assert abs(e0.mean()) <= 1.5e-4, f"channel-0 mean signed error {e0.mean():.2e}"
    rest = res["got"][:, :, 1:] - res["ref"][:, :, 1:]
    assert abs(rest.mean()) <= 1.5e-4


def test_tiny_workload():
    w = synth.WORKLOADS["tiny"]
    tables, n = synth.block_tables(w)
    _run(w, synth.seq_lens(w), tables[0], n)


def test_many_splits_long_sequence():
    # one sequence of 20000 tokens: 156 pages + a 32-token tail -> many splits
    w = synth.scaled(synth.WORKLOADS["long_context"], batch=1, seq=20000, hkv=2, hq=8)
    lens = torch.tensor([20000], dtype=torch.int32)
    g = torch.Generator().manual_seed(3)
    table = torch.randperm(157, generator=g).to(torch.int32).reshape(1, 157)
    res, state = _run(w, lens, table, 157)
    # the workspace tickets are left at zero: a second call gives the same output
    cfg, q, pool, table, lens, tk, tv, out, ws, max_seq = state
    import quantized_decode_attention_blocks_b300 as kv
    out2 = torch.empty_like(out)
    kv.kvarn_decode_attention(cfg, q.to(DEV), pool, table.to(DEV), lens.to(DEV), max_seq, tk, tv,
                              out2, ws)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)


def test_max_seq_larger_than_lengths():
    # the grid is sized from max_seq; shorter sequences finish early
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=3, seq=700, hkv=2, hq=8)
    lens = torch.tensor([700, 5, 260], dtype=torch.int32)
    table = torch.arange(3 * 40, dtype=torch.int32).reshape(3, 40)
    _run(w, lens, table, 120, max_seq=5000)


def test_bad_page_reported():
    import quantized_decode_attention_blocks_b300 as kv
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=1, seq=512, hkv=2, hq=8)
    k, v = synth.kv(w, device=DEV)
    cfg = config(w.hq, w.hkv)
    lens = torch.tensor([512], dtype=torch.int32)
    pool, tk, tv, _ = prefill(cfg, k, v, lens, torch.tensor([[0, 1, 2, 3]], dtype=torch.int32),
                              4)
    bad = torch.tensor([[0, 1, -5, 3]], dtype=torch.int32)
    out, st, _ = decode(cfg, synth.queries(w), pool, bad, lens, tk, tv)
    torch.cuda.synchronize()
    assert int(st.item()) & kv.kvarn.STATUS_BAD_PAGE
    assert torch.isfinite(out.float()).all()


def test_scale_argument():
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=2, seq=400, hkv=2, hq=8)
    lens = torch.tensor([400, 333], dtype=torch.int32)
    table = torch.arange(8, dtype=torch.int32).reshape(2, 4)
    k, v = synth.kv(w, device=DEV)
    cfg = config(w.hq, w.hkv)
    pool, tk, tv, _ = prefill(cfg, k, v, lens, table, 8)
    q = synth.queries(w)
    import quantized_decode_attention_blocks_b300 as kv
    out = torch.empty((2, 8, 128), dtype=torch.float16, device=DEV)
    ws = kv.alloc_decode_workspace(cfg, 2, 400, DEV)
    kv.kvarn_decode_attention(cfg, q.to(DEV), pool, table.to(DEV), lens.to(DEV), 400, tk, tv,
                              out, ws, softmax_scale=0.3)
    torch.cuda.synchronize()
    ref = kvref.decode_attention(host(q), host(pool), host(table), host(lens), host(tk), host(tv),
                                 8, 2, scale=0.3, route=1)
    parity.compare_attention(host(out), ref)


@pytest.mark.parametrize("hq,hkv,fmt", [(4, 1, {}), (12, 2, {}), (4, 1, {"k8": True}),
                                        (8, 2, {"g64": True}), (4, 1, {"v4": True}),
                                        (6, 1, {"m16": True})])
def test_ragged_batch_that_runs_in_several_waves(hq, hkv, fmt):
    # More (sequence, KV head) pairs than resident CTAs: the plan cuts the
    # long sequences into runs of at most 32 pages merged through the
    # workspace (no clusters), while short sequences end in their first run.
    # Whole sequences of every length class are checked against the oracle.
    import quantized_decode_attention_blocks_b300 as kv
    from tests.test_gpu_workloads import _check_sampled_decode
    B = 600 if hkv == 1 else 300
    max_seq = 6000
    g = torch.Generator().manual_seed(97 + hq)
    lens = torch.randint(1, max_seq + 1, (B,), generator=g, dtype=torch.int32)
    lens[:4] = torch.tensor([max_seq, 4096, 129, 0], dtype=torch.int32)
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=B, seq=max_seq, hkv=hkv, hq=hq)
    cfg = config(hq, hkv, **fmt)
    pps, ns, _ = kv.decode_split_plan(cfg, B, max_seq, 0)
    assert ns > 1 and pps <= 32   # the several-waves plan
    mb = (max_seq + 127) // 128
    table = torch.randperm(B * mb, generator=g).to(torch.int32).reshape(B, mb)
    k, v = synth.kv(w, device=DEV)
    pool, tk, tv, st = prefill(cfg, k, v, lens, table, B * mb, max_seq=max_seq)
    del k, v
    q = synth.queries(w)
    out, st2, _ = decode(cfg, q, pool, table, lens, tk, tv, max_seq=max_seq)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(st2.item()) == 0
    seqs = [0, 1, 2, 3] + sorted(torch.randperm(B - 4, generator=g)[:12].add(4).tolist())
    _check_sampled_decode(cfg, q.to(DEV), out, pool, table.to(DEV), lens.to(DEV), tk, tv, seqs,
                          **fmt)
    assert not torch.isnan(out.float()).any()
