"""Quantization on the GPU against the float64 oracle (tile by tile).

KVarN page (blog.edumints.com), "KVarN Nasil Calisir?": rotation, log-domain
Sinkhorn-like normalization and asymmetric RTN with 4-bit K / 2-bit V.
"""
import numpy as np
import pytest
import torch

from oracle import kvref
from tests import parity
from tests.gpu_helpers import DEV, bits16, config, host, prefill
from workloads import synth

pytestmark = pytest.mark.gpu


def _check_prefill(w, lens, table, num_pages, iters=2, k=None, v=None, rms=False, m16=False,
                   pc=False, g64=False, v4=False, k8=False):
    if k is None:
        k, v = synth.kv(w, device=DEV)
    cfg = config(w.hq, w.hkv, iters, rms=rms, m16=m16, pc=pc, g64=g64, v4=v4, k8=k8)
    pool, tk, tv, status = prefill(cfg, k, v, lens, table, num_pages, max_seq=w.seq)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    kh, vh = host(k), host(v)
    ref = kvref.quantize_blocks(kh, vh, host(lens), host(table), num_pages, iters, want_u=True,
                                rms=rms, meta16=m16, pc=pc, g64=g64, v4=v4, k8=k8)
    ref32 = (kvref.quantize_blocks(kh, vh, host(lens), host(table), num_pages, iters, rms=rms)
             if m16 else None)
    got_pool = host(pool)
    stats = {}
    nfull = host(lens) // 128
    for b in range(w.batch):
        for j in range(int(nfull[b])):
            page = int(table[b, j])
            for h in range(w.hkv):
                parity.compare_record(got_pool[page, h], ref["pool"][page, h],
                                      ref["u_k"][b, j, h], ref["u_v"][b, j, h], stats, meta16=m16,
                                      ref32=ref32["pool"][page, h] if m16 else None, pc=pc,
                                      g64=g64, v4=v4, k8=k8)
    parity.check_flip_rate(stats)
    _check_prefill.last = (pool, tk, tv, cfg)
    # leftover tokens copied verbatim into the tails
    for b in range(w.batch):
        rem = int(host(lens)[b]) % 128
        assert np.array_equal(bits16(tk)[b, :, :rem], ref["tail_k"][b, :, :rem])
        assert np.array_equal(bits16(tv)[b, :, :rem], ref["tail_v"][b, :, :rem])
    return stats


def test_tiny_workload():
    w = synth.WORKLOADS["tiny"]
    lens = synth.seq_lens(w)
    tables, n = synth.block_tables(w)
    _check_prefill(w, lens, tables[0], n)


def test_ragged_lengths_permuted_pages():
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=4, seq=1000)
    lens = torch.tensor([1000, 128, 517, 0], dtype=torch.int32)
    g = torch.Generator().manual_seed(5)
    table = torch.randperm(4 * 8, generator=g).to(torch.int32).reshape(4, 8)
    stats = _check_prefill(w, lens, table, 32)
    assert stats["k_codes"] == (7 + 1 + 4) * 8 * 128 * 128


@pytest.mark.parametrize("iters", [0, 1, 4])
def test_other_iteration_counts(iters):
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=1, seq=384, hkv=2, hq=8)
    lens = torch.tensor([384], dtype=torch.int32)
    table = torch.tensor([[2, 0, 1]], dtype=torch.int32)
    _check_prefill(w, lens, table, 3, iters=iters)


@pytest.mark.parametrize("iters", [1, 2, 4])
def test_rms_variant(iters):
    # format variant "_rms" (uncentred Sinkhorn statistic): same record, the
    # scales and codes of the oracle's variant; then decode reads it
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=3, seq=700, hkv=2, hq=8)
    lens = torch.tensor([700, 256, 300], dtype=torch.int32)
    g = torch.Generator().manual_seed(9)
    table = torch.randperm(3 * 6, generator=g).to(torch.int32).reshape(3, 6)
    _check_prefill(w, lens, table, 18, iters=iters, rms=True)
    pool, tk, tv, cfg = _check_prefill.last
    assert cfg.sinkhorn_rms == 1 and cfg.sinkhorn_iters == iters
    from tests.gpu_helpers import decode
    q = synth.queries(w)
    out, st, _ = decode(cfg, q, pool, table, lens, tk, tv)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = kvref.decode_attention(host(q), host(pool), host(table), host(lens), host(tk),
                                 host(tv), w.hq, w.hkv)
    parity.compare_attention(host(out), ref)


@pytest.mark.parametrize("variant", ["f32", "g64", "k8"])
def test_strided_input(variant):
    # K/V as views into a [B][S][2*Hkv][128] buffer (every other head), and a
    # batch stride larger than S*Hkv*128
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=2, seq=256, hkv=4, hq=8)
    kf, vf = synth.kv(synth.scaled(w, hkv=8), device=DEV)
    big_k = torch.zeros((2, 300, 8, 128), dtype=torch.float16, device=DEV)
    big_v = torch.zeros_like(big_k)
    big_k[:, :256] = kf
    big_v[:, :256] = vf
    k = big_k[:, :256, ::2]
    v = big_v[:, :256, ::2]
    lens = torch.tensor([256, 200], dtype=torch.int32)
    table = torch.tensor([[0, 1], [2, 3]], dtype=torch.int32)
    _check_prefill(w, lens, table, 4, k=k, v=v, **({} if variant == "f32" else {variant: True}))


@pytest.mark.parametrize("variant", ["f32", "m16", "pc", "g64", "v4", "k8"])
def test_special_tiles(variant):
    # zero tile, constant tile, a huge random-sign outlier channel, fp16
    # extremes, in every record format
    fmt = {} if variant == "f32" else {variant: True}
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=1, seq=512, hkv=1, hq=1)
    k, v = synth.kv(w, device=DEV)
    k[0, :128] = 0
    v[0, :128] = 0
    k[0, 128:256] = 1.5
    v[0, 128:256, :, 7] = -3.0
    sign = torch.where(k[0, 256:384, 0, 5] > 0, 1.0, -1.0)
    k[0, 256:384, 0, 5] = (60000.0 * sign).half()
    v[0, 384:512] = torch.where(v[0, 384:512] > 0, 65504.0, -65504.0).half()
    lens = torch.tensor([512], dtype=torch.int32)
    table = torch.tensor([[3, 2, 1, 0]], dtype=torch.int32)
    _check_prefill(w, lens, table, 4, k=k, v=v, **fmt)


def test_ill_conditioned_constant_offset_tile():
    """A channel holding the same huge value in every token makes every rotated
    column a large constant plus small variation (|mean|/std ~ 5e2 here).  fp32
    holds each rotated value only to 2^-24 of the offset, so a column std can
    only be known to about 2^-24 |mean|/std relative: the bound below is that
    conditioning limit (with a 64x margin for the accumulation), not the 1e-5
    rule.  End to end, decode attention over this page still meets the
    attention tolerance."""
    import quantized_decode_attention_blocks_b300 as kv
    from tests.gpu_helpers import decode
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=1, seq=256, hkv=1, hq=4)
    k, v = synth.kv(w, device=DEV)
    k[0, :128, 0, 5] = 60000.0
    cfg = config(w.hq, w.hkv)
    lens = torch.tensor([256], dtype=torch.int32)
    table = torch.tensor([[1, 0]], dtype=torch.int32)
    pool, tk, tv, st = prefill(cfg, k, v, lens, table, 2)
    torch.cuda.synchronize()
    tile = host(k)[0, :128, 0]
    ref = kvref.quantize_tile(tile, False, 2)
    a, b = ref["a"], ref["b"]
    Z = ref["Y"] * np.exp(-a)[:, None]
    kappa = np.abs(Z.mean(0)) / Z.std(0)
    _, _, _, cg = kvref.unpack_part(host(pool)[1, 0], False)
    cr = np.exp(b)
    rel = np.abs(cg - cr) / cr
    assert np.all(rel <= 1e-5 + 64 * 2.0 ** -24 * kappa), rel.max()
    assert kappa.max() > 100          # the tile is as ill-conditioned as intended
    q = synth.queries(w)
    out, st2, _ = decode(cfg, q, pool, table, lens, tk, tv)
    torch.cuda.synchronize()
    refo = kvref.decode_attention(host(q), host(pool), host(table), host(lens), host(tk),
                                  host(tv), w.hq, w.hkv, route=1)
    parity.compare_attention(host(out), refo)


def test_dequantize_pages_matches_oracle():
    import quantized_decode_attention_blocks_b300 as kv
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=1, seq=256, hkv=2, hq=8)
    k, v = synth.kv(w, device=DEV)
    cfg = config(w.hq, w.hkv)
    pool, _, _, _ = prefill(cfg, k, v, torch.tensor([256], dtype=torch.int32),
                            torch.tensor([[0, 1]], dtype=torch.int32), 2)
    yk, yv = kv.kvarn_dequantize_pages(pool.reshape(-1, 15360))
    torch.cuda.synchronize()
    recs = host(pool).reshape(-1, 15360)
    for i in range(recs.shape[0]):
        for is_v, y in ((False, yk), (True, yv)):
            ref = kvref.dequant_part(recs[i], is_v)
            got = host(y[i]).astype(np.float64)
            assert np.all(np.abs(got - ref) <= 1e-6 * np.abs(ref) + 1e-30)


@pytest.mark.parametrize("variant", ["f32", "m16", "pc", "g64", "v4", "k8"])
def test_dequantize_records_of_every_format_match_oracle(variant):
    # kvarn_dequantize_records against the oracle's dequantization of the same
    # records, for each record format; the tolerance is relative to the
    # largest value of the element's row and column (the two terms of yhat can
    # cancel)
    import quantized_decode_attention_blocks_b300 as kv
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=1, seq=256, hkv=2, hq=8)
    k, v = synth.kv(w, device=DEV)
    fmt = {} if variant == "f32" else {variant: True}
    cfg = config(w.hq, w.hkv, **fmt)
    pool, _, _, _ = prefill(cfg, k, v, torch.tensor([256], dtype=torch.int32),
                            torch.tensor([[0, 1]], dtype=torch.int32), 2)
    nb = cfg.page_bytes
    yk, yv = kv.kvarn_dequantize_records(cfg, pool.reshape(-1, nb))
    torch.cuda.synchronize()
    recs = host(pool).reshape(-1, nb)
    okw = {} if variant == "f32" else {("meta16" if variant == "m16" else variant): True}
    for i in range(recs.shape[0]):
        for is_v, y in ((False, yk), (True, yv)):
            ref = kvref.dequant_part(recs[i], is_v, **okw)
            got = host(y[i]).astype(np.float64)
            a = np.abs(ref)
            scale = np.maximum(a.max(axis=1, keepdims=True), a.max(axis=0, keepdims=True))
            assert np.all(np.abs(got - ref) <= 2e-6 * (a + scale)), (variant, is_v, i)


def test_bad_page_sets_status_and_skips():
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=2, seq=256, hkv=2, hq=8)
    k, v = synth.kv(w, device=DEV)
    cfg = config(w.hq, w.hkv)
    table = torch.tensor([[0, 1], [2, 99]], dtype=torch.int32)   # 99 outside a 4-page pool
    lens = torch.tensor([256, 256], dtype=torch.int32)
    pool, _, _, status = prefill(cfg, k, v, lens, table, 4)
    torch.cuda.synchronize()
    assert int(status.item()) & 1          # KVARN_STATUS_BAD_PAGE
    assert not host(pool)[3].any()         # nothing written for the bad block
    # a length beyond max_seq is reported too
    pool, _, _, status = prefill(cfg, k, v, torch.tensor([256, 300], dtype=torch.int32),
                                 torch.tensor([[0, 1], [2, 3]], dtype=torch.int32), 4,
                                 max_seq=256)
    torch.cuda.synchronize()
    assert int(status.item()) & 2          # KVARN_STATUS_BAD_LENGTH


@pytest.mark.parametrize("rms", [False, True])
def test_m16_variant(rms):
    # format variant "_m16" (fp16 metadata, 13824-byte records): the same
    # codes as the fp32 format, the metadata rounded once more to fp16; ragged
    # lengths on permuted pages
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=3, seq=1100, hkv=2, hq=8)
    lens = torch.tensor([1100, 300, 640], dtype=torch.int32)
    g = torch.Generator().manual_seed(71)
    table = torch.randperm(3 * 9, generator=g).to(torch.int32).reshape(3, 9)
    stats = _check_prefill(w, lens, table, 27, rms=rms, m16=True)
    assert stats["k_codes"] == (8 + 2 + 5) * 2 * 128 * 128
    pool = _check_prefill.last[0]
    assert pool.shape[-1] == 13824


@pytest.mark.parametrize("rms,iters", [(False, 2), (True, 2), (False, 0)])
def test_pc_variant(rms, iters):
    # format variant "_pc" (per-channel RTN groups, r_t stored per token):
    # ragged lengths on permuted pages, the special tiles included
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=3, seq=1100, hkv=2, hq=8)
    k, v = synth.kv(w, device=DEV)
    k[0, :128, 0] = 0                       # a zero tile
    v[1, :128, 1] = 1.5                     # a constant tile
    k[2, 300, 1, 7] = 30000.0               # a single outlier
    lens = torch.tensor([1100, 300, 640], dtype=torch.int32)
    g = torch.Generator().manual_seed(73)
    table = torch.randperm(3 * 9, generator=g).to(torch.int32).reshape(3, 9)
    _check_prefill(w, lens, table, 27, iters=iters, k=k, v=v, rms=rms, pc=True)


@pytest.mark.parametrize("rms,iters", [(False, 2), (True, 2), (False, 0)])
def test_g64_variant(rms, iters):
    # format variant "k4v2_g64" (two RTN groups per token): ragged lengths on
    # permuted pages, the special tiles included
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=3, seq=1100, hkv=2, hq=8)
    k, v = synth.kv(w, device=DEV)
    k[0, :128, 0] = 0                       # a zero tile
    v[1, :128, 1] = 1.5                     # a constant tile
    k[2, 300, 1, 7] = 30000.0               # a single outlier
    lens = torch.tensor([1100, 300, 640], dtype=torch.int32)
    g = torch.Generator().manual_seed(74)
    table = torch.randperm(3 * 9, generator=g).to(torch.int32).reshape(3, 9)
    _check_prefill(w, lens, table, 27, iters=iters, k=k, v=v, rms=rms, g64=True)
    assert _check_prefill.last[0].shape[-1] == 17408


@pytest.mark.parametrize("rms,iters", [(False, 2), (True, 2), (False, 0)])
def test_v4_variant(rms, iters):
    # format variant "k4v4_g128" (4-bit values): ragged lengths on permuted
    # pages, the special tiles included
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=3, seq=1100, hkv=2, hq=8)
    k, v = synth.kv(w, device=DEV)
    k[0, :128, 0] = 0                       # a zero tile
    v[1, :128, 1] = 1.5                     # a constant tile
    v[2, 300, 1, 7] = 30000.0               # a single outlier (in V)
    lens = torch.tensor([1100, 300, 640], dtype=torch.int32)
    g = torch.Generator().manual_seed(75)
    table = torch.randperm(3 * 9, generator=g).to(torch.int32).reshape(3, 9)
    _check_prefill(w, lens, table, 27, iters=iters, k=k, v=v, rms=rms, v4=True)
    assert _check_prefill.last[0].shape[-1] == 19456


@pytest.mark.parametrize("rms,iters", [(False, 2), (True, 2), (False, 0)])
def test_k8_variant(rms, iters):
    # format variant "k8v4_g128" (8-bit keys, 4-bit values): ragged lengths on
    # permuted pages, the special tiles included
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=3, seq=1100, hkv=2, hq=8)
    k, v = synth.kv(w, device=DEV)
    k[0, :128, 0] = 0                       # a zero tile
    v[1, :128, 1] = 1.5                     # a constant tile
    k[2, 300, 1, 7] = 30000.0               # a single outlier (in K)
    lens = torch.tensor([1100, 300, 640], dtype=torch.int32)
    g = torch.Generator().manual_seed(76)
    table = torch.randperm(3 * 9, generator=g).to(torch.int32).reshape(3, 9)
    stats = _check_prefill(w, lens, table, 27, iters=iters, k=k, v=v, rms=rms, k8=True)
    assert _check_prefill.last[0].shape[-1] == 27648
    print(f"k8 boundary flips: {stats['k_flips']} of {stats['k_codes']} K codes, "
          f"widest {stats.get('k_flip_dist', 0.0):.2e} from a boundary")
