"""The C-ABI library: loads, exports every symbol include/kvarn.h declares, and
rejects bad arguments on the host before any launch (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

import quantized_decode_attention_blocks_b300 as kv
from quantized_decode_attention_blocks_b300 import kvarn as K

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvarn.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvarn_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    L = kv.lib()
    names = declared_symbols()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n
    nm = subprocess.run(["nm", "-D", "--defined-only", K.LIB_PATH], capture_output=True,
                        text=True).stdout
    exported = set(re.findall(r" T (kvarn_\w+)", nm))
    assert set(names) <= exported
    assert set(names) == set(K.SIGNATURES)


def test_header_constants_match_binding():
    text = open(HEADER).read()
    for name, val in (("KVARN_PAGE_BYTES", K.PAGE_BYTES),
                      ("KVARN_PAGE_BYTES_M16", K.PAGE_BYTES_M16),
                      ("KVARN_PAGE_BYTES_G64", K.PAGE_BYTES_G64),
                      ("KVARN_PAGE_BYTES_V4", K.PAGE_BYTES_V4),
                      ("KVARN_PAGE_BYTES_K8", K.PAGE_BYTES_K8), ("KVARN_OK", K.OK),
                      ("KVARN_ERR_INVALID_ARG", K.ERR_INVALID_ARG),
                      ("KVARN_ERR_UNSUPPORTED", K.ERR_UNSUPPORTED),
                      ("KVARN_ERR_WORKSPACE", K.ERR_WORKSPACE), ("KVARN_ERR_LAUNCH", K.ERR_LAUNCH),
                      ("KVARN_STATUS_BAD_PAGE", K.STATUS_BAD_PAGE),
                      ("KVARN_STATUS_BAD_LENGTH", K.STATUS_BAD_LENGTH),
                      ("KVARN_STATUS_TIMEOUT", K.STATUS_TIMEOUT)):
        m = re.search(rf"#define {name} \(?(-?\d+)\)?", text)
        assert m and int(m.group(1)) == val, name
    m = re.search(r"#define KVARN_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", text)
    assert m and int(m.group(1)) << int(m.group(2)) == K.NOALLOC_SCRATCH_BYTES


def test_config_parsing():
    c = kv.config_from_string("kvarn_k4v2_g128", 32, 8)
    assert (c.head_dim, c.block_tokens, c.group, c.k_bits, c.v_bits) == (128, 128, 128, 4, 2)
    assert c.sinkhorn_iters == 2 and c.g == 4
    assert kv.config_from_string("k4v2_g128_s7", 12, 2).sinkhorn_iters == 7
    assert c.sinkhorn_rms == 0
    r = kv.config_from_string("kvarn_k4v2_g128_rms_s3", 12, 2)
    assert r.sinkhorn_rms == 1 and r.sinkhorn_iters == 3
    assert kv.config_from_string("k4v2_g128_rms", 12, 2).sinkhorn_iters == 2
    for bad in ("k4v2_g128_s3_rms", "k4v2_g128_rm", "k4v2_g128_rms_"):
        with pytest.raises(kv.KvarnError):
            kv.config_from_string(bad, 12, 2)
    r.sinkhorn_rms = 2
    assert kv.config_validate(r) == K.ERR_UNSUPPORTED
    # the fp16-metadata variant, alone or with "_rms", either order
    assert c.meta_fp16 == 0
    for fmt in ("k4v2_g128_m16", "kvarn_k4v2_g128_m16_s3", "k4v2_g128_rms_m16", "k4v2_g128_m16_rms_s1"):
        m = kv.config_from_string(fmt, 12, 2)
        assert m.meta_fp16 == 1 and m.sinkhorn_rms == ("rms" in fmt)
        assert kv.page_bytes(m) == 13824 == 108 * 128 == m.page_bytes
    for bad in ("k4v2_g128_m16_m16", "k4v2_g128_rms_rms", "k4v2_g128_s2_m16", "k4v2_g128_m8"):
        with pytest.raises(kv.KvarnError):
            kv.config_from_string(bad, 12, 2)
    m.meta_fp16 = 3
    assert kv.config_validate(m) == K.ERR_UNSUPPORTED
    # per-channel groups, alone or with "_rms", any order; never with "_m16"
    for fmt in ("k4v2_g128_pc", "k4v2_g128_rms_pc_s3", "k4v2_g128_pc_rms"):
        p = kv.config_from_string(fmt, 12, 2)
        assert p.per_channel == 1 and p.meta_fp16 == 0 and p.sinkhorn_rms == ("rms" in fmt)
        assert kv.page_bytes(p) == 15360
    for bad in ("k4v2_g128_pc_m16", "k4v2_g128_m16_pc", "k4v2_g128_pcx", "k4v2_g128_pc_pc"):
        with pytest.raises(kv.KvarnError):
            kv.config_from_string(bad, 12, 2)
    p.meta_fp16 = 1
    assert kv.config_validate(p) == K.ERR_UNSUPPORTED
    # groups of 64 channels: "k4v2_g64", with "_rms" but not "_m16" / "_pc"
    g = kv.config_from_string("kvarn_k4v2_g64_rms_s3", 12, 2)
    assert g.group == 64 and g.sinkhorn_rms == 1 and g.sinkhorn_iters == 3
    assert kv.page_bytes(g) == 17408 == 136 * 128 == g.page_bytes
    for bad in ("k4v2_g64_m16", "k4v2_g64_pc", "k4v2_g32"):
        with pytest.raises(kv.KvarnError):
            kv.config_from_string(bad, 12, 2)
    # 4-bit values: "k4v4_g128", with "_rms" but not "_m16" / "_pc"
    v4 = kv.config_from_string("kvarn_k4v4_g128_rms", 12, 2)
    assert v4.v_bits == 4 and v4.group == 128 and v4.sinkhorn_rms == 1
    assert kv.page_bytes(v4) == 19456 == 152 * 128 == v4.page_bytes
    for bad in ("k4v4_g128_m16", "k4v4_g128_pc", "k4v4_g64"):
        with pytest.raises(kv.KvarnError):
            kv.config_from_string(bad, 12, 2)
    # 8-bit keys, 4-bit values: "k8v4_g128", with "_rms" but not "_m16" / "_pc"
    k8 = kv.config_from_string("kvarn_k8v4_g128_rms_s1", 12, 2)
    assert (k8.k_bits, k8.v_bits, k8.group, k8.sinkhorn_rms, k8.sinkhorn_iters) == (8, 4, 128, 1, 1)
    assert kv.page_bytes(k8) == 27648 == 216 * 128 == k8.page_bytes
    for bad in ("k8v4_g128_m16", "k8v4_g128_pc", "k8v4_g64", "k8v2_g128"):
        with pytest.raises(kv.KvarnError):
            kv.config_from_string(bad, 12, 2)
    k8.v_bits = 2
    assert kv.config_validate(k8) == K.ERR_UNSUPPORTED
    for bad in ("k2v2_g128", "k4v2_g96", "k4v2_g128_x", "k4v2_g128_s", "k4v2_g128_s999"):
        with pytest.raises(kv.KvarnError) as e:
            kv.config_from_string(bad, 32, 8)
        assert e.value.code == K.ERR_UNSUPPORTED
    with pytest.raises(kv.KvarnError) as e:
        kv.config_from_string("k4v2_g128", 30, 8)
    assert e.value.code == K.ERR_INVALID_ARG
    with pytest.raises(kv.KvarnError) as e:
        kv.config_from_string("k4v2_g128", 64, 2)        # group of 32 > 16
    assert e.value.code == K.ERR_UNSUPPORTED
    c.head_dim = 64
    assert kv.config_validate(c) == K.ERR_UNSUPPORTED
    assert kv.page_bytes(c) == 0


B300_SMS = 148


def _ws(c, batch, max_seq, sms=B300_SMS):
    return kv.decode_split_plan(c, batch, max_seq, sms)[2]


def test_page_bytes_and_workspace_sizes():
    c = kv.config_from_string("k4v2_g128", 32, 8)
    assert kv.page_bytes(c) == 15360 == 120 * 128
    with pytest.raises(kv.KvarnError):
        kv.decode_split_plan(c, 0, 100, B300_SMS)
    small = _ws(c, 1, 200)
    big = _ws(c, 16, 131072)
    assert big > small >= 0
    assert big % 256 == 0


@pytest.mark.parametrize("sms", [148, 132, 160])
@pytest.mark.parametrize("g", [1, 4, 6, 8, 12])
def test_split_plan_fills_one_wave_and_covers_every_page(sms, g):
    # The plan follows the SM count it is given: it cuts each (sequence, KV
    # head) into at most as many splits as keep the whole grid resident (the
    # tensor-core kernel is planned at 2 CTAs per SM, the CUDA-core one at 3),
    # covers every page, and leaves no split empty.  When the pairs alone
    # outnumber one wave (tensor-core kernel), runs are cut to at most 32
    # pages as far as the partial states fit the no-alloc scratch.
    per_sm = 2 if g <= 8 else 3
    resident = 3 if g <= 4 else 2   # one head tile: three fit an SM
    for hkv in (1, 2, 8):
        c = kv.config_from_string("k4v2_g128", g * hkv, hkv)
        for batch in (1, 3, 16, 48, 64, 1000):
            for max_seq in (100, 128, 4097, 131072):
                pps, ns, ws = kv.decode_split_plan(c, batch, max_seq, sms)
                pages = max(max_seq // 128, 1)
                assert pps * ns >= pages and pps * (ns - 1) < pages
                assert (ws == 0) == (ns == 1)
                if batch * hkv <= sms * resident or g > 8:
                    assert ns == 1 or batch * hkv * ns <= sms * per_sm
                else:
                    assert ws <= K.NOALLOC_SCRATCH_BYTES
                    more = ns + 1   # one more split would pass the scratch
                    assert pps <= 32 or (batch * g * hkv * more * 132 * 4
                                         > K.NOALLOC_SCRATCH_BYTES - 256 - 4 * batch * hkv)


def test_split_plan_of_a_ragged_serving_batch_runs_in_several_waves():
    # 128 sequences of up to 32768 tokens, 8 KV heads: 1024 (sequence, KV
    # head) pairs against 296 resident CTAs.  One CTA per pair would leave the
    # longest sequences straggling; the plan cuts them into runs of about 32
    # pages whose partial states fit the no-alloc scratch.
    c = kv.config_from_string("k4v2_g128", 32, 8)
    pps, ns, ws = kv.decode_split_plan(c, 128, 32768, B300_SMS)
    assert ns > 4 and pps <= 48
    assert 0 < ws <= K.NOALLOC_SCRATCH_BYTES
    # a batch that fills one wave keeps the one-wave plan, also where its
    # pairs fill more than the plan's two CTAs per SM but fit the three that
    # can be resident
    pps, ns, ws = kv.decode_split_plan(c, 16, 4096, B300_SMS)
    assert (pps, ns) == (16, 2)
    assert kv.decode_split_plan(c, 48, 8192, B300_SMS)[:2] == (64, 1)
    assert kv.decode_split_plan(c, 64, 8192, B300_SMS)[:2] == (32, 2)


def test_split_plan_of_8bit_keys_follows_its_shared_memory():
    # the 27648-byte records of "k8v4_g128" leave shared memory for two
    # tensor-core CTAs per SM with one head tile (g <= 4) and one with two,
    # and the plan sizes its wave by that
    for g in (1, 4, 6, 8):
        per_sm = 2 if g <= 4 else 1
        c = kv.config_from_string("k8v4_g128", g * 2, 2)
        for batch in (1, 3, 16):
            pps, ns, ws = kv.decode_split_plan(c, batch, 131072, B300_SMS)
            assert ns > 1 and batch * 2 * ns <= B300_SMS * per_sm
            assert pps * ns >= 1024 and pps * (ns - 1) < 1024


def test_split_plan_grows_with_the_sm_count():
    c = kv.config_from_string("k4v2_g128", 32, 8)
    n = [kv.decode_split_plan(c, 1, 131072, sms)[1] for sms in (74, 148, 296)]
    assert n[0] < n[1] < n[2]


@pytest.mark.parametrize("fmt", ["k4v2_g128_m16", "k4v2_g128_pc", "k4v2_g64", "k4v4_g128",
                                 "k8v4_g128"])
def test_several_wave_plans_of_every_format_fit_the_scratch(fmt):
    # every record format sets its own resident CTAs per SM; a ragged batch
    # of many pairs is cut into short runs, its partial states within the
    # no-alloc scratch
    for g in (1, 4, 6, 8):
        c = kv.config_from_string(fmt, g * 8, 8)
        for batch in (64, 128, 1000):
            for max_seq in (8192, 32768, 131072):
                pps, ns, ws = kv.decode_split_plan(c, batch, max_seq, B300_SMS)
                pages = max_seq // 128
                assert pps * ns >= pages and pps * (ns - 1) < pages
                assert ws <= K.NOALLOC_SCRATCH_BYTES


@pytest.mark.parametrize("g", [1, 2, 4, 6, 8, 12, 16])
def test_noalloc_scratch_covers_every_group_up_to_sixteen(g):
    # a plan of one wave, or one of several waves sized to the scratch: the
    # partial states of every (batch, length) with at most 16 query heads per
    # KV head fit in the built-in scratch of the no-alloc decode on a B300 (a
    # host-only computation)
    for hkv in (1, 2, 8, 32):
        c = kv.config_from_string("k4v2_g128", g * hkv, hkv)
        for batch in (1, 3, 64, 1000, 65535):
            for max_seq in (128, 4097, 131072, 1 << 22):
                need = _ws(c, batch, max_seq)
                assert need <= K.NOALLOC_SCRATCH_BYTES, (g, hkv, batch, max_seq, need)


def test_no_workspace_when_the_batch_fills_the_gpu():
    # enough (sequence, KV head) pairs for one CTA each: no split, no partials
    c = kv.config_from_string("k4v2_g128", 32, 8)
    assert _ws(c, 4096, 32768) == 0


def test_status_strings():
    for code in (0, -1, -2, -3, -4, 1, 2, 4, 3, -99):
        s = kv.status_string(code)
        assert isinstance(s, str) and s
    assert kv.version().count(".") == 2


def _cfg():
    return kv.config_from_string("k4v2_g128", 8, 2)


def test_host_validation_quantize():
    L = kv.lib()
    c = _cfg()
    P = ctypes.c_void_p
    a16 = P(4096)          # fake aligned addresses: validation must fail before any use
    mis = P(4098)
    call = lambda **kw: L.kvarn_quantize_blocks(
        ctypes.byref(kw.get("cfg", c)), kw.get("k", a16), kw.get("v", a16),
        kw.get("sb", 128 * 2 * 256), kw.get("st", 256), kw.get("sh", 128), kw.get("batch", 1),
        kw.get("lens", a16), kw.get("max_seq", 256), kw.get("table", a16),
        kw.get("max_blocks", 2), kw.get("pool", a16), kw.get("num_pages", 2),
        kw.get("tk", a16), kw.get("tv", a16), None, None)
    assert call(k=None) == K.ERR_INVALID_ARG
    assert call(lens=None) == K.ERR_INVALID_ARG
    assert call(k=mis) == K.ERR_INVALID_ARG
    assert call(st=100) == K.ERR_INVALID_ARG          # not a multiple of 8
    assert call(sh=4) == K.ERR_INVALID_ARG
    assert call(max_blocks=1) == K.ERR_INVALID_ARG    # 256 tokens need 2 blocks
    assert call(batch=-1) == K.ERR_INVALID_ARG
    assert call(pool=None) == K.ERR_INVALID_ARG
    assert call(batch=0, k=None) == K.OK              # nothing to do
    bad = _cfg()
    bad.k_bits = 8
    assert call(cfg=bad) == K.ERR_UNSUPPORTED


def test_host_validation_append_and_decode():
    L = kv.lib()
    c = _cfg()
    P = ctypes.c_void_p
    a16 = P(4096)
    assert L.kvarn_append_token(ctypes.byref(c), None, a16, a16, 1, a16, 2, a16, 2, a16, a16,
                                None, None) == K.ERR_INVALID_ARG
    assert L.kvarn_append_token(ctypes.byref(c), a16, a16, a16, 1, a16, 0, a16, 2, a16, a16,
                                None, None) == K.ERR_INVALID_ARG
    dec = lambda **kw: L.kvarn_decode_attention(
        ctypes.byref(c), kw.get("q", a16), a16, 4, a16, 4, a16, kw.get("batch", 2),
        kw.get("max_seq", 512), a16, a16, kw.get("scale", 0.088), kw.get("out", a16),
        kw.get("ws", None), kw.get("ws_bytes", 0), None, None)
    assert dec(q=None) == K.ERR_INVALID_ARG
    assert dec(out=P(4097)) == K.ERR_INVALID_ARG
    assert dec(scale=0.0) == K.ERR_INVALID_ARG
    assert dec(scale=float("nan")) == K.ERR_INVALID_ARG
    if torch.cuda.is_available():
        need = kv.decode_workspace_bytes(c, 2, 512)
        if need:
            assert dec() == K.ERR_WORKSPACE
            assert dec(ws=a16, ws_bytes=need - 1) == K.ERR_WORKSPACE
    else:
        # the split plan needs the device's SM count: with no device the call
        # fails before anything could launch
        assert kv.decode_workspace_bytes(c, 2, 512) == 0
        assert dec() == K.ERR_LAUNCH
    assert dec(batch=0) == K.OK
    assert L.kvarn_dequantize_pages(a16, -1, a16, a16, None) == K.ERR_INVALID_ARG
    assert L.kvarn_dequantize_pages(None, 3, a16, a16, None) == K.ERR_INVALID_ARG
    k8 = kv.config_from_string("k8v4_g128", 8, 2)
    assert L.kvarn_dequantize_records(ctypes.byref(k8), a16, -1, a16, a16, None) == K.ERR_INVALID_ARG
    assert L.kvarn_dequantize_records(ctypes.byref(k8), None, 3, a16, a16, None) == K.ERR_INVALID_ARG
    assert L.kvarn_dequantize_records(ctypes.byref(k8), a16, 0, a16, a16, None) == K.OK
    k8.k_bits = 6
    assert L.kvarn_dequantize_records(ctypes.byref(k8), a16, 3, a16, a16, None) == K.ERR_UNSUPPORTED
    assert L.kvarn_dequantize_records(None, a16, 3, a16, a16, None) == K.ERR_INVALID_ARG
    # the bounded-wait check: arguments refused before any launch
    assert L.kvarn_wait_check(None, 0, 1000, None) == K.ERR_INVALID_ARG
    assert L.kvarn_wait_check(a16, 2, 1000, None) == K.ERR_INVALID_ARG
    assert L.kvarn_wait_check(a16, 0, 0, None) == K.ERR_INVALID_ARG
    assert L.kvarn_wait_check(a16, 0, 1000001, None) == K.ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors():
    c = _cfg()
    k = torch.zeros((1, 128, 2, 128), dtype=torch.float16)
    with pytest.raises(ValueError):
        kv.kvarn_quantize_blocks(c, k, k, torch.zeros(1, dtype=torch.int32), 128,
                                 torch.zeros((1, 1), dtype=torch.int32),
                                 torch.zeros((1, 2, 15360), dtype=torch.uint8), k, k)


def test_host_validation_fp16_cache():
    # the FP16-cache baseline's calls check their arguments on the host too;
    # every call here is invalid, so none reaches a launch
    L = kv.lib()
    P = ctypes.c_void_p
    a16, mis = P(4096), P(4100)
    wr = lambda **kw: L.kvarn_fp16_write_blocks(
        kw.get("k", a16), kw.get("v", a16), kw.get("sb", 256 * 2 * 128), kw.get("st", 256),
        kw.get("sh", 128), kw.get("batch", 1), kw.get("hkv", 2), kw.get("lens", a16),
        kw.get("max_seq", 256), kw.get("table", a16), kw.get("max_blocks", 2),
        kw.get("pool", a16), kw.get("num_pages", 2), None, None)
    assert wr(k=None) == K.ERR_INVALID_ARG
    assert wr(v=mis) == K.ERR_INVALID_ARG
    assert wr(hkv=0) == K.ERR_INVALID_ARG
    assert wr(st=100) == K.ERR_INVALID_ARG            # not a multiple of 8 elements
    assert wr(max_blocks=1) == K.ERR_INVALID_ARG      # 256 tokens need 2 pages
    assert wr(num_pages=0) == K.ERR_INVALID_ARG
    assert wr(batch=0, k=None) == K.OK                # nothing to do
    dec = lambda **kw: L.kvarn_fp16_decode_attention(
        kw.get("q", a16), kw.get("hq", 8), kw.get("hkv", 2), kw.get("pool", a16), 40, a16,
        kw.get("max_blocks", 40), a16, kw.get("batch", 1), kw.get("max_seq", 5000),
        kw.get("scale", 0.088), kw.get("out", a16), kw.get("ws", None),
        kw.get("ws_bytes", 0), None, None)
    assert dec(hq=7) == K.ERR_INVALID_ARG             # not a multiple of hkv
    assert dec(hq=18) == K.ERR_UNSUPPORTED            # groups above 8
    assert dec(q=None) == K.ERR_INVALID_ARG
    assert dec(out=mis) == K.ERR_INVALID_ARG
    assert dec(max_blocks=39) == K.ERR_INVALID_ARG    # 5000 tokens need 40 pages
    assert dec(scale=-1.0) == K.ERR_INVALID_ARG
    if torch.cuda.is_available():
        need = kv.fp16_decode_workspace_bytes(8, 2, 1, 5000)
        assert need > 0                               # one long sequence is split
        assert dec() == K.ERR_WORKSPACE
        assert dec(ws=a16, ws_bytes=need - 1) == K.ERR_WORKSPACE
    else:
        assert kv.fp16_decode_workspace_bytes(8, 2, 1, 5000) == 0
        assert dec() == K.ERR_LAUNCH                  # no device to plan for
    assert dec(batch=0) == K.OK
    assert kv.fp16_decode_workspace_bytes(8, 3, 1, 5000) == 0      # bad group


def test_host_validation_snapkv():
    # SnapKV-style selection and gather: every call here is invalid (or has
    # nothing to do), so none reaches a launch
    L = kv.lib()
    c = _cfg()
    P = ctypes.c_void_p
    a16, mis = P(4096), P(4100)
    ws = kv.snapkv_workspace_bytes(c, 2, 32, 5000)
    # statistics: 2 x 2 heads x 2 row tiles (32 x 4 rows) x 3 chunks x 1 KB,
    # pooled votes: 2 x 2 x 5000 floats
    assert ws == 2 * 2 * 1 * 3 * 1024 + ((2 * 2 * 5000 * 4 + 255) & ~255)
    assert kv.snapkv_workspace_bytes(c, 0, 32, 5000) == 0
    sel = lambda **kw: L.kvarn_snapkv_select(
        ctypes.byref(c), kw.get("q", a16), kw.get("W", 32), kw.get("k", a16), 5000 * 256, 256,
        128, kw.get("lens", a16), kw.get("batch", 2), 5000, kw.get("cap", 1024),
        kw.get("kern", 7), kw.get("scale", 0.088), kw.get("votes", a16), kw.get("idx", a16),
        kw.get("ws", a16), kw.get("ws_bytes", ws), None, None)
    assert sel(q=None) == K.ERR_INVALID_ARG
    assert sel(k=mis) == K.ERR_INVALID_ARG
    assert sel(votes=P(4098)) == K.ERR_INVALID_ARG
    assert sel(W=0) == K.ERR_INVALID_ARG
    assert sel(cap=31) == K.ERR_INVALID_ARG           # smaller than the window
    assert sel(kern=4) == K.ERR_INVALID_ARG           # even pooling width
    assert sel(scale=0.0) == K.ERR_INVALID_ARG
    assert sel(ws_bytes=ws - 1) == K.ERR_WORKSPACE
    assert sel(batch=0, q=None) == K.OK
    gat = lambda **kw: L.kvarn_snapkv_gather(
        kw.get("k", a16), a16, 5000 * 256, kw.get("st", 256), 128, 2, 5000, kw.get("hkv", 2),
        a16, kw.get("cap", 1024), kw.get("ko", a16), a16, None)
    assert gat(k=None) == K.ERR_INVALID_ARG
    assert gat(ko=mis) == K.ERR_INVALID_ARG
    assert gat(st=100) == K.ERR_INVALID_ARG
    assert gat(hkv=0) == K.ERR_INVALID_ARG
    assert gat(cap=0, k=None) == K.OK
