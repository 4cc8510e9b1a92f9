"""Argument checks of the Python binding, on the CPU.

The C ABI addresses every buffer from its base pointer with a fixed layout
(include/kvarn.h), so the binding must refuse a tensor whose dtype, shape,
contiguity or device does not fit that layout before anything is launched.
Here the library is replaced by a recorder and the CUDA-device requirement is
lifted, so the checks run on CPU tensors: a valid call reaches the recorder
with the sizes the ABI expects, an invalid one raises and reaches nothing.
"""
import pytest
import torch

import quantized_decode_attention_blocks_b300 as kv
from quantized_decode_attention_blocks_b300 import kvarn as K

B, S, HKV, HQ, MB, PAGES = 2, 300, 2, 8, 3, 6


class _Recorder:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def fn(*args):
            self.calls.append((name, args))
            return K.OK
        return fn


class _Stream:
    cuda_stream = 0


@pytest.fixture
def rec(monkeypatch):
    cfg = kv.config_from_string("k4v2_g128", HQ, HKV)   # the real library, host-only call
    r = _Recorder()
    monkeypatch.setattr(K, "_REQUIRE_CUDA", False)
    monkeypatch.setattr(K, "lib", lambda: r)
    r.cfg = cfg
    return r


def _prefill_args():
    k = torch.zeros((B, S, HKV, 128), dtype=torch.float16)
    return dict(k=k, v=torch.zeros_like(k), seq_lens=torch.tensor([300, 255], dtype=torch.int32),
                max_seq=301, block_table=torch.zeros((B, MB), dtype=torch.int32),
                pool=torch.zeros((PAGES, HKV, K.PAGE_BYTES), dtype=torch.uint8),
                tail_k=torch.zeros((B, HKV, 128, 128), dtype=torch.float16),
                tail_v=torch.zeros((B, HKV, 128, 128), dtype=torch.float16),
                status=torch.zeros(1, dtype=torch.int32), stream=_Stream())


def _decode_args():
    a = _prefill_args()
    for name in ("k", "v"):
        del a[name]
    a["q"] = torch.zeros((B, HQ, 128), dtype=torch.float16)
    a["out"] = torch.zeros((B, HQ, 128), dtype=torch.float16)
    a["workspace"] = torch.zeros(1024, dtype=torch.uint8)
    return a


def _append_args():
    a = _prefill_args()
    for name in ("k", "v", "max_seq", "seq_lens"):
        del a[name]
    a["k_new"] = torch.zeros((B, HKV, 128), dtype=torch.float16)
    a["v_new"] = torch.zeros((B, HKV, 128), dtype=torch.float16)
    a["pos"] = torch.tensor([300, 255], dtype=torch.int32)
    return a


def test_valid_calls_reach_the_library_with_the_abi_sizes(rec):
    kv.kvarn_quantize_blocks(rec.cfg, **_prefill_args())
    name, args = rec.calls[-1]
    assert name == "kvarn_quantize_blocks"
    # strides in elements, batch, max_seq, max_blocks, num_pages
    assert args[3:7] == (S * HKV * 128, HKV * 128, 128, B)
    assert args[8] == 301 and args[10] == MB and args[12] == PAGES

    kv.kvarn_append_token(rec.cfg, **_append_args())
    name, args = rec.calls[-1]
    assert name == "kvarn_append_token" and args[4] == B and args[6] == MB and args[8] == PAGES

    kv.kvarn_decode_attention(rec.cfg, **_decode_args())
    name, args = rec.calls[-1]
    assert name == "kvarn_decode_attention"
    assert args[3] == PAGES and args[5] == MB and args[7] == B and args[8] == 301
    assert args[14] == 1024                      # workspace bytes

    a = _decode_args()
    del a["workspace"]
    kv.kvarn_decode_attention_noalloc(rec.cfg, **a)
    assert rec.calls[-1][0] == "kvarn_decode_attention_noalloc"

    kv.kvarn_dequantize_pages(torch.zeros((5, K.PAGE_BYTES), dtype=torch.uint8), stream=_Stream())
    assert rec.calls[-1][0] == "kvarn_dequantize_pages" and rec.calls[-1][1][1] == 5


def test_valid_edge_forms_are_accepted(rec):
    # max_seq above the prefill allocation (the device lengths stay within it),
    # longer lengths/table/tails than the batch, no status, no workspace,
    # k and v as strided views with a dense last dim
    a = _prefill_args()
    a["max_seq"] = 5000
    a["seq_lens"] = torch.zeros(B + 3, dtype=torch.int32)
    a["block_table"] = torch.zeros((B + 1, 40), dtype=torch.int32)
    a["status"] = None
    big = torch.zeros((B, S, 2 * HKV, 128), dtype=torch.float16)
    a["k"], a["v"] = big[:, :, :HKV], big[:, :, HKV:]
    kv.kvarn_quantize_blocks(rec.cfg, **a)
    assert rec.calls[-1][1][3:6] == (S * 2 * HKV * 128, 2 * HKV * 128, 128)
    d = _decode_args()
    d["workspace"] = None
    d["tail_k"] = torch.zeros((B + 2, HKV, 128, 128), dtype=torch.float16)
    d["tail_v"] = torch.zeros((B + 2, HKV, 128, 128), dtype=torch.float16)
    kv.kvarn_decode_attention(rec.cfg, **d)
    assert rec.calls[-1][1][14] == 0


def _variants():
    """(entry point, argument builder, argument to replace, bad value, why)."""
    i32, i64 = torch.int32, torch.int64
    p = _prefill_args
    d = _decode_args
    ap = _append_args
    return [
        ("q", d, "seq_lens", torch.zeros(B, dtype=i64), "int64 lengths"),
        ("q", d, "seq_lens", torch.zeros(B - 1, dtype=i32), "fewer lengths than sequences"),
        ("q", d, "block_table", torch.zeros((B, MB), dtype=i64), "int64 table"),
        ("q", d, "block_table", torch.zeros((MB, B), dtype=i32).t(), "transposed table"),
        ("q", d, "block_table", torch.zeros(MB, dtype=i32), "1-D table"),
        ("q", d, "block_table", torch.zeros((B - 1, MB), dtype=i32), "too few table rows"),
        ("q", d, "pool", torch.zeros((PAGES, HKV + 1, K.PAGE_BYTES), dtype=torch.uint8),
         "pool with other KV heads"),
        ("q", d, "pool", torch.zeros((PAGES, HKV, K.PAGE_BYTES - 16), dtype=torch.uint8),
         "pool pages of another size"),
        ("q", d, "pool", torch.zeros((PAGES, HKV, K.PAGE_BYTES // 2), dtype=torch.int16),
         "int16 pool"),
        ("q", d, "tail_k", torch.zeros((B, HKV, 128, 64), dtype=torch.float16), "tail shape"),
        ("q", d, "tail_v", torch.zeros((B, HKV, 128, 128), dtype=torch.float32), "fp32 tail"),
        ("q", d, "tail_k", torch.zeros((B - 1, HKV, 128, 128), dtype=torch.float16),
         "too few tail rows"),
        ("q", d, "out", torch.zeros((B, HQ, 64), dtype=torch.float16), "out shape"),
        ("q", d, "out", torch.zeros((B, HQ, 128), dtype=torch.float32), "fp32 out"),
        ("q", d, "q", torch.zeros((B, HQ // 2, 128), dtype=torch.float16), "q with other heads"),
        ("q", d, "q", torch.zeros((128, HQ, B), dtype=torch.float16).transpose(0, 2),
         "non-contiguous q"),
        ("q", d, "status", torch.zeros(1, dtype=i64), "int64 status"),
        ("q", d, "status", torch.zeros(0, dtype=i32), "empty status"),
        ("q", d, "workspace", torch.zeros(16, dtype=torch.uint8, device="meta"),
         "workspace on another device"),
        ("q", d, "seq_lens", [300, 255], "a list for lengths"),
        ("k", p, "k", torch.zeros((B, S, HKV + 1, 128), dtype=torch.float16), "k heads"),
        ("k", p, "v", torch.zeros((B, S + 1, HKV, 128), dtype=torch.float16), "v shape"),
        ("k", p, "k", torch.zeros((B, S, HKV, 256), dtype=torch.float16)[..., ::2],
         "strided last dim"),
        ("k", p, "pool", torch.zeros((PAGES, HKV, K.PAGE_BYTES), dtype=torch.uint8,
                                     device="meta"), "pool on another device"),
        ("k_new", ap, "k_new", torch.zeros((B, HKV, 64), dtype=torch.float16), "k_new shape"),
        ("k_new", ap, "v_new", torch.zeros((B + 1, HKV, 128), dtype=torch.float16),
         "v_new rows"),
        ("k_new", ap, "pos", torch.zeros(B, dtype=i64), "int64 positions"),
    ]


@pytest.mark.parametrize("case", range(len(_variants())))
def test_invalid_arguments_are_refused_before_the_library(rec, case):
    first, build, name, bad, why = _variants()[case]
    a = build()
    a[name] = bad
    call = {"q": kv.kvarn_decode_attention, "k": kv.kvarn_quantize_blocks,
            "k_new": kv.kvarn_append_token}[first]
    with pytest.raises((ValueError, TypeError)):
        call(rec.cfg, **a)
    assert rec.calls == [], why


def test_fp16_cache_calls_are_checked_too(rec):
    k = torch.zeros((B, S, HKV, 128), dtype=torch.float16)
    lens = torch.tensor([300, 255], dtype=torch.int32)
    table = torch.zeros((B, MB), dtype=torch.int32)
    pool16 = torch.zeros((PAGES, HKV, K.FP16_PAGE_BYTES), dtype=torch.uint8)
    kv.kvarn_fp16_write_blocks(k, k, lens, 300, table, pool16, stream=_Stream())
    assert rec.calls[-1][0] == "kvarn_fp16_write_blocks" and rec.calls[-1][1][6] == HKV
    q = torch.zeros((B, HQ, 128), dtype=torch.float16)
    kv.kvarn_fp16_decode_attention(q, HKV, pool16, table, lens, 300, torch.zeros_like(q), None,
                                   stream=_Stream())
    assert rec.calls[-1][0] == "kvarn_fp16_decode_attention"
    n = len(rec.calls)
    with pytest.raises(ValueError):   # a quantized pool where the fp16 one belongs
        kv.kvarn_fp16_decode_attention(
            q, HKV, torch.zeros((PAGES, HKV, K.PAGE_BYTES), dtype=torch.uint8), table, lens,
            300, torch.zeros_like(q), None, stream=_Stream())
    with pytest.raises(ValueError):
        kv.kvarn_fp16_write_blocks(k, k, lens.long(), 300, table, pool16, stream=_Stream())
    assert len(rec.calls) == n


def test_cuda_tensors_are_required_outside_these_tests():
    cfg = kv.config_from_string("k4v2_g128", HQ, HKV)
    with pytest.raises(ValueError, match="CUDA"):
        kv.kvarn_decode_attention(cfg, **_decode_args())
