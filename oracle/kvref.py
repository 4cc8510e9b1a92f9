"""Python face of the float64 CPU oracle (``kvref.c``).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  It does not import
the product package and the product package does not import it; the two sides
share nothing but the seeded input generators in ``workloads/``.

What the oracle computes, and where each step comes from, is written in the
header of ``kvref.c``: the four stages of "KVarN Nasil Calisir?" (How KVarN
works) on the KVarN page (blog.edumints.com) and decode attention over a paged
cache as in "KV Cache (Anahtar-Deger Onbellegi)" (yapayzekasozluk.tr).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkvref.so")
SRC_PATH = os.path.join(HERE, "kvref.c")

NCH = 128
NTOK = 128
REC_BYTES = 15360
REC_BYTES_M16 = 13824      # format variant "_m16": metadata stored as fp16
REC_BYTES_G64 = 17408      # format variant "k4v2_g64": two groups per token
REC_BYTES_V4 = 19456       # format variant "k4v4_g128": 4-bit values
REC_BYTES_K8 = 27648       # format variant "k8v4_g128": 8-bit keys, 4-bit values


def _fmt(meta16: bool = False, pc: bool = False, g64: bool = False, v4: bool = False,
         k8: bool = False) -> int:
    """Record format code of the C oracle: 0 fp32 metadata, 1 "_m16", 2 "_pc",
    3 "g64", 4 "k4v4", 5 "k8v4"; the variants do not combine."""
    if int(meta16) + int(pc) + int(g64) + int(v4) + int(k8) > 1:
        raise ValueError("the _m16, _pc, g64, k4v4 and k8v4 variants do not combine")
    return 5 if k8 else 4 if v4 else 3 if g64 else 2 if pc else 1 if meta16 else 0


def rec_bytes(meta16: bool = False, pc: bool = False, g64: bool = False, v4: bool = False,
              k8: bool = False) -> int:
    return {0: REC_BYTES, 1: REC_BYTES_M16, 2: REC_BYTES, 3: REC_BYTES_G64,
            4: REC_BYTES_V4, 5: REC_BYTES_K8}[_fmt(meta16, pc, g64, v4, k8)]

_lib = None


def build(force: bool = False) -> str:
    """Compile kvref.c with gcc (-O2, OpenMP, no intrinsics) into libkvref.so."""
    if force or not os.path.exists(LIB_PATH) or os.path.getmtime(LIB_PATH) < os.path.getmtime(SRC_PATH):
        cmd = ["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", SRC_PATH, "-o", LIB_PATH + ".tmp", "-lm"]
        subprocess.check_call(cmd)
        os.replace(LIB_PATH + ".tmp", LIB_PATH)
    return LIB_PATH


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.c_void_p
        L.kvref_half_to_double.restype = ctypes.c_double
        L.kvref_half_to_double.argtypes = [ctypes.c_uint16]
        L.kvref_hadamard.argtypes = [ctypes.c_int, P]
        L.kvref_rotate_tile.argtypes = [P, ctypes.c_long, P, P]
        L.kvref_sinkhorn.argtypes = [P, ctypes.c_int, P, P, P]
        L.kvref_sinkhorn_stat.argtypes = [P, ctypes.c_int, ctypes.c_int, P, P, P]
        L.kvref_rtn.argtypes = [P, P, P, ctypes.c_int, P, P, P, P]
        L.kvref_pack_part.argtypes = [P, ctypes.c_int, P, P, P, P]
        L.kvref_pack_part_fmt.argtypes = [P, ctypes.c_int, P, P, P, P, ctypes.c_int]
        L.kvref_unpack_part_fmt.argtypes = [P, ctypes.c_int, P, P, P, P, ctypes.c_int]
        L.kvref_dequant_part_fmt.argtypes = [P, ctypes.c_int, ctypes.c_int, P]
        L.kvref_pack_part_pc.argtypes = [P, ctypes.c_int, P, P, P, P]
        L.kvref_unpack_part_pc.argtypes = [P, ctypes.c_int, P, P, P, P]
        L.kvref_rtn_pc.argtypes = [P, P, P, ctypes.c_int, P, P, P, P, P]
        L.kvref_rtn_g64.argtypes = [P, P, P, ctypes.c_int, P, P, P, P]
        L.kvref_v4_code_pos.argtypes = [ctypes.c_int, ctypes.c_int, P, P]
        L.kvref_k8_code_pos.argtypes = [ctypes.c_int, ctypes.c_int]
        L.kvref_k8_code_pos.restype = ctypes.c_int
        L.kvref_pack_part_g64.argtypes = [P, ctypes.c_int, P, P, P, P]
        L.kvref_unpack_part_g64.argtypes = [P, ctypes.c_int, P, P, P, P]
        L.kvref_f32_to_f16.argtypes = [ctypes.c_float]
        L.kvref_f32_to_f16.restype = ctypes.c_uint16
        L.kvref_record_bytes.argtypes = [ctypes.c_int]
        L.kvref_record_bytes.restype = ctypes.c_long
        L.kvref_quantize_tile_fmt.argtypes = [P, ctypes.c_long, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, P, P, P, P, P, P]
        L.kvref_quantize_blocks_fmt.argtypes = [P, P, ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                                ctypes.c_int, P, P, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_int, ctypes.c_int, P,
                                                ctypes.c_long, P, P, P, P]
        L.kvref_append_token_fmt.argtypes = [P, P, P, ctypes.c_int, P, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_int, P,
                                             ctypes.c_long, P, P]
        L.kvref_decode_attention_fmt.argtypes = [P, P, ctypes.c_long, P, ctypes.c_int, P,
                                                 ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P,
                                                 ctypes.c_double, ctypes.c_int, ctypes.c_int, P]
        L.kvref_unpack_part.argtypes = [P, ctypes.c_int, P, P, P, P]
        L.kvref_dequant_part.argtypes = [P, ctypes.c_int, P]
        L.kvref_quantize_tile.argtypes = [P, ctypes.c_long, ctypes.c_int, ctypes.c_int, P, P, P,
                                          P, P, P]
        L.kvref_quantize_tile_stat.argtypes = [P, ctypes.c_long, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, P, P, P, P, P, P]
        L.kvref_quantize_blocks_stat.restype = ctypes.c_int
        L.kvref_quantize_blocks_stat.argtypes = [P, P, ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                                 ctypes.c_int, P, P, ctypes.c_int, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_int, P, ctypes.c_long, P,
                                                 P, P, P]
        L.kvref_append_token_stat.restype = ctypes.c_int
        L.kvref_append_token_stat.argtypes = [P, P, P, ctypes.c_int, P, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, P, ctypes.c_long, P, P]
        L.kvref_decode_attention.restype = ctypes.c_int
        L.kvref_decode_attention.argtypes = [P, P, ctypes.c_long, P, ctypes.c_int, P,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P,
                                             ctypes.c_double, ctypes.c_int, P]
        L.kvref_e4m3_decode.restype = ctypes.c_double
        L.kvref_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.kvref_e4m3_encode.restype = ctypes.c_uint8
        L.kvref_e4m3_encode.argtypes = [ctypes.c_float]
        L.kvref_fp8_quantize_token.argtypes = [P, P, P]
        L.kvref_fp8_write_blocks.restype = ctypes.c_int
        L.kvref_fp8_write_blocks.argtypes = [P, P, ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                             ctypes.c_int, ctypes.c_int, P, P, ctypes.c_int, P,
                                             ctypes.c_long]
        L.kvref_fp8_decode_attention.restype = ctypes.c_int
        L.kvref_fp8_decode_attention.argtypes = [P, P, ctypes.c_long, P, ctypes.c_int, P,
                                                 ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                 ctypes.c_double, P]
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _bits16(x):
    """fp16 array (or uint16 bit patterns) -> contiguous uint16 bit patterns."""
    x = np.asarray(x)
    if x.dtype == np.float16:
        return np.ascontiguousarray(x).view(np.uint16)
    return _c(x, np.uint16)


# ---------------------------------------------------------------- stages --

def half_to_double(bits: int) -> float:
    return lib().kvref_half_to_double(int(bits))


def hadamard(n: int = NCH) -> np.ndarray:
    H = np.zeros((n, n), dtype=np.float64)
    lib().kvref_hadamard(n, _p(H))
    return H


def rotate_tile(x) -> np.ndarray:
    """Stage 2 on one 128x128 fp16 tile: rows y_t = H x_t (float64)."""
    xb = _bits16(x).reshape(NTOK, NCH)
    H = hadamard(NCH)
    Y = np.zeros((NTOK, NCH), dtype=np.float64)
    lib().kvref_rotate_tile(_p(xb), NCH, _p(H), _p(Y))
    return Y


def sinkhorn(Y, iters: int, rms: bool = False):
    """Stage 3: log row scales a, log column scales b, and the per-iteration
    trace [iters][4] = (row max|log sigma|, row spread, column max|log sigma|,
    column spread).  rms: the uncentred statistic of the "_rms" variant."""
    Y = _c(Y, np.float64).reshape(NTOK, NCH)
    a = np.zeros(NTOK)
    b = np.zeros(NCH)
    tr = np.zeros(max(4 * iters, 1))
    lib().kvref_sinkhorn_stat(_p(Y), iters, int(rms), _p(a), _p(b), _p(tr))
    return a, b, tr[:4 * iters].reshape(iters, 4)


def rtn(Y, r, c32, bits: int):
    """Stage 4: codes q, fp32 s', z' and pre-rounding u."""
    Y = _c(Y, np.float64).reshape(NTOK, NCH)
    r = _c(r, np.float64)
    c32 = _c(c32, np.float32)
    q = np.zeros((NTOK, NCH), dtype=np.uint8)
    s = np.zeros(NTOK, dtype=np.float32)
    z = np.zeros(NTOK, dtype=np.float32)
    u = np.zeros((NTOK, NCH), dtype=np.float64)
    lib().kvref_rtn(_p(Y), _p(r), _p(c32), bits, _p(q), _p(s), _p(z), _p(u))
    return q, s, z, u


def f32_to_f16(x: float) -> int:
    """binary16 bits of the float32 value x, round to nearest even."""
    return int(lib().kvref_f32_to_f16(float(np.float32(x))))


def v4_code_pos(c: int, t: int):
    """Format "k4v4": (byte, bit shift) of the 4-bit V code of (channel, token)."""
    byte, shift = ctypes.c_int(0), ctypes.c_int(0)
    lib().kvref_v4_code_pos(c, t, ctypes.byref(byte), ctypes.byref(shift))
    return byte.value, shift.value


def k8_code_pos(d: int, t: int) -> int:
    """Format "k8v4": byte of the 8-bit K code of (channel, token)."""
    return lib().kvref_k8_code_pos(d, t)


def pack_part(rec, is_v: bool, q, s32, z32, c32, meta16: bool = False, v4: bool = False,
              k8: bool = False):
    lib().kvref_pack_part_fmt(_p(rec), int(is_v), _p(_c(q, np.uint8)), _p(_c(s32, np.float32)),
                              _p(_c(z32, np.float32)), _p(_c(c32, np.float32)),
                              _fmt(meta16, v4=v4, k8=k8))


def unpack_part(rec, is_v: bool, meta16: bool = False, v4: bool = False, k8: bool = False):
    q = np.zeros((NTOK, NCH), dtype=np.uint8)
    s = np.zeros(NTOK, dtype=np.float32)
    z = np.zeros(NTOK, dtype=np.float32)
    c = np.zeros(NCH, dtype=np.float32)
    lib().kvref_unpack_part_fmt(_p(_c(rec, np.uint8)), int(is_v), _p(q), _p(s), _p(z), _p(c),
                                _fmt(meta16, v4=v4, k8=k8))
    return q, s, z, c


def pack_part_pc(rec, is_v: bool, q, r32, cs32, cz32):
    lib().kvref_pack_part_pc(_p(rec), int(is_v), _p(_c(q, np.uint8)), _p(_c(r32, np.float32)),
                             _p(_c(cs32, np.float32)), _p(_c(cz32, np.float32)))


def unpack_part_pc(rec, is_v: bool):
    """Format "_pc": (codes, r_t, cs_d, cz_d)."""
    q = np.zeros((NTOK, NCH), dtype=np.uint8)
    r = np.zeros(NTOK, dtype=np.float32)
    cs = np.zeros(NCH, dtype=np.float32)
    cz = np.zeros(NCH, dtype=np.float32)
    lib().kvref_unpack_part_pc(_p(_c(rec, np.uint8)), int(is_v), _p(q), _p(r), _p(cs), _p(cz))
    return q, r, cs, cz


def rtn_pc(Y, r, c32, bits: int):
    """Format "_pc": RTN with one group per channel; (q, r32, cs32, cz32, u)."""
    Y = _c(Y, np.float64)
    q = np.zeros((NTOK, NCH), dtype=np.uint8)
    r32 = np.zeros(NTOK, dtype=np.float32)
    cs = np.zeros(NCH, dtype=np.float32)
    cz = np.zeros(NCH, dtype=np.float32)
    u = np.zeros((NTOK, NCH))
    lib().kvref_rtn_pc(_p(Y), _p(_c(r, np.float64)), _p(_c(c32, np.float32)), bits, _p(q),
                       _p(r32), _p(cs), _p(cz), _p(u))
    return q, r32, cs, cz, u


def rtn_g64(Y, r, c32, bits: int):
    """Format "g64": RTN with two groups of 64 channels per token;
    (q, s32 [128][2], z32 [128][2], u)."""
    Y = _c(Y, np.float64)
    q = np.zeros((NTOK, NCH), dtype=np.uint8)
    s = np.zeros((NTOK, 2), dtype=np.float32)
    z = np.zeros((NTOK, 2), dtype=np.float32)
    u = np.zeros((NTOK, NCH))
    lib().kvref_rtn_g64(_p(Y), _p(_c(r, np.float64)), _p(_c(c32, np.float32)), bits, _p(q),
                        _p(s), _p(z), _p(u))
    return q, s, z, u


def unpack_part_g64(rec, is_v: bool):
    """Format "g64": (codes, s' [128][2], z' [128][2], c)."""
    q = np.zeros((NTOK, NCH), dtype=np.uint8)
    s = np.zeros((NTOK, 2), dtype=np.float32)
    z = np.zeros((NTOK, 2), dtype=np.float32)
    c = np.zeros(NCH, dtype=np.float32)
    lib().kvref_unpack_part_g64(_p(_c(rec, np.uint8)), int(is_v), _p(q), _p(s), _p(z), _p(c))
    return q, s, z, c


def dequant_part(rec, is_v: bool, meta16: bool = False, pc: bool = False,
                 g64: bool = False, v4: bool = False, k8: bool = False) -> np.ndarray:
    y = np.zeros((NTOK, NCH), dtype=np.float64)
    lib().kvref_dequant_part_fmt(_p(_c(rec, np.uint8)), int(is_v), _fmt(meta16, pc, g64, v4, k8),
                                 _p(y))
    return y


def quantize_tile(x, is_v: bool, iters: int, rms: bool = False, meta16: bool = False,
                  pc: bool = False, g64: bool = False, v4: bool = False, k8: bool = False):
    """All four stages on one tile; returns a dict of every intermediate."""
    xb = _bits16(x).reshape(NTOK, NCH)
    rec = np.zeros(rec_bytes(meta16, pc, g64, v4, k8), dtype=np.uint8)
    Y = np.zeros((NTOK, NCH))
    a = np.zeros(NTOK)
    b = np.zeros(NCH)
    q = np.zeros((NTOK, NCH), dtype=np.uint8)
    u = np.zeros((NTOK, NCH))
    lib().kvref_quantize_tile_fmt(_p(xb), NCH, int(is_v), iters, int(rms), _fmt(meta16, pc, g64, v4, k8),
                                  _p(rec), _p(Y), _p(a), _p(b), _p(q), _p(u))
    return {"rec": rec, "Y": Y, "a": a, "b": b, "q": q, "u": u}


# ------------------------------------------------------------ whole ops --

def quantize_blocks(k, v, seq_lens, block_table, num_pages: int, iters: int, pool=None,
                    tail_k=None, tail_v=None, want_u: bool = False, rms: bool = False,
                    meta16: bool = False, pc: bool = False, g64: bool = False,
                    v4: bool = False, k8: bool = False):
    """Prefill: k, v fp16 [B][S][Hkv][128] (contiguous).  Returns a dict with
    the pool [num_pages][Hkv][15360] uint8 ([..][13824] with meta16), the fp16
    tails [B][Hkv][128][128] and, with want_u, the pre-rounding values
    [B][max_blocks][Hkv][128][128]."""
    kb = _bits16(k)
    vb = _bits16(v)
    B, S, hkv, d = kb.shape
    assert d == NCH
    seq_lens = _c(seq_lens, np.int32)
    block_table = _c(block_table, np.int32)
    max_blocks = block_table.shape[1]
    if pool is None:
        pool = np.zeros((num_pages, hkv, rec_bytes(meta16, pc, g64, v4, k8)), dtype=np.uint8)
    if tail_k is None:
        tail_k = np.zeros((B, hkv, NTOK, NCH), dtype=np.uint16)
    if tail_v is None:
        tail_v = np.zeros((B, hkv, NTOK, NCH), dtype=np.uint16)
    u_k = u_v = None
    if want_u:
        u_k = np.zeros((B, max_blocks, hkv, NTOK, NCH))
        u_v = np.zeros((B, max_blocks, hkv, NTOK, NCH))
    assert pool.shape[-1] == rec_bytes(meta16, pc, g64, v4, k8)
    rc = lib().kvref_quantize_blocks_fmt(_p(kb), _p(vb), S * hkv * NCH, hkv * NCH, NCH, B,
                                         _p(seq_lens), _p(block_table), max_blocks, hkv, iters,
                                         int(rms), _fmt(meta16, pc, g64, v4, k8), _p(pool), num_pages,
                                         _p(tail_k),
                                         _p(tail_v), _p(u_k), _p(u_v))
    return {"rc": rc, "pool": pool, "tail_k": tail_k, "tail_v": tail_v, "u_k": u_k, "u_v": u_v}


def append_token(k_new, v_new, pos, block_table, iters: int, pool, tail_k, tail_v,
                 rms: bool = False, meta16: bool = False, pc: bool = False, g64: bool = False,
                 v4: bool = False, k8: bool = False):
    """Decode-time append (in place on pool / tails).  Returns the status."""
    kb = _bits16(k_new)
    vb = _bits16(v_new)
    B, hkv, d = kb.shape
    pos = _c(pos, np.int32)
    block_table = _c(block_table, np.int32)
    assert pool.flags["C_CONTIGUOUS"] and tail_k.flags["C_CONTIGUOUS"]
    assert pool.shape[-1] == rec_bytes(meta16, pc, g64, v4, k8)
    return lib().kvref_append_token_fmt(_p(kb), _p(vb), _p(pos), B, _p(block_table),
                                        block_table.shape[1], hkv, iters, int(rms),
                                        _fmt(meta16, pc, g64, v4, k8),
                                        _p(pool), pool.shape[0], _p(tail_k), _p(tail_v))


def decode_attention(q, pool, block_table, seq_lens, tail_k, tail_v, hq: int, hkv: int,
                     scale: float = 1.0 / np.sqrt(128.0), route: int = 1, meta16: bool = False,
                     pc: bool = False, g64: bool = False, v4: bool = False, k8: bool = False):
    """Decode attention, float64 output [B][Hq][128].  route 0 = textbook
    (un-rotate every token), route 1 = rotated space with one final H."""
    qb = _bits16(q)
    B = qb.shape[0]
    pool = _c(pool, np.uint8)
    block_table = _c(block_table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    out = np.zeros((B, hq, NCH))
    assert pool.shape[-1] == rec_bytes(meta16, pc, g64, v4, k8)
    rc = lib().kvref_decode_attention_fmt(_p(qb), _p(pool), pool.shape[0], _p(block_table),
                                          block_table.shape[1], _p(seq_lens), B, hq, hkv,
                                          _p(_bits16(tail_k)), _p(_bits16(tail_v)), float(scale),
                                          int(route), _fmt(meta16, pc, g64, v4, k8), _p(out))
    if rc != 0:
        raise ValueError("oracle: page id outside the pool")
    return out


def attention_fp16(q, k, v, seq_lens, hq: int, hkv: int,
                   scale: float = 1.0 / np.sqrt(128.0)) -> np.ndarray:
    """Decode attention over an uncompressed fp16 cache, float64 output
    [B][Hq][128]: out[b][h] = sum_t softmax_t(scale q[b][h] . k[b][t][h/g]) v[b][t][h/g]
    over t < seq_lens[b], the textbook definition ("KV Cache (Anahtar-Deger
    Onbellegi)", yapayzekasozluk.tr, "KV Cache Nasil Calisir?") written out in
    numpy float64 (max-subtracted softmax).  q: fp16 [B][Hq][128]; k, v: fp16
    [B][S][Hkv][128]; fp16 values are taken exactly."""
    def f64(x):
        if hasattr(x, "numpy"):
            x = x.cpu().numpy()
        x = np.asarray(x)
        if x.dtype == np.uint16:
            x = x.view(np.float16)
        return x.astype(np.float64)

    qd, kd, vd = f64(q), f64(k), f64(v)
    lens = np.asarray(seq_lens.cpu().numpy() if hasattr(seq_lens, "numpy") else seq_lens)
    B = qd.shape[0]
    g = hq // hkv
    out = np.zeros((B, hq, NCH))
    for b in range(B):
        n = int(lens[b])
        if n <= 0:
            continue
        for h in range(hq):
            kh = kd[b, :n, h // g, :]
            vh = vd[b, :n, h // g, :]
            s = (kh @ qd[b, h]) * scale
            p = np.exp(s - s.max())
            out[b, h] = (p @ vh) / p.sum()
    return out


def chunk_attention(q, start, chunk_lens, pool, block_table, tail_k, tail_v, hq: int, hkv: int,
                    scale: float = 1.0 / np.sqrt(128.0), meta16: bool = False,
                    pc: bool = False, g64: bool = False, v4: bool = False,
                    k8: bool = False) -> np.ndarray:
    """Attention of a chunk of new query tokens over the quantized cache
    (chunked prefill), float64 output [B][M][Hq][128].

    Sequence b holds start[b] tokens before the chunk and chunk_lens[b] <= M
    new ones; the cache (pool pages + fp16 tails) is its state after the
    chunk's tokens were appended, n_b = start[b] + chunk_lens[b] tokens.
    Query i sits at position P = start[b] + i and attends causally to tokens
    0..P: out = sum_{t<=P} softmax_t(scale q . k_t) v_t, the textbook
    definition ("KV Cache (Anahtar-Deger Onbellegi)", yapayzekasozluk.tr, "KV
    Cache Nasil Calisir?") with the decode reading "append, then attend"
    applied to a whole chunk.  Token t is read, in plain space, from its page
    (x = H yhat, stage-4 dequantization of the KVarN page, blog.edumints.com)
    when its block is full in the cache, else from tail slot t mod 128.  Rows
    i >= chunk_lens[b] are zero.  q: fp16 [B][M][Hq][128]."""
    qd = np.asarray(q)
    if qd.dtype == np.uint16:
        qd = qd.view(np.float16)
    qd = qd.astype(np.float64)
    tk = np.asarray(tail_k)
    tv = np.asarray(tail_v)
    tk = (tk.view(np.float16) if tk.dtype == np.uint16 else tk).astype(np.float64)
    tv = (tv.view(np.float16) if tv.dtype == np.uint16 else tv).astype(np.float64)
    start = np.asarray(start, dtype=np.int64)
    chunk_lens = np.asarray(chunk_lens, dtype=np.int64)
    block_table = np.asarray(block_table)
    B, M = qd.shape[0], qd.shape[1]
    g = hq // hkv
    H = hadamard(NCH)
    out = np.zeros((B, M, hq, NCH))
    for b in range(B):
        n = int(start[b] + chunk_lens[b])
        if chunk_lens[b] <= 0 or n <= 0:
            continue
        nfull = n // NTOK
        K = np.zeros((hkv, n, NCH))
        V = np.zeros((hkv, n, NCH))
        for j in range(nfull):
            page = int(block_table[b, j])
            if page < 0 or page >= pool.shape[0]:
                raise ValueError("oracle: page id outside the pool")
            for h in range(hkv):
                K[h, j * NTOK:(j + 1) * NTOK] = dequant_part(pool[page, h], False, meta16, pc,
                                                             g64, v4, k8) @ H
                V[h, j * NTOK:(j + 1) * NTOK] = dequant_part(pool[page, h], True, meta16, pc,
                                                             g64, v4, k8) @ H
        r = n - nfull * NTOK
        K[:, nfull * NTOK:] = tk[b, :, :r]
        V[:, nfull * NTOK:] = tv[b, :, :r]
        for i in range(int(chunk_lens[b])):
            P = int(start[b]) + i
            for h in range(hq):
                s = (K[h // g, :P + 1] @ qd[b, i, h]) * scale
                p = np.exp(s - s.max())
                out[b, i, h] = (p / p.sum()) @ V[h // g, :P + 1]
    return out


# ------------------------------------------------------------ FP8 cache --
# The FP8 paged cache the quantized one is compared with (per-token e4m3 with
# an fp32 absmax scale; layout and readings in the header of that part of
# kvref.c).

FP8_PAGE_BYTES = 33792


def e4m3_decode(code: int) -> float:
    return lib().kvref_e4m3_decode(int(code))


def e4m3_encode(u: float) -> int:
    return int(lib().kvref_e4m3_encode(float(u)))


def fp8_quantize_token(x):
    """fp16 [128] -> (codes uint8 [128], fp32 scale)."""
    xb = _bits16(x).reshape(NCH)
    codes = np.zeros(NCH, dtype=np.uint8)
    s = np.zeros(1, dtype=np.float32)
    lib().kvref_fp8_quantize_token(_p(xb), _p(codes), _p(s))
    return codes, float(s[0])


def fp8_write_blocks(k, v, seq_lens, block_table, num_pages: int):
    """fp16 k, v [B][S][Hkv][128] -> pool uint8 [num_pages][Hkv][33792]."""
    kb, vb = _bits16(k), _bits16(v)
    B, S, hkv, _ = kb.shape
    seq_lens = _c(seq_lens, np.int32)
    block_table = _c(block_table, np.int32)
    pool = np.zeros((num_pages, hkv, FP8_PAGE_BYTES), dtype=np.uint8)
    rc = lib().kvref_fp8_write_blocks(_p(kb), _p(vb), S * hkv * NCH, hkv * NCH, NCH, B, hkv,
                                      _p(seq_lens), _p(block_table), block_table.shape[1],
                                      _p(pool), num_pages)
    if rc != 0:
        raise ValueError("oracle: page id outside the pool")
    return pool


def fp8_decode_attention(q, pool, block_table, seq_lens, hq: int, hkv: int,
                         scale: float = 1.0 / np.sqrt(128.0)) -> np.ndarray:
    """Decode attention over the fp8 pages, float64 [B][Hq][128]."""
    qb = _bits16(q)
    B = qb.shape[0]
    pool = _c(pool, np.uint8)
    block_table = _c(block_table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    out = np.zeros((B, hq, NCH))
    rc = lib().kvref_fp8_decode_attention(_p(qb), _p(pool), pool.shape[0], _p(block_table),
                                          block_table.shape[1], _p(seq_lens), B, hq, hkv,
                                          float(scale), _p(out))
    if rc != 0:
        raise ValueError("oracle: page id outside the pool")
    return out


# ------------------------------------------------- SnapKV-style selection --
# "Makale Bulteni - SnapKV" (cmlonder.com): at the end of prefill the
# attention of the prompt's last 32 or 64 tokens (the observation window) over
# the earlier tokens is scanned once, and each head keeps its most critical,
# clustered KV positions (pooling, then selection); the rest of the cache is
# dropped and decode runs on a compact cache of fixed size, each head with its
# own positions.  Readings (the page fixes none of the numbers below):
#   * votes of KV head h: v_t = sum over the window queries i (positions
#     P_i = n - W + i) and the query heads of h's group of
#     softmax_{t' <= P_i}(scale q . k_t')[t], for the prefix positions
#     t < n - W (scale 1/sqrt(128), the decode attention's);
#   * clustering: a 1-D max pooling of the votes with an odd kernel (7 unless
#     given), the window [t - K//2, t + K//2] clipped to the prefix;
#   * selection: the capacity - W prefix positions with the largest pooled
#     votes, ties to the lower position, then the W window positions, all in
#     increasing order; a prefix no longer than capacity - W is kept whole;
#   * compaction: the kept tokens' K and V, in that order.

def snapkv_votes(q_window, k, seq_lens, hq: int, hkv: int,
                 scale: float = 1.0 / np.sqrt(128.0)) -> np.ndarray:
    """Votes [B][Hkv][S] (float64; zero at and beyond n - W).  q_window: fp16
    [B][W][Hq][128] (the queries of the last W prompt tokens); k: fp16
    [B][S][Hkv][128]; seq_lens: prompt lengths n (window included)."""
    qd = np.asarray(q_window)
    qd = (qd.view(np.float16) if qd.dtype == np.uint16 else qd).astype(np.float64)
    kd = np.asarray(k)
    kd = (kd.view(np.float16) if kd.dtype == np.uint16 else kd).astype(np.float64)
    B, W = qd.shape[0], qd.shape[1]
    S = kd.shape[1]
    g = hq // hkv
    votes = np.zeros((B, hkv, S))
    for b in range(B):
        n = int(seq_lens[b])
        if n <= W:
            continue
        for h in range(hkv):
            for i in range(W):
                P = n - W + i
                for hh in range(g):
                    s = (kd[b, :P + 1, h] @ qd[b, i, h * g + hh]) * scale
                    p = np.exp(s - s.max())
                    p /= p.sum()
                    votes[b, h, :n - W] += p[:n - W]
    return votes


def snapkv_pool(votes_1d, kernel: int = 7) -> np.ndarray:
    """1-D max pooling over a prefix of votes (window clipped to its ends)."""
    v = np.asarray(votes_1d, dtype=np.float64)
    n = len(v)
    r = kernel // 2
    return np.array([v[max(0, t - r):min(n, t + r + 1)].max() for t in range(n)])


def snapkv_select(votes, seq_lens, window: int, capacity: int, kernel: int = 7):
    """Kept positions [B][Hkv][capacity] (int32, increasing; -1 past a short
    sequence's n) from the votes of snapkv_votes."""
    votes = np.asarray(votes)
    B, hkv, _ = votes.shape
    out = np.full((B, hkv, capacity), -1, dtype=np.int32)
    for b in range(B):
        n = int(seq_lens[b])
        npre = max(n - window, 0)
        keep_pre = capacity - window
        for h in range(hkv):
            if npre <= keep_pre:
                kept = list(range(n))
            else:
                pooled = snapkv_pool(votes[b, h, :npre], kernel)
                # largest first, ties to the lower position
                order = sorted(range(npre), key=lambda t: (-pooled[t], t))
                kept = sorted(order[:keep_pre]) + list(range(npre, n))
            out[b, h, :len(kept)] = kept
    return out
