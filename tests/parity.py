"""Comparison rules between the CUDA path and the float64 oracle.

  * codes: bit-exact, except elements whose oracle pre-rounding value u lies
    within 1e-5 of a rounding boundary (k + 1/2); such flips must be at most
    1e-4 of all elements.  For 8-bit codes ("k8v4") u spans 0..255 instead
    of 0..15 and fp32 carries 17 times the absolute error there, so the
    window is 1e-5 x 255 / 15;
  * s' and c: |gpu - ref| <= 1e-5 |ref| (1e-12 absolute when ref = 0);
  * z': |gpu - ref| <= 1e-5 (|z'| + s' (2^b - 1));
  * fp16 metadata (format "_m16"): equal to the oracle's fp16 value, or one
    fp16 spacing away from it with the oracle's fp32 value within 1e-5
    (relative) of the midpoint between the two (a rounding boundary of the
    second rounding);
  * attention output (fp16): |gpu - ref| <= 2e-3 + 1e-3 |ref| elementwise, the
    oracle being fed the GPU's own pool so that decode is judged apart from
    boundary flips in quantization.
"""
from __future__ import annotations

import numpy as np

from oracle import kvref

BOUNDARY = 1e-5
FLIP_RATE = 1e-4


def near_boundary(u, bits: int = 4):
    window = BOUNDARY * (255 / 15 if bits == 8 else 1)
    return np.abs(u - np.floor(u) - 0.5) < window


def _compare_meta16(tag, got16, ref16, ref32):
    """fp16 metadata: the same rounding of nearly the same fp32 value."""
    g, r = got16.astype(np.float64), ref16.astype(np.float64)
    same = g == r
    if same.all():
        return
    r32 = ref32.astype(np.float64)
    spacing = np.spacing(ref16.astype(np.float16)).astype(np.float64)
    mid = 0.5 * (g + r)
    near = (np.abs(g - r) <= spacing * 1.0000001) & (np.abs(r32 - mid) <= 1e-5 * np.abs(mid))
    bad = ~same & ~near
    assert not bad.any(), (f"{tag}: {int(bad.sum())} fp16 values differ away from a rounding "
                           f"boundary, e.g. gpu={g[bad][:3]}, ref={r[bad][:3]}, "
                           f"ref fp32={r32[bad][:3]}")


def _compare_pc(tag, got, ref, is_v, bits):
    """Format "_pc" metadata: r_t and cs_d within 1e-5 relative, cz_d within
    1e-5 (|cz| + cs (2^b - 1)) (the z' rule with the per-channel step)."""
    _, rg, csg, czg = kvref.unpack_part_pc(got, is_v)
    _, rr, csr, czr = kvref.unpack_part_pc(ref, is_v)
    for name, g_, r_ in (("r", rg, rr), ("cs", csg, csr)):
        gd, rd = g_.astype(np.float64), r_.astype(np.float64)
        tol = np.where(rd == 0, 1e-12, 1e-5 * np.abs(rd))
        err = np.abs(gd - rd)
        assert np.all(err <= tol), (f"{tag}.{name}: worst rel err "
                                    f"{(err / np.maximum(np.abs(rd), 1e-30)).max():.3e}")
    tolz = np.maximum(1e-5 * (np.abs(czr.astype(np.float64))
                              + np.abs(csr.astype(np.float64)) * (2 ** bits - 1)), 1e-12)
    errz = np.abs(czg.astype(np.float64) - czr.astype(np.float64))
    assert np.all(errz <= tolz), f"{tag}.cz: worst err {errz.max():.3e}"


def _compare_g64(tag, got, ref, is_v, bits):
    """Format "g64": the s', c and z' rules of the default format, per group."""
    _, sg, zg, cg = kvref.unpack_part_g64(got, is_v)
    _, sr, zr, cr = kvref.unpack_part_g64(ref, is_v)
    for name, g_, r_ in (("s", sg, sr), ("c", cg, cr)):
        gd, rd = g_.astype(np.float64), r_.astype(np.float64)
        tol = np.where(rd == 0, 1e-12, 1e-5 * np.abs(rd))
        err = np.abs(gd - rd)
        assert np.all(err <= tol), (f"{tag}.{name}: worst rel err "
                                    f"{(err / np.maximum(np.abs(rd), 1e-30)).max():.3e}")
    tolz = np.maximum(1e-5 * (np.abs(zr.astype(np.float64))
                              + sr.astype(np.float64) * (2 ** bits - 1)), 1e-12)
    errz = np.abs(zg.astype(np.float64) - zr.astype(np.float64))
    assert np.all(errz <= tolz), f"{tag}.z: worst err {errz.max():.3e}"


def compare_record(got: np.ndarray, ref: np.ndarray, u_k=None, u_v=None, stats=None,
                   meta16: bool = False, ref32: np.ndarray = None, pc: bool = False,
                   g64: bool = False, v4: bool = False, k8: bool = False):
    """Compares one record (GPU) with the oracle's.  u_k, u_v: oracle
    pre-rounding values [128][128] (token, channel).  meta16: the "_m16"
    format, whose metadata is judged against ref32, the oracle's record of
    the same tile in the fp32 format; pc: the "_pc" format.  Returns a dict."""
    out = {} if stats is None else stats
    for is_v, u in ((False, u_k), (True, u_v)):
        bits = (4 if v4 or k8 else 2) if is_v else (8 if k8 else 4)
        if pc or g64:
            unpack = kvref.unpack_part_pc if pc else kvref.unpack_part_g64
            qg = unpack(got, is_v)[0]
            qr = unpack(ref, is_v)[0]
        else:
            qg, sg, zg, cg = kvref.unpack_part(got, is_v, meta16, v4, k8=k8)
            qr, sr, zr, cr = kvref.unpack_part(ref, is_v, meta16, v4, k8=k8)
        tag = "v" if is_v else "k"
        diff = qg != qr
        n_diff = int(diff.sum())
        if n_diff:
            assert u is not None, f"{tag}: {n_diff} code mismatches and no u to judge them"
            ok = near_boundary(u, bits)
            bad = diff & ~ok
            assert not bad.any(), (f"{tag}: {int(bad.sum())} code mismatches away from a "
                                   f"rounding boundary, e.g. u={u[bad][:4]}, gpu={qg[bad][:4]}, "
                                   f"ref={qr[bad][:4]}")
        if n_diff:   # the widest distance from a boundary among the flips
            dist = float(np.abs(u[diff] - np.floor(u[diff]) - 0.5).max())
            out[f"{tag}_flip_dist"] = max(out.get(f"{tag}_flip_dist", 0.0), dist)
        out[f"{tag}_flips"] = out.get(f"{tag}_flips", 0) + n_diff
        out[f"{tag}_codes"] = out.get(f"{tag}_codes", 0) + qg.size
        if pc:
            _compare_pc(tag, got, ref, is_v, bits)
            continue
        if g64:
            _compare_g64(tag, got, ref, is_v, bits)
            continue
        if meta16:
            _, s32, z32, c32 = kvref.unpack_part(ref32, is_v)
            for name, g_, r_, r32 in (("s", sg, sr, s32), ("z", zg, zr, z32), ("c", cg, cr, c32)):
                _compare_meta16(f"{tag}.{name}", g_, r_, r32)
            continue
        for name, g_, r_ in (("s", sg, sr), ("c", cg, cr)):
            gd, rd = g_.astype(np.float64), r_.astype(np.float64)
            tol = np.where(rd == 0, 1e-12, 1e-5 * np.abs(rd))
            err = np.abs(gd - rd)
            assert np.all(err <= tol), (f"{tag}.{name}: worst rel err "
                                        f"{(err / np.maximum(np.abs(rd), 1e-30)).max():.3e}")
        tolz = 1e-5 * (np.abs(zr.astype(np.float64)) + sr.astype(np.float64) * (2 ** bits - 1))
        tolz = np.maximum(tolz, 1e-12)
        errz = np.abs(zg.astype(np.float64) - zr.astype(np.float64))
        assert np.all(errz <= tolz), f"{tag}.z: worst err {errz.max():.3e}"
    return out


def check_flip_rate(stats):
    for tag in ("k", "v"):
        if stats.get(f"{tag}_codes"):
            rate = stats[f"{tag}_flips"] / stats[f"{tag}_codes"]
            assert rate <= FLIP_RATE, f"{tag}: boundary flips {rate:.2e} > {FLIP_RATE}"


def compare_attention(got: np.ndarray, ref: np.ndarray):
    got = got.astype(np.float64)
    err = np.abs(got - ref)
    tol = 2e-3 + 1e-3 * np.abs(ref)
    assert np.all(err <= tol), (f"attention: {int((err > tol).sum())} of {err.size} outside "
                                f"2e-3 + 1e-3|ref|; max abs err {err.max():.3e}")
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert rel <= 1e-3, f"attention: relative norm error {rel:.3e}"
    return {"max_abs": float(err.max()), "rel_norm": float(rel)}
