"""Pins of the float64 oracle against facts the pages and mathematics fix.

None of these re-types the oracle's formulas: each checks a property that a
plausible mistake (a dropped term, a wrong sign or index, a transposed operand,
a mis-packed bit) would break.

Sources: the KVarN page (blog.edumints.com), "KVarN Nasil Calisir?" (stage 2:
orthonormal Hadamard rotation along channels that keeps attention scores;
stage 3: log-domain Sinkhorn-like row/column variance normalization; stage 4:
asymmetric RTN, 4-bit K / 2-bit V, group 128); "KV Cache (Anahtar-Deger
Onbellegi)" (yapayzekasozluk.tr) for decode attention over the cache.
"""
import json
import os

import numpy as np
import pytest
import torch

from workloads import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _tile(seed, sigma=1.0, outliers=2, fac=20.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((128, 128)) * np.exp(sigma * rng.standard_normal(128))
    idx = rng.choice(128, outliers, replace=False)
    x[:, idx] *= fac
    return x.astype(np.float16)


# ------------------------------------------------------------------ fp16 --

def test_half_decode_matches_numpy_for_every_pattern(oracle):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits[::7]])
    r = ref[::7]
    finite = np.isfinite(r)
    assert np.array_equal(got[finite], r[finite])
    assert np.all(np.isnan(got[np.isnan(r)]))
    assert oracle.half_to_double(0x3C00) == 1.0
    assert oracle.half_to_double(0xC000) == -2.0
    assert oracle.half_to_double(0x0001) == 2.0 ** -24
    assert oracle.half_to_double(0x7BFF) == 65504.0


# -------------------------------------------------------------- Hadamard --

def test_hadamard_orthonormal_symmetric_self_inverse(oracle):
    H = oracle.hadamard(128)
    assert np.abs(H @ H.T - np.eye(128)).max() < 1e-15 * 4
    assert np.array_equal(H, H.T)
    assert np.abs(H @ H - np.eye(128)).max() < 1e-15 * 4


def test_hadamard_closed_form_sylvester_order(oracle):
    # Sylvester order: H[i, j] = (-1)^popcount(i & j) / sqrt(n)
    for n in (1, 2, 8, 128):
        H = oracle.hadamard(n)
        i = np.arange(n)[:, None]
        j = np.arange(n)[None, :]
        pc = np.vectorize(lambda v: bin(int(v)).count("1"))(i & j)
        assert np.array_equal(H * np.sqrt(n), (-1.0) ** pc)


def test_hadamard_first_basis_vector_and_norm(oracle):
    H = oracle.hadamard(128)
    e0 = np.zeros(128)
    e0[0] = 1
    assert np.allclose(H @ e0, np.full(128, 1 / np.sqrt(128)), atol=1e-16, rtol=0)
    x = np.random.default_rng(1).standard_normal(128) * 50
    assert abs(np.linalg.norm(H @ x) - np.linalg.norm(x)) < 1e-12 * np.linalg.norm(x)


def _fwht_recursive(x):
    """Textbook recursive fast Walsh-Hadamard transform (unnormalised)."""
    n = len(x)
    if n == 1:
        return x.copy()
    a = _fwht_recursive(x[: n // 2])
    b = _fwht_recursive(x[n // 2:])
    return np.concatenate([a + b, a - b])


def test_rotate_tile_equals_recursive_fwht(oracle):
    x = _tile(3)
    Y = oracle.rotate_tile(x)
    xd = x.astype(np.float64)
    for t in (0, 1, 77, 127):
        ref = _fwht_recursive(xd[t]) / np.sqrt(128)
        assert np.abs(Y[t] - ref).max() <= 1e-12 * np.abs(ref).max()


def test_rotation_preserves_attention_scores(oracle):
    # stage 2: "attention scores are preserved" -> (Hq).(Hk) = q.k
    H = oracle.hadamard(128)
    rng = np.random.default_rng(2)
    for _ in range(5):
        q = rng.standard_normal(128)
        k = rng.standard_normal(128) * 30
        assert abs((H @ q) @ (H @ k) - q @ k) < 1e-12 * np.linalg.norm(q) * np.linalg.norm(k)


# -------------------------------------------------------------- Sinkhorn --

@pytest.mark.parametrize("iters", [1, 2, 4])
def test_final_column_step_gives_unit_column_std(oracle, iters):
    Y = oracle.rotate_tile(_tile(4))
    a, b, _ = oracle.sinkhorn(Y, iters)
    Z = Y * np.exp(-a)[:, None] * np.exp(-b)[None, :]
    assert np.abs(Z.std(axis=0) - 1).max() < 1e-12


def test_sinkhorn_spread_converges(oracle):
    w = synth.WORKLOADS["tiny"]
    k, v = synth.kv(w)
    for x in (k[0, :128, 0].numpy(), v[0, 128:256, 0].numpy(), _tile(5, sigma=1.0, outliers=4,
                                                                       fac=30.0)):
        Y = oracle.rotate_tile(x)
        _, _, tr = oracle.sinkhorn(Y, 64)
        row_spread = tr[:, 1]
        col_spread = tr[:, 3]
        assert row_spread[-1] < 1e-9 and col_spread[-1] < 1e-9
        # non-increasing in practice (allow round-off once converged)
        assert np.all(np.diff(row_spread) <= 1e-12)
        assert np.all(np.diff(col_spread) <= 1e-12)


def test_sinkhorn_row_equivariance(oracle):
    # rows first: scaling token rows by alpha > 0 changes only a (by log alpha)
    Y = oracle.rotate_tile(_tile(6))
    alpha = np.exp(np.random.default_rng(7).standard_normal(128))
    a, b, _ = oracle.sinkhorn(Y, 3)
    a2, b2, _ = oracle.sinkhorn(Y * alpha[:, None], 3)
    assert np.abs(b2 - b).max() < 1e-12
    assert np.abs(a2 - (a + np.log(alpha))).max() < 1e-12


def test_sinkhorn_rank_one_closed_form(oracle):
    # Y = u v^T with u > 0: row t has centred std u_t * std(v); after the row
    # step every column is constant, so the column step is skipped (b = 0),
    # and later row steps see unit std (a unchanged).
    rng = np.random.default_rng(8)
    u = np.exp(rng.standard_normal(128))
    v = rng.standard_normal(128)
    Y = np.outer(u, v)
    for iters in (1, 2, 5):
        a, b, _ = oracle.sinkhorn(Y, iters)
        assert np.abs(b).max() == 0.0
        assert np.abs(a - (np.log(u) + np.log(v.std()))).max() < 1e-12


def _row_std(Z):
    return Z.std(axis=1)


@pytest.mark.parametrize("k", [1, 2, 3])
def test_row_step_normalizes_rows_against_current_column_scales(oracle, k):
    # The row step of iteration k+1 starts from the state (a_k, b_k) that k
    # whole iterations leave and changes only a.  After it, every row of
    # Z = Y exp(-a_{k+1}) exp(-b_k) must have centred std exactly 1: that is
    # what normalizing a row means (KVarN page, "KVarN Nasil Calisir?", stage
    # "Normalize Edilmis Onbellek"; rows first, centred population std).  A
    # row step that ignored the current column scales would leave these rows
    # at std(Y_t e^-b) / std(Y_t), not 1.
    for x in (_tile(41), _tile(42, sigma=1.5, outliers=4, fac=30.0)):
        Y = oracle.rotate_tile(x)
        a_k, b_k, _ = oracle.sinkhorn(Y, k)
        a_next, b_next, _ = oracle.sinkhorn(Y, k + 1)
        assert np.abs(b_k).max() > 1e-3   # the column scales are not trivial
        Z = Y * np.exp(-a_next)[:, None] * np.exp(-b_k)[None, :]
        assert np.abs(_row_std(Z) - 1.0).max() < 1e-12
        # ... and the column step that follows then gives unit column std
        Z2 = Y * np.exp(-a_next)[:, None] * np.exp(-b_next)[None, :]
        assert np.abs(Z2.std(axis=0) - 1.0).max() < 1e-12


def test_sinkhorn_limit_has_equal_row_and_unit_column_stds(oracle):
    # At the limit of the alternating normalization both steps are no-ops up
    # to a common factor: columns of Z have std 1 and the rows all share one
    # std (the common offset between r and c does not vanish for centred
    # statistics).  Checked on Z rebuilt from the returned scales.
    for x in (_tile(43), _tile(44, sigma=1.0, outliers=4, fac=25.0)):
        Y = oracle.rotate_tile(x)
        a, b, _ = oracle.sinkhorn(Y, 64)
        Z = Y * np.exp(-a)[:, None] * np.exp(-b)[None, :]
        rs = _row_std(Z)
        assert np.abs(Z.std(axis=0) - 1.0).max() < 1e-12
        assert (rs.max() - rs.min()) / rs.mean() < 1e-9
        # and the rows are not already equal after the first iteration: the
        # later row steps have work to do
        a1, b1, _ = oracle.sinkhorn(Y, 1)
        rs1 = _row_std(Y * np.exp(-a1)[:, None] * np.exp(-b1)[None, :])
        assert (rs1.max() - rs1.min()) / rs1.mean() > 1e-3


def test_sinkhorn_second_row_step_has_positive_spread(oracle):
    # On a tile that is not separable the column step of iteration 1 unsettles
    # the rows again, so the row step of iteration 2 moves them by different
    # amounts (its spread of log sigma is > 0).
    Y = oracle.rotate_tile(_tile(45, sigma=1.0, outliers=4, fac=30.0))
    _, _, tr = oracle.sinkhorn(Y, 3)
    assert tr[1, 1] > 1e-4 and tr[2, 1] > 0.0


def _near_constant(n, c, rel, rng):
    """n values c (1 + rel s_i), s_i = +-1 in equal numbers: centred variance
    over mean square = rel^2 / (1 + rel^2)."""
    s = np.array([1.0, -1.0] * (n // 2))
    rng.shuffle(s)
    return c * (1.0 + rel * s)


def test_sinkhorn_skip_threshold_rows(oracle):
    # The skip rule leaves a row alone only when its variance is at most
    # 1e-10 of its mean square.  A row at var/msq ~ 1e-8 must be normalized
    # (a_t = log of its std, as the first row step sees Y itself); one at
    # ~ 1e-12 must be skipped (a_t stays exactly 0).
    rng = np.random.default_rng(46)
    Y = rng.standard_normal((128, 128)) * 2.0
    Y[5] = _near_constant(128, 3.0, 1e-4, rng)    # var/msq ~ 1e-8: updated
    Y[9] = _near_constant(128, -7.0, 1e-6, rng)   # var/msq ~ 1e-12: skipped
    Y[17] = _near_constant(128, 2.0, 3e-5, rng)   # var/msq ~ 9e-10: updated
    Y[23] = _near_constant(128, 1.5, 3e-6, rng)   # var/msq ~ 9e-12: skipped
    a, _, _ = oracle.sinkhorn(Y, 1)
    assert a[9] == 0.0 and a[23] == 0.0
    for t in (5, 17):
        assert abs(a[t] - np.log(Y[t].std())) < 1e-9
        assert a[t] < -5.0


def test_sinkhorn_skip_threshold_columns(oracle):
    # Same rule for columns.  Every row is a permutation of one vector w
    # outside columns 0..3, so the first row step scales all rows alike and
    # leaves the near-constant columns near-constant: column 1 at var/msq
    # ~ 1e-8 must get b = log of its std, columns 2 and 3 at ~ 1e-12 and
    # ~ 9e-12 must keep b = 0.
    rng = np.random.default_rng(47)
    w = rng.standard_normal(124) * 3.0
    Y = np.empty((128, 128))
    for t in range(128):
        Y[t, 4:] = np.roll(w, t)
    Y[:, 0] = 5.0
    Y[:, 1] = _near_constant(128, 4.0, 1e-4, rng)
    Y[:, 2] = _near_constant(128, -6.0, 1e-6, rng)
    Y[:, 3] = _near_constant(128, 2.5, 3e-6, rng)
    a, b, _ = oracle.sinkhorn(Y, 1)
    Z = Y * np.exp(-a)[:, None]
    assert b[0] == 0.0 and b[2] == 0.0 and b[3] == 0.0
    assert abs(b[1] - np.log(Z[:, 1].std())) < 1e-9
    assert b[1] < -5.0


# ------------------------------------------- uncentred (RMS) variant ----
# Format variant "_rms": each step divides by the root mean square instead of
# the centred std, i.e. the Sinkhorn-Knopp scaling of the squared tile (the
# plain-Sinkhorn reading of "Sinkhorn-like variance normalization", KVarN
# page, "KVarN Nasil Calisir?", stage "Normalize Edilmis Onbellek").

def _rms(Z, axis):
    return np.sqrt((Z * Z).mean(axis=axis))


def test_rms_variant_rank_one_fixed_point(oracle):
    # Y = u v^T, u > 0, no zero in v: the row step leaves every column
    # constant in magnitude, |v_d| / rms(v); the column step then makes every
    # |Z| = 1, a fixed point of both steps.
    rng = np.random.default_rng(48)
    u = np.exp(rng.standard_normal(128))
    v = rng.standard_normal(128)
    Y = np.outer(u, v)
    rv = np.sqrt((v * v).mean())
    for iters in (1, 2, 5):
        a, b, _ = oracle.sinkhorn(Y, iters, rms=True)
        assert np.abs(a - (np.log(u) + np.log(rv))).max() < 1e-12
        assert np.abs(b - (np.log(np.abs(v)) - np.log(rv))).max() < 1e-12


@pytest.mark.parametrize("k", [1, 2, 3])
def test_rms_row_and_column_steps_give_unit_rms(oracle, k):
    for x in (_tile(49), _tile(50, sigma=1.5, outliers=4, fac=30.0)):
        Y = oracle.rotate_tile(x)
        a_k, b_k, _ = oracle.sinkhorn(Y, k, rms=True)
        a_n, b_n, _ = oracle.sinkhorn(Y, k + 1, rms=True)
        assert np.abs(_rms(Y * np.exp(-a_n)[:, None] * np.exp(-b_k)[None, :], 1) - 1).max() < 1e-12
        assert np.abs(_rms(Y * np.exp(-a_n)[:, None] * np.exp(-b_n)[None, :], 0) - 1).max() < 1e-12


def test_rms_variant_converges_to_a_doubly_normalized_tile(oracle):
    # Sinkhorn-Knopp on a positive matrix (the squares) converges to a scaling
    # with all row and all column sums equal: every row and every column of Z
    # reaches RMS 1 (no common offset, unlike the centred statistic)
    for x in (_tile(51), _tile(52, sigma=1.0, outliers=4, fac=25.0)):
        Y = oracle.rotate_tile(x)
        a, b, _ = oracle.sinkhorn(Y, 64, rms=True)
        Z = Y * np.exp(-a)[:, None] * np.exp(-b)[None, :]
        assert np.abs(_rms(Z, 0) - 1).max() < 1e-12
        assert np.abs(_rms(Z, 1) - 1).max() < 1e-9


def test_rms_variant_skips_only_zero_rows(oracle):
    rng = np.random.default_rng(53)
    Y = rng.standard_normal((128, 128))
    Y[3] = 0.0                      # zero row: skipped, stays zero
    Y[7] = 2.5                      # constant row: updated (centred would skip it)
    a, b, _ = oracle.sinkhorn(Y, 1, rms=True)
    assert a[3] == 0.0
    assert abs(a[7] - np.log(2.5)) < 1e-12
    ac, _, _ = oracle.sinkhorn(Y, 1)
    assert ac[7] == 0.0


def test_rms_variant_quantizes_through_all_stages(oracle):
    # the variant changes only the scales: codes stay within half a step of
    # the tile normalized by the variant's own scales
    x = _tile(54)
    r = oracle.quantize_tile(x, False, 2, rms=True)
    a, b, _ = oracle.sinkhorn(r["Y"], 2, rms=True)
    assert np.array_equal(r["a"], a) and np.array_equal(r["b"], b)
    c = oracle.quantize_tile(x, False, 2)
    assert not np.array_equal(r["b"], c["b"])


def test_sinkhorn_zero_and_constant_tiles_are_skipped(oracle):
    a, b, _ = oracle.sinkhorn(np.zeros((128, 128)), 3)
    assert not a.any() and not b.any()
    a, b, _ = oracle.sinkhorn(np.full((128, 128), 3.5), 3)
    assert not a.any() and not b.any()
    a, b, _ = oracle.sinkhorn(oracle.rotate_tile(_tile(9)), 0)
    assert not a.any() and not b.any()


# ------------------------------------------------------------------- RTN --

@pytest.mark.parametrize("bits", [4, 2])
def test_rtn_half_step_bound_argmin_and_endpoints(oracle, bits):
    Y = oracle.rotate_tile(_tile(10))
    a, b, _ = oracle.sinkhorn(Y, 2)
    r = np.exp(a)
    c32 = np.exp(b).astype(np.float32)
    q, s32, z32, u = oracle.rtn(Y, r, c32, bits)
    xn = Y / (r[:, None] * c32.astype(np.float64)[None, :])
    mn = xn.min(1)
    mx = xn.max(1)
    s = (mx - mn) / (2 ** bits - 1)
    deq = s[:, None] * q + mn[:, None]
    assert np.all(np.abs(xn - deq) <= s[:, None] / 2 + 1e-12)
    # brute force: q is the nearest level (ties excepted)
    levels = np.arange(2 ** bits)
    dist = np.abs(xn[..., None] - (s[:, None, None] * levels + mn[:, None, None]))
    best = dist.argmin(-1)
    tie = np.abs(u - np.floor(u) - 0.5) < 1e-9
    assert np.array_equal(best[~tie], q[~tie])
    # the row minimum maps to 0 and the row maximum to 2^b - 1
    assert np.all(q[np.arange(128), xn.argmin(1)] == 0)
    assert np.all(q[np.arange(128), xn.argmax(1)] == 2 ** bits - 1)
    # stored metadata is the row scale folded in, rounded to fp32
    assert np.array_equal(s32, (r * s).astype(np.float32))
    assert np.array_equal(z32, (r * mn).astype(np.float32))


@pytest.mark.parametrize("bits", [4, 2])
def test_rtn_sign_symmetry(oracle, bits):
    Y = oracle.rotate_tile(_tile(11))
    r = np.exp(np.random.default_rng(12).standard_normal(128))
    c32 = np.exp(np.random.default_rng(13).standard_normal(128)).astype(np.float32)
    q, _, _, u = oracle.rtn(Y, r, c32, bits)
    q2, _, _, _ = oracle.rtn(-Y, r, c32, bits)
    tie = np.abs(u - np.floor(u) - 0.5) < 1e-9
    assert np.array_equal(q2[~tie], (2 ** bits - 1) - q[~tie])


def test_rtn_constant_row(oracle):
    Y = oracle.rotate_tile(_tile(14))
    Y[5, :] = 2.25
    q, s32, z32, u = oracle.rtn(Y, np.ones(128), np.ones(128, np.float32), 4)
    assert s32[5] == 0.0 and z32[5] == np.float32(2.25)
    assert not q[5].any() and not u[5].any()


@pytest.mark.parametrize("is_v", [False, True])
def test_reconstruction_error_same_in_both_spaces(oracle, is_v):
    # orthonormal H: ||x_t - H yhat_t|| = ||y_t - yhat_t|| for every token
    x = _tile(15)
    out = oracle.quantize_tile(x, is_v, 2)
    yhat = oracle.dequant_part(out["rec"], is_v)
    H = oracle.hadamard(128)
    xhat = yhat @ H.T
    e_x = np.linalg.norm(x.astype(np.float64) - xhat, axis=1)
    e_y = np.linalg.norm(out["Y"] - yhat, axis=1)
    assert np.abs(e_x - e_y).max() < 1e-9 * max(1.0, e_y.max())


@pytest.mark.parametrize("is_v", [False, True])
def test_dequant_within_half_step_of_rotated_tile(oracle, is_v):
    x = _tile(16)
    out = oracle.quantize_tile(x, is_v, 2)
    q, s32, z32, c32 = oracle.unpack_part(out["rec"], is_v)
    yhat = oracle.dequant_part(out["rec"], is_v)
    half = 0.5 * np.abs(s32.astype(np.float64))[:, None] * c32.astype(np.float64)[None, :]
    # fp32 rounding of s', z', c adds a few ulps on top of the half step
    slack = 1e-6 * (np.abs(out["Y"]) + np.abs(yhat)) + 1e-9
    assert np.all(np.abs(out["Y"] - yhat) <= half + slack)


# ------------------------------------------------------------------ pack --

def test_pack_unpack_roundtrip(oracle):
    rng = np.random.default_rng(17)
    for is_v, bits in ((False, 4), (True, 2)):
        q = rng.integers(0, 2 ** bits, (128, 128)).astype(np.uint8)
        s = rng.standard_normal(128).astype(np.float32)
        z = rng.standard_normal(128).astype(np.float32)
        c = np.exp(rng.standard_normal(128)).astype(np.float32)
        rec = np.zeros(15360, np.uint8)
        oracle.pack_part(rec, is_v, q, s, z, c)
        q2, s2, z2, c2 = oracle.unpack_part(rec, is_v)
        assert np.array_equal(q, q2) and np.array_equal(s, s2)
        assert np.array_equal(z, z2) and np.array_equal(c, c2)


def test_pack_golden_bytes(oracle):
    g = json.load(open(os.path.join(GOLDEN, "pack_examples.json")))
    off = g["record_offsets"]
    # K: token 0 channel codes 0..15 repeated
    q = np.zeros((128, 128), np.uint8)
    q[0] = np.tile(np.arange(16), 8)
    q[1, :4] = g["k_row_alternating_15_0"]["codes_first_4_channels"]
    rec = np.zeros(15360, np.uint8)
    oracle.pack_part(rec, False, q, np.zeros(128, np.float32), np.zeros(128, np.float32),
                     np.zeros(128, np.float32))
    want = [int(h, 16) for h in g["k_row_codes_0_to_15_repeated"]["bytes_first_8"]]
    assert list(rec[off["k_codes"]:off["k_codes"] + 8]) == want
    want = [int(h, 16) for h in g["k_row_alternating_15_0"]["bytes_first_2"]]
    assert list(rec[off["k_codes"] + 64:off["k_codes"] + 66]) == want
    # V: hand-derived positions of single codes in the permuted layout
    s = np.arange(128, dtype=np.float32)
    z = -np.arange(128, dtype=np.float32)
    c = np.arange(128, dtype=np.float32) + 0.5
    for ex in g["v_examples"]:
        q = np.zeros((128, 128), np.uint8)
        q[ex["tokens"], ex["channel"]] = ex["codes"]
        rec = np.zeros(15360, np.uint8)
        oracle.pack_part(rec, True, q, s, z, c)
        want = [int(h, 16) for h in ex["bytes"]]
        base = off["v_codes"] + ex["byte_offset"]
        assert list(rec[base:base + len(want)]) == want, ex["_derivation"]
        # and nothing else in the code region is set
        assert int(rec[off["v_codes"]:off["v_scale_zero"]].astype(np.int64).sum()) == sum(want)
    # metadata offsets: {s', z'} per token, then column scales
    sz = rec[off["v_scale_zero"]:off["v_scale_zero"] + 1024].view(np.float32).reshape(128, 2)
    assert np.array_equal(sz[:, 0], s) and np.array_equal(sz[:, 1], z)
    assert np.array_equal(rec[off["v_col_scale"]:off["v_col_scale"] + 512].view(np.float32), c)
    assert off["record_bytes"] == oracle.REC_BYTES
    per = g["bytes_per_token_head"]
    assert per["total"] * 128 == oracle.REC_BYTES
    assert 3.0 <= per["fp16_total"] / per["total"] <= 5.0    # "3-5x capacity"


# ------------------------------------------------------------- attention --

def _small_state(oracle, B=2, S=(300, 517), hkv=2, hq=4, iters=2, seed=21):
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=B, seq=max(S), hkv=hkv, hq=hq,
                     seed=seed)
    k, v = synth.kv(w)
    lens = np.array(S, dtype=np.int32)
    mb = (max(S) + 127) // 128
    table = np.arange(B * mb, dtype=np.int32).reshape(B, mb)[:, ::-1].copy()   # reversed pages
    st = oracle.quantize_blocks(k.numpy(), v.numpy(), lens, table, B * mb, iters)
    q = synth.queries(w).numpy()
    return w, k.numpy(), v.numpy(), q, lens, table, st


def test_attention_routes_agree(oracle):
    w, k, v, q, lens, table, st = _small_state(oracle)
    oa = oracle.decode_attention(q, st["pool"], table, lens, st["tail_k"], st["tail_v"], w.hq,
                                 w.hkv, route=0)
    ob = oracle.decode_attention(q, st["pool"], table, lens, st["tail_k"], st["tail_v"], w.hq,
                                 w.hkv, route=1)
    assert np.abs(oa - ob).max() <= 1e-12 * np.abs(oa).max()


def test_attention_matches_torch_softmax(oracle):
    w, k, v, q, lens, table, st = _small_state(oracle)
    out = oracle.decode_attention(q, st["pool"], table, lens, st["tail_k"], st["tail_v"], w.hq,
                                  w.hkv, route=0)
    H = torch.tensor(oracle.hadamard(128))
    g = w.hq // w.hkv
    for b in range(w.batch):
        n = int(lens[b])
        nfull = n // 128
        for h in range(w.hq):
            kvh = h // g
            keys, vals = [], []
            for j in range(nfull):
                rec = st["pool"][table[b, j], kvh]
                keys.append(torch.tensor(oracle.dequant_part(rec, False)) @ H)   # rows H yhat
                vals.append(torch.tensor(oracle.dequant_part(rec, True)) @ H)
            keys.append(torch.tensor(k[b, nfull * 128:n, kvh].astype(np.float64)))
            vals.append(torch.tensor(v[b, nfull * 128:n, kvh].astype(np.float64)))
            K = torch.cat(keys)
            V = torch.cat(vals)
            p = torch.softmax(K @ torch.tensor(q[b, h].astype(np.float64)) / np.sqrt(128.0), 0)
            ref = (p[:, None] * V).sum(0).numpy()
            assert np.abs(out[b, h] - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


def test_attention_special_cases(oracle):
    rng = np.random.default_rng(22)
    B, hkv, hq = 3, 1, 2
    pool = np.zeros((4, hkv, 15360), np.uint8)
    table = np.zeros((B, 4), np.int32)
    tk = rng.standard_normal((B, hkv, 128, 128)).astype(np.float16)
    tv = rng.standard_normal((B, hkv, 128, 128)).astype(np.float16)
    q = rng.standard_normal((B, hq, 128)).astype(np.float16)
    tk[2, 0, :50] = tk[2, 0, 0]                  # all 50 keys equal
    lens = np.array([0, 1, 50], np.int32)
    out = oracle.decode_attention(q, pool, table, lens, tk, tv, hq, hkv)
    assert not out[0].any()                                       # empty sequence
    assert np.array_equal(out[1, 0], tv[1, 0, 0].astype(np.float64))  # one token
    assert np.abs(out[2] - tv[2, 0, :50].astype(np.float64).mean(0)).max() < 1e-13
    # GQA: both query heads read KV head 0, so equal queries give equal outputs
    q[:, 1] = q[:, 0]
    out = oracle.decode_attention(q, pool, table, lens, tk, tv, hq, hkv)
    assert np.array_equal(out[:, 0], out[:, 1])


def test_softmax_shift_invariance(oracle):
    # adding the same constant to every score leaves o unchanged; realise it by
    # adding an integer delta to channel j of every (tail) key: the score of
    # token t moves by scale * q_j * delta for all t alike.  Channel j holds
    # small integers so the fp16 keys stay exact.
    rng = np.random.default_rng(23)
    q = rng.standard_normal((1, 1, 128)).astype(np.float16)
    tk = rng.standard_normal((1, 1, 128, 128)).astype(np.float16)
    tv = rng.standard_normal((1, 1, 128, 128)).astype(np.float16)
    j = 17
    tk[0, 0, :, j] = rng.integers(-8, 8, 128).astype(np.float16)
    tk2 = tk.copy()
    tk2[0, 0, :, j] = (tk[0, 0, :, j].astype(np.float64) + 5.0).astype(np.float16)
    lens = np.array([100], np.int32)
    pool = np.zeros((1, 1, 15360), np.uint8)
    table = np.zeros((1, 1), np.int32)
    o1 = oracle.decode_attention(q, pool, table, lens, tk, tv, 1, 1)
    o2 = oracle.decode_attention(q, pool, table, lens, tk2, tv, 1, 1)
    assert np.abs(o1 - o2).max() < 1e-13


# ------------------------------------------------------- prefill / append --

def test_prefill_tail_copy_and_page_placement(oracle):
    w, k, v, q, lens, table, st = _small_state(oracle)
    for b in range(w.batch):
        n = int(lens[b])
        nfull, rem = n // 128, n % 128
        assert np.array_equal(st["tail_k"][b, :, :rem].transpose(1, 0, 2),
                              k[b, nfull * 128:n].view(np.uint16))
        assert np.array_equal(st["tail_v"][b, :, :rem].transpose(1, 0, 2),
                              v[b, nfull * 128:n].view(np.uint16))
        # page j of sequence b holds exactly the tile quantized alone
        for j in range(nfull):
            for h in range(w.hkv):
                solo = oracle.quantize_tile(k[b, j * 128:(j + 1) * 128, h], False, 2)["rec"]
                got = st["pool"][table[b, j], h]
                assert np.array_equal(got[:9728], solo[:9728])   # the whole K part


def test_append_fills_page_like_prefill(oracle):
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=2, seq=256, hkv=2, hq=4, seed=31)
    k, v = synth.kv(w)
    k, v = k.numpy(), v.numpy()
    lens = np.array([256, 256], np.int32)
    table = np.array([[0, 1], [2, 3]], np.int32)
    ref = oracle.quantize_blocks(k, v, lens, table, 4, 2)
    pool = np.zeros((4, 2, 15360), np.uint8)
    tk = np.zeros((2, 2, 128, 128), np.uint16)
    tv = np.zeros((2, 2, 128, 128), np.uint16)
    for pos in range(256):
        rc = oracle.append_token(k[:, pos], v[:, pos], np.array([pos, pos], np.int32), table, 2,
                                 pool, tk, tv)
        assert rc == 0
    assert np.array_equal(pool, ref["pool"])
    # idle slots (pos < 0) are untouched
    before = tk.copy()
    oracle.append_token(k[:, 0], v[:, 0], np.array([-1, -1], np.int32), table, 2, pool, tk, tv)
    assert np.array_equal(before, tk)


# --------------------------------------------------- method sanity (info) --

def test_method_beats_plain_rtn_on_outlier_keys(oracle):
    """Rotation + normalization lower the K reconstruction error against plain
    per-token 4-bit RTN of the raw tile (stage 2's outlier spreading).  The
    size of the gain is not pinned: the pages print no accuracy figures."""
    x = _tile(40, sigma=1.0, outliers=4, fac=30.0)
    out = oracle.quantize_tile(x, False, 2)
    H = oracle.hadamard(128)
    xhat = oracle.dequant_part(out["rec"], False) @ H.T
    err_kvarn = np.linalg.norm(x.astype(np.float64) - xhat)
    q, s32, z32, _ = oracle.rtn(x.astype(np.float64), np.ones(128), np.ones(128, np.float32), 4)
    plain = s32.astype(np.float64)[:, None] * q + z32.astype(np.float64)[:, None]
    err_plain = np.linalg.norm(x.astype(np.float64) - plain)
    assert err_kvarn < 0.5 * err_plain


# ------------------------------------------- the FP16 baseline's attention --

def test_fp16_attention_matches_torch_sdpa(oracle):
    """attention_fp16 equals torch's scaled_dot_product_attention (a library
    routine) in float64, with GQA and ragged lengths (keys beyond the length
    masked out)."""
    import torch
    g = torch.Generator().manual_seed(5)
    B, S, hq, hkv = 3, 37, 6, 2
    q = torch.randn(B, hq, 128, generator=g).half()
    k = torch.randn(B, S, hkv, 128, generator=g).half()
    v = torch.randn(B, S, hkv, 128, generator=g).half()
    lens = np.array([37, 5, 20])
    got = oracle.attention_fp16(q, k, v, lens, hq, hkv)
    for b in range(B):
        n = int(lens[b])
        kk = k[b, :n].double().repeat_interleave(hq // hkv, dim=1).permute(1, 0, 2)
        vv = v[b, :n].double().repeat_interleave(hq // hkv, dim=1).permute(1, 0, 2)
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[b].double()[:, None, :], kk, vv, scale=128 ** -0.5)[:, 0, :]
        assert np.abs(got[b] - ref.numpy()).max() < 1e-12


def test_fp16_attention_special_cases(oracle):
    import torch
    g = torch.Generator().manual_seed(6)
    q = torch.randn(2, 2, 128, generator=g).half()
    k = torch.randn(2, 4, 1, 128, generator=g).half()
    v = torch.randn(2, 4, 1, 128, generator=g).half()
    out = oracle.attention_fp16(q, k, v, np.array([1, 0]), 2, 1)
    # one token: its value; no token: zeros
    assert np.array_equal(out[0, 0], v[0, 0, 0].double().numpy())
    assert np.array_equal(out[1], np.zeros((2, 128)))
    # equal keys: the mean of the values
    k[:] = k[0, 0, 0]
    out = oracle.attention_fp16(q, k, v, np.array([4, 4]), 2, 1)
    assert np.abs(out[0, 1] - v[0, :, 0].double().mean(0).numpy()).max() < 1e-12


# ------------------------------------------------- chunked prefill (next) --

def _chunk_state(oracle, start=(250, 100, 0), m=(150, 60, 60), hkv=2, hq=4, seed=31):
    """Caches holding start + m tokens (the chunk already appended: a page is
    what 128 appends make, pinned above), and M = max(m) query rows."""
    n = [s + c for s, c in zip(start, m)]
    B, M = len(n), max(m)
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=B, seq=max(n), hkv=hkv, hq=hq,
                     seed=seed)
    k, v = synth.kv(w)
    lens = np.array(n, dtype=np.int32)
    mb = (max(n) + 127) // 128
    table = np.arange(B * mb, dtype=np.int32).reshape(B, mb)[:, ::-1].copy()
    st = oracle.quantize_blocks(k.numpy(), v.numpy(), lens, table, B * mb, 2)
    q = np.random.default_rng(seed).standard_normal((B, M, hq, 128)).astype(np.float16)
    return k.numpy(), v.numpy(), q, np.array(start), np.array(m), table, st


def test_chunk_rows_at_whole_pages_and_the_last_row_equal_decode(oracle):
    # a query whose prefix is whole pages, or the whole cache, sees exactly
    # what decode attention over that many tokens sees
    k, v, q, start, m, table, st = _chunk_state(oracle)
    hq, hkv = q.shape[2], st["pool"].shape[1]
    out = oracle.chunk_attention(q, start, m, st["pool"], table, st["tail_k"], st["tail_v"], hq,
                                 hkv)
    checked = 0
    for b in range(len(start)):
        for i in range(int(m[b])):
            P = int(start[b]) + i
            if (P + 1) % 128 and i != m[b] - 1:
                continue
            ref = oracle.decode_attention(q[b:b + 1, i], st["pool"], table[b:b + 1],
                                          np.array([P + 1], np.int32), st["tail_k"][b:b + 1],
                                          st["tail_v"][b:b + 1], hq, hkv, route=0)[0]
            assert np.abs(out[b, i] - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())
            checked += 1
    assert checked == 6     # P + 1 = 256, 384, 400 | 128, 160 | 60
    assert not out[1, 60:].any() and not out[2, 60:].any()   # rows past the chunk


def test_chunk_within_one_block_is_causal_fp16_attention(oracle):
    # sequence 2 has 60 tokens, all in the fp16 tail: row i is plain attention
    # over the first i + 1 raw tokens (the fp16 oracle, pinned to torch above)
    k, v, q, start, m, table, st = _chunk_state(oracle)
    hq, hkv = q.shape[2], st["pool"].shape[1]
    out = oracle.chunk_attention(q, start, m, st["pool"], table, st["tail_k"], st["tail_v"], hq,
                                 hkv)
    for i in (0, 1, 17, 59):
        ref = oracle.attention_fp16(q[2:3, i], k[2:3], v[2:3], np.array([i + 1]), hq, hkv)[0]
        assert np.abs(out[2, i] - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())
    assert np.array_equal(out[2, 0, 0], v[2, 0, 0].astype(np.float64))   # one token: its value


def test_chunk_attention_is_causal(oracle):
    # changing token 394 (tail slot 10 of sequence 0) moves rows P >= 394 only
    k, v, q, start, m, table, st = _chunk_state(oracle)
    hq, hkv = q.shape[2], st["pool"].shape[1]
    args = (st["pool"], table)
    o1 = oracle.chunk_attention(q, start, m, *args, st["tail_k"], st["tail_v"], hq, hkv)
    tk, tv = st["tail_k"].copy(), st["tail_v"].copy()
    tk[0, :, 10] = tk[0, :, 3]
    tv[0, :, 10] = (tv[0, :, 10].view(np.float16) * 3).view(tv.dtype)
    o2 = oracle.chunk_attention(q, start, m, *args, tk, tv, hq, hkv)
    cut = 394 - int(start[0])
    assert np.array_equal(o1[0, :cut], o2[0, :cut])
    assert (np.abs(o1[0, cut:150] - o2[0, cut:150]).max(axis=(1, 2)) > 0).all()
    assert np.array_equal(o1[1:], o2[1:])


def test_chunk_attention_gqa_heads_share_their_kv_head(oracle):
    k, v, q, start, m, table, st = _chunk_state(oracle)
    hq, hkv = q.shape[2], st["pool"].shape[1]
    q[:, :, 1] = q[:, :, 0]      # heads 0 and 1 read KV head 0 (g = 2)
    q[:, :, 3] = q[:, :, 0]      # head 3 reads KV head 1
    out = oracle.chunk_attention(q, start, m, st["pool"], table, st["tail_k"], st["tail_v"], hq,
                                 hkv)
    assert np.array_equal(out[:, :, 0], out[:, :, 1])
    assert not np.array_equal(out[0, :150, 0], out[0, :150, 3])


# ---------------------------------------------------------- FP8 cache --
# The FP8 paged cache (the glossary's INT8/FP8 KV quantization, "KV Cache
# (Anahtar-Deger Onbellegi)", "Sik Sorulan Sorular"): e4m3 codes with a
# per-token absmax scale.  Its arithmetic is pinned to torch's float8_e4m3fn
# conversion (round to nearest even) and to textbook attention.

def test_e4m3_decode_matches_torch_for_every_code(oracle):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_decode(c) for c in range(256)])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin]) and np.all(np.isnan(got[~fin]))
    assert oracle.e4m3_decode(0x7E) == 448.0 and oracle.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_encode_matches_torch_rounding(oracle):
    rng = np.random.default_rng(60)
    u = np.concatenate([rng.standard_normal(4000) * 30, rng.uniform(-463.9, 463.9, 2000),
                        rng.standard_normal(2000) * 1e-2, rng.standard_normal(500) * 1e-3])
    # every midpoint between neighbouring codes: ties go to the even code
    vals = np.array([oracle.e4m3_decode(c) for c in range(0x7F)])
    mids = (vals[:-1] + vals[1:]) / 2
    u = np.concatenate([u, mids, -mids]).astype(np.float32)
    ref = torch.from_numpy(u).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(x) for x in u], dtype=np.uint8)
    same = (got == ref) | ((got & 0x7F) == 0) & ((ref & 0x7F) == 0)   # +-0
    assert same.all(), (u[~same][:5], got[~same][:5], ref[~same][:5])


def test_e4m3_encode_saturates(oracle):
    for x, c in ((464.0, 0x7E), (1e6, 0x7E), (-1e6, 0xFE), (448.0, 0x7E), (-449.0, 0xFE)):
        assert oracle.e4m3_encode(x) == c


def test_fp8_token_scale_and_half_step_bound(oracle):
    rng = np.random.default_rng(61)
    x = (rng.standard_normal(128) * np.exp(rng.standard_normal(128))).astype(np.float16)
    codes, s = oracle.fp8_quantize_token(x)
    xd = x.astype(np.float64)
    assert s == np.float32(np.float32(np.abs(xd).max()) / np.float32(448.0))
    deq = np.array([oracle.e4m3_decode(c) for c in codes]) * s
    # the largest element maps to the top code; every element lies within
    # half a code step (relative 2^-4) of its decoded value, or half the
    # smallest subnormal step below 2^-6
    assert abs(deq[np.argmax(np.abs(xd))]) == pytest.approx(np.abs(xd).max(), rel=2 ** -4)
    assert np.all(np.abs(deq - xd) <= np.maximum(np.abs(xd) * 2 ** -4, s * 2 ** -10) + 1e-12)
    codes0, s0 = oracle.fp8_quantize_token(np.zeros(128, np.float16))
    assert s0 == 0.0 and not codes0.any()


def test_fp8_attention_matches_torch_sdpa_on_dequantized_cache(oracle):
    rng = np.random.default_rng(62)
    B, S, hkv, hq = 2, 300, 2, 8
    k = (rng.standard_normal((B, S, hkv, 128)) * 3).astype(np.float16)
    v = rng.standard_normal((B, S, hkv, 128)).astype(np.float16)
    q = rng.standard_normal((B, hq, 128)).astype(np.float16)
    lens = np.array([300, 129], dtype=np.int32)
    table = np.array([[0, 1, 2], [3, 4, 5]], dtype=np.int32)
    pool = oracle.fp8_write_blocks(k, v, lens, table, 6)
    out = oracle.fp8_decode_attention(q, pool, table, lens, hq, hkv)
    for b in range(B):
        n = int(lens[b])
        for kvh in range(hkv):
            K = np.zeros((n, 128))
            V = np.zeros((n, 128))
            for t in range(n):
                pg = pool[table[b, t // 128], kvh]
                sk = pg[32768 + 4 * (t % 128):32772 + 4 * (t % 128)].view(np.float32)[0]
                sv = pg[33280 + 4 * (t % 128):33284 + 4 * (t % 128)].view(np.float32)[0]
                kc = torch.from_numpy(pg[(t % 128) * 128:(t % 128 + 1) * 128].copy())
                vc = torch.from_numpy(pg[16384 + (t % 128) * 128:16384 + (t % 128 + 1) * 128].copy())
                K[t] = kc.view(torch.float8_e4m3fn).to(torch.float64).numpy() * sk
                V[t] = vc.view(torch.float8_e4m3fn).to(torch.float64).numpy() * sv
            qq = torch.from_numpy(q[b, kvh * 4:(kvh + 1) * 4].astype(np.float64))[None, :, None]
            ref = torch.nn.functional.scaled_dot_product_attention(
                qq, torch.from_numpy(K)[None, None].expand(1, 4, n, 128),
                torch.from_numpy(V)[None, None].expand(1, 4, n, 128))
            assert np.abs(out[b, kvh * 4:(kvh + 1) * 4] - ref[0, :, 0].numpy()).max() < 1e-12


# ------------------------------------------------- SnapKV-style selection --
# "Makale Bulteni - SnapKV" (cmlonder.com): the observation window's attention
# over the prefix, pooled, then each head's top positions kept.

def _snap_inputs(seed, B=2, S=300, hkv=2, hq=8, W=16):
    rng = np.random.default_rng(seed)
    k = (rng.standard_normal((B, S, hkv, 128)) * 2).astype(np.float16)
    q = rng.standard_normal((B, W, hq, 128)).astype(np.float16)
    return q, k


def test_snapkv_votes_are_softmax_mass_on_the_prefix(oracle):
    # each window query's softmax sums to 1 over its causal context, so the
    # votes of a KV head plus that mass on the window tokens is W x g
    q, k = _snap_inputs(70)
    lens = np.array([300, 200])
    W, g = 16, 4
    votes = oracle.snapkv_votes(q, k, lens, 8, 2)
    for b in range(2):
        n = int(lens[b])
        for h in range(2):
            win_mass = 0.0
            for i in range(W):
                P = n - W + i
                for hh in range(g):
                    qq = torch.from_numpy(q[b, i, h * g + hh].astype(np.float64))
                    kk = torch.from_numpy(k[b, :P + 1, h].astype(np.float64))
                    a = torch.softmax(kk @ qq / np.sqrt(128.0), 0).numpy()
                    win_mass += a[n - W:].sum()
            assert abs(votes[b, h].sum() + win_mass - W * g) < 1e-9
            assert not votes[b, h, n - W:].any()


def test_snapkv_pool_equals_scipy_maximum_filter(oracle):
    from scipy.ndimage import maximum_filter1d
    v = np.random.default_rng(71).random(257)
    for kern in (1, 3, 7, 9):
        ref = maximum_filter1d(v, size=kern, mode="nearest")
        assert np.array_equal(oracle.snapkv_pool(v, kern), ref)


def test_snapkv_select_brute_force_and_ties(oracle):
    rng = np.random.default_rng(72)
    votes = rng.random((1, 2, 100))
    votes[0, 1, :] = 0.5                                  # all tied: lowest positions
    lens = np.array([90])
    idx = oracle.snapkv_select(votes, lens, window=10, capacity=30, kernel=1)
    pooled = votes[0, 0, :80]
    assert np.array_equal(idx[0, 0, :20], np.sort(np.argsort(-pooled, kind="stable")[:20]))
    assert np.array_equal(idx[0, 0, 20:], np.arange(80, 90))
    assert np.array_equal(idx[0, 1], np.concatenate([np.arange(20), np.arange(80, 90)]))
    # a short prompt is kept whole, the rest marked -1
    idx = oracle.snapkv_select(votes, np.array([25]), window=10, capacity=30)
    assert np.array_equal(idx[0, 0, :25], np.arange(25)) and (idx[0, 0, 25:] == -1).all()


def test_snapkv_keeps_the_cluster_around_a_planted_key(oracle):
    # a key aligned with every window query at position 100 draws the votes;
    # pooling with kernel 7 spreads its score to 97..103, which are kept
    q, k = _snap_inputs(73, B=1, S=300, hkv=1, hq=2)
    qm = q.astype(np.float64).mean(axis=(1, 2))[0]
    k[0, 100, 0] = (qm / np.linalg.norm(qm) * 40).astype(np.float16)
    votes = oracle.snapkv_votes(q, k, np.array([300]), 2, 1)
    assert votes[0, 0].argmax() == 100
    idx = oracle.snapkv_select(votes, np.array([300]), window=16, capacity=40, kernel=7)
    assert set(range(97, 104)) <= set(idx[0, 0].tolist())


# ------------------------------------------- format variant: fp16 metadata --
# Format variant "_m16" (the metadata of the KVarN record stored as fp16,
# 108 B per token-head instead of 120): the KVarN page (blog.edumints.com),
# "KVarN Nasil Calisir?", stage "Kuantize Edilmis Onbellek", fixes the codes;
# the metadata width is a reading.  Pinned against numpy's own float16
# rounding, the fp32 record, and attention on the dequantized cache.

def test_f32_to_f16_matches_numpy_rounding(oracle):
    rng = np.random.default_rng(41)
    vals = np.concatenate([
        rng.standard_normal(3000) * np.exp(rng.uniform(-20, 12, 3000)),   # every binade
        rng.uniform(-1e-7, 1e-7, 500),                                     # subnormals
        np.array([0.0, -0.0, 1.0, -2.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -24,
                  2.0 ** -25, 1.5 * 2.0 ** -25, 2.0 ** -14 - 2.0 ** -25, 6.1e-5]),
    ]).astype(np.float32)
    # exact ties between two fp16 neighbours, both parities
    base = rng.integers(0x0400, 0x7BFF, 400).astype(np.uint16).view(np.float16).astype(np.float64)
    ulp = np.spacing(base.astype(np.float16)).astype(np.float64)
    ties = (base + 0.5 * ulp).astype(np.float32)
    with np.errstate(over="ignore"):
        for x in np.concatenate([vals, ties]):
            want = int(np.array([x], np.float32).astype(np.float16).view(np.uint16)[0])
            assert oracle.f32_to_f16(x) == want, (x, hex(want))


def test_m16_record_is_the_fp32_record_with_fp16_metadata(oracle):
    x = _tile(42)
    for is_v in (False, True):
        a = oracle.quantize_tile(x, is_v, 2)
        b = oracle.quantize_tile(x, is_v, 2, meta16=True)
        assert b["rec"].size == oracle.REC_BYTES_M16 == 108 * 128
        q32, s32, z32, c32 = oracle.unpack_part(a["rec"], is_v)
        q16, s16, z16, c16 = oracle.unpack_part(b["rec"], is_v, meta16=True)
        assert np.array_equal(q32, q16)                      # the same codes
        for m32, m16 in ((s32, s16), (z32, z16), (c32, c16)):
            assert np.array_equal(m32.astype(np.float16).astype(np.float32), m16)
        # the raw bytes at the stated offsets: codes, {s', z'} pairs, c
        rec = b["rec"]
        if not is_v:
            assert np.array_equal(rec[:8192], a["rec"][:8192])
            sz = rec[8192:8704].view(np.float16).reshape(128, 2)
            cc = rec[8704:8960].view(np.float16)
        else:
            assert np.array_equal(rec[8960:13056], a["rec"][9728:13824])
            sz = rec[13056:13568].view(np.float16).reshape(128, 2)
            cc = rec[13568:13824].view(np.float16)
        assert np.array_equal(sz[:, 0], s32.astype(np.float16))
        assert np.array_equal(sz[:, 1], z32.astype(np.float16))
        assert np.array_equal(cc, c32.astype(np.float16))


def test_m16_dequant_within_fp16_rounding_of_the_fp32_record(oracle):
    x = _tile(43)
    for is_v in (False, True):
        a = oracle.quantize_tile(x, is_v, 2)
        b = oracle.quantize_tile(x, is_v, 2, meta16=True)
        y32 = oracle.dequant_part(a["rec"], is_v)
        y16 = oracle.dequant_part(b["rec"], is_v, meta16=True)
        q, s, z, c = oracle.unpack_part(a["rec"], is_v)
        s, z, c = (np.abs(t.astype(np.float64)) for t in (s, z, c))
        # each of c, s', z' moves by at most half an fp16 ulp (2^-11 relative)
        u = 2.0 ** -11
        bound = c[None, :] * (s[:, None] * q + z[:, None]) * (2 * u + u * u) + 1e-12
        assert np.all(np.abs(y16 - y32) <= bound)
        assert np.abs(y16 - y32).max() > 0                   # the rounding is really there


def test_m16_attention_matches_torch_softmax_on_dequantized_cache(oracle):
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=2, seq=517, hkv=2, hq=4, seed=44)
    k, v = synth.kv(w)
    k, v = k.numpy(), v.numpy()
    lens = np.array([300, 517], np.int32)
    table = np.array([[5, 1, 3, 7, 0], [2, 6, 4, 8, 9]], np.int32)
    st = oracle.quantize_blocks(k, v, lens, table, 10, 2, meta16=True)
    assert st["pool"].shape == (10, 2, 13824) and st["rc"] == 0
    q = synth.queries(w).numpy()
    o1 = oracle.decode_attention(q, st["pool"], table, lens, st["tail_k"], st["tail_v"], 4, 2,
                                 meta16=True)
    o0 = oracle.decode_attention(q, st["pool"], table, lens, st["tail_k"], st["tail_v"], 4, 2,
                                 route=0, meta16=True)
    assert np.abs(o0 - o1).max() <= 1e-12 * np.abs(o0).max()
    H = torch.tensor(oracle.hadamard(128))
    for b in range(2):
        n = int(lens[b])
        nfull = n // 128
        for h in range(4):
            keys, vals = [], []
            for j in range(nfull):
                rec = st["pool"][table[b, j], h // 2]
                keys.append(torch.tensor(oracle.dequant_part(rec, False, True)) @ H)
                vals.append(torch.tensor(oracle.dequant_part(rec, True, True)) @ H)
            keys.append(torch.tensor(k[b, nfull * 128:n, h // 2].astype(np.float64)))
            vals.append(torch.tensor(v[b, nfull * 128:n, h // 2].astype(np.float64)))
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.tensor(q[b, h].astype(np.float64))[None, None, None],
                torch.cat(keys)[None, None], torch.cat(vals)[None, None])[0, 0, 0].numpy()
            assert np.abs(o1[b, h] - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())
    # and the fp32-metadata cache of the same tokens gives nearly the same output
    st32 = oracle.quantize_blocks(k, v, lens, table, 10, 2)
    o32 = oracle.decode_attention(q, st32["pool"], table, lens, st32["tail_k"], st32["tail_v"],
                                  4, 2)
    assert np.abs(o32 - o1).max() <= 1e-2 * np.abs(o32).max()


def test_m16_append_fills_page_like_prefill(oracle):
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=1, seq=256, hkv=2, hq=4, seed=45)
    k, v = synth.kv(w)
    k, v = k.numpy(), v.numpy()
    table = np.array([[1, 0]], np.int32)
    ref = oracle.quantize_blocks(k, v, np.array([256], np.int32), table, 2, 2, meta16=True)
    st = oracle.quantize_blocks(k, v, np.array([250], np.int32), table, 2, 2, meta16=True)
    for t in range(250, 256):
        rc = oracle.append_token(k[:, t], v[:, t], np.array([t], np.int32), table, 2, st["pool"],
                                 st["tail_k"], st["tail_v"], meta16=True)
        assert rc == 0
    assert np.array_equal(st["pool"], ref["pool"])


# ---------------------------------------- format variant: per-channel groups --
# Format variant "_pc" (per-channel grouping): after the same
# rotation and normalization, one RTN group is one channel's 128 tokens; the
# row scale r_t is stored per token and c_d folds into the per-channel scale
# and zero (yhat_td = r_t (cs_d q_td + cz_d)).  The KVarN page (blog.edumints.com,
# "KVarN Nasil Calisir?", stage "Kuantize Edilmis Onbellek") fixes per-token
# groups; the variant is a reading.

def test_pc_rtn_is_the_per_token_rtn_of_the_transposed_tile(oracle):
    # with r exactly representable in fp32, swapping the roles of tokens and
    # channels (and of r and c) turns per-channel groups into per-token ones:
    # the same x_td, so the same codes and the same scale and zero products
    rng = np.random.default_rng(51)
    Y = rng.standard_normal((128, 128)) * np.exp(rng.standard_normal(128))[None, :]
    r = np.exp(rng.standard_normal(128)).astype(np.float32).astype(np.float64)
    c32 = np.exp(0.5 * rng.standard_normal(128)).astype(np.float32)
    for bits in (4, 2):
        q, r32, cs, cz, u = oracle.rtn_pc(Y, r, c32, bits)
        qt, st, zt, ut = oracle.rtn(Y.T.copy(), c32.astype(np.float64), r.astype(np.float32), bits)
        assert np.array_equal(q, qt.T) and np.array_equal(u, ut.T)
        assert np.array_equal(cs, st) and np.array_equal(cz, zt)
        assert np.array_equal(r32, r.astype(np.float32))


def test_pc_rtn_half_step_bound_and_endpoints(oracle):
    x = _tile(52)
    for is_v, bits in ((False, 4), (True, 2)):
        out = oracle.quantize_tile(x, is_v, 2, pc=True)
        q, r, cs, cz = oracle.unpack_part_pc(out["rec"], is_v)
        yhat = oracle.dequant_part(out["rec"], is_v, pc=True)
        r64, cs64 = r.astype(np.float64), cs.astype(np.float64)
        half = 0.5 * np.abs(r64)[:, None] * np.abs(cs64)[None, :]
        slack = 1e-6 * (np.abs(out["Y"]) + np.abs(yhat)) + 1e-9
        assert np.all(np.abs(out["Y"] - yhat) <= half + slack)
        # every channel uses both ends of its range
        assert np.all(q.min(axis=0) == 0) and np.all(q.max(axis=0) == 2 ** bits - 1)


def test_pc_record_bytes_at_the_stated_offsets(oracle):
    x = _tile(53)
    for is_v, qmax in ((False, 15), (True, 3)):
        out = oracle.quantize_tile(x, is_v, 2, pc=True)
        rec = out["rec"]
        assert rec.size == 15360
        codes = (9728, 13824) if is_v else (0, 8192)
        rr = rec[(13824 if is_v else 8192):(14336 if is_v else 8704)].view(np.float32)
        pairs = rec[(14336 if is_v else 8704):(15360 if is_v else 9728)].view(np.float32)
        pairs = pairs.reshape(128, 2)
        a = np.exp(out["a"])
        c32 = np.exp(out["b"]).astype(np.float32)
        assert np.array_equal(rr, a.astype(np.float32))                 # r_t = e^{a_t}
        # the code region is the shared packer's output for these codes
        rec_q = np.zeros(15360, np.uint8)
        oracle.pack_part(rec_q, is_v, out["q"], np.zeros(128, np.float32),
                         np.zeros(128, np.float32), np.zeros(128, np.float32))
        assert np.array_equal(rec[codes[0]:codes[1]], rec_q[codes[0]:codes[1]])
        # {cs_d, cz_d} = c_d times the channel's step and minimum
        xd = out["Y"] / (a[:, None] * c32.astype(np.float64)[None, :])
        step = (xd.max(axis=0) - xd.min(axis=0)) / qmax
        assert np.allclose(pairs[:, 0] / c32, step, rtol=1e-6)
        assert np.allclose(pairs[:, 1] / c32, xd.min(axis=0), rtol=1e-6, atol=1e-12)


def test_pc_attention_matches_torch_sdpa_on_dequantized_cache(oracle):
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=2, seq=517, hkv=2, hq=4, seed=54)
    k, v = synth.kv(w)
    k, v = k.numpy(), v.numpy()
    lens = np.array([300, 517], np.int32)
    table = np.array([[5, 1, 3, 7, 0], [2, 6, 4, 8, 9]], np.int32)
    st = oracle.quantize_blocks(k, v, lens, table, 10, 2, pc=True)
    assert st["rc"] == 0
    q = synth.queries(w).numpy()
    o1 = oracle.decode_attention(q, st["pool"], table, lens, st["tail_k"], st["tail_v"], 4, 2,
                                 pc=True)
    o0 = oracle.decode_attention(q, st["pool"], table, lens, st["tail_k"], st["tail_v"], 4, 2,
                                 route=0, pc=True)
    assert np.abs(o0 - o1).max() <= 1e-12 * np.abs(o0).max()
    H = torch.tensor(oracle.hadamard(128))
    for b in range(2):
        n = int(lens[b])
        nfull = n // 128
        for h in range(4):
            keys, vals = [], []
            for j in range(nfull):
                rec = st["pool"][table[b, j], h // 2]
                keys.append(torch.tensor(oracle.dequant_part(rec, False, pc=True)) @ H)
                vals.append(torch.tensor(oracle.dequant_part(rec, True, pc=True)) @ H)
            keys.append(torch.tensor(k[b, nfull * 128:n, h // 2].astype(np.float64)))
            vals.append(torch.tensor(v[b, nfull * 128:n, h // 2].astype(np.float64)))
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.tensor(q[b, h].astype(np.float64))[None, None, None],
                torch.cat(keys)[None, None], torch.cat(vals)[None, None])[0, 0, 0].numpy()
            assert np.abs(o1[b, h] - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


def test_pc_append_fills_page_like_prefill(oracle):
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=1, seq=256, hkv=2, hq=4, seed=55)
    k, v = synth.kv(w)
    k, v = k.numpy(), v.numpy()
    table = np.array([[1, 0]], np.int32)
    ref = oracle.quantize_blocks(k, v, np.array([256], np.int32), table, 2, 2, pc=True)
    st = oracle.quantize_blocks(k, v, np.array([250], np.int32), table, 2, 2, pc=True)
    for t in range(250, 256):
        assert oracle.append_token(k[:, t], v[:, t], np.array([t], np.int32), table, 2,
                                   st["pool"], st["tail_k"], st["tail_v"], pc=True) == 0
    assert np.array_equal(st["pool"], ref["pool"])


def test_rotation_of_a_constant_tile_is_exact(oracle):
    # H x for a constant x is (sqrt(128) x0, 0, ..., 0): the zero channels
    # must come out exactly zero, since the skip rules of the normalization
    # (and the "_rms" rule above all: only all-zero columns are skipped) act
    # on exact zeros
    for v in (1.5, -0.3, 65504.0):
        Y = oracle.rotate_tile(np.full((128, 128), v, np.float16))
        assert np.all(Y[:, 1:] == 0.0)
        assert np.allclose(Y[:, 0], np.sqrt(128.0) * np.float64(np.float16(v)), rtol=1e-15)


def test_rms_variant_constant_tile_closed_form(oracle):
    # y_t = (v sqrt(128), 0, ...): row 1 gives r = |v|, column 1 c_0 = sqrt(128)
    # (the zero columns are skipped), row 2 r = |v| / sqrt(128), column 2
    # c_0 = 128
    for v in (1.5, -2.0):
        Y = oracle.rotate_tile(np.full((128, 128), v, np.float16))
        a, b, _ = oracle.sinkhorn(Y, 2, rms=True)
        assert np.allclose(np.exp(a), abs(v) / np.sqrt(128.0), rtol=1e-12)
        assert np.isclose(np.exp(b[0]), 128.0, rtol=1e-12) and np.all(b[1:] == 0.0)


# ---------------------------------------------- format variant: group size 64 --
# Format variant "k4v2_g64" (group size 64; the KVarN page names the
# format kvarn_k4v2_g128 in "Yazilim Gelistirme ve Ogrenme Acisindan Pratik
# Cikarimlar", g the group size): two RTN groups per token, channels 0-63 and
# 64-127, each with its own scale and zero; everything else as the default.

def test_g64_rtn_is_the_g128_rtn_of_each_half(oracle):
    # a row whose two halves are the same 64 values has the same range in each
    # half as in the whole row: g64 and g128 then give the same codes, and
    # each group's {s', z'} equals the row's
    rng = np.random.default_rng(61)
    half = rng.standard_normal((128, 64)) * np.exp(rng.standard_normal(64))[None, :]
    Y = np.concatenate([half, half], axis=1)
    r = np.exp(rng.standard_normal(128))
    c_half = np.exp(0.5 * rng.standard_normal(64)).astype(np.float32)
    c32 = np.concatenate([c_half, c_half])
    for bits in (4, 2):
        q64, s64, z64, u64 = oracle.rtn_g64(Y, r, c32, bits)
        q, s, z, u = oracle.rtn(Y, r, c32, bits)
        assert np.array_equal(q64, q) and np.array_equal(u64, u)
        for g in (0, 1):
            assert np.array_equal(s64[:, g], s) and np.array_equal(z64[:, g], z)


def test_g64_half_step_bound_and_group_endpoints(oracle):
    x = _tile(62)
    for is_v, bits in ((False, 4), (True, 2)):
        out = oracle.quantize_tile(x, is_v, 2, g64=True)
        q, s, z, c = oracle.unpack_part_g64(out["rec"], is_v)
        yhat = oracle.dequant_part(out["rec"], is_v, g64=True)
        sg = np.repeat(np.abs(s.astype(np.float64)), 64, axis=1)      # [t][d] step of d's group
        half = 0.5 * sg * c.astype(np.float64)[None, :]
        slack = 1e-6 * (np.abs(out["Y"]) + np.abs(yhat)) + 1e-9
        assert np.all(np.abs(out["Y"] - yhat) <= half + slack)
        for g in (0, 1):
            qg = q[:, 64 * g:64 * (g + 1)]
            assert np.all(qg.min(axis=1) == 0) and np.all(qg.max(axis=1) == 2 ** bits - 1)


def test_g64_record_bytes_at_the_stated_offsets(oracle):
    x = _tile(63)
    for is_v in (False, True):
        out = oracle.quantize_tile(x, is_v, 2, g64=True)
        rec = out["rec"]
        assert rec.size == 17408 == 136 * 128
        codes = (10752, 14848) if is_v else (0, 8192)
        sz = rec[(14848 if is_v else 8192):(16896 if is_v else 10240)].view(np.float32)
        cc = rec[(16896 if is_v else 10240):(17408 if is_v else 10752)].view(np.float32)
        r = np.exp(out["a"])
        c32 = np.exp(out["b"]).astype(np.float32)
        q, s, z, u = oracle.rtn_g64(out["Y"], r, c32, 2 if is_v else 4)
        assert np.array_equal(q, out["q"])
        assert np.array_equal(sz.reshape(128, 2, 2)[:, :, 0], s)
        assert np.array_equal(sz.reshape(128, 2, 2)[:, :, 1], z)
        assert np.array_equal(cc, c32)
        rec_q = np.zeros(15360, np.uint8)
        oracle.pack_part(rec_q, is_v, out["q"], np.zeros(128, np.float32),
                         np.zeros(128, np.float32), np.zeros(128, np.float32))
        lo = 9728 if is_v else 0
        assert np.array_equal(rec[codes[0]:codes[1]], rec_q[lo:lo + codes[1] - codes[0]])


def test_g64_attention_matches_torch_sdpa_on_dequantized_cache(oracle):
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=2, seq=517, hkv=2, hq=4, seed=64)
    k, v = synth.kv(w)
    k, v = k.numpy(), v.numpy()
    lens = np.array([300, 517], np.int32)
    table = np.array([[5, 1, 3, 7, 0], [2, 6, 4, 8, 9]], np.int32)
    st = oracle.quantize_blocks(k, v, lens, table, 10, 2, g64=True)
    assert st["rc"] == 0 and st["pool"].shape == (10, 2, 17408)
    q = synth.queries(w).numpy()
    o1 = oracle.decode_attention(q, st["pool"], table, lens, st["tail_k"], st["tail_v"], 4, 2,
                                 g64=True)
    o0 = oracle.decode_attention(q, st["pool"], table, lens, st["tail_k"], st["tail_v"], 4, 2,
                                 route=0, g64=True)
    assert np.abs(o0 - o1).max() <= 1e-12 * np.abs(o0).max()
    H = torch.tensor(oracle.hadamard(128))
    for b in range(2):
        n = int(lens[b])
        nfull = n // 128
        for h in range(4):
            keys, vals = [], []
            for j in range(nfull):
                rec = st["pool"][table[b, j], h // 2]
                keys.append(torch.tensor(oracle.dequant_part(rec, False, g64=True)) @ H)
                vals.append(torch.tensor(oracle.dequant_part(rec, True, g64=True)) @ H)
            keys.append(torch.tensor(k[b, nfull * 128:n, h // 2].astype(np.float64)))
            vals.append(torch.tensor(v[b, nfull * 128:n, h // 2].astype(np.float64)))
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.tensor(q[b, h].astype(np.float64))[None, None, None],
                torch.cat(keys)[None, None], torch.cat(vals)[None, None])[0, 0, 0].numpy()
            assert np.abs(o1[b, h] - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


def test_g64_append_fills_page_like_prefill(oracle):
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=1, seq=256, hkv=2, hq=4, seed=65)
    k, v = synth.kv(w)
    k, v = k.numpy(), v.numpy()
    table = np.array([[1, 0]], np.int32)
    ref = oracle.quantize_blocks(k, v, np.array([256], np.int32), table, 2, 2, g64=True)
    st = oracle.quantize_blocks(k, v, np.array([250], np.int32), table, 2, 2, g64=True)
    for t in range(250, 256):
        assert oracle.append_token(k[:, t], v[:, t], np.array([t], np.int32), table, 2,
                                   st["pool"], st["tail_k"], st["tail_v"], g64=True) == 0
    assert np.array_equal(st["pool"], ref["pool"])


# --------------------------------------------- format variant: 4-bit values --
# Format variant "k4v4_g128" (4-bit values): the KVarN page fixes 4-bit
# keys and 2-bit values ("Kuantize Edilmis Onbellek"); the variant quantizes
# values at 4 bits too, with a 4-bit V code permutation of its own.

def test_v4_code_positions_golden_and_a_bijection(oracle):
    g = json.load(open(os.path.join(GOLDEN, "pack_v4_examples.json")))
    for ex in g["examples"]:
        assert oracle.v4_code_pos(ex["channel"], ex["token"]) == (ex["byte"], ex["shift"]), \
            ex["_derivation"]
    seen = set()
    for c in range(128):
        for t in range(128):
            byte, shift = oracle.v4_code_pos(c, t)
            assert 0 <= byte < 8192 and shift in (0, 4)
            seen.add((byte, shift))
    assert len(seen) == 128 * 128


def test_v4_values_quantize_like_keys(oracle):
    # at 4 bits the V part runs the same stages as the K part: the same codes,
    # scales and zeros for the same tile
    x = _tile(71)
    k = oracle.quantize_tile(x, False, 2)
    v = oracle.quantize_tile(x, True, 2, v4=True)
    assert np.array_equal(k["q"], v["q"]) and v["q"].max() == 15
    qk, sk, zk, ck = oracle.unpack_part(k["rec"], False)
    qv, sv, zv, cv = oracle.unpack_part(v["rec"], True, v4=True)
    assert np.array_equal(qk, qv)
    assert np.array_equal(sk, sv) and np.array_equal(zk, zv) and np.array_equal(ck, cv)
    assert v["rec"].size == 19456 == 152 * 128
    # the V part's bytes at the stated offsets
    rec = v["rec"]
    assert np.array_equal(rec[17920:18944].view(np.float32).reshape(128, 2)[:, 0], sv)
    assert np.array_equal(rec[18944:19456].view(np.float32), cv)
    for c, t in ((0, 0), (37, 90), (127, 127), (64, 3)):
        byte, shift = oracle.v4_code_pos(c, t)
        assert (rec[9728 + byte] >> shift) & 15 == qv[t, c]


def test_v4_half_step_bound(oracle):
    x = _tile(72)
    out = oracle.quantize_tile(x, True, 2, v4=True)
    q, s, z, c = oracle.unpack_part(out["rec"], True, v4=True)
    yhat = oracle.dequant_part(out["rec"], True, v4=True)
    half = 0.5 * np.abs(s.astype(np.float64))[:, None] * c.astype(np.float64)[None, :]
    slack = 1e-6 * (np.abs(out["Y"]) + np.abs(yhat)) + 1e-9
    assert np.all(np.abs(out["Y"] - yhat) <= half + slack)


def test_v4_attention_matches_torch_sdpa_on_dequantized_cache(oracle):
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=2, seq=517, hkv=2, hq=4, seed=74)
    k, v = synth.kv(w)
    k, v = k.numpy(), v.numpy()
    lens = np.array([300, 517], np.int32)
    table = np.array([[5, 1, 3, 7, 0], [2, 6, 4, 8, 9]], np.int32)
    st = oracle.quantize_blocks(k, v, lens, table, 10, 2, v4=True)
    assert st["rc"] == 0 and st["pool"].shape == (10, 2, 19456)
    q = synth.queries(w).numpy()
    o1 = oracle.decode_attention(q, st["pool"], table, lens, st["tail_k"], st["tail_v"], 4, 2,
                                 v4=True)
    o0 = oracle.decode_attention(q, st["pool"], table, lens, st["tail_k"], st["tail_v"], 4, 2,
                                 route=0, v4=True)
    assert np.abs(o0 - o1).max() <= 1e-12 * np.abs(o0).max()
    H = torch.tensor(oracle.hadamard(128))
    for b in range(2):
        n = int(lens[b])
        nfull = n // 128
        for h in range(4):
            keys, vals = [], []
            for j in range(nfull):
                rec = st["pool"][table[b, j], h // 2]
                keys.append(torch.tensor(oracle.dequant_part(rec, False, v4=True)) @ H)
                vals.append(torch.tensor(oracle.dequant_part(rec, True, v4=True)) @ H)
            keys.append(torch.tensor(k[b, nfull * 128:n, h // 2].astype(np.float64)))
            vals.append(torch.tensor(v[b, nfull * 128:n, h // 2].astype(np.float64)))
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.tensor(q[b, h].astype(np.float64))[None, None, None],
                torch.cat(keys)[None, None], torch.cat(vals)[None, None])[0, 0, 0].numpy()
            assert np.abs(o1[b, h] - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


def test_v4_append_fills_page_like_prefill(oracle):
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=1, seq=256, hkv=2, hq=4, seed=75)
    k, v = synth.kv(w)
    k, v = k.numpy(), v.numpy()
    table = np.array([[1, 0]], np.int32)
    ref = oracle.quantize_blocks(k, v, np.array([256], np.int32), table, 2, 2, v4=True)
    st = oracle.quantize_blocks(k, v, np.array([250], np.int32), table, 2, 2, v4=True)
    for t in range(250, 256):
        assert oracle.append_token(k[:, t], v[:, t], np.array([t], np.int32), table, 2,
                                   st["pool"], st["tail_k"], st["tail_v"], v4=True) == 0
    assert np.array_equal(st["pool"], ref["pool"])


# ------------------------------------ format variant: 8-bit keys, 4-bit values --
# Format variant "k8v4_g128" (8-bit keys, 4-bit values, the "k" and "v" of the
# KVarN page's format name kvarn_k4v2_g128): the same stages with 8-bit RTN on
# K; V as in "k4v4_g128".  K codes are token-major bytes, the 16-byte chunks
# of odd tokens swapped pairwise.

def test_k8_code_positions_golden_and_a_bijection(oracle):
    g = json.load(open(os.path.join(GOLDEN, "pack_k8_examples.json")))
    for ex in g["examples"]:
        assert oracle.k8_code_pos(ex["channel"], ex["token"]) == ex["byte"], ex["_derivation"]
    seen = {oracle.k8_code_pos(d, t) for d in range(128) for t in range(128)}
    assert seen == set(range(128 * 128))


def test_k8_keys_share_zero_and_range_with_k4(oracle):
    # the normalization does not depend on the bit width: for the same tile the
    # 8-bit keys have the 4-bit keys' zero and c_d and a step 15/255 of theirs;
    # every token's codes reach 0 and 255; the V part is the k4v4 V part
    x = _tile(81)
    k4 = oracle.quantize_tile(x, False, 2)
    k8 = oracle.quantize_tile(x, False, 2, k8=True)
    assert np.array_equal(k4["a"], k8["a"]) and np.array_equal(k4["b"], k8["b"])
    q4, s4, z4, c4 = oracle.unpack_part(k4["rec"], False)
    q8, s8, z8, c8 = oracle.unpack_part(k8["rec"], False, k8=True)
    assert np.array_equal(z4, z8) and np.array_equal(c4, c8)
    assert np.allclose(s8.astype(np.float64) * 255, s4.astype(np.float64) * 15, rtol=2e-7)
    assert np.array_equal(q8, k8["q"]) and np.all(q8.min(axis=1) == 0) and np.all(q8.max(axis=1) == 255)
    # 8-bit codes round the same values on a 17x finer grid
    assert np.all(np.abs(q8 / 255.0 - q4 / 15.0) <= 0.5 / 15 + 0.5 / 255 + 1e-12)
    rec = k8["rec"]
    assert rec.size == 27648 == 216 * 128
    assert np.array_equal(rec[16384:17408].view(np.float32).reshape(128, 2)[:, 0], s8)
    assert np.array_equal(rec[17408:17920].view(np.float32), c8)
    for d, t in ((0, 0), (17, 1), (127, 126), (64, 99)):
        assert rec[oracle.k8_code_pos(d, t)] == q8[t, d]
    v4 = oracle.quantize_tile(x, True, 2, v4=True)
    v8 = oracle.quantize_tile(x, True, 2, k8=True)
    assert np.array_equal(v4["rec"][9728:], v8["rec"][17920:])


def test_k8_half_step_bound(oracle):
    x = _tile(82)
    out = oracle.quantize_tile(x, False, 2, k8=True)
    q, s, z, c = oracle.unpack_part(out["rec"], False, k8=True)
    yhat = oracle.dequant_part(out["rec"], False, k8=True)
    half = 0.5 * np.abs(s.astype(np.float64))[:, None] * c.astype(np.float64)[None, :]
    slack = 1e-6 * (np.abs(out["Y"]) + np.abs(yhat)) + 1e-9
    assert np.all(np.abs(out["Y"] - yhat) <= half + slack)
    # and 17x tighter than the 4-bit keys on average
    e4 = np.abs(out["Y"] - oracle.dequant_part(oracle.quantize_tile(x, False, 2)["rec"], False))
    assert np.abs(out["Y"] - yhat).mean() < e4.mean() / 10


def test_k8_attention_matches_torch_sdpa_on_dequantized_cache(oracle):
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=2, seq=517, hkv=2, hq=4, seed=84)
    k, v = synth.kv(w)
    k, v = k.numpy(), v.numpy()
    lens = np.array([300, 517], np.int32)
    table = np.array([[5, 1, 3, 7, 0], [2, 6, 4, 8, 9]], np.int32)
    st = oracle.quantize_blocks(k, v, lens, table, 10, 2, k8=True)
    assert st["rc"] == 0 and st["pool"].shape == (10, 2, 27648)
    q = synth.queries(w).numpy()
    o1 = oracle.decode_attention(q, st["pool"], table, lens, st["tail_k"], st["tail_v"], 4, 2,
                                 k8=True)
    o0 = oracle.decode_attention(q, st["pool"], table, lens, st["tail_k"], st["tail_v"], 4, 2,
                                 route=0, k8=True)
    assert np.abs(o0 - o1).max() <= 1e-12 * np.abs(o0).max()
    H = torch.tensor(oracle.hadamard(128))
    for b in range(2):
        n = int(lens[b])
        nfull = n // 128
        for h in range(4):
            keys, vals = [], []
            for j in range(nfull):
                rec = st["pool"][table[b, j], h // 2]
                keys.append(torch.tensor(oracle.dequant_part(rec, False, k8=True)) @ H)
                vals.append(torch.tensor(oracle.dequant_part(rec, True, k8=True)) @ H)
            keys.append(torch.tensor(k[b, nfull * 128:n, h // 2].astype(np.float64)))
            vals.append(torch.tensor(v[b, nfull * 128:n, h // 2].astype(np.float64)))
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.tensor(q[b, h].astype(np.float64))[None, None, None],
                torch.cat(keys)[None, None], torch.cat(vals)[None, None])[0, 0, 0].numpy()
            assert np.abs(o1[b, h] - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


def test_k8_append_fills_page_like_prefill(oracle):
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=1, seq=256, hkv=2, hq=4, seed=85)
    k, v = synth.kv(w)
    k, v = k.numpy(), v.numpy()
    table = np.array([[1, 0]], np.int32)
    ref = oracle.quantize_blocks(k, v, np.array([256], np.int32), table, 2, 2, k8=True)
    st = oracle.quantize_blocks(k, v, np.array([250], np.int32), table, 2, 2, k8=True)
    for t in range(250, 256):
        assert oracle.append_token(k[:, t], v[:, t], np.array([t], np.int32), table, 2,
                                   st["pool"], st["tail_k"], st["tail_v"], k8=True) == 0
    assert np.array_equal(st["pool"], ref["pool"])
