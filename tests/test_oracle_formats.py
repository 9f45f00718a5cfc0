"""Pins of the oracle's code tables, rounding and quantisers (CPU only).

Each check compares the oracle with something other than itself: the OCP MX
code tables typed in as published literals, torch's float8 conversions
(library routines), an independent binade-wise round-half-even built on
numpy, and the invariants the format definitions fix.
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _table(name):
    """Element magnitudes of the positive codes, as published (tests/golden, cited there)."""
    vals = []
    for line in open(os.path.join(GOLDEN, name)):
        if not line.startswith("#"):
            vals += [float(v) for v in line.split()]
    return vals


# OCP Microscaling Formats (MX) v1.0: element magnitudes of the positive codes.
E2M1_TABLE = _table("e2m1_magnitudes.txt")
E2M3_TABLE = _table("e2m3_magnitudes.txt")
assert len(E2M1_TABLE) == 8 and len(E2M3_TABLE) == 32


def test_e2m1_table_exhaustive():
    for c in range(16):
        v = oracle.e2m1_value(c)
        ref = E2M1_TABLE[c & 7] * (-1.0 if c & 8 else 1.0)
        assert v == ref, (c, v, ref)
    assert np.signbit(oracle.e2m1_value(8))  # code 8 is -0


def test_e2m3_table_exhaustive():
    for c in range(64):
        v = oracle.e2m3_value(c)
        ref = E2M3_TABLE[c & 31] * (-1.0 if c & 32 else 1.0)
        assert v == ref, (c, v, ref)


def test_e4m3_table_matches_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_value(c) for c in range(256)])
    nan = np.isnan(ref)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert oracle.e4m3_value(0x7E) == 448.0


def test_ue8m0_matches_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).double().numpy()
    got = np.array([oracle.ue8m0_value(b) for b in range(256)])
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert np.array_equal(got[:255], ref[:255])


# ---------------------------------------------------------------- rounding
def _binade_rne(v, steps):
    """Independent RNE onto a grid made of uniform-step segments.

    steps: list of (lo, hi, step); within [lo, hi] the grid is lo + n*step and
    round-half-even of v/step picks the neighbour (numpy's np.round is
    half-to-even).  Above the last hi the value saturates.
    """
    a = abs(float(v))
    for lo, hi, step in steps:
        if a <= hi + step / 2 and a >= lo:
            q = float(np.round(np.float64(a) / step)) * step
            return min(q, steps[-1][1])
    return steps[-1][1]


E2M1_STEPS = [(0.0, 2.0, 0.5), (2.0, 4.0, 1.0), (4.0, 6.0, 2.0)]
E2M3_STEPS = [(0.0, 2.0, 0.125), (2.0, 4.0, 0.25), (4.0, 7.5, 0.5)]


def _sample_points(table, rng, n_random):
    mids = [(table[i] + table[i + 1]) / 2 for i in range(len(table) - 1)]
    pts = []
    for m in mids + table:
        f = np.float32(m)
        pts += [f, np.nextafter(f, np.float32(-1)), np.nextafter(f, np.float32(100))]
    pts += list(rng.uniform(0, table[-1] * 1.3, n_random).astype(np.float32))
    pts += [np.float32(table[-1] * 2), np.float32(1e-30), np.float32(0)]
    return [p for p in pts if p >= 0]


@pytest.mark.parametrize("name,table,steps,sign_bit",
                         [("e2m1", E2M1_TABLE, E2M1_STEPS, 8), ("e2m3", E2M3_TABLE, E2M3_STEPS, 32)])
def test_element_rne_against_binade_rounding(name, table, steps, sign_bit):
    rng = np.random.default_rng(1)
    rne = oracle.e2m1_rne if name == "e2m1" else oracle.e2m3_rne
    val = oracle.e2m1_value if name == "e2m1" else oracle.e2m3_value
    for p in _sample_points(table, rng, 20000):
        for s in (1.0, -1.0):
            v = np.float32(p * s)
            code = rne(float(v))
            ref = _binade_rne(v, steps)
            assert abs(val(code)) == ref, (name, float(v), code, ref)
            if ref == 0.0:
                assert code == 0, "zero must be +0"
            else:
                assert bool(code & sign_bit) == (s < 0)


def test_e2m1_ties_go_to_even_code():
    # the published midpoints and where round-half-even sends them
    for v, want in [(0.25, 0.0), (0.75, 1.0), (1.25, 1.0), (1.75, 2.0), (2.5, 2.0), (3.5, 4.0),
                    (5.0, 4.0), (7.0, 6.0), (100.0, 6.0)]:
        assert oracle.e2m1_value(oracle.e2m1_rne(v)) == want, v


def test_e4m3_rne_matches_torch():
    rng = np.random.default_rng(2)
    table = [oracle.e4m3_value(c) for c in range(127)]
    pts = _sample_points(table, rng, 20000)
    pts += list((2.0 ** rng.uniform(-12, 8.8, 20000)).astype(np.float32))
    v = np.array([p for p in pts if p <= 448], dtype=np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_rne(float(x)) for x in v], dtype=np.uint8)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(v[i]), got[i], ref[i]) for i in bad[:5]]
    assert oracle.e4m3_rne(460.0) == 0x7E and oracle.e4m3_rne(1e9) == 0x7E  # saturation


# ---------------------------------------------------------------- quantisers
def _unpack_nibbles(codes):
    lo = codes & 15
    hi = codes >> 4
    out = np.empty((codes.shape[0], codes.shape[1] * 2), np.uint8)
    out[:, 0::2] = lo
    out[:, 1::2] = hi
    return out


def _e2m1_values(q):
    mag = np.array(E2M1_TABLE)[q & 7]
    return np.where(q & 8, -mag, mag)


def _random_matrix(rng, rows, K, scale=0.02):
    W = (rng.standard_normal((rows, K)) * scale).astype(np.float32)
    W[0, :16] = 0.0                          # an all-zero block
    W[1, 16:32] = np.float32(1e-12)          # a block far below the tensor's range
    W[2, 5] = np.float32(scale * 9)          # an outlier sets the tensor amax
    return W


def test_nvfp4_quantizer_recipe():
    rng = np.random.default_rng(3)
    rows, K = 24, 96
    W = _random_matrix(rng, rows, K)
    codes, scales, ts = oracle.quantize_nvfp4(W)
    A = np.float32(np.abs(W).max())
    assert np.float32(ts) == np.float32(A / np.float32(2688.0))          # amax / (6 * 448)
    blocks = np.abs(W).reshape(rows, K // 16, 16).max(axis=2).astype(np.float32)
    sv = (blocks / np.float32(6.0)) / np.float32(ts)                      # fp32, as specified
    ref_s = torch.from_numpy(sv.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8)
    assert np.array_equal(scales, ref_s.numpy())
    assert scales.max() <= 0x7E
    q = _unpack_nibbles(codes)
    sval = torch.from_numpy(scales).view(torch.float8_e4m3fn).float().numpy()
    for r in range(rows):
        for c in range(K):
            s = sval[r, c // 16]
            if s == 0:
                assert q[r, c] == 0
                continue
            v = W[r, c] / np.float32(np.float32(s) * np.float32(ts))
            assert abs(_e2m1_values(q[r, c])) == _binade_rne(v, E2M1_STEPS), (r, c)
            assert ((q[r, c] & 8) != 0) == bool(v < 0 and _binade_rne(v, E2M1_STEPS) > 0)
    assert np.all(q[0, :16] == 0) and scales[0, 0] == 0


def test_nvfp4_all_zero_matrix():
    codes, scales, ts = oracle.quantize_nvfp4(np.zeros((16, 32), np.float32))
    assert ts == 0.0 and not codes.any() and not scales.any()


def test_nvfp4_dequant_matches_tables():
    rng = np.random.default_rng(4)
    W = _random_matrix(rng, 16, 64)
    codes, scales, ts = oracle.quantize_nvfp4(W)
    D = oracle.dequant_nvfp4(codes, scales, ts, 16, 64)
    sval = torch.from_numpy(scales).view(torch.float8_e4m3fn).float().numpy()
    q = _unpack_nibbles(codes)
    cs = (_e2m1_values(q) * np.repeat(sval, 16, axis=1)).astype(np.float32)
    ref = cs * np.float32(ts)
    assert np.array_equal(D, ref.astype(np.float32))
    # quantisation error: at most half a step of the block's grid, plus saturation never hit
    err = np.abs(D - W)
    step = np.repeat(sval, 16, axis=1) * ts * 2.0  # the widest e2m1 step is 2 units
    assert np.all(err <= step / 2 + 1e-9)


def test_fp6_quantizer_exponent_minimal_and_codes_nearest():
    rng = np.random.default_rng(5)
    rows, K = 8, 256
    W = _random_matrix(rng, rows, K)
    W[3, 128:256] *= 1e3
    codes, exps = oracle.quantize_fp6(W)
    amax = np.abs(W).reshape(rows, K // 128, 128).max(axis=2).astype(np.float64)
    E = exps.astype(np.int64) - 127
    for r in range(rows):
        for b in range(K // 128):
            if amax[r, b] == 0:
                assert exps[r, b] == 127
                continue
            assert amax[r, b] <= 7.5 * 2.0 ** E[r, b]
            assert amax[r, b] > 7.5 * 2.0 ** (E[r, b] - 1)   # minimal
    vals = np.array(E2M3_TABLE)
    for r in range(rows):
        for c in range(K):
            e = E[r, c // 128]
            v = np.float32(np.ldexp(np.float64(W[r, c]), -int(e)))
            code = codes[r, c]
            assert code < 64
            assert vals[code & 31] == _binade_rne(v, E2M3_STEPS), (r, c)
            assert ((code & 32) != 0) == bool(v < 0 and vals[code & 31] > 0)


def test_fp6_all_zero_block_and_dequant():
    W = np.zeros((2, 128), np.float32)
    W[1, 7] = -0.3
    codes, exps = oracle.quantize_fp6(W)
    assert exps[0, 0] == 127 and not codes[0].any()
    D = oracle.dequant_fp6(codes, exps, 2, 128)
    assert np.all(D[0] == 0)
    # 0.3 <= 7.5 * 2^-4 but 0.3 > 7.5 * 2^-5, so E = -4; -0.3 * 16 = -4.8 -> -5.0 (step 0.5)
    assert exps[1, 0] == 127 - 4 and D[1, 7] == np.float32(-5.0 * 2.0 ** -4)


def test_fp6_vs_nvfp4_byte_ratio():
    # "fp6 spends about 1.4x the weight bytes" (knivesysl README, "formats")
    nvfp4 = 0.5 + 1 / 16          # e2m1 code + one e4m3 scale per 16
    fp6 = 0.75 + 1 / 128          # e2m3 code + one exponent byte per 128
    assert 1.3 < fp6 / nvfp4 < 1.45


# ---------------------------------------------------------------- MXFP4 (OCP MX v1.0 FP4)
def test_mxfp4_quantizer_scale_rule_and_codes_nearest():
    """Shared scale X = 2^(floor(log2 amax) - 2) per 32 weights, written as the
    binade bracket 2^(E+2) <= amax < 2^(E+3); codes = the binade-wise
    round-half-even of w / X on the e2m1 grid, saturating at 6."""
    rng = np.random.default_rng(7)
    rows, K = 6, 256
    W = _random_matrix(rng, rows, K)
    W[2, 64:96] *= 1e4          # a loud block
    W[4, 0:32] *= 1e-6          # a quiet one
    W[5, 160:192] = 0.0         # an all-zero one
    W[1, 32] = np.float32(2.0 ** -3 * 6.0)  # an exact power-of-two edge: amax = 0.75 -> E = -3
    W[1, 33:64] = 0.0
    codes, exps = oracle.quantize_mxfp4(W)
    amax = np.abs(W).reshape(rows, K // 32, 32).max(axis=2).astype(np.float64)
    E = exps.astype(np.int64) - 127
    for r in range(rows):
        for b in range(K // 32):
            if amax[r, b] == 0:
                assert exps[r, b] == 127
                continue
            assert 2.0 ** (E[r, b] + 2) <= amax[r, b] < 2.0 ** (E[r, b] + 3), (r, b)
    assert E[1, 1] == -3
    vals = np.array(E2M1_TABLE)
    for r in range(rows):
        for c in range(K):
            byte = codes[r, c // 2]
            code = (byte & 15) if c % 2 == 0 else (byte >> 4)
            v = np.float32(np.ldexp(np.float64(W[r, c]), -int(E[r, c // 32])))
            assert vals[code & 7] == _binade_rne(v, E2M1_STEPS), (r, c)
            assert ((code & 8) != 0) == bool(v < 0 and vals[code & 7] > 0)


def test_mxfp4_saturation_and_dequant_values():
    W = np.zeros((1, 64), np.float32)
    W[0, 0] = 7.5          # amax 7.5: E = floor(log2 7.5) - 2 = 0, 7.5 saturates to 6
    W[0, 1] = -5.0         # midpoint of 4 and 6: ties to the even code (4)
    W[0, 2] = 0.25         # midpoint of 0 and 0.5: ties to 0, never -0
    W[0, 3] = -0.25
    W[0, 32] = 1.0 / 1024  # second block: E = -10 - 2 = -12, 2^-10 / 2^-12 = 4
    codes, exps = oracle.quantize_mxfp4(W)
    assert exps[0, 0] == 127 and exps[0, 1] == 127 - 12
    D = oracle.dequant_mxfp4(codes, exps, 1, 64)
    assert D[0, 0] == 6.0 and D[0, 1] == -4.0 and D[0, 2] == 0.0 and D[0, 3] == 0.0
    assert (codes[0, 1] >> 4) == 0  # -0.25 -> +0
    assert D[0, 32] == np.float32(1.0 / 1024)
    assert np.all(D[0, 4:32] == 0) and np.all(D[0, 33:] == 0)


def test_mxfp4_error_bound():
    """Away from saturation the error is at most half a grid step of the
    element's binade times X (0.25 X below 2, 0.5 X below 4, X below 6)."""
    rng = np.random.default_rng(9)
    W = _random_matrix(rng, 16, 512)
    codes, exps = oracle.quantize_mxfp4(W)
    D = oracle.dequant_mxfp4(codes, exps, 16, 512).astype(np.float64)
    X = np.repeat(2.0 ** (exps.astype(np.float64) - 127), 32, axis=1)
    a = np.abs(W.astype(np.float64)) / X
    step = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
    err = np.abs(D - W) / X
    inside = a <= 6.0
    assert np.all(err[inside] <= step[inside] / 2 + 1e-12)
    assert np.all(err[~inside] == a[~inside] - 6.0)  # saturated: clipped to 6 X
