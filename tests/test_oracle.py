"""Pins of the CPU oracle against what the source pages and mathematics fix.

Each test checks the oracle against something other than itself: constants
the pages print (tests/golden), IEEE binary16 as implemented by numpy, an
independent cast library where installed, closed forms, brute force on tiny
inputs, and statistical laws.  CPU only.
"""

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import mx, pertensor, gemm, philox
from block_scaled_precision_02_gb300 import inputs

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold():
    with open(os.path.join(GOLD, "pages_constants.json")) as fh:
        return json.load(fh)


# ----------------------------------------------------------------- formats
def test_e4m3_printed_constants():
    g = gold()
    t = F.E4M3.table
    fin = t[np.isfinite(t)]
    assert F.E4M3.max_finite == g["e4m3_max"]["value"] == 1.75 * 2 ** 8
    assert F.E4M3.min_subnormal == g["e4m3_min_positive"]["value"] == 2.0 ** -9
    binades = math.log2(F.E4M3.max_finite / F.E4M3.min_subnormal)
    assert round(binades, 1) == g["e4m3_binades"]["value"]
    nan_codes = [c for c in range(256) if math.isnan(t[c])]
    assert nan_codes == [0x7F, 0xFF]                      # one pattern up to sign
    assert len({c & 0x7F for c in nan_codes}) == g["e4m3_nan_patterns_up_to_sign"]["value"]
    assert not np.any(np.isinf(t))                         # no infinities
    assert len(fin) == 254


def test_e5m2_is_top_byte_of_ieee_half():
    """E5M2 follows IEEE-754 specials; its codes are exactly the upper byte of
    IEEE binary16 (checked against numpy's float16)."""
    assert gold()["e5m2_ieee_specials"]["value"]
    h = (np.arange(256, dtype=np.uint16) << 8).view(np.float16).astype(np.float64)
    t = F.E5M2.table
    same = (t == h) | (np.isnan(t) & np.isnan(h))
    assert same.all()
    assert np.isinf(t[0x7C]) and t[0x7C] > 0 and np.isinf(t[0xFC]) and t[0xFC] < 0
    assert F.E5M2.max_finite == 57344.0


def test_e8m0_range():
    g = gold()
    codes = np.arange(256)
    v = F.e8m0_decode(codes)
    assert v[0] == 2.0 ** g["e8m0_min"]["value_log2"]
    assert v[254] == 2.0 ** g["e8m0_max"]["value_log2"]
    assert np.isnan(v[255]) and g["e8m0_has_nan"]["value"]
    assert np.all(v[1:255] / v[:254] == 2.0)               # exponent-only
    assert np.all(v[:255] > 0)                             # no sign


def test_e2m1_invariants():
    t = F.E2M1.table
    assert len(t) == 16 and np.all(np.isfinite(t))
    pos = t[:8]
    assert np.all(np.diff(pos) > 0)                        # monotone
    assert pos[0] == 0.0 and t[8] == 0.0 and np.signbit(t[8])
    assert np.all(t[8:] == -t[:8])
    assert F.E2M1.max_finite == 6.0


def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 1 << 16, size=4096, dtype=np.uint32).astype(np.uint16)
    mine = F.bf16_bits_to_f64(bits)
    tt = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    same = (mine == tt) | (np.isnan(mine) & np.isnan(tt))
    assert same.all()


def test_cross_check_cast_library():
    """Decode tables and in-range RNE encode against ml_dtypes (independent)."""
    mld = pytest.importorskip("ml_dtypes")
    for f, dt in ((F.E4M3, mld.float8_e4m3fn), (F.E5M2, mld.float8_e5m2)):
        ref = np.arange(256, dtype=np.uint8).view(dt).astype(np.float64)
        same = (ref == f.table) | (np.isnan(ref) & np.isnan(f.table))
        assert same.all(), f.name
        rng = np.random.default_rng(1)
        y = rng.standard_normal(200000) * rng.choice([1e-4, 1e-2, 1, 30, 300], 200000)
        y = y[np.abs(y) < f.max_finite]
        mine = F.encode_rne_sat(f, y)
        theirs = y.astype(dt).view(np.uint8)
        assert np.array_equal(mine, theirs), f.name
    ref4 = np.arange(16, dtype=np.uint8).view(mld.float4_e2m1fn).astype(np.float64)
    assert np.array_equal(ref4, F.E2M1.table)
    y = np.random.default_rng(2).uniform(-6, 6, 50000)
    assert np.array_equal(F.encode_rne_sat(F.E2M1, y),
                          y.astype(mld.float4_e2m1fn).view(np.uint8) & 0xF)
    e8 = np.arange(255, dtype=np.uint8).view(mld.float8_e8m0fnu).astype(np.float64)
    assert np.array_equal(e8, F.e8m0_decode(np.arange(255)))


@pytest.mark.parametrize("f", [F.E4M3, F.E5M2, F.E2M1])
def test_rne_midpoints_brute_force(f):
    vals, codes = F._positive_grid(f)
    for i in range(len(vals) - 1):
        lo, hi = vals[i], vals[i + 1]
        mid = (lo + hi) / 2
        even = codes[i] if codes[i] % 2 == 0 else codes[i + 1]
        assert F.encode_rne_sat(f, np.array([mid]))[0] == even
        eps = (hi - lo) / 64
        assert F.encode_rne_sat(f, np.array([mid - eps]))[0] == codes[i]
        assert F.encode_rne_sat(f, np.array([mid + eps]))[0] == codes[i + 1]
        neg = F.encode_rne_sat(f, np.array([-mid]))[0]
        assert neg == even | (1 << (f.nbits - 1))
    # idempotent on the grid, sign kept on zero
    assert np.array_equal(F.encode_rne_sat(f, vals), codes)
    assert F.encode_rne_sat(f, np.array([-0.0]))[0] == 1 << (f.nbits - 1)
    assert F.encode_rne_sat(f, np.array([-vals[1] / 4]))[0] == 1 << (f.nbits - 1)


@pytest.mark.parametrize("f", [F.E4M3, F.E5M2, F.E2M1])
def test_saturation(f):
    big = np.array([f.max_finite * 1.01, f.max_finite * 1e6, np.inf, -np.inf, -f.max_finite * 3])
    dec = F.decode(f, F.encode_rne_sat(f, big))
    assert np.array_equal(dec, [f.max_finite, f.max_finite, f.max_finite, -f.max_finite, -f.max_finite])


# ----------------------------------------------------------------- scales
def _brute_floor_log2(a: Fraction) -> int:
    e = 0
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    return e


@pytest.mark.parametrize("f", [F.E4M3, F.E5M2, F.E2M1])
def test_scale_exponent_brute_force(f):
    rng = np.random.default_rng(5)
    amax = np.concatenate([np.exp2(rng.uniform(-40, 40, 300)),
                           np.array([1.0, 1.5, 1.75, 1.7578125, 448.0, 449.0, 6.0, 7.0, 2.0 ** -133])])
    amax = amax.astype(np.float32).astype(np.float64)
    dm = Fraction(f.max_finite)
    ef = mx.scale_exponent(amax, f, mx.FLOOR)
    ec = mx.scale_exponent(amax, f, mx.CEIL)
    for a, a_f, a_c in zip(amax, ef, ec):
        A = Fraction(float(a))
        want_floor = _brute_floor_log2(A) - _brute_floor_log2(dm)
        e = -200                                       # smallest e with A * 2^-e <= destmax
        while A / Fraction(2) ** e > dm:
            e += 1
        while A / Fraction(2) ** (e - 1) <= dm:
            e -= 1
        assert a_f == max(-127, min(127, want_floor))
        assert a_c == max(-127, min(127, e))


@pytest.mark.parametrize("f", [F.E4M3, F.E5M2, F.E2M1])
def test_ceil_never_saturates_floor_saturates_iff_mantissa(f):
    rng = np.random.default_rng(6)
    amax = np.exp2(rng.uniform(-20, 20, 5000))
    ec = mx.scale_exponent(amax, f, mx.CEIL)
    ef = mx.scale_exponent(amax, f, mx.FLOOR)
    assert np.all(amax * np.exp2(-ec) <= f.max_finite)
    assert np.all(amax * np.exp2(-(ec - 1)) > f.max_finite)      # minimal
    _, ma = mx.exponent_mantissa(amax)
    _, md = mx.exponent_mantissa(np.float64(f.max_finite))
    assert np.array_equal(amax * np.exp2(-ef) > f.max_finite, ma > md)


def test_zero_block_and_nan_block():
    z = np.zeros((1, 32))
    z[0, 3] = -0.0
    q, s = mx.quantize_blocks(z, F.E4M3, mx.FLOOR)
    assert s[0] == 0 and np.all(q[0] & 0x7F == 0)
    assert q[0, 3] == 0x80 and q[0, 0] == 0x00          # signed zeros kept
    n = np.ones((1, 32))
    n[0, 5] = np.nan
    q, s = mx.quantize_blocks(n, F.E4M3, mx.FLOOR)
    assert s[0] == 0xFF and np.all(q == 0)


def test_metadata_bits_per_block():
    """8 scale bits per 32 elements: 256b -> 264b with E8M0, 288b with an FP32
    scale; 75 % less scale traffic."""
    g = gold()
    x = inputs.small_rowwise(32, 32).float().numpy().astype(np.float64)
    out = mx.quantize(x[:1], F.E4M3, mx.ROW)
    bits = out["q_row"].nbytes * 8 + out["s_row"].nbytes * 8
    assert bits == g["block_bits_e8m0"]["value"]
    assert out["q_row"].nbytes * 8 + 32 == g["block_bits_fp32_scale"]["value"]
    assert 1 - 8 / 32 == g["scale_metadata_saving"]["value"]


@pytest.mark.parametrize("f", [F.E4M3, F.E5M2, F.E2M1])
@pytest.mark.parametrize("mode", [mx.FLOOR, mx.CEIL])
def test_dequant_bound(f, mode):
    """q_i * X ~= V_i: |v_hat - v| <= half the grid spacing at y, times X,
    unless the element saturated (floor mode only)."""
    x = inputs.small_rowwise(64, 128, seed=3).float().numpy().astype(np.float64)
    out = mx.quantize(x, f, mx.ROW, mode)
    vh = mx.dequantize(out["q_row"], out["s_row"], f)
    X = np.repeat(F.e8m0_decode(out["s_row"]), 32, axis=1)
    y = x / X
    lo, hi = F.neighbours(f, np.minimum(np.abs(y), f.max_finite))
    sat = np.abs(y) > f.max_finite
    if mode == mx.CEIL:
        assert not sat.any()
    bound = (hi - lo) / 2 * X
    ok = (np.abs(vh - x) <= bound) | sat
    assert ok.all()
    assert np.all(np.abs(vh[sat]) == f.max_finite * X[sat])


def test_col_is_row_of_transpose():
    x = inputs.small_rowwise(96, 64, seed=4).float().numpy().astype(np.float64)
    for f in (F.E4M3, F.E5M2, F.E2M1):
        d = mx.quantize(x, f, mx.DUAL, mx.CEIL)
        r = mx.quantize(np.ascontiguousarray(x.T), f, mx.ROW, mx.CEIL)
        assert np.array_equal(d["q_col"], r["q_row"]) and np.array_equal(d["s_col"], r["s_row"])
        only = mx.quantize(x, f, mx.ROW, mx.CEIL)
        assert np.array_equal(d["q_row"], only["q_row"])


def test_sf_mma_layout_is_a_bijection():
    rng = np.random.default_rng(3)
    s = rng.integers(0, 256, size=(256, 8)).astype(np.uint8)
    flat = mx.sf_to_mma(s)
    assert np.array_equal(mx.sf_from_mma(flat, 256, 8), s)
    # row 37, k-block 5 -> chunk (0, 1), byte 5*16 + 1*4 + 1
    assert flat[512 + 5 * 16 + 4 + 1] == s[37, 5]


# ----------------------------------------------------------------- Hadamard
def test_hadamard_orthogonal_and_involution():
    H = mx.sylvester(32)
    assert np.array_equal(H @ H.T, 32 * np.eye(32, dtype=np.int64))
    Hn = H / math.sqrt(32)
    assert np.allclose(Hn @ Hn, np.eye(32), atol=1e-15)


def test_fwht_matches_dense_sylvester_exactly():
    """Small-integer inputs keep every butterfly exact in float32, so the
    oracle's FWHT must equal c * H * D * v to the last bit."""
    rng = np.random.default_rng(9)
    v = rng.integers(-8, 9, size=(50, 32)).astype(np.float32)
    seed = 7
    s = philox.hadamard_signs(seed)
    got = mx.hadamard32_blocks(v, seed).astype(np.float64)
    dense = (v.astype(np.float64) * s) @ mx.sylvester(32).T     # exact integers
    want = (dense.astype(np.float32) * mx.HADAMARD_C).astype(np.float64)
    assert np.array_equal(got, want)
    # the transform is orthonormal: it keeps each block's energy
    y = got
    assert np.allclose(np.sum(y * y, axis=1), np.sum(v.astype(np.float64) ** 2, axis=1), rtol=1e-6)
    # its transpose undoes it: D H^T (H D v) / 32 == v
    back = (dense @ mx.sylvester(32)) * philox.hadamard_signs(seed) / 32.0
    assert np.array_equal(back, v.astype(np.float64))


def _fwht_tie_blocks():
    """Two blocks whose butterflies produce a float32 tie: 1 and 2^-24 meet
    at the first stage (positions 0 and 1) or at the last (0 and 16)."""
    v = np.zeros((2, 32), dtype=np.float32)
    v[:, 0] = 1.0
    v[0, 1] = 2.0 ** -24
    v[1, 16] = 2.0 ** -24
    return v


def _fwht_tie_expected(seed=7):
    """Expected outputs of _fwht_tie_blocks, worked by hand.

    Block 0: the h = 1 butterfly gives u0 = s0 + s1 e and u1 = s0 - s1 e
    (e = 2^-24).  One of them has magnitude 1 + e, the midpoint of 1 and the
    next float32 1 + 2^-23, so it rounds to magnitude 1 (even mantissa); the
    other, 1 - e, is a float32.  Every later butterfly pairs a value with a
    zero, (u, 0) -> (u, u), which is exact, so y_j = RN32(w_(j mod 2) * c).
    Block 1: stages h = 1..8 copy s0 over positions 0..15 and s16 e over
    16..31 (exact); stage 16 gives s0 + s16 e on 0..15 and s0 - s16 e on
    16..31, rounded as above, so y_j = RN32(w_(j >= 16) * c).
    With c in [1/8, 1/4) (float32 step 2^-26) and c e = 0.707.. * 2^-26:
    RN32(1 * c) = c and RN32((1 - e) c) = c - 2^-26.  (A float64 transform
    rounded once would give RN32((1 + e) c) = c + 2^-26 instead of c.)
    The signs s_j are the pinned seed-7 signs."""
    s = philox.hadamard_signs(seed)
    c = float(mx.HADAMARD_C)
    step = 2.0 ** -26
    assert 0.125 <= c < 0.25

    def pair(sa, sb):
        # (value on the "+" side, value on the "-" side) after RN32 of each
        # butterfly output times c
        plus, minus = (c, c - step) if sa == sb else (c - step, c)
        return sa * plus, sa * minus

    out = np.zeros((2, 32))
    p0, m0 = pair(s[0], s[1])
    out[0, 0::2], out[0, 1::2] = p0, m0
    p1, m1 = pair(s[0], s[16])
    out[1, :16], out[1, 16:] = p1, m1
    return out


def test_fwht_rounds_every_butterfly_to_float32():
    """The Hadamard rounds each butterfly output to float32 (ties to even),
    at the first stage and at the last, then RN32(u * c): the hand-worked
    values of _fwht_tie_expected."""
    got = mx.hadamard32_blocks(_fwht_tie_blocks(), 7).astype(np.float64)
    want = _fwht_tie_expected(7)
    assert np.array_equal(got, want)
    assert np.all(np.abs(got) > 0)


def test_hadamard_constant_is_nearest_float32():
    c = Fraction(float(mx.HADAMARD_C))
    ulp = Fraction(2) ** (math.frexp(float(mx.HADAMARD_C))[1] - 24)
    lo, hi = c - ulp / 2, c + ulp / 2
    assert lo * lo < Fraction(1, 32) < hi * hi


def test_hadamard_signs_from_seed7_are_fixed():
    s = philox.hadamard_signs(7)
    w = int(philox.philox4x32_10(np.zeros(4, np.uint32), (7, 0))[0])
    assert np.array_equal(s < 0, [(w >> j) & 1 == 1 for j in range(32)])
    assert 0 < np.sum(s < 0) < 32


# ----------------------------------------------------------------- Philox / SR
def test_philox_known_answers():
    with open(os.path.join(GOLD, "philox4x32_10_kat.txt")) as fh:
        rows = [ln.split() for ln in fh if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 3
    for r in rows:
        w = [int(v, 16) for v in r]
        out = philox.philox4x32_10(np.array(w[:4], dtype=np.uint32), (w[4], w[5]))
        assert [int(v) for v in out] == w[6:]


def _kat_rows():
    with open(os.path.join(GOLD, "philox4x32_10_kat.txt")) as fh:
        return [[int(v, 16) for v in ln.split()] for ln in fh if ln.strip() and not ln.startswith("#")]


def test_sr_draw4_known_answers():
    """Four-draws-per-call option: indices 0..3 with key 0 take words 0..3 of
    the published counter-0 / key-0 vector, in order."""
    w = _kat_rows()[0]
    assert w[:6] == [0] * 6
    assert [int(v) for v in philox.sr_draw4(0, np.arange(4))] == w[6:]


def test_sr_draw4_counter_is_index_over_four():
    """Index 4c + j takes word j of the call with counter c: word 0 equals the
    one-draw-per-call draw for index c (itself pinned by the known answers),
    also when c needs the counter's high word."""
    for seed in (0, 7, 0x123456789):
        for c in (0, 1, 5, 2 ** 32 + 5, 2 ** 40 + 3):
            assert int(philox.sr_draw4(seed, np.array([4 * c]))[0]) == int(philox.sr_draw(seed, np.array([c]))[0])
    d = philox.sr_draw4(3, np.arange(64))
    assert len(set(int(v) for v in d)) == 64                     # the four words differ


def test_planted_sr4_word_mistake_is_caught():
    """Taking word 0 for all four indices of a call (a plausible slip) fails
    the known-answer check above."""
    w = _kat_rows()[0]
    wrong = [int(philox.sr_draw(0, np.array([i >> 2]))[0]) for i in range(4)]
    assert wrong != w[6:]


@pytest.mark.parametrize("f", [F.E2M1])
def test_sr4_unbiased(f):
    rng = np.random.default_rng(13)
    y = rng.uniform(-f.max_finite * 0.9, f.max_finite * 0.9, 20)
    n = 20000
    idx = np.arange(n, dtype=np.int64)
    for yi in y:
        r = philox.sr_draw4(5, idx)
        s = F.decode(f, mx.stochastic_round(f, np.full(n, yi), r))
        lo, hi = F.neighbours(f, np.array([abs(yi)]))
        p = (abs(yi) - lo[0]) / (hi[0] - lo[0]) if hi[0] > lo[0] else 0.0
        sd = (hi[0] - lo[0]) * math.sqrt(max(p * (1 - p), 1e-12) / n)
        assert abs(np.mean(s) - yi) <= 5 * sd + 1e-12


def test_sr_on_grid_values_are_kept():
    for f in (F.E4M3, F.E5M2, F.E2M1):
        vals, codes = F._positive_grid(f)
        r = np.full(vals.shape, 0xFFFFFFFF, dtype=np.uint32)
        assert np.array_equal(mx.stochastic_round(f, vals, r), codes)
        r0 = np.zeros(vals.shape, dtype=np.uint32)
        assert np.array_equal(mx.stochastic_round(f, vals, r0), codes)


def test_sr_threshold_exact_and_direction():
    f = F.E2M1
    y = np.array([0.75, 0.625, 2.5, 5.0, -1.25])
    lo, hi, t = mx.sr_threshold(f, y)
    assert list(t) == [2 ** 31, 2 ** 30, 2 ** 31, 2 ** 31, 2 ** 31]
    # r < t rounds up (probability t / 2^32 = distance fraction)
    q_up = mx.stochastic_round(f, y, np.zeros(5, dtype=np.uint32))
    q_dn = mx.stochastic_round(f, y, np.full(5, 2 ** 31, dtype=np.uint32))
    assert list(F.decode(f, q_up)) == [1.0, 1.0, 3.0, 6.0, -1.5]
    assert list(F.decode(f, q_dn)) == [0.5, 0.5, 2.0, 4.0, -1.0]


@pytest.mark.parametrize("f", [F.E2M1, F.E4M3])
def test_sr_unbiased(f):
    rng = np.random.default_rng(12)
    y = rng.uniform(-f.max_finite * 0.9, f.max_finite * 0.9, 40)
    n = 20000
    idx = np.arange(n, dtype=np.int64)
    for yi in y:
        acc = []
        for seed in (1, 2):
            r = philox.sr_draw(seed, idx)
            acc.append(F.decode(f, mx.stochastic_round(f, np.full(n, yi), r)))
        s = np.concatenate(acc)
        lo, hi = F.neighbours(f, np.array([abs(yi)]))
        p = (abs(yi) - lo[0]) / (hi[0] - lo[0]) if hi[0] > lo[0] else 0.0
        sd = (hi[0] - lo[0]) * math.sqrt(max(p * (1 - p), 1e-12) / s.size)
        assert abs(s.mean() - yi) <= 6 * sd + 1e-12


# ----------------------------------------------------------------- per-tensor + ring
def test_pertensor_transposed_byte_equality_and_amax():
    x = inputs.small_rowwise(64, 96, seed=7).float().numpy().astype(np.float64)
    for f in (F.E4M3, F.E5M2):
        x8, x8T, amax = pertensor.quantize_pertensor(x, 0.5, f)
        assert np.array_equal(x8T, x8.T)
        assert amax == np.max(np.abs(x))
        # multiplier 1 and values on the grid are kept exactly
        g = F.decode(f, np.arange(0, 0x70)).astype(np.float64)
        assert np.array_equal(F.decode(f, pertensor.quantize_pertensor(g[None, :], 1.0, f)[0])[0], g)


def _pt_cases():
    """(x, m, fmt, code under RN32 of the product, code of the exact product)
    -- the hand-worked cases of test_pertensor_product_is_rounded_to_float32."""
    x = 1.0 + 2.0 ** -7                          # a bf16 value: 129 * 2^-7
    return [
        (x, 8843804 * 2.0 ** -23, F.E4M3, 0x38, 0x39),
        (x, 9884251 * 2.0 ** -23, F.E4M3, 0x3A, 0x39),
        (x, 9364028 * 2.0 ** -23, F.E5M2, 0x3C, 0x3D),
        (-x, 8843804 * 2.0 ** -23, F.E4M3, 0xB8, 0xB9),
    ]


def test_pertensor_product_is_rounded_to_float32():
    """x8 = encode(RN32(x * m)): the product is rounded to float32 once, and
    that rounding can land on an element-grid midpoint, where the tie goes to
    the even code.  Hand-worked (x = 129 * 2^-7, m = k * 2^-23, so
    x * m = 129 k * 2^-30 exactly; a float32 step in [1, 2) is 128 * 2^-30):

    * E4M3, k = 8843804: x * m = 1140850716 * 2^-30 = 1.0625 + 28 * 2^-30.
      28 < 64, so RN32 gives 1.0625, the midpoint of 1.0 (0x38, mantissa 000)
      and 1.125 (0x39, mantissa 001): even code 0x38.  The exact product lies
      above the midpoint and would encode to 0x39.
    * E4M3, k = 9884251: x * m = 1275068379 * 2^-30 = 1.1875 - 37 * 2^-30.
      RN32 gives 1.1875, the midpoint of 1.125 (0x39) and 1.25 (0x3A,
      mantissa 010): 0x3A.  The exact product lies below it: 0x39.
    * E5M2, k = 9364028: x * m = 1207959612 * 2^-30 = 1.125 + 60 * 2^-30.
      RN32 gives 1.125, the midpoint of 1.0 (0x3C) and 1.25 (0x3D): 0x3C.
      The exact product: 0x3D.
    * the first case negated: the sign bit is set, 0xB8 (exact product 0xB9).
    """
    for x, m, f, want, _ in _pt_cases():
        assert np.float32(m) == m                 # m is a float32 multiplier
        x8, x8T, amax = pertensor.quantize_pertensor(np.array([[x]]), m, f)
        assert int(x8[0, 0]) == want and int(x8T[0, 0]) == want
        assert amax == abs(x)


def test_ring_fold_sixteen_steps_closed_form():
    g = gold()
    n, fp8_max, margin = 16, g["fp8_max_default"]["value"], g["pow2_margin_default"]["value"]
    rng = np.random.default_rng(3)
    amaxes = [float(np.float32(v)) for v in np.exp2(rng.uniform(-8, 4, 40))]
    ring = pertensor.ring_new(n)
    assert list(ring[n:]) == [1.0, 1.0, 0.0, 0.0]
    for t, a in enumerate(amaxes):
        ring = pertensor.ring_fold(ring, a, t % n, fp8_max, margin)
        window = amaxes[max(0, t - n + 1): t + 1]
        M = Fraction(max(window))
        sc = Fraction(float(ring[n]))
        exact1 = M / Fraction(fp8_max)
        # the published scale is the float32 nearest the exact quotient (margin 1)
        ulp = Fraction(2) ** (math.frexp(float(ring[n]))[1] - 24)
        assert abs(sc - exact1) <= ulp / 2
        leg = Fraction(float(ring[n + 1]))
        ulp2 = Fraction(2) ** (math.frexp(float(ring[n + 1]))[1] - 24)
        assert abs(leg - 1 / sc) <= ulp2 / 2
        assert ring[n + 2] == 0 and ring[n + 3] == 0
        assert list(ring[:n]).count(0.0) == max(0, n - (t + 1))


def test_ring_fold_zero_history_publishes_nothing():
    ring = pertensor.ring_new(4)
    r2 = pertensor.ring_fold(ring, 0.0, 0)
    assert r2[4] == 1.0 and r2[5] == 1.0


# ----------------------------------------------------------------- GEMM reference
def test_gemm_unit_rows_pick_columns():
    rng = np.random.default_rng(4)
    M, N, K = 64, 32, 128
    a = rng.standard_normal((M, K))
    A = mx.quantize(a, F.E4M3, mx.ROW)
    b = np.zeros((N, K))
    cols = rng.choice(K, N, replace=False)
    b[np.arange(N), cols] = 4.0
    B = mx.quantize(b, F.E4M3, mx.ROW)
    ref = gemm.reference(A["q_row"], A["s_row"], B["q_row"], B["s_row"], F.E4M3)
    deqA = mx.dequantize(A["q_row"], A["s_row"], F.E4M3)
    assert np.array_equal(ref, 4.0 * deqA[:, cols])


def test_gemm_mixed_formats_decode_each_operand():
    """A in E4M3 times B in E5M2 with unit rows: C[:, n] is a column of A's
    dequantized values times B's value.  After block scaling B's single
    non-zero per row is the E5M2 element 1.5 * 2^15, far outside E4M3's
    range, so decoding B with A's format (a plausible slip) fails."""
    rng = np.random.default_rng(14)
    M, N, K = 64, 32, 128
    a = rng.standard_normal((M, K))
    A = mx.quantize(a, F.E4M3, mx.ROW)
    b = np.zeros((N, K))
    cols = rng.choice(K, N, replace=False)
    vals = np.array([1.5 * 2.0 ** e for e in rng.integers(-12, 15, N)])
    b[np.arange(N), cols] = vals
    B = mx.quantize(b, F.E5M2, mx.ROW)
    deqA = mx.dequantize(A["q_row"], A["s_row"], F.E4M3)
    ref = gemm.reference(A["q_row"], A["s_row"], B["q_row"], B["s_row"], F.E4M3, F.E5M2)
    assert np.array_equal(ref, deqA[:, cols] * vals)
    wrong = gemm.reference(A["q_row"], A["s_row"], B["q_row"], B["s_row"], F.E4M3)
    assert not np.array_equal(wrong, ref)
    sub = gemm.reference_rows_cols(A["q_row"], A["s_row"], B["q_row"], B["s_row"], F.E4M3,
                                   np.arange(5), np.arange(7), F.E5M2)
    assert np.array_equal(sub, ref[:5, :7])


def test_gemm_fp8_x_fp4_unpacks_the_packed_operand():
    """A in E4M3 times B in packed E2M1 (two codes per byte, low nibble the
    even column) with unit rows: C[:, n] is A's dequantized column cols[n]
    times B's value, each value a top-binade E2M1 element after its block
    scale.  The non-zeros sit at odd and even columns, so a swapped nibble
    order moves them to the neighbouring column; decoding B with A's format
    fails too.  The operands swapped give the transpose."""
    rng = np.random.default_rng(17)
    M, N, K = 64, 32, 128
    a = rng.standard_normal((M, K))
    A = mx.quantize(a, F.E4M3, mx.ROW)
    cols = rng.choice(K, N, replace=False)
    assert len(set(cols % 2)) == 2
    vals = rng.choice([1.0, 1.5, 3.0, -6.0], N) * np.exp2(rng.integers(-6, 7, N))
    b = np.zeros((N, K))
    b[np.arange(N), cols] = vals
    B = mx.quantize(b, F.E2M1, mx.ROW)
    assert B["q_row"].shape == (N, K // 2)
    deqA = mx.dequantize(A["q_row"], A["s_row"], F.E4M3)
    ref = gemm.reference(A["q_row"], A["s_row"], B["q_row"], B["s_row"], F.E4M3, F.E2M1)
    assert np.array_equal(ref, deqA[:, cols] * vals)
    ref_t = gemm.reference(B["q_row"], B["s_row"], A["q_row"], A["s_row"], F.E2M1, F.E4M3)
    assert np.array_equal(ref_t, ref.T)
    swapped = ((B["q_row"] >> 4) | (B["q_row"] << 4)).astype(np.uint8)
    assert not np.array_equal(gemm.reference(A["q_row"], A["s_row"], swapped, B["s_row"], F.E4M3, F.E2M1), ref)


def test_mm_fp8_reference_one_hot_rows_index_b():
    """One-hot A rows (code for 1.0 at column perm[m]) pick B's columns:
    C[m, n] = dec(b)[n, perm[m]] * scale + bias[n], read off by indexing
    (no product), so a transposed operand, a missing scale or a bias added
    per row instead of per column fails."""
    rng = np.random.default_rng(15)
    for f in (F.E4M3, F.E5M2):
        M, N, K = 6, 9, 16
        one = F.encode_rne_sat(f, np.array([1.0]))[0]
        perm = rng.permutation(K)[:M]
        a8 = np.zeros((M, K), dtype=np.uint8)
        a8[np.arange(M), perm] = one
        b8 = rng.integers(0, 0x70, (N, K), dtype=np.uint8) | (rng.integers(0, 2, (N, K), dtype=np.uint8) << 7)
        bias = rng.standard_normal(N)
        C = gemm.mm_fp8_reference(a8, b8, f, 0.25, bias)
        db = F.decode(f, b8)
        want = np.array([[db[n, perm[m]] * 0.25 + bias[n] for n in range(N)] for m in range(M)])
        assert np.array_equal(C, want)


def test_mm_fp8_reference_batch_broadcast():
    """A leading batch axis on A with a shared B equals the per-batch products."""
    rng = np.random.default_rng(16)
    a8 = rng.integers(0, 0x70, (3, 4, 8), dtype=np.uint8)
    b8 = rng.integers(0, 0x70, (5, 8), dtype=np.uint8)
    C = gemm.mm_fp8_reference(a8, b8, F.E4M3, 2.0)
    for i in range(3):
        assert np.array_equal(C[i], gemm.mm_fp8_reference(a8[i], b8, F.E4M3, 2.0))
    ones = np.full((2, 8), F.encode_rne_sat(F.E4M3, np.array([1.0]))[0], dtype=np.uint8)
    assert np.array_equal(gemm.mm_fp8_reference(ones, ones, F.E4M3, 0.5), np.full((2, 2), 4.0))


def test_gemm_pm_one_integer_sums():
    rng = np.random.default_rng(5)
    M, N, K = 32, 32, 256
    a = rng.choice([-1.0, 1.0], (M, K))
    b = rng.choice([-1.0, 1.0], (N, K))
    A = mx.quantize(a, F.E2M1, mx.ROW)
    B = mx.quantize(b, F.E2M1, mx.ROW)
    ref = gemm.reference(A["q_row"], A["s_row"], B["q_row"], B["s_row"], F.E2M1)
    assert np.array_equal(ref, a @ b.T)


def test_gate_accepts_bf16_rounding_and_rejects_errors():
    rng = np.random.default_rng(6)
    ref = rng.standard_normal(10000)
    c = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    assert gemm.gate_error(c, ref) == 0.0
    c2 = c.copy()
    c2[17] *= 1.01
    assert gemm.gate_error(c2, ref) > 2e-3


# ----------------------------------------------------------------- planted mistakes
def test_planted_fwht_sign_error_is_caught(monkeypatch):
    """A butterfly with a swapped difference must fail the Sylvester pin."""
    orig = mx.hadamard32_blocks

    def wrong(v32, seed):
        s = philox.hadamard_signs(seed).astype(np.float32)
        u = (np.asarray(v32, dtype=np.float32) * s).astype(np.float32)
        h = 1
        while h < 32:
            nu = u.copy()
            for i in range(32):
                if i & h == 0:
                    a, b = u[..., i], u[..., i + h]
                    nu[..., i], nu[..., i + h] = a + b, b - a
            u = nu
            h *= 2
        return (u * mx.HADAMARD_C).astype(np.float32)

    v = np.random.default_rng(9).integers(-8, 9, size=(5, 32)).astype(np.float32)
    dense = (v.astype(np.float64) * philox.hadamard_signs(7)) @ mx.sylvester(32).T
    want = (dense.astype(np.float32) * mx.HADAMARD_C)
    assert np.array_equal(orig(v, 7), want)
    assert not np.array_equal(wrong(v, 7), want)


def test_planted_fwht_rounded_once_is_caught():
    """A transform done exactly in float64 and rounded to float32 only at the
    end must fail the per-butterfly rounding pin."""
    def rounded_once(v32, seed):
        u = np.asarray(v32, dtype=np.float64) * philox.hadamard_signs(seed)
        y = u @ mx.sylvester(32).T.astype(np.float64)             # exact sums
        return (y * np.float64(mx.HADAMARD_C)).astype(np.float32)

    v = _fwht_tie_blocks()
    want = _fwht_tie_expected(7)
    assert np.array_equal(mx.hadamard32_blocks(v, 7).astype(np.float64), want)
    assert not np.array_equal(rounded_once(v, 7).astype(np.float64), want)


def test_planted_pertensor_exact_product_is_caught():
    """Encoding the exact float64 product x * m (no float32 rounding first)
    must fail the per-tensor pin."""
    for x, m, f, want, exact_code in _pt_cases():
        wrong = F.encode_rne_sat(f, np.array([[x]]) * np.float64(np.float32(m)))
        assert int(wrong[0, 0]) == exact_code != want
        assert int(pertensor.quantize_pertensor(np.array([[x]]), m, f)[0][0, 0]) == want


def test_planted_sr_direction_error_is_caught():
    f = F.E2M1
    y = np.full(40000, 0.625)                  # 1/4 of the way from 0.5 to 1.0
    r = philox.sr_draw(3, np.arange(y.size))
    lo, hi, t = mx.sr_threshold(f, y)
    wrong = np.where(r.astype(np.uint64) >= t, hi, lo)   # flipped comparison
    right = F.decode(f, mx.stochastic_round(f, y, r))
    assert abs(right.mean() - 0.625) < 0.01
    assert abs(wrong.mean() - 0.625) > 0.1
