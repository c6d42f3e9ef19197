"""Pins for the CPU oracle: every oracle function is checked against something other than
itself -- the e2m1 format definition, hand-worked blocks, exhaustive comparison with an
independent encoder, the scale formula in its literal log2 form and as an interval
characterisation, error-bound invariants, exact closed-form GEMMs and brute force on tiny
inputs with exact rational arithmetic.

Pages: amd-mxfp4-mm submission 711914 (``_mxfp4_quant_tile``), submission 608632
(``_hw_mxfp4_quant_op``: direct-exponent scale form and nibble order).
"""
import json
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle
from block_scaled_mxfp4_bf16_gb300 import workloads

GOLD = os.path.join(os.path.dirname(__file__), "golden", "hand_blocks.json")
GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]   # e2m1 magnitudes as stated for the method


def f32_of(u: int) -> float:
    return struct.unpack("<f", struct.pack("<I", u & 0xFFFFFFFF))[0]


def bf16_of_float(x: float) -> int:
    """Exact float -> bf16 pattern; asserts the value is representable."""
    u = struct.unpack("<I", struct.pack("<f", x))[0]
    assert u & 0xFFFF == 0, x
    return u >> 16


# ----------------------------------------------------------------------------- e2m1 format

def test_e2m1_decode_is_the_stated_grid():
    for c in range(8):
        assert oracle.e2m1_decode(c) == GRID[c]
        neg = oracle.e2m1_decode(c | 8)
        assert neg == -GRID[c] and math.copysign(1.0, neg) == -1.0


def test_encode_grid_points_round_trip():
    for c in range(16):
        v = oracle.e2m1_decode(c)
        assert oracle.e2m1_encode(v) == c
        assert oracle.e2m1_encode_count(v) == c


@pytest.mark.parametrize("qx,code", [
    (0.25, 0), (0.2500001, 1), (0.75, 2), (0.7499999, 1), (1.25, 2), (1.75, 4), (2.5, 4),
    (3.5, 6), (5.0, 6), (5.0000005, 7), (6.0, 7), (7.0, 7), (1e30, 7), (-0.25, 8), (-5.0, 14),
    (-1e-45, 8), (1e-45, 0), (-0.0, 8), (0.0, 0),
])
def test_encode_ties_and_saturation(qx, code):
    # round to nearest, ties to the even code; saturate at 6; sign kept on zero results
    assert oracle.e2m1_encode(qx) == code


def test_encode_exhaustive_below_8_matches_midpoint_count():
    # every fp32 bit pattern with |x| < 8, both signs: the nearest-grid search vs an
    # independently built encoder that counts the grid midpoints below |x|
    bad, first = oracle.encode_selfcheck(0, 0x41000000, 1)
    assert bad == 0, hex(first)


def test_encode_sweep_large_and_subnormal():
    bad, first = oracle.encode_selfcheck(0x41000000, 0x7F800000, 127)
    assert bad == 0, hex(first)
    bad, first = oracle.encode_selfcheck(0, 0x00800000, 1)
    assert bad == 0, hex(first)


# ----------------------------------------------------------------------------- hand blocks

def _load_blocks():
    with open(GOLD) as f:
        return json.load(f)["blocks"]


@pytest.mark.parametrize("blk", _load_blocks(), ids=lambda b: b["name"])
def test_hand_worked_blocks(blk):
    fill = int(blk.get("fill", "0000"), 16)
    x = [int(h, 16) for h in blk["x"]] + [fill] * (32 - len(blk["x"]))
    codes = blk["codes"] + [blk.get("code_fill", 0)] * (32 - len(blk["codes"]))
    q, s = oracle.quantize(np.array([x], np.uint16))
    assert int(s[0, 0]) == blk["scale_byte"]
    assert bytes(q[0]).hex() == blk["packed_hex"]
    got = [(q[0, i // 2] >> (4 * (i & 1))) & 15 for i in range(32)]
    assert got == codes


TAIL_GOLD = os.path.join(os.path.dirname(__file__), "golden", "tail_blocks.json")


def _load_tail_rows():
    with open(TAIL_GOLD) as f:
        return json.load(f)["rows"]


def tail_row_input(row) -> np.ndarray:
    """The fixture row as bf16 bit patterns [1, K] ("a-b" keys fill a range)."""
    x = np.zeros(row["K"], np.uint16)
    for key, h in row["x"].items():
        lo, _, hi = key.partition("-")
        x[int(lo):int(hi or lo) + 1] = int(h, 16)
    return x.reshape(1, -1).copy()


@pytest.mark.parametrize("row", _load_tail_rows(), ids=lambda r: r["name"])
def test_hand_worked_tail_rows(row):
    q, s = oracle.quantize(tail_row_input(row))
    nblk = (row["K"] + 31) // 32
    assert q.shape == (1, nblk * 16) and s.shape == (1, nblk)
    assert [int(v) for v in s[0]] == row["scale_bytes"]
    assert bytes(q[0]).hex() == row["packed_hex"]


def test_block_maximum_at_every_position():
    # Rows of one 1x32 block: 1.0 everywhere except 4.0 at position p (row 2p) or -4.0 at p
    # (row 2p+1). Worked by hand: the block maximum |x| = 4.0 is a power of two, so the
    # rounding keeps it; floor(log2 4) - 2 = 0 gives scale byte 127 and a multiplier of 1;
    # 1.0 encodes as code 2, 4.0 as code 6 and -4.0 as 0xE. A maximum that one position of
    # the block does not reach would leave 1.0 as the maximum (byte 125) at that position.
    x = np.full((64, 32), bf16_of_float(1.0), np.uint16)
    for p in range(32):
        x[2 * p, p] = bf16_of_float(4.0)
        x[2 * p + 1, p] = bf16_of_float(-4.0)
    q, s = oracle.quantize(x)
    assert (s[:, 0] == 127).all(), np.nonzero(s[:, 0] != 127)[0]
    for r in range(64):
        p, neg = divmod(r, 2)
        want = [2] * 32
        want[p] = 0xE if neg else 6
        got = [(int(q[r, i // 2]) >> (4 * (i & 1))) & 15 for i in range(32)]
        assert got == want, r


def test_k_not_multiple_of_8_is_refused():
    with pytest.raises(ValueError):
        oracle.quantize(np.zeros((1, 36), np.uint16))


# ----------------------------------------------------------------------------- scale

def _all_finite_positive_bf16():
    return np.arange(0, 0x7F80, dtype=np.uint16)


def _scale_bytes_for_amax(h: np.ndarray) -> np.ndarray:
    x = np.zeros((h.size, 32), np.uint16)
    x[:, 7] = h
    return oracle.quantize(x)[1][:, 0].astype(int)


def test_scale_formula_literal_log2_for_every_bf16_amax():
    # the method's wording: amax rounded with (bits + 0x200000) & 0xFF800000, then
    # floor(log2(.)) - 2 clamped to [-127, 127], stored +127 -- evaluated with math.log2
    h = _all_finite_positive_bf16()
    got = _scale_bytes_for_amax(h)
    for hv, b in zip(h.tolist(), got.tolist()):
        r = f32_of(((hv << 16) + 0x200000) & 0xFF800000)
        e = -math.inf if r == 0 else (math.inf if math.isinf(r) else math.floor(math.log2(r)))
        s = max(-127, min(127, e - 2))
        assert b == int(s) + 127, hex(hv)


def test_scale_is_the_unique_octave_placing_amax_in_3p5_to_7():
    # Closed form of the rounding rule: the mantissa rounds up exactly when it is >= 1.75,
    # so (unclamped) the scaled block maximum amax * 2^-s lies in [3.5, 7): one octave,
    # hence exactly one s qualifies.
    h = _all_finite_positive_bf16()
    got = _scale_bytes_for_amax(h)
    for hv, b in zip(h.tolist(), got.tolist()):
        amax = Fraction(f32_of(hv << 16))
        s = b - 127
        if amax == 0:
            assert b == 0
            continue
        scaled = amax / (Fraction(2) ** s)
        if -127 < s < 127:
            assert Fraction(7, 2) <= scaled < 7, hex(hv)
        elif s == -127:
            assert scaled < 7, hex(hv)          # clamped at the bottom: amax is tiny
        else:
            # clamped at the top: only an amax that rounds up to +inf (>= 1.75 * 2^127)
            # gets s = 127, leaving the scaled maximum in [1.75, 2)
            assert Fraction(7, 4) <= scaled < 2, hex(hv)


def test_scale_monotone_in_amax():
    h = _all_finite_positive_bf16()
    got = _scale_bytes_for_amax(h)
    assert np.all(np.diff(got) >= 0)
    assert got.min() == 0 and got.max() == 254


def test_direct_exponent_form_agrees_except_at_overflow():
    # submission 608632's integer form: byte = clamp(E - 2, 0, 254) with E the biased
    # exponent of the rounded amax. It equals the log2 form for every finite rounded
    # amax; they differ only where the rounding overflows to +inf (253 vs 254).
    h = _all_finite_positive_bf16()
    got = _scale_bytes_for_amax(h)
    for hv, b in zip(h.tolist(), got.tolist()):
        u = ((hv << 16) + 0x200000) & 0xFF800000
        E = (u >> 23) & 0xFF
        direct = min(max(E - 2, 0), 254)
        if E == 255:
            assert (direct, b) == (253, 254)
        else:
            assert b == direct, hex(hv)


# ----------------------------------------------------------------------------- quantizer

def test_grid_values_at_every_scale_quantize_to_themselves():
    # blocks whose max is +-6 * 2^s quantize with scale s, and every grid value times 2^s
    # comes back as its own code (for every s the bf16 range allows: -127 .. 125)
    rows, want_codes, want_scale = [], [], []
    rng = np.random.default_rng(1)
    for s in range(-127, 126):
        codes = [7 if rng.random() < 0.5 else 15] + list(rng.integers(0, 16, 31))
        vals = [math.ldexp(oracle.e2m1_decode(int(c)), s) for c in codes]
        rows.append([bf16_of_float(v) for v in vals])
        want_codes.append(codes)
        want_scale.append(s + 127)
    q, sc = oracle.quantize(np.array(rows, np.uint16))
    assert sc[:, 0].tolist() == want_scale
    got = np.stack([q & 15, q >> 4], axis=-1).reshape(len(rows), 32)
    # +0.0 and -0.0 are distinct codes (0 and 8); all others exact
    assert got.tolist() == [list(map(int, c)) for c in want_codes]


def _half_step(a: np.ndarray) -> np.ndarray:
    return np.where(a <= 2, 0.25, np.where(a <= 4, 0.5, 1.0))


@pytest.mark.parametrize("name", ["M32_N4096_K512", "M16_N3072_K1536"])
def test_quant_error_bound_and_nearest(name):
    w = workloads.by_name(name)
    a, _ = workloads.make_inputs(w, seed=0)
    x_bits = workloads.bf16_bits(a)
    q, s = oracle.quantize(x_bits)
    x = oracle.bf16_to_f64(x_bits)
    dq = oracle.dequantize(q, s)
    scale = np.repeat(np.ldexp(1.0, s.astype(np.int64) - 127), 32, axis=1)
    qx = x / scale
    err = np.abs(qx - dq / scale)
    assert np.all(err <= _half_step(np.abs(qx)))
    # nearest grid point (ties aside) among all 8 magnitudes
    grid = np.array(GRID)
    best = np.min(np.abs(np.abs(qx)[..., None] - grid), axis=-1)
    assert np.all(np.abs(np.abs(qx) - np.abs(dq / scale)) <= best + 0)
    # the outlier workload really hits saturation and zero-scale blocks
    if w.outlier_blocks:
        assert (s == 0).sum() >= w.M * w.K // 32 * 5 // 100
        assert (np.abs(qx) > 6).any()


# ----------------------------------------------------------------------------- GEMM

def _decode_nibble(byte: int, hi: bool) -> Fraction:
    """Independent e2m1 decode (sign, 2-bit exponent bias 1, 1-bit mantissa)."""
    c = (byte >> 4) if hi else (byte & 15)
    sgn = -1 if c & 8 else 1
    e, m = (c >> 1) & 3, c & 1
    mag = Fraction(m, 2) if e == 0 else Fraction(2 + m, 2) * Fraction(2) ** (e - 1)
    return sgn * mag


def _exact_value(q, s, r, k) -> Fraction:
    return _decode_nibble(int(q[r, k // 2]), bool(k & 1)) * Fraction(2) ** (int(s[r, k // 32]) - 127)


@pytest.mark.parametrize("M,N,K", [(3, 5, 96), (2, 3, 40), (3, 4, 72), (1, 2, 8)])
def test_gemm_closed_form_on_exact_mxfp4_operands(M, N, K):
    # A, B already exact MXFP4 values (block max forced to +-6*2^s among the block's real
    # elements), so quantization is the identity and C = A . B^T exactly over the K real
    # elements, also when K cuts the last block (40, 72, 8); M != N != K catches a transposed
    # operand.
    rng = np.random.default_rng(7 + K)
    def make(rows):
        vals = np.zeros((rows, K))
        for r in range(rows):
            for j in range((K + 31) // 32):
                n = min(32, K - 32 * j)
                s = int(rng.integers(-4, 5))
                codes = rng.integers(0, 16, n)
                codes[int(rng.integers(0, n))] = 7 if rng.random() < 0.5 else 15
                for i in range(n):
                    vals[r, 32 * j + i] = math.ldexp(oracle.e2m1_decode(int(codes[i])), s)
        return vals
    a, b = make(M), make(N)
    ab = np.vectorize(bf16_of_float, otypes=[np.uint16])(a)
    bb = np.vectorize(bf16_of_float, otypes=[np.uint16])(b)
    aq, as_ = oracle.quantize(ab)
    bq, bs = oracle.quantize(bb)
    assert np.array_equal(oracle.dequantize(aq, as_)[:, :K], a)
    assert np.array_equal(oracle.dequantize(bq, bs)[:, :K], b)
    assert not oracle.dequantize(aq, as_)[:, K:].any()    # padding decodes to zero
    c = oracle.mxfp4_gemm_ref(aq, as_, bq, bs)
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(a[m, k]) * Fraction(b[n, k]) for k in range(K))
            assert Fraction(c[m, n]) == exact


def test_gemm_brute_force_tiny_random():
    # random bf16 operands, quantized by the oracle, then an exact rational triple loop over
    # an independent decode of the packed bytes
    M, N, K = 4, 6, 128
    a = workloads.random_bf16(M, K, seed=11)
    b = workloads.random_bf16(N, K, seed=12, scale=3.0)
    aq, as_ = oracle.quantize(workloads.bf16_bits(a))
    bq, bs = oracle.quantize(workloads.bf16_bits(b))
    c = oracle.mxfp4_gemm_ref(aq, as_, bq, bs)
    idx_m = np.repeat(np.arange(M), N)
    idx_n = np.tile(np.arange(N), M)
    ce = oracle.gemm_entries(aq, as_, bq, bs, idx_m, idx_n).reshape(M, N)
    for m in range(M):
        for n in range(N):
            exact = sum(_exact_value(aq, as_, m, k) * _exact_value(bq, bs, n, k) for k in range(K))
            assert abs(Fraction(c[m, n]) - exact) <= abs(exact) * Fraction(1, 2 ** 50)
            assert ce[m, n] == c[m, n]


def test_gemm_single_product_lands_in_place():
    # one nonzero in A (row 2, k=37) and one in B (row 4, k=37): only C[2,4] is nonzero
    M, N, K = 3, 6, 64
    a = np.zeros((M, K), np.uint16)
    b = np.zeros((N, K), np.uint16)
    a[2, 37] = bf16_of_float(3.0)
    b[4, 37] = bf16_of_float(-0.75)
    b[1, 36] = bf16_of_float(5.0)     # different k: must not meet A's element
    aq, as_ = oracle.quantize(a)
    bq, bs = oracle.quantize(b)
    c = oracle.mxfp4_gemm_ref(aq, as_, bq, bs)
    want = np.zeros((M, N))
    want[2, 4] = 3.0 * -0.75
    assert np.array_equal(c, want)


# ----------------------------------------------------------------------------- bf16 output

def _bf16_rne_exact(d: float) -> int:
    """Nearest bf16 (8 significant bits) to d by exact rational comparison, ties to even."""
    if d == 0:
        return 0x8000 if math.copysign(1, d) < 0 else 0
    sgn = 0x8000 if d < 0 else 0
    x = Fraction(abs(d))
    m, e = math.frexp(abs(d))          # abs(d) = m * 2^e, m in [0.5, 1)
    ulp = Fraction(2) ** (e - 8)
    lo = (x // ulp) * ulp
    hi = lo + ulp
    if x - lo < hi - x:
        v = lo
    elif x - lo > hi - x:
        v = hi
    else:
        v = lo if (lo / ulp) % 2 == 0 else hi
    return sgn | bf16_of_float(float(v))


@pytest.mark.parametrize("d,h", [
    (1.0, 0x3F80), (1 + 2 ** -8, 0x3F80), (1 + 3 * 2 ** -8, 0x3F82),
    (1 + 2 ** -8 + 2 ** -30, 0x3F81),          # a double rounding via fp32 would give 0x3F80
    (-(1 + 2 ** -8 + 2 ** -40), 0xBF81), (0.0, 0x0000), (-0.0, 0x8000),
    (2.0 ** -133, 0x0001), (3.4e38, 0x7F80), (-3.3e38, 0xFF78),
])
def test_bf16_rounding_pins(d, h):
    assert int(oracle.to_bf16(np.array([d]))[0]) == h


def test_bf16_rounding_matches_exact_rational_rounding():
    rng = np.random.default_rng(3)
    d = rng.standard_normal(4000) * np.ldexp(1.0, rng.integers(-60, 60, 4000))
    # also values a hair away from bf16 ties
    t = (rng.integers(1 << 7, 1 << 8, 2000) * 2 + 1).astype(np.float64) * 2.0 ** -9
    d = np.concatenate([d, t, t * (1 + 2.0 ** -40), t * (1 - 2.0 ** -40)])
    got = oracle.to_bf16(d)
    for x, g in zip(d.tolist(), got.tolist()):
        assert g == _bf16_rne_exact(x), x


def test_tolerance_helper():
    ref = np.array([1.0, -2.0, 0.0, 4.0])
    ok, worst = oracle.tolerance_ok(ref * (1 + 7e-3), ref)
    assert ok and worst < 1
    ok, _ = oracle.tolerance_ok(ref + np.array([0, 0, 0.01, 0]), ref)
    assert not ok
