"""The oracle's pins must catch a plausible mistake anywhere in it. Each case plants one mistake
in a copy of the oracle's C source (on the CPU: the copy is compiled with the oracle's own flags
and loaded in place of the oracle for the duration of the case), runs the fast pins of
test_oracle_pins.py against it, and requires at least one of them to fail."""
import ctypes
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

# (name, text in mxfp4_oracle.c, the same text with the mistake planted)
MUTANTS = [
    ("nibble order swapped",
     "(uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4))", "(uint8_t)(codes[2 * i + 1] | (codes[2 * i] << 4))"),
    ("amax rounding constant", "bits_of(amax) + 0x200000u", "bits_of(amax) + 0x400000u"),
    ("scale offset", "    e -= 2;\n", "    e -= 1;\n"),
    ("overflow clamp", "if (amax_r_bits >= 0x7F800000u) return 127;", "if (amax_r_bits >= 0x7F800000u) return 126;"),
    ("scale applied inverted", "mul = ldexpf(1.0f, -s);", "mul = ldexpf(1.0f, s);"),
    ("amax without |x|", "amax = fmaxf(amax, fabsf(xs[i]));", "amax = fmaxf(amax, xs[i]);"),
    ("amax misses the last element", "amax = fmaxf(amax, fabsf(xs[i]));",
     "if (i < 31) amax = fmaxf(amax, fabsf(xs[i]));"),
    ("saturation: the search stops below 6", "for (c = 1; c < 8; ++c) {", "for (c = 1; c < 7; ++c) {"),
    ("ties go to the odd code", "int tie_to_even = (a == mid) && (c & 1) == 0 && (best & 1) == 1;",
     "int tie_to_even = (a == mid) && (c & 1) == 1 && (best & 1) == 0;"),
    ("ties always round up", "int c_nearer = (g_c > g_best) ? (a > mid) : (a < mid);",
     "int c_nearer = (g_c > g_best) ? (a >= mid) : (a < mid);"),
    ("sign dropped", "return (uint8_t)(best | (signbit(qx) ? 8 : 0));", "return (uint8_t)(best);"),
    ("decode exponent bias", "(1.0 + 0.5 * m) * (double)(1 << (e - 1))", "(1.0 + 0.5 * m) * (double)(1 << e)"),
    ("dequantize scale bias", "ldexp(1.0, (int)srow[k / 32] - 127)", "ldexp(1.0, (int)srow[k / 32] - 126)"),
    ("B transposed in the GEMM", "acc += a[m * K + k] * b[n * K + k];", "acc += a[m * K + k] * b[k * N + n];"),
    ("bf16 output rounds half up", "u += 0x7FFFu + ((u >> 16) & 1u);", "u += 0x8000u;"),
]


def _pins():
    """The pins of test_oracle_pins.py that run in well under a second each."""
    out = [("hand block " + b["name"], lambda b=b: pins.test_hand_worked_blocks(b)) for b in pins._load_blocks()]
    out += [("tail row " + r["name"], lambda r=r: pins.test_hand_worked_tail_rows(r)) for r in pins._load_tail_rows()]
    out += [(f"closed-form GEMM {s}", lambda s=s: pins.test_gemm_closed_form_on_exact_mxfp4_operands(*s))
            for s in ((3, 5, 96), (2, 3, 40), (3, 4, 72), (1, 2, 8))]
    out += [
        ("decode grid", pins.test_e2m1_decode_is_the_stated_grid),
        ("grid round trip", pins.test_encode_grid_points_round_trip),
        ("scale formula, every bf16 amax", pins.test_scale_formula_literal_log2_for_every_bf16_amax),
        ("unique octave", pins.test_scale_is_the_unique_octave_placing_amax_in_3p5_to_7),
        ("block maximum at every position", pins.test_block_maximum_at_every_position),
        ("single product", pins.test_gemm_single_product_lands_in_place),
        ("brute-force GEMM", pins.test_gemm_brute_force_tiny_random),
        ("bf16 rounding", pins.test_bf16_rounding_matches_exact_rational_rounding),
        ("encoder vs midpoint count, |x| < 8 (every 97th pattern)",
         lambda: _assert_selfcheck(0, 0x41000000, 97)),
    ]
    return out


def _assert_selfcheck(lo: int, hi: int, step: int) -> None:
    bad, first = oracle.encode_selfcheck(lo, hi, step)
    assert bad == 0, hex(first)


@pytest.fixture(scope="module")
def source() -> str:
    with open(oracle._SRC) as fh:
        return fh.read()


def test_real_oracle_passes_every_pin():
    failed = []
    for label, fn in _pins():
        try:
            fn()
        except AssertionError:
            failed.append(label)
    assert not failed, failed


@pytest.mark.parametrize("name,orig,planted", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(name, orig, planted, source, tmp_path, monkeypatch):
    assert source.count(orig) == 1, f"{name}: the text to mutate is not in the oracle once"
    src = tmp_path / "mutant.c"
    src.write_text(source.replace(orig, planted))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math", "-ffp-contract=off",
                    "-o", str(so), str(src), "-lm"], check=True)
    monkeypatch.setattr(oracle, "_LIB", oracle.configure(ctypes.CDLL(str(so))))
    failed = []
    for label, fn in _pins():
        try:
            fn()
        except AssertionError:
            failed.append(label)
    assert failed, f"planted mistake '{name}' passed every pin"
