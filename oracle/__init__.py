"""CPU oracle for the MXFP4 GEMM: C = MXFP4(A) . MXFP4(B)^T -> bf16.

TEST INFRASTRUCTURE ONLY. The product package never imports this module; it is loaded by
the tests, by ``__graft_entry__.smoke()`` and by the CPU-baseline leg of ``bench.py``.

The arithmetic lives in ``mxfp4_oracle.c`` (plain C: the fp32 block scale as the pages
spell it out, the element encode from the e2m1 definition, fp64 GEMM); this module only
compiles it with gcc and marshals numpy arrays.
It shares no code with the CUDA path.

Sources (the "amd-mxfp4-mm" leaderboard submissions):
  * quantizer: submission 711914, ``_mxfp4_quant_tile``; scale form cross-checked against
    submission 608632, ``_hw_mxfp4_quant_op`` (step 1, direct exponent);
  * nibble order: submission 608632, ``_hw_mxfp4_quant_op`` (step 3: evens low, odds high);
  * GEMM: ``dot_scaled`` of the two e2m1 operands with their e8m0 scales, fp32 accumulate
    in the pages; fp64 here, rounded once to bf16 (round to nearest even).

Pins (tests/test_oracle_pins.py): the e2m1 grid, an exhaustive fp32 cross-check of the
nearest-value encoder against an independently built midpoint-counting encoder, hand-worked
blocks (tests/golden/hand_blocks.json) and rows
whose K cuts the last block (tests/golden/tail_blocks.json), the block maximum at every
position of a block, the scale formula as the method states it, evaluated literally for every
bf16 amax, an error-bound invariant, exact closed-form GEMMs and brute-force tiny GEMMs.
tests/test_oracle_mutants.py plants fifteen plausible mistakes in copies of mxfp4_oracle.c and
checks that each fails a pin. No oracle function is "parity
unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxfp4_oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
_LOCK = threading.Lock()
_LIB = None

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile mxfp4_oracle.c into liboracle.so next to it (gcc, OpenMP, no fast-math)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def configure(L: ctypes.CDLL) -> ctypes.CDLL:
    """Declare the C signatures on a loaded oracle library (this one, or a test's variant)."""
    L.oracle_round_amax_bits.restype = ctypes.c_uint32
    L.oracle_round_amax_bits.argtypes = [ctypes.c_float]
    L.oracle_scale_exponent.restype = ctypes.c_int
    L.oracle_scale_exponent.argtypes = [ctypes.c_uint32]
    L.oracle_e2m1_encode.restype = ctypes.c_uint8
    L.oracle_e2m1_encode.argtypes = [ctypes.c_float]
    L.oracle_e2m1_encode_count.restype = ctypes.c_uint8
    L.oracle_e2m1_encode_count.argtypes = [ctypes.c_float]
    L.oracle_e2m1_decode.restype = ctypes.c_double
    L.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
    L.oracle_quantize.restype = None
    L.oracle_quantize.argtypes = [_u16p, _i64, _i64, _i64, _u8p, _u8p]
    L.oracle_dequantize.restype = None
    L.oracle_dequantize.argtypes = [_u8p, _u8p, _i64, _i64, _f64p]
    L.oracle_gemm_f64.restype = None
    L.oracle_gemm_f64.argtypes = [_f64p, _f64p, _i64, _i64, _i64, _f64p]
    L.oracle_gemm_entries.restype = None
    L.oracle_gemm_entries.argtypes = [_u8p, _u8p, _u8p, _u8p, _i64, _i64p, _i64p, _i64, _f64p]
    L.oracle_f64_to_bf16.restype = ctypes.c_uint16
    L.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
    L.oracle_f64_to_bf16_array.restype = None
    L.oracle_f64_to_bf16_array.argtypes = [_f64p, _i64, _u16p]
    L.oracle_encode_selfcheck.restype = ctypes.c_int64
    L.oracle_encode_selfcheck.argtypes = [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32,
                                          ctypes.POINTER(ctypes.c_uint32)]
    L.oracle_num_threads.restype = ctypes.c_int
    L.oracle_num_threads.argtypes = []
    L.oracle_set_num_threads.restype = None
    L.oracle_set_num_threads.argtypes = [ctypes.c_int]
    return L


def lib() -> ctypes.CDLL:
    global _LIB
    with _LOCK:
        if _LIB is None:
            build()
            _LIB = configure(ctypes.CDLL(_SO))
    return _LIB


def _p(a: np.ndarray, t):
    assert a.flags["C_CONTIGUOUS"], "oracle expects C-contiguous arrays"
    return a.ctypes.data_as(t)


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads the oracle's parallel loops use from now on (for timing it on one core)."""
    lib().oracle_set_num_threads(int(n))


def quantize(x_bf16: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """bf16 bit patterns [rows, K] (uint16) -> (q uint8 [rows, nblk*16], scales uint8 [rows, nblk]),
    nblk = ceil(K/32).

    When K is not a multiple of 32 the row is first widened to 32*nblk elements with zeros:
    submission 711914's `_standalone_quant_kernel` loads A under the mask offs_k < K with 0.0
    as the fill value, so the missing elements of the last block are zeros to the block
    maximum and to the encoder (zero codes). K must be a multiple of 8 (the library's bf16
    rows move in 16-byte pieces)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    rows, K = x.shape
    if K % 8:
        raise ValueError("K must be a multiple of 8")
    if K % 32:
        x = np.concatenate([x, np.zeros((rows, 32 - K % 32), np.uint16)], axis=1)
        K = x.shape[1]
    q = np.empty((rows, K // 2), np.uint8)
    s = np.empty((rows, K // 32), np.uint8)
    if rows and K:
        lib().oracle_quantize(_p(x, _u16p), rows, K, K, _p(q, _u8p), _p(s, _u8p))
    return q, s


def dequantize(q: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Packed e2m1 [rows, K/2] + e8m0 [rows, K/32] -> fp64 [rows, K] (K = 32 * whole blocks; a
    K-tail matrix comes back with its zero padding)."""
    q = np.ascontiguousarray(q, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    rows, K = q.shape[0], q.shape[1] * 2
    out = np.empty((rows, K), np.float64)
    if rows and K:
        lib().oracle_dequantize(_p(q, _u8p), _p(scales, _u8p), rows, K, _p(out, _f64p))
    return out


def gemm_f64(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """C[m,n] = sum_k a[m,k] * b[n,k] in fp64 (plain loop in C)."""
    a = np.ascontiguousarray(a, np.float64)
    b = np.ascontiguousarray(b, np.float64)
    M, K = a.shape
    N = b.shape[0]
    c = np.zeros((M, N), np.float64)
    if M and N:
        lib().oracle_gemm_f64(_p(a, _f64p), _p(b, _f64p), M, N, K, _p(c, _f64p))
    return c


def mxfp4_gemm_ref(aq, as_, bq, bs) -> np.ndarray:
    """fp64 C = dequant(A) . dequant(B)^T from packed operands."""
    return gemm_f64(dequantize(aq, as_), dequantize(bq, bs))


def gemm_entries(aq, as_, bq, bs, idx_m, idx_n) -> np.ndarray:
    """fp64 C[idx_m[i], idx_n[i]] one by one from packed operands."""
    aq = np.ascontiguousarray(aq, np.uint8)
    as_ = np.ascontiguousarray(as_, np.uint8)
    bq = np.ascontiguousarray(bq, np.uint8)
    bs = np.ascontiguousarray(bs, np.uint8)
    im = np.ascontiguousarray(idx_m, np.int64)
    inn = np.ascontiguousarray(idx_n, np.int64)
    K = aq.shape[1] * 2
    out = np.empty(im.shape[0], np.float64)
    lib().oracle_gemm_entries(_p(aq, _u8p), _p(as_, _u8p), _p(bq, _u8p), _p(bs, _u8p), K,
                              _p(im, _i64p), _p(inn, _i64p), im.shape[0], _p(out, _f64p))
    return out


def to_bf16(c: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 bit patterns (uint16), one round-to-nearest-even rounding."""
    c = np.ascontiguousarray(c, np.float64)
    out = np.empty(c.shape, np.uint16)
    if c.size:
        lib().oracle_f64_to_bf16_array(_p(c, _f64p), c.size, _p(out, _u16p))
    return out


def bf16_to_f64(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp64 (exact)."""
    h = np.asarray(h, np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def e2m1_encode(qx: float) -> int:
    return int(lib().oracle_e2m1_encode(float(qx)))


def e2m1_encode_count(v: float) -> int:
    """The self-check's second encoder (midpoints counted), for the pins."""
    return int(lib().oracle_e2m1_encode_count(float(v)))


def e2m1_decode(code: int) -> float:
    return float(lib().oracle_e2m1_decode(code))


def scale_byte_of_amax(amax: float) -> int:
    s = lib().oracle_scale_exponent(lib().oracle_round_amax_bits(float(amax)))
    return int(s) + 127


def encode_selfcheck(lo: int, hi: int, step: int = 1) -> tuple[int, int]:
    first = ctypes.c_uint32(0)
    bad = lib().oracle_encode_selfcheck(lo, hi, step, ctypes.byref(first))
    return int(bad), int(first.value)


def tolerance_ok(c: np.ndarray, c_ref: np.ndarray, rel: float = 8e-3, rms_frac: float = 1e-3):
    """The acceptance bound |C - C_ref| <= rel*|C_ref| + rms_frac*rms(C_ref), elementwise.
    Returns (all_ok, worst_ratio) where worst_ratio = max |C-C_ref| / bound."""
    c = np.asarray(c, np.float64)
    c_ref = np.asarray(c_ref, np.float64)
    rms = float(np.sqrt(np.mean(c_ref * c_ref))) if c_ref.size else 0.0
    bound = rel * np.abs(c_ref) + rms_frac * rms
    err = np.abs(c - c_ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / np.where(bound > 0, bound, 1), np.where(err > 0, np.inf, 0))
    worst = float(ratio.max()) if ratio.size else 0.0
    return bool(np.all(err <= bound)), worst
