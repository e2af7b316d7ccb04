"""CPU oracle for the weight-only quantized decode GEMM (TEST INFRASTRUCTURE).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The CUDA library never imports it, and it
imports nothing from the CUDA library.

The arithmetic lives in ``qgemm_oracle.c`` (plain C, ``-ffp-contract=off``),
compiled on first use into ``oracle/_build/liboracle.so``.  This module adds
numpy marshalling and the comparison criterion:

* ``bf16_ord`` / ``fp16_ord`` -- ordinal of a bit pattern, so that ULP
  distance is a difference of ordinals (the "atlas" m16_tc page's oracle
  module exports a BF16 ordinal for exactly this use).
* ``within_budget`` -- the one pass/fail rule.  An element passes if its
  ordinal distance to the reference is at most ``MAX_ULP`` (= 2, the page's
  "<= 2 BF16 ULP per element" contract, section NUMERICS) **or** its
  absolute error is at most the floor
  ``FLOOR_MARGIN * 2**-24 * A[m, n]``, where ``A`` is the absolute mass of
  the sum (see ``fp8_abs_mass`` / ``lut3_abs_mass``).  The floor is the
  page's mixed absolute/relative criterion for outputs that cancel to near
  zero (section "THE ROUND-6 M=32 RED CELL WAS THE ORACLE"); the page does not
  print its constant, so ``FLOOR_MARGIN = 32`` is this oracle's reading,
  fixed before any GPU kernel existed.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

__all__ = [
    "MAX_ULP", "FLOOR_MARGIN", "lib", "build", "e4m3_to_float", "bf16_to_float",
    "fp16_to_float", "float_to_bf16", "float_to_fp16", "qgemm_fp8_block",
    "qgemm_fp8_block_sample", "fp8_abs_mass", "lut3_dequant", "lut3_dequant_matrix",
    "qgemm_lut3", "qgemm_lut3_sample", "lut3_abs_mass", "pack_lut3", "unpack_lut3",
    "lut3_packed_bytes", "bf16_ord", "fp16_ord", "within_budget", "BudgetReport",
    "gemm_bf16", "gemm_bf16_sample", "bf16_abs_mass", "float_to_e4m3", "quantize_act_e4m3",
    "qgemm_w8a8_block", "w8a8_abs_mass",
    "max_threads",
]

MAX_ULP = 2
FLOOR_MARGIN = 32.0

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qgemm_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, no FP contraction). Returns the .so path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    tmp = _SO + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c99", "-D_DEFAULT_SOURCE", "-ffp-contract=off", "-fno-fast-math",
           "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_int64

_SIGS = {
    "oracle_e4m3_to_float": (ctypes.c_float, [ctypes.c_uint8]),
    "oracle_bf16_to_float": (ctypes.c_float, [ctypes.c_uint16]),
    "oracle_fp16_to_float": (ctypes.c_float, [ctypes.c_uint16]),
    "oracle_float_to_bf16_rne": (ctypes.c_uint16, [ctypes.c_float]),
    "oracle_float_to_fp16_rne": (ctypes.c_uint16, [ctypes.c_float]),
    "oracle_max_threads": (_I, []),
    "oracle_e4m3_to_float_array": (None, [_L, _P, _P]),
    "oracle_fp16_to_float_array": (None, [_L, _P, _P]),
    "oracle_float_to_bf16_array": (None, [_L, _P, _P]),
    "oracle_float_to_fp16_array": (None, [_L, _P, _P]),
    "oracle_qgemm_fp8_block": (None, [_I, _I, _I, _P, _L, _P, _L, _P, _L, _P, _P, _L, _I]),
    "oracle_qgemm_fp8_block_sample": (None, [_I, _I, _I, _P, _L, _P, _L, _P, _L, _P, _P, _L, _P, _P, _I]),
    "oracle_fp8_abs_mass": (None, [_I, _I, _I, _P, _L, _P, _L, _P, _L, _P, _P, _L, _P, _I]),
    "oracle_float_to_e4m3_rne_sat": (ctypes.c_uint8, [ctypes.c_float]),
    "oracle_quantize_act_e4m3": (None, [_I, _I, _P, _L, _P, _L, _P, _L]),
    "oracle_qgemm_w8a8_block": (None, [_I, _I, _I, _P, _L, _P, _L, _P, _L, _P, _L, _P, _P, _L, _I]),
    "oracle_w8a8_abs_mass": (None, [_I, _I, _I, _P, _L, _P, _L, _P, _L, _P, _L, _P, _I]),
    "oracle_gemm_bf16": (None, [_I, _I, _I, _P, _L, _P, _L, _P, _P, _L, _I]),
    "oracle_gemm_bf16_sample": (None, [_I, _I, _I, _P, _L, _P, _L, _P, _P, _L, _P, _P, _I]),
    "oracle_bf16_abs_mass": (None, [_I, _I, _I, _P, _L, _P, _L, _P, _P, _L, _P, _I]),
    "oracle_lut3_dequant": (ctypes.c_uint16, [ctypes.c_uint8, _P, ctypes.c_uint16]),
    "oracle_lut3_dequant_matrix": (None, [_I, _I, _P, _L, _P, _P, _L, _P, _L]),
    "oracle_qgemm_lut3": (None, [_I, _I, _I, _P, _L, _P, _L, _P, _P, _L, _P, _P, _L, _I]),
    "oracle_qgemm_lut3_sample": (None, [_I, _I, _I, _P, _L, _P, _L, _P, _P, _L, _P, _P, _L, _P, _P, _I]),
    "oracle_lut3_abs_mass": (None, [_I, _I, _I, _P, _L, _P, _L, _P, _P, _L, _P, _P, _L, _P, _I]),
    "oracle_lut3_packed_bytes": (_L, [_I, _I]),
    "oracle_pack_lut3": (None, [_I, _I, _P, _P]),
    "oracle_unpack_lut3": (None, [_I, _I, _P, _P]),
}


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            handle = ctypes.CDLL(path)
            for name, (res, args) in _SIGS.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def max_threads() -> int:
    return int(lib().oracle_max_threads())


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- scalars
def e4m3_to_float(codes) -> np.ndarray:
    c = _c(codes, np.uint8).ravel()
    out = np.empty(c.size, dtype=np.float32)
    lib().oracle_e4m3_to_float_array(c.size, _ptr(c), _ptr(out))
    return out.reshape(np.shape(codes))


def bf16_to_float(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def fp16_to_float(bits) -> np.ndarray:
    b = _c(bits, np.uint16).ravel()
    out = np.empty(b.size, dtype=np.float32)
    lib().oracle_fp16_to_float_array(b.size, _ptr(b), _ptr(out))
    return out.reshape(np.shape(bits))


def float_to_bf16(x) -> np.ndarray:
    v = _c(x, np.float32).ravel()
    out = np.empty(v.size, dtype=np.uint16)
    lib().oracle_float_to_bf16_array(v.size, _ptr(v), _ptr(out))
    return out.reshape(np.shape(x))


def float_to_fp16(x) -> np.ndarray:
    v = _c(x, np.float32).ravel()
    out = np.empty(v.size, dtype=np.uint16)
    lib().oracle_float_to_fp16_array(v.size, _ptr(v), _ptr(out))
    return out.reshape(np.shape(x))


# ---------------------------------------------------------------- W8A8
def float_to_e4m3(x) -> np.ndarray:
    """E4M3FN codes of float32 values: round to nearest even, saturating at +-448."""
    a = np.ascontiguousarray(x, dtype=np.float32).ravel()
    f = lib().oracle_float_to_e4m3_rne_sat
    return np.array([f(float(v)) for v in a], dtype=np.uint8).reshape(np.shape(x))


def quantize_act_e4m3(X):
    """Per (row, 128-wide K block) activation quantiser: returns (Xq uint8
    [M, K] E4M3 codes, Sx float32 [ceil(K/128), M] scales)."""
    X = _c(X, np.uint16)
    M, K = X.shape
    KB = -(-K // 128)
    Xq = np.empty((M, K), dtype=np.uint8)
    Sx = np.empty((KB, M), dtype=np.float32)
    lib().oracle_quantize_act_e4m3(M, K, _ptr(X), K, _ptr(Xq), K, _ptr(Sx), M)
    return Xq, Sx


def qgemm_w8a8_block(Xq, Sx, W, S, nthreads: int = 0, want_f32: bool = False):
    """Y = bf16(two-level fold of E4M3 Xq[M,K] . W[N,K]^T with block factor
    Sx[kb, m] * S[n/128, kb])."""
    Xq = _c(Xq, np.uint8); Sx = _c(Sx, np.float32); W = _c(W, np.uint8); S = _c(S, np.float32)
    M, K = Xq.shape
    N = W.shape[0]
    assert W.shape[1] == K and S.shape == (-(-N // 128), -(-K // 128)) and Sx.shape == (-(-K // 128), M)
    Y = np.empty((M, N), dtype=np.uint16)
    Yf = np.empty((M, N), dtype=np.float32) if want_f32 else None
    lib().oracle_qgemm_w8a8_block(M, N, K, _ptr(Xq), K, _ptr(Sx), M, _ptr(W), K, _ptr(S), S.shape[1],
                                  _ptr(Y), _ptr(Yf), N, nthreads)
    return (Y, Yf) if want_f32 else Y


def w8a8_abs_mass(Xq, Sx, W, S, nthreads: int = 0) -> np.ndarray:
    Xq = _c(Xq, np.uint8); Sx = _c(Sx, np.float32); W = _c(W, np.uint8); S = _c(S, np.float32)
    M, K = Xq.shape
    N = W.shape[0]
    A = np.empty((M, N), dtype=np.float64)
    lib().oracle_w8a8_abs_mass(M, N, K, _ptr(Xq), K, _ptr(Sx), M, _ptr(W), K, _ptr(S), S.shape[1], _ptr(A),
                               nthreads)
    return A


# ---------------------------------------------------------------- dense BF16 GEMM
def gemm_bf16(X, W, nthreads: int = 0, want_f32: bool = False):
    """Y = bf16(X[M,K] . W[N,K]^T), FP32 sums in strict K order (BF16 bits in
    and out)."""
    X = _c(X, np.uint16); W = _c(W, np.uint16)
    M, K = X.shape
    N = W.shape[0]
    assert W.shape[1] == K
    Y = np.empty((M, N), dtype=np.uint16)
    Yf = np.empty((M, N), dtype=np.float32) if want_f32 else None
    lib().oracle_gemm_bf16(M, N, K, _ptr(X), K, _ptr(W), K, _ptr(Y), _ptr(Yf), N, nthreads)
    return (Y, Yf) if want_f32 else Y


def gemm_bf16_sample(X, W, ms, ns, nthreads: int = 0, want_f32: bool = False):
    X = _c(X, np.uint16); W = _c(W, np.uint16)
    M, K = X.shape
    N = W.shape[0]
    ms = _c(ms, np.int32); ns = _c(ns, np.int32)
    Y = np.empty(ms.size, dtype=np.uint16)
    Yf = np.empty(ms.size, dtype=np.float32) if want_f32 else None
    lib().oracle_gemm_bf16_sample(M, N, K, _ptr(X), K, _ptr(W), K, _ptr(ms), _ptr(ns), ms.size, _ptr(Y),
                                  _ptr(Yf), nthreads)
    return (Y, Yf) if want_f32 else Y


def bf16_abs_mass(X, W, ms=None, ns=None, nthreads: int = 0) -> np.ndarray:
    X = _c(X, np.uint16); W = _c(W, np.uint16)
    M, K = X.shape
    N = W.shape[0]
    if ms is None:
        A = np.empty((M, N), dtype=np.float64)
        lib().oracle_bf16_abs_mass(M, N, K, _ptr(X), K, _ptr(W), K, None, None, 0, _ptr(A), nthreads)
        return A
    ms = _c(ms, np.int32); ns = _c(ns, np.int32)
    A = np.empty(ms.size, dtype=np.float64)
    lib().oracle_bf16_abs_mass(M, N, K, _ptr(X), K, _ptr(W), K, _ptr(ms), _ptr(ns), ms.size, _ptr(A), nthreads)
    return A


# ---------------------------------------------------------------- FP8 GEMM
def qgemm_fp8_block(X, W, S, nthreads: int = 0, want_f32: bool = False):
    """Y = bf16(two-level fold of X[M,K] . dequant(W)[N,K]^T).  Returns BF16 bits
    [M, N] (and the FP32 pre-rounding values if ``want_f32``)."""
    X = _c(X, np.uint16); W = _c(W, np.uint8); S = _c(S, np.float32)
    M, K = X.shape
    N = W.shape[0]
    assert W.shape[1] == K and S.shape == (-(-N // 128), -(-K // 128))
    Y = np.empty((M, N), dtype=np.uint16)
    Yf = np.empty((M, N), dtype=np.float32) if want_f32 else None
    lib().oracle_qgemm_fp8_block(M, N, K, _ptr(X), K, _ptr(W), K, _ptr(S), S.shape[1],
                                 _ptr(Y), _ptr(Yf), N, nthreads)
    return (Y, Yf) if want_f32 else Y


def qgemm_fp8_block_sample(X, W, S, ms, ns, nthreads: int = 0, want_f32: bool = False):
    X = _c(X, np.uint16); W = _c(W, np.uint8); S = _c(S, np.float32)
    M, K = X.shape
    N = W.shape[0]
    ms = _c(ms, np.int32); ns = _c(ns, np.int32)
    Y = np.empty(ms.size, dtype=np.uint16)
    Yf = np.empty(ms.size, dtype=np.float32) if want_f32 else None
    lib().oracle_qgemm_fp8_block_sample(M, N, K, _ptr(X), K, _ptr(W), K, _ptr(S), S.shape[1],
                                        _ptr(ms), _ptr(ns), ms.size, _ptr(Y), _ptr(Yf), nthreads)
    return (Y, Yf) if want_f32 else Y


def fp8_abs_mass(X, W, S, ms=None, ns=None, nthreads: int = 0) -> np.ndarray:
    X = _c(X, np.uint16); W = _c(W, np.uint8); S = _c(S, np.float32)
    M, K = X.shape
    N = W.shape[0]
    if ms is None:
        A = np.empty((M, N), dtype=np.float64)
        lib().oracle_fp8_abs_mass(M, N, K, _ptr(X), K, _ptr(W), K, _ptr(S), S.shape[1],
                                  None, None, 0, _ptr(A), nthreads)
        return A
    ms = _c(ms, np.int32); ns = _c(ns, np.int32)
    A = np.empty(ms.size, dtype=np.float64)
    lib().oracle_fp8_abs_mass(M, N, K, _ptr(X), K, _ptr(W), K, _ptr(S), S.shape[1],
                              _ptr(ms), _ptr(ns), ms.size, _ptr(A), nthreads)
    return A


# ---------------------------------------------------------------- LUT3 GEMM
def lut3_dequant(code: int, qmap, scale_bits: int) -> int:
    q = _c(qmap, np.uint16)
    return int(lib().oracle_lut3_dequant(int(code), _ptr(q), int(scale_bits)))


def lut3_dequant_matrix(codes, qmap, scales) -> np.ndarray:
    codes = _c(codes, np.uint8); q = _c(qmap, np.uint16); sc = _c(scales, np.uint16)
    N, K = codes.shape
    D = np.empty((N, K), dtype=np.uint16)
    lib().oracle_lut3_dequant_matrix(N, K, _ptr(codes), K, _ptr(q), _ptr(sc), sc.shape[1],
                                     _ptr(D), K)
    return D


def qgemm_lut3(X, codes, qmap, scales, nthreads: int = 0, want_f32: bool = False):
    X = _c(X, np.uint16); codes = _c(codes, np.uint8)
    q = _c(qmap, np.uint16); sc = _c(scales, np.uint16)
    M, K = X.shape
    N = codes.shape[0]
    Y = np.empty((M, N), dtype=np.uint16)
    Yf = np.empty((M, N), dtype=np.float32) if want_f32 else None
    lib().oracle_qgemm_lut3(M, N, K, _ptr(X), K, _ptr(codes), K, _ptr(q), _ptr(sc), sc.shape[1],
                            _ptr(Y), _ptr(Yf), N, nthreads)
    return (Y, Yf) if want_f32 else Y


def qgemm_lut3_sample(X, codes, qmap, scales, ms, ns, nthreads: int = 0, want_f32: bool = False):
    X = _c(X, np.uint16); codes = _c(codes, np.uint8)
    q = _c(qmap, np.uint16); sc = _c(scales, np.uint16)
    M, K = X.shape
    N = codes.shape[0]
    ms = _c(ms, np.int32); ns = _c(ns, np.int32)
    Y = np.empty(ms.size, dtype=np.uint16)
    Yf = np.empty(ms.size, dtype=np.float32) if want_f32 else None
    lib().oracle_qgemm_lut3_sample(M, N, K, _ptr(X), K, _ptr(codes), K, _ptr(q), _ptr(sc),
                                   sc.shape[1], _ptr(ms), _ptr(ns), ms.size, _ptr(Y), _ptr(Yf),
                                   nthreads)
    return (Y, Yf) if want_f32 else Y


def lut3_abs_mass(X, codes, qmap, scales, ms=None, ns=None, nthreads: int = 0) -> np.ndarray:
    X = _c(X, np.uint16); codes = _c(codes, np.uint8)
    q = _c(qmap, np.uint16); sc = _c(scales, np.uint16)
    M, K = X.shape
    N = codes.shape[0]
    if ms is None:
        A = np.empty((M, N), dtype=np.float64)
        lib().oracle_lut3_abs_mass(M, N, K, _ptr(X), K, _ptr(codes), K, _ptr(q), _ptr(sc),
                                   sc.shape[1], None, None, 0, _ptr(A), nthreads)
        return A
    ms = _c(ms, np.int32); ns = _c(ns, np.int32)
    A = np.empty(ms.size, dtype=np.float64)
    lib().oracle_lut3_abs_mass(M, N, K, _ptr(X), K, _ptr(codes), K, _ptr(q), _ptr(sc),
                               sc.shape[1], _ptr(ms), _ptr(ns), ms.size, _ptr(A), nthreads)
    return A


def lut3_packed_bytes(N: int, K: int) -> int:
    return int(lib().oracle_lut3_packed_bytes(N, K))


def pack_lut3(codes) -> np.ndarray:
    codes = _c(codes, np.uint8)
    N, K = codes.shape
    out = np.empty(lut3_packed_bytes(N, K), dtype=np.uint8)
    lib().oracle_pack_lut3(N, K, _ptr(codes), _ptr(out))
    return out


def unpack_lut3(packed, N: int, K: int) -> np.ndarray:
    p = _c(packed, np.uint8).view(np.uint8).ravel()
    assert p.size == lut3_packed_bytes(N, K)
    out = np.empty((N, K), dtype=np.uint8)
    lib().oracle_unpack_lut3(N, K, _ptr(p), _ptr(out))
    return out


# ---------------------------------------------------------------- criterion
def bf16_ord(bits) -> np.ndarray:
    """Ordinal of BF16 bit patterns: +0 and -0 map to 0, adjacent values differ by 1."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def fp16_ord(bits) -> np.ndarray:
    """Ordinal of FP16 bit patterns (same construction as :func:`bf16_ord`)."""
    return bf16_ord(bits)


@dataclass
class BudgetReport:
    count: int
    over_budget: int
    max_ulp: int
    max_ulp_outside_floor: int
    sign_flips: int
    rel_rms: float
    max_rel_err: float
    fro_rel: float

    @property
    def ok(self) -> bool:
        return self.over_budget == 0


def within_budget(gpu_bits, ref_bits, abs_mass, fmt: str = "bf16",
                  max_ulp: int = MAX_ULP, margin: float = FLOOR_MARGIN):
    """Evaluate the comparison rule; returns (pass_mask, BudgetReport).

    ``fmt`` is "bf16" or "fp16" and fixes how the bit patterns decode and
    which ULP grid ``max_ulp`` counts on.
    """
    g = np.asarray(gpu_bits, dtype=np.uint16).ravel()
    r = np.asarray(ref_bits, dtype=np.uint16).ravel()
    A = np.asarray(abs_mass, dtype=np.float64).ravel()
    if fmt == "bf16":
        gv = bf16_to_float(g).astype(np.float64)
        rv = bf16_to_float(r).astype(np.float64)
    elif fmt == "fp16":
        gv = g.view(np.float16).astype(np.float64)
        rv = r.view(np.float16).astype(np.float64)
    else:
        raise ValueError(fmt)
    ulp = np.abs(bf16_ord(g) - bf16_ord(r))
    floor = margin * 2.0 ** -24 * A
    err = np.abs(gv - rv)
    finite = np.isfinite(gv) & np.isfinite(rv)
    in_floor = finite & (err <= floor)
    ok = finite & ((ulp <= max_ulp) | in_floor)
    flips = int(np.sum((np.sign(gv) * np.sign(rv) < 0) & ~in_floor))
    denom = np.maximum(np.abs(rv), floor)
    with np.errstate(divide="ignore", invalid="ignore"):
        rel = np.where(denom > 0, err / denom, np.where(err > 0, np.inf, 0.0))
    ref_rms = float(np.sqrt(np.mean(rv ** 2))) if rv.size else 0.0
    rel_rms = float(np.sqrt(np.mean(err ** 2)) / ref_rms) if ref_rms > 0 else 0.0
    fro = float(np.linalg.norm(gv - rv) / np.linalg.norm(rv)) if rv.size and np.linalg.norm(rv) > 0 else 0.0
    rep = BudgetReport(
        count=int(g.size),
        over_budget=int(np.sum(~ok)),
        max_ulp=int(ulp.max()) if ulp.size else 0,
        max_ulp_outside_floor=int(ulp[~in_floor].max()) if np.any(~in_floor) else 0,
        sign_flips=flips,
        rel_rms=rel_rms,
        max_rel_err=float(rel.max()) if rel.size else 0.0,
        fro_rel=fro,
    )
    return ok.reshape(np.shape(gpu_bits)), rep
