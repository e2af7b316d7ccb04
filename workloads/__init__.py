"""Seeded synthetic inputs for the weight-only quantized decode GEMM.

This module only *produces input bytes*.  It holds none of the GEMM's
arithmetic (no dequantisation, no accumulation, no output rounding); the CUDA
path and the CPU oracle both consume the arrays made here and share nothing
else.

Workloads (the five configurations of the weight-only decode GEMM study):

* ``fp8_small``  -- W8A16 FP8 block-scaled, M=1, N=256, K=512.
* ``fp8_gateup`` -- FFN gate/up shape, N=17408, K=5120, M=16 (and M=8).
* ``fp8_down``   -- FFN down shape, N=5120, K=17408, M=16 (and M=32).
* ``fp8_attn``   -- small-N attention shapes N in {1024, 5120, 6144},
  K=5120, M in {1,2,4,5,8,16,17,24,32}.
* ``lut3``       -- 3-bit learned-LUT, N=28672, K=8192, M in {1,4,8,16}.
* ``bf16_lm_head`` -- unquantised BF16 decode GEMM of an output-projection
  (lm_head) shape, N=32768, K=5120, M in {1,16,32}.

Input recipe (identical for every consumer):

* FP8 weights: W ~ N(0, 0.02) in float32; each
  [128 x 128] block (ragged at the N/K edges) gets the FP32 scale
  ``s = fl32(amax / 448)`` (448 is the largest finite E4M3 value), and every
  weight becomes ``e4m3_rne_satfinite(fl32(w / s))``.  A block whose amax is
  zero gets ``s = 1`` and all-zero codes.  The E4M3 encoding is PyTorch's
  ``float8_e4m3fn`` conversion (round to nearest even) after clamping to
  [-448, 448], i.e. saturating to the largest finite value.
* Activations: X ~ N(0, 1), rounded to BF16 (FP8 path) or FP16 (LUT path)
  with round-to-nearest-even.
* BF16 weights (dense path): W ~ N(0, 0.02) rounded to BF16.
* LUT3: codes uniform on 0..7; the 8-entry FP16 map is the standard-normal
  quantiles at (i + 0.5) / 8, sorted ascending; per-(row, 128-K group)
  scales ~ U[0.005, 0.02] rounded to FP16.

Random numbers come from numpy's PCG64 bit generator (``standard_normal`` in
float32, ``random``, ``integers``), one stream per tensor, seeded with
``0x51A7E000 + 16 * config_id + tensor_id``.  Every consumer in a run reads
the same arrays; no stored expected value depends on these streams.
"""
from __future__ import annotations

import statistics
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "SEED_BASE", "seed_for", "uniform01", "normal", "uniform_codes", "bf16_bits_from_f32",
    "fp16_bits_from_f32", "e4m3_codes_from_f32", "Fp8Problem", "Lut3Problem", "Bf16Problem", "make_bf16_problem",
    "make_fp8_problem", "make_w8a8_problem", "make_lut3_problem", "lut3_qmap_bits", "WORKLOADS",
]

SEED_BASE = 0x51A7E000


def seed_for(config_id: int, tensor_id: int) -> int:
    return SEED_BASE + 16 * config_id + tensor_id


def _gen(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def uniform01(seed: int, count: int) -> np.ndarray:
    """``count`` doubles in [0, 1) from the stream ``seed``."""
    return _gen(seed).random(count)


def normal(seed: int, count: int) -> np.ndarray:
    """``count`` standard normal float32 values from the stream ``seed``."""
    return _gen(seed).standard_normal(count, dtype=np.float32)


def uniform_codes(seed: int, count: int, levels: int = 8) -> np.ndarray:
    """``count`` integers uniform on 0..levels-1 (uint8) from the stream ``seed``."""
    return _gen(seed).integers(0, levels, size=count, dtype=np.uint8)


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to BF16 (nearest even); returns uint16 bit patterns."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def fp16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to IEEE FP16 (nearest even); returns uint16 bits."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def e4m3_codes_from_f32(v: np.ndarray) -> np.ndarray:
    """Saturating round-to-nearest-even encoding of float32 values as E4M3FN."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).clamp(-448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


@dataclass
class Fp8Problem:
    M: int
    N: int
    K: int
    X: np.ndarray        # uint16 [M, K]  BF16 bits
    W: np.ndarray        # uint8  [N, K]  E4M3 codes
    S: np.ndarray        # float32 [ceil(N/128), ceil(K/128)]
    W_f32: np.ndarray | None = field(default=None, repr=False)  # the pre-quantisation draw


@dataclass
class Lut3Problem:
    M: int
    N: int
    K: int
    X: np.ndarray        # uint16 [M, K]  FP16 bits
    codes: np.ndarray    # uint8 [N, K], values 0..7
    qmap: np.ndarray     # uint16 [8] FP16 bits, ascending
    scales: np.ndarray   # uint16 [N, ceil(K/128)] FP16 bits


def quantize_blockwise_e4m3(w: np.ndarray, block: int = 128) -> tuple[np.ndarray, np.ndarray]:
    """Per-[block x block] amax/448 scaling and E4M3 encoding of a float32 [N,K] matrix."""
    N, K = w.shape
    nb, kb = -(-N // block), -(-K // block)
    S = np.empty((nb, kb), dtype=np.float32)
    codes = np.empty((N, K), dtype=np.uint8)
    for i in range(nb):
        r0, r1 = i * block, min(N, (i + 1) * block)
        rows = w[r0:r1]
        for j in range(kb):
            c0, c1 = j * block, min(K, (j + 1) * block)
            blk = rows[:, c0:c1]
            amax = np.float32(np.max(np.abs(blk)))
            if amax == 0:
                S[i, j] = np.float32(1.0)
                codes[r0:r1, c0:c1] = 0
                continue
            s = np.float32(amax / np.float32(448.0))
            S[i, j] = s
            codes[r0:r1, c0:c1] = e4m3_codes_from_f32((blk / s).astype(np.float32))
    return codes, S


def _quantize_fast(w: np.ndarray, block: int = 128) -> tuple[np.ndarray, np.ndarray]:
    """Same result as :func:`quantize_blockwise_e4m3`, vectorised for shapes
    that are multiples of the block size."""
    N, K = w.shape
    if N % block or K % block:
        return quantize_blockwise_e4m3(w, block)
    nb, kb = N // block, K // block
    v = w.reshape(nb, block, kb, block)
    amax = np.abs(v).max(axis=(1, 3)).astype(np.float32)
    S = np.where(amax == 0, np.float32(1.0), (amax / np.float32(448.0)).astype(np.float32)).astype(np.float32)
    codes = np.empty((N, K), dtype=np.uint8)
    cv = codes.reshape(nb, block, kb, block)
    step = max(1, (1 << 22) // (block * K))
    for i0 in range(0, nb, step):
        i1 = min(nb, i0 + step)
        q = (v[i0:i1] / S[i0:i1, None, :, None]).astype(np.float32)
        cv[i0:i1] = e4m3_codes_from_f32(q)
    zero = amax == 0
    if zero.any():
        for i, j in zip(*np.nonzero(zero)):
            cv[i, :, j, :] = 0
    return codes, S


def make_fp8_problem(M: int, N: int, K: int, config_id: int = 0, keep_float: bool = False,
                     x_seed_tensor: int = 0, w_seed_tensor: int = 1) -> Fp8Problem:
    w = (normal(seed_for(config_id, w_seed_tensor), N * K) * np.float32(0.02)).reshape(N, K)
    codes, S = _quantize_fast(w)
    x = normal(seed_for(config_id, x_seed_tensor), M * K).reshape(M, K)
    X = bf16_bits_from_f32(x).reshape(M, K)
    return Fp8Problem(M, N, K, X, codes, S, w if keep_float else None)


@dataclass
class Bf16Problem:
    M: int
    N: int
    K: int
    X: np.ndarray        # uint16 [M, K]  BF16 bits
    W: np.ndarray        # uint16 [N, K]  BF16 bits


def make_w8a8_problem(M: int, N: int, K: int, config_id: int = 6) -> Fp8Problem:
    """Inputs of the W8A8 path: the FP8 weight generator and BF16 N(0,1)
    activations (quantised to E4M3 by the path itself)."""
    return make_fp8_problem(M, N, K, config_id=config_id)


def make_bf16_problem(M: int, N: int, K: int, config_id: int = 5, x_seed_tensor: int = 0,
                      w_seed_tensor: int = 1) -> Bf16Problem:
    w = (normal(seed_for(config_id, w_seed_tensor), N * K) * np.float32(0.02)).reshape(N, K)
    x = normal(seed_for(config_id, x_seed_tensor), M * K).reshape(M, K)
    return Bf16Problem(M, N, K, bf16_bits_from_f32(x).reshape(M, K), bf16_bits_from_f32(w).reshape(N, K))


def lut3_qmap_bits() -> np.ndarray:
    """FP16 bits of the standard-normal quantiles at (i + 0.5)/8, i = 0..7."""
    nd = statistics.NormalDist()
    q = np.array([nd.inv_cdf((i + 0.5) / 8.0) for i in range(8)], dtype=np.float64)
    return fp16_bits_from_f32(np.sort(q).astype(np.float32))


def make_lut3_problem(M: int, N: int, K: int, config_id: int = 4,
                      x_seed_tensor: int = 0, code_seed_tensor: int = 2,
                      scale_seed_tensor: int = 3) -> Lut3Problem:
    G = -(-K // 128)
    codes = uniform_codes(seed_for(config_id, code_seed_tensor), N * K).reshape(N, K)
    u = uniform01(seed_for(config_id, scale_seed_tensor), N * G)
    scales = fp16_bits_from_f32((0.005 + 0.015 * u).astype(np.float32)).reshape(N, G)
    x = normal(seed_for(config_id, x_seed_tensor), M * K).reshape(M, K)
    X = fp16_bits_from_f32(x).reshape(M, K)
    return Lut3Problem(M, N, K, X, codes, lut3_qmap_bits(), scales)


# name -> (kind, config_id, N, K, list of M)
WORKLOADS = {
    "fp8_small": ("fp8", 0, 256, 512, [1]),
    "fp8_gateup": ("fp8", 1, 17408, 5120, [16, 8]),
    "fp8_down": ("fp8", 2, 5120, 17408, [16, 32]),
    "fp8_attn_1024": ("fp8", 3, 1024, 5120, [1, 2, 4, 5, 8, 16, 17, 24, 32]),
    "fp8_attn_5120": ("fp8", 3, 5120, 5120, [1, 2, 4, 5, 8, 16, 17, 24, 32]),
    "fp8_attn_6144": ("fp8", 3, 6144, 5120, [1, 2, 4, 5, 8, 16, 17, 24, 32]),
    "lut3": ("lut3", 4, 28672, 8192, [1, 4, 8, 16]),
    "bf16_lm_head": ("bf16", 5, 32768, 5120, [1, 16, 32]),
    # W8A8 beyond the decode tier: the gate/up layer at prefill batch sizes
    "w8a8_gateup": ("w8a8", 6, 17408, 5120, [64, 128, 256, 512]),
}
