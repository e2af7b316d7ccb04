"""Helpers shared by the GPU tests: move generated problems to the device,
call the library through its binding, and grade against the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle

_cache = {}


def cached(key, make):
    if key not in _cache:
        _cache[key] = make()
    return _cache[key]


def qg():
    import __graft_entry__
    __graft_entry__.build_library()
    import weight_only_quantized_qgemm_gb300 as q
    return q


def bits_to_bf16(a: np.ndarray, pad_cols: int = 0) -> torch.Tensor:
    M, K = a.shape
    t = torch.zeros((M, K + pad_cols), dtype=torch.int16)
    t[:, :K] = torch.from_numpy(a.view(np.int16))
    return t.view(torch.bfloat16).cuda()


def bits_to_f16(a: np.ndarray, pad_cols: int = 0) -> torch.Tensor:
    M, K = a.shape
    t = torch.zeros((M, K + pad_cols), dtype=torch.int16)
    t[:, :K] = torch.from_numpy(a.view(np.int16))
    return t.view(torch.float16).cuda()


def to_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


class Fp8Device:
    def __init__(self, p, copies: int = 1):
        self.p = p
        self.W = [torch.from_numpy(p.W).cuda() for _ in range(copies)]
        self.S = torch.from_numpy(p.S).cuda()

    def run(self, X_bits=None, x_pad=0, y_pad=0, canary=True, copy=0, q=None):
        q = q or qg()
        Xb = self.p.X if X_bits is None else X_bits
        M, K = Xb.shape
        N = self.p.N
        Xd = bits_to_bf16(Xb, x_pad)
        Y = torch.empty((M, N + y_pad), dtype=torch.bfloat16, device="cuda")
        if canary:
            Y.view(torch.int16).fill_(0x7FC1)  # a NaN pattern
        q.qgemm_fp8_block(Xd[:, :K], self.W[copy], self.S, Y=Y[:, :N])
        return Y


def grade_fp8(p, y_bits, X_bits=None, ms=None, ns=None, nthreads=0):
    X = p.X if X_bits is None else X_bits
    if ms is None:
        ref = oracle.qgemm_fp8_block(X, p.W, p.S, nthreads=nthreads)
        A = oracle.fp8_abs_mass(X, p.W, p.S, nthreads=nthreads)
        got = y_bits
    else:
        ref = oracle.qgemm_fp8_block_sample(X, p.W, p.S, ms, ns, nthreads=nthreads)
        A = oracle.fp8_abs_mass(X, p.W, p.S, ms, ns, nthreads=nthreads)
        got = y_bits[ms, ns]
    return oracle.within_budget(got, ref, A, fmt="bf16")


class Lut3Device:
    def __init__(self, p, q=None):
        q = q or qg()
        self.p = p
        self.Wq = torch.from_numpy(q.pack_lut3(p.codes)).cuda()
        self.qmap = torch.from_numpy(p.qmap.view(np.int16)).view(torch.float16).cuda()
        self.scales = torch.from_numpy(p.scales.view(np.int16)).view(torch.float16).cuda()

    def run(self, x_pad=0, y_pad=0, canary=True, q=None, X_bits=None):
        q = q or qg()
        Xb = self.p.X if X_bits is None else X_bits
        M, K = Xb.shape
        N = self.p.N
        Xd = bits_to_f16(Xb, x_pad)
        Y = torch.empty((M, N + y_pad), dtype=torch.float16, device="cuda")
        if canary:
            Y.view(torch.int16).fill_(0x7E01)
        q.qgemm_lut3(Xd[:, :K], self.Wq, self.qmap, self.scales, N, Y=Y[:, :N])
        return Y


def grade_lut3(p, y_bits, X_bits=None, ms=None, ns=None, nthreads=0):
    X = p.X if X_bits is None else X_bits
    if ms is None:
        ref = oracle.qgemm_lut3(X, p.codes, p.qmap, p.scales, nthreads=nthreads)
        A = oracle.lut3_abs_mass(X, p.codes, p.qmap, p.scales, nthreads=nthreads)
        got = y_bits
    else:
        ref = oracle.qgemm_lut3_sample(X, p.codes, p.qmap, p.scales, ms, ns, nthreads=nthreads)
        A = oracle.lut3_abs_mass(X, p.codes, p.qmap, p.scales, ms, ns, nthreads=nthreads)
        got = y_bits[ms, ns]
    return oracle.within_budget(got, ref, A, fmt="fp16")


def sample_indices(M, N, count, seed=0):
    rng = np.random.default_rng(seed)
    ms = rng.integers(0, M, count)
    ns = rng.integers(0, N, count)
    # always include the corners and the ragged tail
    ms = np.concatenate([ms, [0, M - 1, 0, M - 1]])
    ns = np.concatenate([ns, [0, 0, N - 1, N - 1]])
    return ms.astype(np.int32), ns.astype(np.int32)


def assert_counters_clear(q, ws, kind, M, N, K):
    """The workspace's arrival counters (everything from the counter offset
    on, for every shape) are zero, as the header promises after a call."""
    need = q.workspace_bytes(kind, M, N, K)
    assert need > 0
    cnt_bytes = (16 * (-(-N // 128)) + 255) // 256 * 256
    off = need - cnt_bytes
    assert int(ws.buf[off:].count_nonzero()) == 0
