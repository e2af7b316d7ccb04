"""Dense BF16 decode GEMM (qgemm_bf16) on the GPU against the CPU oracle,
element by element: small and ragged shapes in full, an output-projection
(lm_head) shape N=32768, K=5120 in full at M = 1, 16, 32."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import cached, qg, to_bits

pytestmark = pytest.mark.gpu


def _dev(bits: np.ndarray, pad_cols: int = 0) -> torch.Tensor:
    R, C = bits.shape
    t = torch.zeros((R, C + pad_cols), dtype=torch.int16)
    t[:, :C] = torch.from_numpy(bits.view(np.int16))
    return t.view(torch.bfloat16).cuda()


def _grade(p, y, X=None):
    """The comparison rule of the numerics contract (2 BF16 ULP, or the
    absolute floor for outputs that cancel) and the Frobenius gate.  The
    FP8 tests' extra bound on the relative error of near-cancelling outputs
    is not asserted here: the oracle sums all K terms in one strict-order FP32
    chain (no 128-wide blocks), whose own rounding error grows like
    sqrt(K) * 2^-24 * sum|x w|, so an output that cancels to ~1e-4 of that
    mass can differ from it by a few percent while staying inside the floor."""
    X = p.X if X is None else X
    ref = oracle.gemm_bf16(X, p.W)
    A = oracle.bf16_abs_mass(X, p.W)
    ok, rep = oracle.within_budget(y, ref, A, fmt="bf16")
    assert rep.ok, rep
    assert rep.fro_rel <= 2e-3, rep
    return rep


def _run(q, p, x_pad=0, y_pad=0, W=None, X=None):
    Xb = p.X if X is None else X
    M, K = Xb.shape
    Xd = _dev(Xb, x_pad)
    Wd = _dev(p.W) if W is None else W
    Y = torch.empty((M, p.N + y_pad), dtype=torch.bfloat16, device="cuda")
    Y.view(torch.int16).fill_(0x7FC1)
    q.qgemm_bf16(Xd[:, :K], Wd, Y=Y[:, :p.N])
    assert q.last_device_status() == 0
    return Y


@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (16, 1024, 5120), (32, 640, 1024), (5, 200, 336), (7, 77, 8),
                                   (20, 3000, 1040), (17, 128, 4096)])
def test_bf16_shapes(M, N, K):
    q = qg()
    p = cached(("bf16", M, N, K), lambda: wl.make_bf16_problem(M, N, K, config_id=20))
    Y = _run(q, p)
    _grade(p, to_bits(Y))


def test_bf16_strided_and_padding_untouched():
    q = qg()
    p = wl.make_bf16_problem(6, 1000, 2056, config_id=21)
    Y = _run(q, p, x_pad=24, y_pad=40)
    _grade(p, to_bits(Y[:, :1000]))
    assert np.all(to_bits(Y[:, 1000:]) == 0x7FC1)


@pytest.mark.parametrize("M", [1, 16, 32])
def test_bf16_lm_head_full(M):
    """N=32768, K=5120 (320 MB of BF16 weights), every element."""
    q = qg()
    p = cached(("bf16", 32, 32768, 5120), lambda: wl.make_bf16_problem(32, 32768, 5120, config_id=5))
    W = cached(("bf16dev", 32768, 5120), lambda: _dev(p.W))
    Xb = p.X[:M]
    Y = _run(q, p, W=W, X=Xb)
    _grade(p, to_bits(Y), X=Xb)


def test_bf16_deterministic_and_split_grids_agree():
    """Same bits call after call; a split-K grid and the one-CTA-per-tile grid
    both within budget."""
    q = qg()
    M, N, K = 16, 5120, 5120
    p = cached(("bf16", M, N, K), lambda: wl.make_bf16_problem(M, N, K, config_id=22))
    Xd, Wd = _dev(p.X), _dev(p.W)
    ws = q.Workspace()
    try:
        for G in (None, 40, 152):
            if G is not None:
                q.dispatch_set(q.KIND_BF16, M, N, K, G)
            outs = [to_bits(q.qgemm_bf16(Xd, Wd, workspace=ws)) for _ in range(3)]
            assert q.last_device_status() == 0
            assert all(np.array_equal(o, outs[0]) for o in outs[1:])
            _grade(p, outs[0])
    finally:
        q.dispatch_clear()
