"""3-bit learned-LUT GEMM on the GPU against the CPU oracle, through the C ABI
(FP16 output: <= 2 FP16 ULP per element or within the near-zero floor, and a
Frobenius relative error within the page's 2e-3 gate)."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import Lut3Device, cached, grade_lut3, qg, sample_indices, to_bits

pytestmark = pytest.mark.gpu


def _problem(M, N, K, cid=4):
    return cached(("lut3", M, N, K, cid), lambda: wl.make_lut3_problem(M, N, K, config_id=cid))


def _check(p, Y, X_bits=None, ms=None, ns=None):
    q = qg()
    assert q.last_device_status() == 0
    y = to_bits(Y)
    ok, rep = grade_lut3(p, y, X_bits=X_bits, ms=ms, ns=ns)
    assert rep.ok, rep
    assert rep.fro_rel <= 2e-3, rep
    return y, rep


@pytest.mark.parametrize("M", [1, 4, 8, 16, 17, 32])
def test_small_full(M):
    p = _problem(32, 512, 2048, 31)
    dev = cached(("lut3dev", 512, 2048), lambda: Lut3Device(p))
    Xb = p.X[:M]
    _check(p, dev.run(X_bits=Xb), X_bits=Xb)


@pytest.mark.parametrize("N,K", [(200, 384), (130, 128), (1000, 1152), (77, 4096), (28672 // 8, 8192)])
@pytest.mark.parametrize("M", [1, 9])
def test_ragged_shapes(M, N, K):
    p = _problem(M, N, K, 32)
    _check(p, Lut3Device(p).run())


@pytest.mark.parametrize("M", [1, 4, 8, 16])
def test_full_size_sampled(M):
    """N=28672, K=8192 (the page's largest shape), 4096 sampled elements plus
    corners; the whole output is checked for unwritten (NaN canary) entries."""
    p = _problem(16, 28672, 8192)
    dev = cached(("lut3dev", 28672, 8192), lambda: Lut3Device(p))
    Xb = p.X[:M]
    Y = dev.run(X_bits=Xb)
    ms, ns = sample_indices(M, 28672, 4096, seed=M)
    y, _ = _check(p, Y, X_bits=Xb, ms=ms, ns=ns)
    assert not np.any((y & 0x7C00) == 0x7C00)


def test_full_size_rows_complete():
    """Two complete rows of the M=16 full-size product."""
    p = _problem(16, 28672, 8192)
    dev = cached(("lut3dev", 28672, 8192), lambda: Lut3Device(p))
    Y = dev.run()
    N = 28672
    ms = np.repeat(np.array([0, 15], dtype=np.int32), N)
    ns = np.tile(np.arange(N, dtype=np.int32), 2)
    _check(p, Y, ms=ms, ns=ns)


def test_strided_and_padding_untouched():
    p = _problem(3, 384, 1024, 33)
    Y = Lut3Device(p).run(x_pad=8, y_pad=24)
    _check(p, Y[:, :384])
    assert np.all(to_bits(Y[:, 384:]) == 0x7E01)


def test_back_to_back_calls_bit_identical():
    """48 calls in a row at N=28672, K=8192, M=16 give the same bits every
    time (deterministic result; a pipeline hazard would show as a difference);
    two rows of the first result are graded in full."""
    q = qg()
    p = _problem(16, 28672, 8192)
    dev = cached(("lut3dev", 28672, 8192), lambda: Lut3Device(p))
    Xd = torch.from_numpy(p.X.view(np.int16)).view(torch.float16).cuda()
    ws = q.Workspace()
    outs = [q.qgemm_lut3(Xd, dev.Wq, dev.qmap, dev.scales, p.N, workspace=ws) for _ in range(48)]
    assert q.last_device_status() == 0
    first = to_bits(outs[0])
    for i, Y in enumerate(outs[1:], 1):
        y = to_bits(Y)
        assert np.array_equal(y, first), f"call {i}: {int((y != first).sum())} elements differ"
    ms = np.repeat(np.array([3, 12], dtype=np.int32), p.N)
    ns = np.tile(np.arange(p.N, dtype=np.int32), 2)
    _check(p, outs[0], ms=ms, ns=ns)
