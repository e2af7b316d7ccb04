"""Several FP8 GEMMs sharing X in one launch (qgemm_fp8_block_multi): the
attention projections Q (N=6144 here), K and V (N=1024 each) at K=5120, and
ragged segments.  Each segment is graded against the oracle on its own, in
full; outputs may go to separate buffers or to column ranges of one fused
buffer (per-segment row strides)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import cached, grade_fp8, qg, to_bits

pytestmark = pytest.mark.gpu


def _segments(M, Ns, K, cid0):
    ps = [cached(("fp8seg", M, N, K, cid0 + j), lambda N=N, j=j: wl.make_fp8_problem(M, N, K, config_id=cid0 + j))
          for j, N in enumerate(Ns)]
    X = ps[0].X
    dev = [(torch.from_numpy(p.W).cuda(), torch.from_numpy(p.S).cuda()) for p in ps]
    return X, ps, dev


@pytest.mark.parametrize("M", [1, 16, 32])
def test_qkv_in_one_launch(M):
    q = qg()
    K = 5120
    X, ps, dev = _segments(32, [6144, 1024, 1024], K, 80)
    Xb = X[:M]
    Xd = torch.from_numpy(Xb.view(np.int16)).view(torch.bfloat16).cuda()
    ws = q.Workspace()
    Ys = [torch.full((M, p.N), float("nan"), dtype=torch.bfloat16, device="cuda") for p in ps]
    outs = []
    for _ in range(3):
        q.qgemm_fp8_block_multi(Xd, dev, Ys=Ys, workspace=ws)
        outs.append([to_bits(Y) for Y in Ys])
    assert q.last_device_status() == 0
    for o in outs[1:]:
        assert all(np.array_equal(a, b) for a, b in zip(o, outs[0]))
    for p, y in zip(ps, outs[0]):
        ok, rep = grade_fp8(p, y, X_bits=Xb)
        assert rep.ok, (p.N, rep)
        assert rep.max_rel_err <= 1e-2, rep


def test_fused_output_buffer_with_strides():
    """The three outputs as column ranges of one [M, 8192 + 24] buffer (row
    stride 8216): the same bits as separate buffers, the padding untouched."""
    q = qg()
    M, K = 16, 5120
    X, ps, dev = _segments(32, [6144, 1024, 1024], K, 80)
    Xd = torch.from_numpy(X[:M].view(np.int16)).view(torch.bfloat16).cuda()
    sep = [to_bits(Y) for Y in q.qgemm_fp8_block_multi(Xd, dev)]
    fused = torch.empty((M, 8192 + 24), dtype=torch.bfloat16, device="cuda")
    fused.view(torch.int16).fill_(0x7FC1)
    views = [fused[:, 0:6144], fused[:, 6144:7168], fused[:, 7168:8192]]
    q.qgemm_fp8_block_multi(Xd, dev, Ys=views)
    assert q.last_device_status() == 0
    for v, ref in zip(views, sep):
        assert np.array_equal(to_bits(v), ref)
    assert np.all(to_bits(fused[:, 8192:]) == 0x7FC1)


@pytest.mark.parametrize("M,Ns,K", [(7, [200, 77, 300], 336), (20, [128, 1000], 2064), (3, [1, 129, 256, 384], 512)])
def test_ragged_segments(M, Ns, K):
    q = qg()
    X, ps, dev = _segments(M, Ns, K, 90)
    Xd = torch.from_numpy(X.view(np.int16)).view(torch.bfloat16).cuda()
    Ys = q.qgemm_fp8_block_multi(Xd, dev)
    assert q.last_device_status() == 0
    for p, Y in zip(ps, Ys):
        ok, rep = grade_fp8(p, to_bits(Y), X_bits=X)
        assert rep.ok, (p.N, rep)


def test_one_segment_is_the_plain_call():
    """One segment runs the plain call's grid: the same bits."""
    q = qg()
    M, N, K = 16, 5120, 5120
    X, ps, dev = _segments(M, [N], K, 95)
    Xd = torch.from_numpy(X.view(np.int16)).view(torch.bfloat16).cuda()
    a = to_bits(q.qgemm_fp8_block_multi(Xd, dev)[0])
    b = to_bits(q.qgemm_fp8_block(Xd, dev[0][0], dev[0][1]))
    assert q.last_device_status() == 0
    assert np.array_equal(a, b)
