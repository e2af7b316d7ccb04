"""The FP8 GEMM with X and Y in pinned host memory (qgemm_fp8_block_host):
a staging kernel reads X over the host link, and the epilogue stores Y into
host memory.  Its results must be those of qgemm_fp8_block on device
buffers, bit for bit, and within the oracle's budget."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import cached, grade_fp8, qg, to_bits

pytestmark = pytest.mark.gpu


def _pinned_bf16(bits: np.ndarray, pad_cols: int = 0) -> torch.Tensor:
    M, K = bits.shape
    t = torch.zeros((M, K + pad_cols), dtype=torch.int16).pin_memory()
    t[:, :K] = torch.from_numpy(bits.view(np.int16))
    return t.view(torch.bfloat16)


def _device_inputs(p):
    W = torch.from_numpy(p.W).cuda()
    S = torch.from_numpy(p.S).cuda()
    return W, S


@pytest.mark.parametrize("M,N,K", [(16, 17408, 5120), (16, 5120, 17408), (32, 1024, 5120), (1, 256, 512),
                                   (7, 200, 336), (20, 3000, 1040)])
def test_host_entry_matches_device_entry(M, N, K):
    """Gate/up and down at M=16 (unsplit and stream-K), the attention shape
    at M=32 (split-K over every SM), the smallest case and ragged tails."""
    q = qg()
    q.set_weight_prefetch_overlap(1)
    p = cached(("fp8host", M, N, K), lambda: wl.make_fp8_problem(M, N, K, config_id=61))
    W, S = _device_inputs(p)
    ws = q.Workspace()
    Xd = torch.from_numpy(p.X.view(np.int16)).view(torch.bfloat16).cuda()
    ref = to_bits(q.qgemm_fp8_block(Xd, W, S, workspace=ws))
    Xh = _pinned_bf16(p.X)
    Yh = torch.empty((M, N), dtype=torch.int16).pin_memory()
    Yh.fill_(0x7FC1)   # a NaN pattern: every element must be written
    q.qgemm_fp8_block_host(Xh, W, S, Y=Yh.view(torch.bfloat16), workspace=ws)
    torch.cuda.synchronize()
    assert q.last_device_status() == 0
    got = Yh.numpy().view(np.uint16)
    np.testing.assert_array_equal(got, ref)
    if M * N * K <= 64 * 1024 * 1024:
        ok, rep = grade_fp8(p, got)
        assert rep.ok, rep


def test_host_entry_strided_rows_and_repeated_calls():
    """Row strides wider than the rows on both sides, and a sequence of calls
    with different X that reuse one staging buffer and one workspace on a
    stream (each call must see its own X, not the previous one's)."""
    q = qg()
    q.set_weight_prefetch_overlap(1)
    M, N, K = 5, 1000, 2064
    p = wl.make_fp8_problem(M, N, K, config_id=62)
    W, S = _device_inputs(p)
    ws = q.Workspace()
    stage = torch.empty(M * K, dtype=torch.bfloat16, device="cuda")
    rng = np.random.default_rng(62)
    xs = [p.X] + [wl.make_fp8_problem(M, N, K, config_id=63 + i).X for i in range(3)]
    outs = []
    for Xb in xs:
        Xh = _pinned_bf16(Xb, pad_cols=8 * int(rng.integers(1, 4)))[:, :K]
        Yfull = torch.empty((M, N + 24), dtype=torch.bfloat16).pin_memory()
        q.qgemm_fp8_block_host(Xh, W, S, Y=Yfull[:, :N], X_stage=stage, workspace=ws)
        outs.append((Xb, Yfull))
    torch.cuda.synchronize()
    assert q.last_device_status() == 0
    for Xb, Yfull in outs:
        Xd = torch.from_numpy(Xb.view(np.int16)).view(torch.bfloat16).cuda()
        ref = to_bits(q.qgemm_fp8_block(Xd, W, S, workspace=ws))
        np.testing.assert_array_equal(to_bits(Yfull[:, :N]), ref)


def test_host_entry_refuses_pageable_memory():
    """Pageable host buffers are refused before anything is enqueued."""
    q = qg()
    M, N, K = 2, 256, 512
    p = wl.make_fp8_problem(M, N, K, config_id=0)
    W, S = _device_inputs(p)
    stage = torch.empty(M * K, dtype=torch.bfloat16, device="cuda")
    Xpage = torch.from_numpy(p.X.view(np.int16).copy()).view(torch.bfloat16)
    Ypage = torch.empty((M, N), dtype=torch.bfloat16)
    fn = q.lib.qgemm_fp8_block_host
    sp = torch.cuda.current_stream().cuda_stream
    rc = fn(Xpage.data_ptr(), K, W.data_ptr(), S.data_ptr(), Ypage.data_ptr(), N, M, N, K, stage.data_ptr(),
            None, 0, sp)
    assert q.STATUS[rc] == "QG_ERR_INVALID_ARG"
    Xh = _pinned_bf16(p.X)
    rc = fn(Xh.data_ptr(), K, W.data_ptr(), S.data_ptr(), Ypage.data_ptr(), N, M, N, K, stage.data_ptr(),
            None, 0, sp)
    assert q.STATUS[rc] == "QG_ERR_INVALID_ARG"
    with pytest.raises(ValueError):
        q.qgemm_fp8_block_host(Xpage, W, S)
    torch.cuda.synchronize()
    assert q.last_device_status() == 0


def test_host_entry_chained_through_host_memory():
    """With launch overlap on, one call's Y_host is the next call's X_host:
    the second call's staging kernel must read the first call's finished
    result (it waits for the preceding grid before it reads X_host), so the
    chain gives exactly the bits of the same chain on device buffers."""
    q = qg()
    q.set_weight_prefetch_overlap(1)
    try:
        M = 16
        pa = cached(("fp8host", M, 5120, 5120), lambda: wl.make_fp8_problem(M, 5120, 5120, config_id=64))
        pb = cached(("fp8host", M, 1024, 5120), lambda: wl.make_fp8_problem(M, 1024, 5120, config_id=65))
        Wa, Sa = _device_inputs(pa)
        Wb, Sb = _device_inputs(pb)
        ws = q.Workspace()
        Xd = torch.from_numpy(pa.X.view(np.int16)).view(torch.bfloat16).cuda()
        ya = q.qgemm_fp8_block(Xd, Wa, Sa, workspace=ws)
        yb = to_bits(q.qgemm_fp8_block(ya, Wb, Sb, workspace=ws))
        ya = to_bits(ya)
        stage = torch.empty(M * 5120, dtype=torch.bfloat16, device="cuda")
        Xh = _pinned_bf16(pa.X)
        outs = []
        for _ in range(3):
            Yh1 = torch.empty((M, 5120), dtype=torch.int16).pin_memory()
            Yh1.fill_(0x7FC1)
            Yh2 = torch.empty((M, 1024), dtype=torch.int16).pin_memory()
            Yh2.fill_(0x7FC1)
            q.qgemm_fp8_block_host(Xh, Wa, Sa, Y=Yh1.view(torch.bfloat16), X_stage=stage, workspace=ws)
            q.qgemm_fp8_block_host(Yh1.view(torch.bfloat16), Wb, Sb, Y=Yh2.view(torch.bfloat16), X_stage=stage,
                                   workspace=ws)
            outs.append((Yh1, Yh2))
        torch.cuda.synchronize()
        assert q.last_device_status() == 0
        for Yh1, Yh2 in outs:
            np.testing.assert_array_equal(Yh1.numpy().view(np.uint16), ya)
            np.testing.assert_array_equal(Yh2.numpy().view(np.uint16), yb)
    finally:
        q.set_weight_prefetch_overlap(0)
