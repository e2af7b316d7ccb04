"""Failure paths on the GPU without faulting it: a wait that runs out reports
QG_ERR_TIMEOUT through the status word, the kernel returns, and the context
stays usable; argument errors never launch anything."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import Fp8Device, Lut3Device, bits_to_bf16, grade_fp8, grade_lut3, qg, to_bits

pytestmark = pytest.mark.gpu


def _timeout_then_recover(run, grade, ws):
    q = qg()
    assert q.last_device_status() == 0
    q.set_wait_timeout_ns(20_000_000)      # 20 ms
    q.set_fault_injection(0)               # CTA 0 never loads its first unit
    try:
        run(ws)
        assert q.last_device_status() == 5  # QG_ERR_TIMEOUT
    finally:
        q.set_fault_injection(-1)
        q.set_wait_timeout_ns(1_000_000_000)
    # the workspace is undefined after an error: zero it, then run normally
    ws.reset()
    Y = run(ws)
    assert q.last_device_status() == 0
    ok, rep = grade(to_bits(Y))
    assert rep.ok, rep


def test_fp8_timeout_reported_and_context_survives():
    q = qg()
    p = wl.make_fp8_problem(4, 1024, 5120, config_id=50)
    dev = Fp8Device(p)
    Xd = torch.from_numpy(p.X.view(np.int16)).view(torch.bfloat16).cuda()
    ws = q.Workspace()
    _timeout_then_recover(lambda w: q.qgemm_fp8_block(Xd, dev.W[0], dev.S, workspace=w),
                          lambda y: grade_fp8(p, y), ws)


def test_lut3_timeout_reported_and_context_survives():
    q = qg()
    p = wl.make_lut3_problem(4, 1024, 4096, config_id=51)
    dev = Lut3Device(p)
    Xd = torch.from_numpy(p.X.view(np.int16)).view(torch.float16).cuda()
    ws = q.Workspace()
    _timeout_then_recover(lambda w: q.qgemm_lut3(Xd, dev.Wq, dev.qmap, dev.scales, 1024, workspace=w),
                          lambda y: grade_lut3(p, y), ws)


def test_bf16_timeout_reported_and_context_survives():
    q = qg()
    p = wl.make_bf16_problem(4, 1024, 5120, config_id=53)
    W = torch.from_numpy(p.W.view(np.int16)).view(torch.bfloat16).cuda()
    Xd = bits_to_bf16(p.X)
    ws = q.Workspace()

    def grade(y):
        return oracle.within_budget(y, oracle.gemm_bf16(p.X, p.W), oracle.bf16_abs_mass(p.X, p.W), fmt="bf16")
    _timeout_then_recover(lambda w: q.qgemm_bf16(Xd, W, workspace=w), grade, ws)


def test_w8a8_timeout_reported_and_context_survives():
    q = qg()
    p = wl.make_w8a8_problem(160, 1152, 2048, config_id=54)
    Xq_ref, Sx_ref = oracle.quantize_act_e4m3(p.X)
    W = torch.from_numpy(p.W).cuda()
    S = torch.from_numpy(p.S).cuda()
    Xq, Sx = q.quantize_act_e4m3(bits_to_bf16(p.X))
    assert q.last_device_status() == 0
    ws = q.Workspace()

    def grade(y):
        return oracle.within_budget(y, oracle.qgemm_w8a8_block(Xq_ref, Sx_ref, p.W, p.S),
                                    oracle.w8a8_abs_mass(Xq_ref, Sx_ref, p.W, p.S), fmt="bf16")
    _timeout_then_recover(lambda w: q.qgemm_w8a8_block(Xq, Sx, W, S, workspace=w), grade, ws)


def test_missing_workspace_is_rejected():
    q = qg()
    p = wl.make_fp8_problem(4, 1024, 5120, config_id=52)
    dev = Fp8Device(p)
    Xd = torch.from_numpy(p.X.view(np.int16)).view(torch.bfloat16).cuda()
    Y = torch.empty((4, 1024), dtype=torch.bfloat16, device="cuda")
    need = q.workspace_bytes(q.KIND_FP8_BLOCK, 4, 1024, 5120)
    assert need > 0
    r = q.lib.qgemm_fp8_block(Xd.data_ptr(), 5120, dev.W[0].data_ptr(), dev.S.data_ptr(), Y.data_ptr(),
                              1024, 4, 1024, 5120, None, 0, None)
    assert r == 6
    small = torch.zeros(need - 256, dtype=torch.uint8, device="cuda")
    r = q.lib.qgemm_fp8_block(Xd.data_ptr(), 5120, dev.W[0].data_ptr(), dev.S.data_ptr(), Y.data_ptr(),
                              1024, 4, 1024, 5120, small.data_ptr(), small.numel(), None)
    assert r == 6
    assert q.last_device_status() == 0
