"""The work decomposition on the device and the dispatch table.

* The unit ranges and split-K bookkeeping the kernels compute (read back with
  the schedule probe, which runs the kernels' own device functions) are
  checked against what they must be: a contiguous cover of all units split
  evenly, and, per tile, the first and last CTA holding its units and the
  slot of the first one's piece, found by brute force from the ranges.
* The same shape run split-K and unsplit (grids forced through the dispatch
  table) gives results within the oracle's budget both ways, each
  deterministic call after call.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import Fp8Device, Lut3Device, cached, grade_fp8, grade_lut3, qg, to_bits

pytestmark = pytest.mark.gpu

SHAPES = [(16, 17408, 5120), (16, 5120, 17408), (32, 5120, 17408), (1, 1024, 5120), (16, 5120, 5120),
          (32, 6144, 5120), (7, 200, 336), (1, 256, 512), (20, 3000, 1040)]


def _check_schedule(ranges, info, U, KB):
    G = ranges.shape[0]
    assert ranges[0, 0] == 0 and ranges[-1, 1] == U
    assert np.all(ranges[1:, 0] == ranges[:-1, 1]), "ranges are not contiguous"
    sizes = ranges[:, 1] - ranges[:, 0]
    assert sizes.min() >= 1 and sizes.max() - sizes.min() <= 1, "units are not split evenly"
    for g in range(G):
        for w, u in ((0, ranges[g, 0]), (1, ranges[g, 1] - 1)):
            t = u // KB
            lo, hi = t * KB, (t + 1) * KB
            holders = np.nonzero((ranges[:, 0] < hi) & (ranges[:, 1] > lo))[0]
            cf, cl = int(holders.min()), int(holders.max())
            slot = 0 if ranges[cf, 0] == lo else 1
            assert tuple(info[g, 3 * w:3 * w + 3]) == (cf, cl, slot), (g, w, t)


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_device_work_split(M, N, K):
    q = qg()
    KB = -(-K // 128)
    U = (-(-N // 128)) * KB
    ranges, info = q.debug_schedule(q.KIND_FP8_BLOCK, M, N, K)
    assert q.last_device_status() == 0
    assert ranges.shape[0] == q.dispatch_get(q.KIND_FP8_BLOCK, M, N, K)
    _check_schedule(ranges, info, U, KB)


@pytest.mark.parametrize("M,N,K", [(64, 17408, 5120), (256, 17408, 5120), (160, 1152, 2048), (100, 300, 272),
                                   (1024, 5120, 17408)])
def test_device_work_split_w8a8(M, N, K):
    """The W8A8 kind's work split: tiles of 128 weight rows x R activation
    rows (R = 64 up to 64 rows, else 128), units of two 128-wide K blocks."""
    q = qg()
    R = 64 if M <= 64 else 128
    KU = -(-K // 256)
    U = (-(-N // 128)) * (-(-M // R)) * KU
    ranges, info = q.debug_schedule(q.KIND_W8A8, M, N, K)
    assert q.last_device_status() == 0
    assert ranges.shape[0] == q.dispatch_get(q.KIND_W8A8, M, N, K)
    _check_schedule(ranges, info, U, KU)


@pytest.mark.parametrize("G", [1, 3, 40, 41, 77, 152])
def test_device_work_split_forced_grids(G):
    q = qg()
    M, N, K = 16, 5120, 5120
    try:
        q.dispatch_set(q.KIND_FP8_BLOCK, M, N, K, G)
        assert q.dispatch_get(q.KIND_FP8_BLOCK, M, N, K) == G
        ranges, info = q.debug_schedule(q.KIND_FP8_BLOCK, M, N, K)
        _check_schedule(ranges, info, 40 * 40, 40)
    finally:
        q.dispatch_clear()
    assert q.dispatch_get(q.KIND_FP8_BLOCK, M, N, K) != 1


def _fp8_runs(q, p, dev, Xd, reps=3):
    ws = q.Workspace()
    outs = [to_bits(q.qgemm_fp8_block(Xd, dev.W[0], dev.S, workspace=ws)) for _ in range(reps)]
    assert q.last_device_status() == 0
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
    return outs[0]


@pytest.mark.parametrize("M,N,K,grids", [(16, 5120, 5120, [152, 40, 80, 120]), (32, 5120, 5120, [152, 40, 100]),
                                         (16, 17408, 5120, [136, 152, 68]), (5, 1024, 5120, [32, 8, 152])])
def test_fp8_split_and_unsplit_agree(M, N, K, grids):
    """Split-K over many CTAs, one CTA per tile, and grids in between: every
    one within the oracle's budget and deterministic."""
    q = qg()
    p = cached(("fp8", M, N, K, 70), lambda: wl.make_fp8_problem(M, N, K, config_id=70))
    dev = Fp8Device(p)
    Xd = torch.from_numpy(p.X.view(np.int16)).view(torch.bfloat16).cuda()
    T = -(-N // 128)
    try:
        for G in grids:
            q.dispatch_set(q.KIND_FP8_BLOCK, M, N, K, G)
            assert q.dispatch_get(q.KIND_FP8_BLOCK, M, N, K) == G
            if G == T:
                assert q.workspace_bytes(q.KIND_FP8_BLOCK, M, N, K) == 0
            y = _fp8_runs(q, p, dev, Xd)
            ok, rep = grade_fp8(p, y)
            assert rep.ok, (G, rep)
    finally:
        q.dispatch_clear()


@pytest.mark.parametrize("grids", [[152, 8, 64]])
def test_lut3_split_and_unsplit_agree(grids):
    q = qg()
    M, N, K = 8, 1024, 4096
    p = cached(("lut3", M, N, K, 71), lambda: wl.make_lut3_problem(M, N, K, config_id=71))
    dev = Lut3Device(p)
    Xd = torch.from_numpy(p.X.view(np.int16)).view(torch.float16).cuda()
    try:
        for G in grids:
            q.dispatch_set(q.KIND_LUT3, M, N, K, G)
            ws = q.Workspace()
            outs = [to_bits(q.qgemm_lut3(Xd, dev.Wq, dev.qmap, dev.scales, N, workspace=ws)) for _ in range(3)]
            assert q.last_device_status() == 0
            assert all(np.array_equal(o, outs[0]) for o in outs[1:])
            ok, rep = grade_lut3(p, outs[0])
            assert rep.ok, (G, rep)
    finally:
        q.dispatch_clear()


def test_fp8_tuner_installs_a_gated_grid():
    """The tuner times the candidate grids that pass its gate, installs the
    fastest in the dispatch table, and later calls use it and stay within the
    oracle's budget."""
    q = qg()
    M, N, K = 16, 5120, 5120
    p = cached(("fp8", M, N, K, 70), lambda: wl.make_fp8_problem(M, N, K, config_id=70))
    dev = Fp8Device(p, copies=2)
    Xd = torch.from_numpy(p.X.view(np.int16)).view(torch.bfloat16).cuda()
    try:
        g, us = q.tune_fp8(Xd, dev.W, dev.S, calls=40)
        assert 1 <= g <= torch.cuda.get_device_properties(0).multi_processor_count and us > 0
        assert q.dispatch_get(q.KIND_FP8_BLOCK, M, N, K) == g
        y = _fp8_runs(q, p, dev, Xd)
        ok, rep = grade_fp8(p, y)
        assert rep.ok, rep
    finally:
        q.dispatch_clear()


def test_lut3_tuner_installs_a_gated_grid():
    q = qg()
    M, N, K = 8, 1024, 4096
    p = cached(("lut3", M, N, K, 71), lambda: wl.make_lut3_problem(M, N, K, config_id=71))
    dev = Lut3Device(p)
    Xd = torch.from_numpy(p.X.view(np.int16)).view(torch.float16).cuda()
    try:
        g, us = q.tune_lut3(Xd, [dev.Wq, dev.Wq.clone()], dev.qmap, dev.scales, N, calls=40)
        assert q.dispatch_get(q.KIND_LUT3, M, N, K) == g and us > 0
        Y = q.qgemm_lut3(Xd, dev.Wq, dev.qmap, dev.scales, N)
        assert q.last_device_status() == 0
        ok, rep = grade_lut3(p, to_bits(Y))
        assert rep.ok, rep
    finally:
        q.dispatch_clear()


def test_bf16_tuner_installs_a_gated_grid():
    q = qg()
    M, N, K = 16, 4096, 5120
    p = cached(("bf16", M, N, K, 72), lambda: wl.make_bf16_problem(M, N, K, config_id=72))
    W = torch.from_numpy(p.W.view(np.int16)).view(torch.bfloat16).cuda()
    Xd = torch.from_numpy(p.X.view(np.int16)).view(torch.bfloat16).cuda()
    try:
        g, us = q.tune_bf16(Xd, [W, W.clone()], calls=40)
        assert q.dispatch_get(q.KIND_BF16, M, N, K) == g and us > 0
        Y = q.qgemm_bf16(Xd, W)
        assert q.last_device_status() == 0
        ref = oracle.gemm_bf16(p.X, p.W)
        ok, rep = oracle.within_budget(to_bits(Y), ref, oracle.bf16_abs_mass(p.X, p.W), fmt="bf16")
        assert rep.ok, rep
    finally:
        q.dispatch_clear()


def test_w8a8_tuner_installs_a_gated_grid():
    q = qg()
    M, N, K = 160, 1152, 2048
    p = cached(("w8a8", M, N, K, 73), lambda: wl.make_w8a8_problem(M, N, K, config_id=73))
    Xq_ref, Sx_ref = oracle.quantize_act_e4m3(p.X)
    W = torch.from_numpy(p.W).cuda()
    S = torch.from_numpy(p.S).cuda()
    Xq, Sx = q.quantize_act_e4m3(torch.from_numpy(p.X.view(np.int16)).view(torch.bfloat16).cuda())
    try:
        g, us = q.tune_w8a8(Xq, Sx, [W, W.clone()], S, calls=20)
        assert q.dispatch_get(q.KIND_W8A8, M, N, K) == g and us > 0
        Y = q.qgemm_w8a8_block(Xq, Sx, W, S)
        assert q.last_device_status() == 0
        ref = oracle.qgemm_w8a8_block(Xq_ref, Sx_ref, p.W, p.S)
        ok, rep = oracle.within_budget(to_bits(Y), ref, oracle.w8a8_abs_mass(Xq_ref, Sx_ref, p.W, p.S), fmt="bf16")
        assert rep.ok, rep
    finally:
        q.dispatch_clear()


def test_default_workspaces_are_per_stream():
    """Split-K calls enqueued on two streams with the binding's default
    workspaces (one per stream) overlap freely and all meet the rule."""
    q = qg()
    pa = cached(("fp8", 4, 1024, 5120, 74), lambda: wl.make_fp8_problem(4, 1024, 5120, config_id=74))
    pb = cached(("fp8", 16, 5120, 5120, 75), lambda: wl.make_fp8_problem(16, 5120, 5120, config_id=75))
    da, db = Fp8Device(pa), Fp8Device(pb)
    Xa = torch.from_numpy(pa.X.view(np.int16)).view(torch.bfloat16).cuda()
    Xb = torch.from_numpy(pb.X.view(np.int16)).view(torch.bfloat16).cuda()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    Ya = [torch.empty((4, 1024), dtype=torch.bfloat16, device="cuda") for _ in range(8)]
    Yb = [torch.empty((16, 5120), dtype=torch.bfloat16, device="cuda") for _ in range(8)]
    for i in range(8):
        q.qgemm_fp8_block(Xa, da.W[0], da.S, Y=Ya[i], stream=sa)
        q.qgemm_fp8_block(Xb, db.W[0], db.S, Y=Yb[i], stream=sb)
    torch.cuda.synchronize()
    assert q.last_device_status() == 0
    for i in range(8):
        ok, rep = grade_fp8(pa, to_bits(Ya[i]))
        assert rep.ok, (i, rep)
        ok, rep = grade_fp8(pb, to_bits(Yb[i]))
        assert rep.ok, (i, rep)
