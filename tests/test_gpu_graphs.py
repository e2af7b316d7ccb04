"""Calls captured in a CUDA graph and replayed, the way a serving loop runs a
decode step: every kind's output on replay equals the eager output bit for
bit, replay after replay, and the split-K arrival counters are back at
zero after each replay (the last piece to arrive resets them, so a replayed
launch finds them as a fresh one does).  The calls launch with programmatic
stream serialization, which capture turns into programmatic graph edges."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import Fp8Device, Lut3Device, assert_counters_clear, bits_to_bf16, bits_to_f16, cached, qg, to_bits

pytestmark = pytest.mark.gpu


def test_decode_step_replays_in_a_cuda_graph():
    q = qg()
    q.set_weight_prefetch_overlap(1)
    ws = q.Workspace()          # FP8, LUT3 and BF16 share a workspace layout
    ws_w8 = q.Workspace()       # the W8A8 kind has its own
    p1 = cached(("fp8", 16, 5120, 5120, 80), lambda: wl.make_fp8_problem(16, 5120, 5120, config_id=80))
    p2 = cached(("fp8", 32, 1024, 5120, 81), lambda: wl.make_fp8_problem(32, 1024, 5120, config_id=81))
    p3 = cached(("lut3", 8, 1024, 4096, 82), lambda: wl.make_lut3_problem(8, 1024, 4096, config_id=82))
    p4 = cached(("bf16", 16, 4096, 1024, 83), lambda: wl.make_bf16_problem(16, 4096, 1024, config_id=83))
    p5 = cached(("w8a8", 256, 2048, 4096, 84), lambda: wl.make_w8a8_problem(256, 2048, 4096, config_id=84))
    d1, d2, d3 = Fp8Device(p1), Fp8Device(p2), Lut3Device(p3)
    X1, X2 = bits_to_bf16(p1.X), bits_to_bf16(p2.X)
    X3 = bits_to_f16(p3.X)
    X4, W4 = bits_to_bf16(p4.X), bits_to_bf16(p4.W)
    X5, W5, S5 = bits_to_bf16(p5.X), torch.from_numpy(p5.W).cuda(), torch.from_numpy(p5.S).cuda()
    Y = [torch.empty((16, 5120), dtype=torch.bfloat16, device="cuda"),
         torch.empty((32, 1024), dtype=torch.bfloat16, device="cuda"),
         torch.empty((8, 1024), dtype=torch.float16, device="cuda"),
         torch.empty((16, 4096), dtype=torch.bfloat16, device="cuda"),
         torch.empty((256, 2048), dtype=torch.bfloat16, device="cuda")]

    def step():
        q.qgemm_fp8_block(X1, d1.W[0], d1.S, Y=Y[0], workspace=ws)       # split-K, 16 rows
        q.qgemm_fp8_block(X2, d2.W[0], d2.S, Y=Y[1], workspace=ws)       # split-K, 32 rows
        q.qgemm_lut3(X3, d3.Wq, d3.qmap, d3.scales, 1024, Y=Y[2], workspace=ws)
        q.qgemm_bf16(X4, W4, Y=Y[3], workspace=ws)
        q.qgemm_w8a8(X5, W5, S5, Y=Y[4], workspace=ws_w8)                 # quantiser + GEMM

    # eager: the reference bits, and workspaces grown to size outside capture
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert q.last_device_status() == 0
    ref = [to_bits(y) for y in Y]

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for y in Y:
        y.view(torch.int16).fill_(0x7FC1)
    for _ in range(4):
        g.replay()
        torch.cuda.synchronize()
        assert q.last_device_status() == 0
        for y, r in zip(Y, ref):
            assert np.array_equal(to_bits(y), r)
        assert_counters_clear(q, ws, q.KIND_FP8_BLOCK, 16, 5120, 5120)
        assert_counters_clear(q, ws, q.KIND_FP8_BLOCK, 32, 1024, 5120)
        for y in Y:
            y.view(torch.int16).fill_(0x7FC1)
