"""W8A16 FP8 block-scaled GEMM on the GPU against the CPU oracle, through the
C ABI.  Every element must satisfy the comparison rule (<= 2 BF16 ULP, or
within the near-zero floor); small shapes are compared in full, the full-size
configurations in full as well (the oracle runs on all host cores)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import Fp8Device, assert_counters_clear, cached, grade_fp8, qg, sample_indices, to_bits

pytestmark = pytest.mark.gpu


def _problem(M, N, K, cid):
    return cached(("fp8", M, N, K, cid), lambda: wl.make_fp8_problem(M, N, K, config_id=cid))


def _check(p, Y, X_bits=None, ms=None, ns=None):
    q = qg()
    assert q.last_device_status() == 0
    y = to_bits(Y)
    ok, rep = grade_fp8(p, y, X_bits=X_bits, ms=ms, ns=ns)
    assert rep.ok, rep
    assert rep.max_rel_err <= 1e-2, rep
    return y, rep


def test_small_config():
    """M=1, N=256, K=512 -- the smallest configuration."""
    p = _problem(1, 256, 512, 0)
    dev = Fp8Device(p)
    _check(p, dev.run())


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 15, 16, 17, 24, 31, 32])
def test_m_sweep_attention_shape(M):
    """N=1024, K=5120 (QKV K/V shape): 8 tiles x 40 blocks, split-K over the SMs."""
    p = _problem(32, 1024, 5120, 3)
    dev = cached(("fp8dev", 32, 1024, 5120), lambda: Fp8Device(p))
    Xb = p.X[:M]
    Y = dev.run(X_bits=Xb)
    _check(p, Y[:M], X_bits=Xb)


@pytest.mark.parametrize("N,K", [(200, 336), (130, 128), (1000, 2064), (128, 16), (77, 4096),
                                 (256, 144), (3000, 1040)])
@pytest.mark.parametrize("M", [1, 7, 20])
def test_ragged_shapes(M, N, K):
    """N not a multiple of 128 and K not a multiple of 128 (partial blocks)."""
    p = _problem(M, N, K, 40)
    _check(p, Fp8Device(p).run())


@pytest.mark.parametrize("N", [5120, 6144])
@pytest.mark.parametrize("M", [1, 5, 16, 32])
def test_attention_shapes(M, N):
    p = _problem(32, N, 5120, 3)
    dev = cached(("fp8dev", 32, N, 5120), lambda: Fp8Device(p))
    Xb = p.X[:M]
    _check(p, dev.run(X_bits=Xb)[:M], X_bits=Xb)


@pytest.mark.parametrize("M", [16, 8])
def test_gateup_full(M):
    """FFN gate/up, N=17408, K=5120 (89 MB of weights), every element."""
    p = _problem(16, 17408, 5120, 1)
    dev = cached(("fp8dev", 16, 17408, 5120), lambda: Fp8Device(p))
    Xb = p.X[:M]
    _check(p, dev.run(X_bits=Xb), X_bits=Xb)


def test_down_full_and_halves():
    """FFN down, N=5120, K=17408: M=16, M=32 in one call, and M=32 as two
    contiguous 16-row halves (plain row offsets of X and Y)."""
    q = qg()
    p = _problem(32, 5120, 17408, 2)
    dev = Fp8Device(p)
    y16, _ = _check(p, dev.run(X_bits=p.X[:16]), X_bits=p.X[:16])
    y32, _ = _check(p, dev.run())
    # two halves through pointer offsets into one X / Y pair
    Xd = torch.from_numpy(p.X.view(np.int16)).view(torch.bfloat16).cuda()
    Y = torch.empty((32, 5120), dtype=torch.bfloat16, device="cuda")
    q.qgemm_fp8_block(Xd[:16], dev.W[0], dev.S, Y=Y[:16])
    q.qgemm_fp8_block(Xd[16:], dev.W[0], dev.S, Y=Y[16:])
    yh, _ = _check(p, Y)
    # the first half of the split is the M=16 call, bit for bit
    assert np.array_equal(yh[:16], y16)


def test_deterministic_and_workspace_left_clean():
    """Same inputs, same bits (the split-K pieces are summed in a fixed order
    whichever CTA finishes last); the arrival counters are back to zero."""
    q = qg()
    p = _problem(16, 5120, 5120, 3)
    dev = Fp8Device(p)
    ws = q.Workspace()
    Xd = torch.from_numpy(p.X[:16].view(np.int16)).view(torch.bfloat16).cuda()
    outs = []
    for _ in range(3):
        outs.append(to_bits(q.qgemm_fp8_block(Xd, dev.W[0], dev.S, workspace=ws)))
    assert q.last_device_status() == 0
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
    assert_counters_clear(q, ws, q.KIND_FP8_BLOCK, 16, 5120, 5120)


def test_shared_workspace_across_shapes():
    """One workspace through a sequence of differently shaped calls (the
    counter region of one shape overlaps the partial sums of another)."""
    q = qg()
    ws = q.Workspace()
    for (M, N, K) in [(32, 1024, 5120), (1, 3000, 1040), (16, 5120, 5120), (5, 6144, 5120), (20, 3000, 1040),
                      (1, 1024, 5120)]:
        p = _problem(M, N, K, 41)
        dev = Fp8Device(p)
        Xd = torch.from_numpy(p.X.view(np.int16)).view(torch.bfloat16).cuda()
        Y = q.qgemm_fp8_block(Xd, dev.W[0], dev.S, workspace=ws)
        _check(p, Y)
        if q.workspace_bytes(q.KIND_FP8_BLOCK, M, N, K):
            assert_counters_clear(q, ws, q.KIND_FP8_BLOCK, M, N, K)


def test_strided_rows_and_padding_untouched():
    """ldx > K and ldy > N: padding columns of Y keep their canary."""
    p = _problem(5, 1024, 5120, 3)
    dev = Fp8Device(p)
    Y = dev.run(x_pad=24, y_pad=40)
    y, _ = _check(p, Y[:, :1024])
    pad = to_bits(Y[:, 1024:])
    assert np.all(pad == 0x7FC1)


def test_k_zero_and_empty():
    q = qg()
    W = torch.zeros((256, 0), dtype=torch.uint8, device="cuda")
    S = torch.zeros((2, 0), dtype=torch.float32, device="cuda")
    X = torch.zeros((3, 8), dtype=torch.bfloat16, device="cuda")[:, :0]
    Y = torch.full((3, 256), 5.0, dtype=torch.bfloat16, device="cuda")
    assert q.lib.qgemm_fp8_block(X.data_ptr() or 16, 8, W.data_ptr() or 16, S.data_ptr() or 16,
                                 Y.data_ptr(), 256, 3, 256, 0, None, 0, None) == 0
    torch.cuda.synchronize()
    assert float(Y.float().abs().max()) == 0.0
    # M == 0 leaves Y alone
    Y.fill_(5.0)
    assert q.lib.qgemm_fp8_block(16, 8, 16, 16, Y.data_ptr(), 256, 0, 256, 128, None, 0, None) == 0
    torch.cuda.synchronize()
    assert float(Y.float().min()) == 5.0


def test_extreme_scales_and_codes():
    """All-448 codes, subnormal codes, zeros, negative zero and tiny/huge block
    scales in one problem."""
    M, N, K = 4, 256, 512
    rng = np.random.default_rng(5)
    W = rng.choice(np.array([0x7E, 0xFE, 0x01, 0x81, 0x07, 0x00, 0x80, 0x3C, 0xBC], dtype=np.uint8),
                   size=(N, K))
    S = np.array([[1e-30, 3e30, 1.0, 2.0 ** -20], [7.0, 1e-3, 4096.0, 0.5]], dtype=np.float32)
    X = wl.bf16_bits_from_f32(rng.standard_normal((M, K)).astype(np.float32) * 8)
    p = wl.Fp8Problem(M, N, K, X, W, S)
    _check(p, Fp8Device(p).run())


def test_overlapped_launches_chain_and_share_workspace():
    """With programmatic overlap on, a GEMM whose X is the previous GEMM's Y
    still reads the finished Y, and calls sharing one workspace stay exact."""
    q = qg()
    pa = _problem(16, 5120, 5120, 42)
    pb = _problem(16, 1024, 5120, 43)
    da, db = Fp8Device(pa), Fp8Device(pb)
    Xa = torch.from_numpy(pa.X.view(np.int16)).view(torch.bfloat16).cuda()
    ws = q.Workspace()
    q.set_weight_prefetch_overlap(True)
    try:
        outs = []
        for _ in range(3):
            Ya = q.qgemm_fp8_block(Xa, da.W[0], da.S, workspace=ws)
            Yb = q.qgemm_fp8_block(Ya, db.W[0], db.S, workspace=ws)
            outs.append((to_bits(Ya), to_bits(Yb)))
        assert q.last_device_status() == 0
    finally:
        q.set_weight_prefetch_overlap(False)
    ya, yb = outs[0]
    ok, rep = grade_fp8(pa, ya)
    assert rep.ok, rep
    ok, rep = grade_fp8(pb, yb, X_bits=ya)
    assert rep.ok, rep
    for a2, b2 in outs[1:]:
        assert np.array_equal(a2, ya) and np.array_equal(b2, yb)
    assert_counters_clear(q, ws, q.KIND_FP8_BLOCK, 16, 5120, 5120)


@pytest.mark.parametrize("M,N,K,cid", [(32, 5120, 17408, 2), (16, 17408, 5120, 1)])
def test_back_to_back_calls_bit_identical(M, N, K, cid):
    """Many calls in a row on one stream give the same bits every time.  The
    result is deterministic, so any pipeline hazard (a weight stage read after
    it was refilled, a partial read before it was written) shows as a
    difference even when it is small; the first result is also graded."""
    q = qg()
    p = _problem(M, N, K, cid)
    dev = cached(("fp8dev", M, N, K), lambda: Fp8Device(p))
    Xd = torch.from_numpy(p.X.view(np.int16)).view(torch.bfloat16).cuda()
    ws = q.Workspace()
    outs = [q.qgemm_fp8_block(Xd, dev.W[0], dev.S, workspace=ws) for _ in range(48)]
    assert q.last_device_status() == 0
    first = to_bits(outs[0])
    for i, Y in enumerate(outs[1:], 1):
        y = to_bits(Y)
        assert np.array_equal(y, first), f"call {i}: {int((y != first).sum())} elements differ"
    _check(p, outs[0])


def _wide_range_x(rng, M, K, binades):
    """BF16 activations whose magnitudes are log-uniform over `binades`
    binades below 4 (random signs), so that every 128-wide block holds values
    far apart in size."""
    mag = np.exp2(rng.uniform(-binades, 0.0, size=(M, K))) * 4.0
    sign = np.where(rng.random((M, K)) < 0.5, -1.0, 1.0)
    return wl.bf16_bits_from_f32((mag * sign).astype(np.float32))


@pytest.mark.parametrize("binades", [12, 24])
def test_wide_dynamic_range_activations(binades):
    """The E4M3 tensor-core path splits each (row, 128-K block) of X into two
    power-of-two-scaled E4M3 planes; values within 2^13 of their block's
    maximum are represented exactly, smaller ones to within 2^-21 of it.  Rows
    spanning 12 binades (all exact) and 24 binades (many elements below the
    exact window) must both meet the comparison rule."""
    M, N, K = 16, 1024, 2048
    rng = np.random.default_rng(77 + binades)
    base = _problem(M, N, K, 44)
    Xb = _wide_range_x(rng, M, K, binades)
    p = wl.Fp8Problem(M, N, K, Xb, base.W, base.S)
    _check(p, Fp8Device(p).run())


def test_zero_rows_and_zero_blocks_in_x():
    """All-zero X rows and all-zero 128-wide blocks inside a row (the split
    takes no exponent from an empty block) alongside normal data."""
    M, N, K = 8, 512, 1024
    base = _problem(M, N, K, 45)
    X = base.X.copy()
    X[3] = 0                    # a whole row of +0
    X[5, 128:256] = 0x8000      # a block of -0
    X[6, :128] = 0
    p = wl.Fp8Problem(M, N, K, X, base.W, base.S)
    y, _ = _check(p, Fp8Device(p).run())
    assert np.all((y[3] & 0x7FFF) == 0)
