"""W8A8 path on the GPU against the CPU oracle: the activation quantiser
bit for bit (codes and scales), and the E4M3 x E4M3 block-scaled GEMM
element by element on small and ragged shapes, on every grid kind (one CTA
per tile, stream-K), with strided operands, and at the gate/up layer shape
N=17408, K=5120 for prefill batches on sampled 128-row tiles."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import bits_to_bf16, cached, qg, to_bits

pytestmark = pytest.mark.gpu


def _quantized(p):
    """The oracle's E4M3 codes and scales of p.X (uint8 [M, K], f32 [KB, M])."""
    return cached(("w8a8q", id(p)), lambda: oracle.quantize_act_e4m3(p.X))


def _problem(M, N, K, cid=40):
    return cached(("w8a8", M, N, K, cid), lambda: wl.make_w8a8_problem(M, N, K, config_id=cid))


def _scales_dev(Sx, ldsx):
    KB, M = Sx.shape
    t = torch.full((KB, ldsx), float("nan"), dtype=torch.float32)
    t[:, :M] = torch.from_numpy(Sx)
    return t.cuda()


def _codes_dev(Xq, pad=0):
    M, K = Xq.shape
    t = torch.zeros((M, K + pad), dtype=torch.uint8)
    t[:, :K] = torch.from_numpy(Xq)
    return t.cuda()[:, :K]


def _grade(Xq, Sx, W, S, y_bits):
    ref = oracle.qgemm_w8a8_block(Xq, Sx, W, S)
    A = oracle.w8a8_abs_mass(Xq, Sx, W, S)
    ok, rep = oracle.within_budget(y_bits, ref, A, fmt="bf16")
    assert rep.ok, rep
    assert rep.max_rel_err <= 1e-2, rep
    return rep


def _run_gemm(q, Xq, Sx, W, S, N, ldsx=None, x_pad=0, y_pad=0):
    M, K = Xq.shape
    ldsx = ldsx or max(32, -(-M // 32) * 32)
    Y = torch.empty((M, N + y_pad), dtype=torch.bfloat16, device="cuda")
    Y.view(torch.int16).fill_(0x7FC1)
    q.qgemm_w8a8_block(_codes_dev(Xq, x_pad), _scales_dev(Sx, ldsx), W, S, Y=Y[:, :N])
    assert q.last_device_status() == 0
    return Y


# ------------------------------------------------------------------ quantiser
def _special_rows(X):
    """Blocks the quantiser treats specially: an all-zero block (scale 1), a
    block of subnormal BF16 values, signed zeros, a block whose largest value
    is huge, and a block holding one value far above the rest."""
    X = X.copy()
    M, K = X.shape
    if M >= 5 and K >= 128:
        X[0, :128] = 0
        X[1, :128] = np.arange(128, dtype=np.uint16) % 127 + 1          # BF16 subnormals
        X[2, :64] = 0x8000                                              # -0.0
        X[3, :128] = (X[3, :128] & 0x807F) | 0x7E00                      # magnitudes ~2^125
        X[4, 5] = 0x4780                                                 # 65536 among N(0,1)
    return X


@pytest.mark.parametrize("M,K", [(1, 128), (5, 16), (33, 5120), (100, 272), (64, 1040), (7, 4096)])
def test_quantize_act_bit_exact(M, K):
    q = qg()
    p = wl.make_w8a8_problem(M, 128, K, config_id=41)
    X = _special_rows(p.X)
    Xq_ref, Sx_ref = oracle.quantize_act_e4m3(X)
    ldsx = -(-M // 32) * 32 + 4
    Xq = torch.full((M, K + 48), 0xAB, dtype=torch.uint8, device="cuda")
    Sx = torch.full((-(-K // 128), ldsx), float("nan"), dtype=torch.float32, device="cuda")
    q.quantize_act_e4m3(bits_to_bf16(X, 8)[:, :K], Xq=Xq[:, :K], X_scale=Sx)
    assert q.last_device_status() == 0
    got_q = Xq.cpu().numpy()
    got_s = Sx.cpu().numpy()
    assert np.array_equal(got_q[:, :K], Xq_ref)
    assert np.array_equal(got_s[:, :M].view(np.uint32), Sx_ref.view(np.uint32))
    assert np.all(got_s[:, M:] == 0.0)
    assert np.all(got_q[:, K:] == 0xAB)


# ------------------------------------------------------------------ GEMM
@pytest.mark.parametrize("M,N,K", [(33, 256, 512), (64, 384, 1024), (100, 300, 272), (1, 128, 128),
                                   (32, 256, 512), (129, 1000, 2064), (256, 2048, 4096), (48, 136, 5120),
                                   (33, 128, 16), (65, 129, 144)])
def test_w8a8_shapes(M, N, K):
    q = qg()
    p = _problem(M, N, K)
    Xq, Sx = _quantized(p)
    W = torch.from_numpy(p.W).cuda()
    S = torch.from_numpy(p.S).cuda()
    Y = _run_gemm(q, Xq, Sx, W, S, N)
    _grade(Xq, Sx, p.W, p.S, to_bits(Y))


def test_w8a8_end_to_end_from_bf16():
    """qgemm_w8a8: the GPU quantiser then the GEMM, against the oracle's
    quantiser then its GEMM."""
    q = qg()
    p = _problem(96, 640, 1536)
    Xq, Sx = _quantized(p)
    Y = q.qgemm_w8a8(bits_to_bf16(p.X), torch.from_numpy(p.W).cuda(), torch.from_numpy(p.S).cuda())
    assert q.last_device_status() == 0
    _grade(Xq, Sx, p.W, p.S, to_bits(Y))


def test_w8a8_strided_and_padding_untouched():
    q = qg()
    M, N, K = 70, 500, 784
    p = _problem(M, N, K)
    Xq, Sx = _quantized(p)
    W = torch.from_numpy(p.W).cuda()
    S = torch.from_numpy(p.S).cuda()
    Y = _run_gemm(q, Xq, Sx, W, S, N, ldsx=132, x_pad=32, y_pad=24)
    _grade(Xq, Sx, p.W, p.S, to_bits(Y[:, :N]))
    assert np.all(to_bits(Y[:, N:]) == 0x7FC1)


@pytest.mark.parametrize("M,N,y_pad,shift", [(70, 504, 8, 0), (130, 248, 24, 0), (33, 384, 0, 0),
                                             (300, 200, 8, 0), (70, 500, 12, 0), (70, 504, 8, 1)])
def test_w8a8_y_store_paths(M, N, y_pad, shift):
    """Y through the TMA store (Y 16-byte aligned, ldy and N multiples of 8:
    ragged last tiles clipped at N and at M, padding columns and the rows
    below Y untouched) and through plain stores (N % 8 != 0; Y starting one
    element in, not 16-byte aligned)."""
    q = qg()
    K = 784
    p = _problem(M, N, K)
    Xq, Sx = _quantized(p)
    W = torch.from_numpy(p.W).cuda()
    S = torch.from_numpy(p.S).cuda()
    ldsx = max(32, -(-M // 32) * 32)
    Y = torch.empty((M + 40, N + y_pad + 8), dtype=torch.bfloat16, device="cuda")
    Y.view(torch.int16).fill_(0x7FC1)
    q.qgemm_w8a8_block(_codes_dev(Xq), _scales_dev(Sx, ldsx), W, S, Y=Y[:M, shift:shift + N])
    assert q.last_device_status() == 0
    bits = to_bits(Y)
    _grade(Xq, Sx, p.W, p.S, bits[:M, shift:shift + N])
    assert np.all(bits[:M, :shift] == 0x7FC1) and np.all(bits[:M, shift + N:] == 0x7FC1)
    assert np.all(bits[M:] == 0x7FC1)


def test_w8a8_grids_agree_and_repeat():
    """Forced grids (one CTA per tile, stream-K over several counts) all meet
    the rule; each grid gives the same bits twice; the workspace's arrival
    counters are zero after every call."""
    q = qg()
    M, N, K = 160, 1152, 2048
    p = _problem(M, N, K)
    Xq, Sx = _quantized(p)
    W = torch.from_numpy(p.W).cuda()
    S = torch.from_numpy(p.S).cuda()
    R = 64 if M <= 64 else 128           # activation rows per tile
    tiles = -(-N // 128) * -(-M // R)
    ws = q.Workspace("cuda")
    try:
        for g in (tiles, 7, 64, 152, 45):
            q.dispatch_set(q.KIND_W8A8, M, N, K, g)
            Y1 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            Y2 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            Xd = _codes_dev(Xq)
            Sd = _scales_dev(Sx, -(-M // 32) * 32)
            q.qgemm_w8a8_block(Xd, Sd, W, S, Y=Y1, workspace=ws)
            q.qgemm_w8a8_block(Xd, Sd, W, S, Y=Y2, workspace=ws)
            assert q.last_device_status() == 0
            assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16)), g
            _grade(Xq, Sx, p.W, p.S, to_bits(Y1))
            need = q.workspace_bytes(q.KIND_W8A8, M, N, K)
            if need:
                cnt = (tiles * (R // 16) * 4 + 255) // 256 * 256
                assert int(ws.buf[need - cnt:need].count_nonzero()) == 0
    finally:
        q.dispatch_clear()


@pytest.mark.parametrize("M", [64, 256])
def test_w8a8_gateup_full_sampled(M):
    """N=17408, K=5120 (89 MB of E4M3 weights) at prefill batch sizes, in the
    grid the built-in rule picks; graded on three whole 128-row tiles (the
    first, a middle one and the last) for a sample of rows, against the
    oracle on that sub-problem (an output depends only on its activation row,
    its scales column, its weight row and that row's block scales)."""
    q = qg()
    N, K = 17408, 5120
    p = cached(("w8a8full", M), lambda: wl.make_w8a8_problem(M, N, K, config_id=6))
    Xq, Sx = _quantized(p)
    W = cached(("w8a8W",), lambda: torch.from_numpy(p.W).cuda())
    S = torch.from_numpy(p.S).cuda()
    Y = q.qgemm_w8a8(bits_to_bf16(p.X), W, S)
    assert q.last_device_status() == 0
    yb = to_bits(Y)
    rng = np.random.default_rng(M)
    ms = np.unique(np.concatenate([[0, 31, 32, M - 1], rng.integers(0, M, 12)]))
    for tn in (0, 67, N // 128 - 1):
        rows = slice(tn * 128, tn * 128 + 128)
        _grade(Xq[ms], np.ascontiguousarray(Sx[:, ms]), p.W[rows], p.S[tn:tn + 1], yb[ms][:, rows])


def test_w8a8_zero_m_is_a_no_op():
    q = qg()
    W = torch.zeros((128, 128), dtype=torch.uint8, device="cuda")
    S = torch.ones((1, 1), dtype=torch.float32, device="cuda")
    Xq = torch.zeros((0, 128), dtype=torch.uint8, device="cuda")
    Sx = torch.zeros((1, 32), dtype=torch.float32, device="cuda")
    Y = q.qgemm_w8a8_block(Xq, Sx, W, S)
    assert Y.shape == (0, 128)
    assert q.last_device_status() == 0


def test_w8a8_and_decode_calls_interleave():
    """Split-K calls of the W8A8 kind (both tile widths) and of the FP8
    decode kind, interleaved on the binding's default workspaces, all meet
    the rule (each family keeps its arrival counters in its own buffer)."""
    q = qg()
    from gpu_util import Fp8Device, grade_fp8
    pf = cached(("fp8il",), lambda: wl.make_fp8_problem(16, 1024, 5120, config_id=42))
    dev = Fp8Device(pf)
    shapes = [(48, 136, 5120), (200, 256, 5120)]
    probs = [_problem(*sh) for sh in shapes]
    mats = [(torch.from_numpy(p.W).cuda(), torch.from_numpy(p.S).cuda()) for p in probs]
    for _ in range(2):
        for p, (W, S) in zip(probs, mats):
            Xq, Sx = _quantized(p)
            Y = _run_gemm(q, Xq, Sx, W, S, p.N)
            _grade(Xq, Sx, p.W, p.S, to_bits(Y))
            Yf = dev.run()
            assert q.last_device_status() == 0
            ok, rep = grade_fp8(pf, to_bits(Yf))
            assert rep.ok, rep


def test_w8a8_k_zero_writes_zeros():
    """K = 0: every output is the empty sum, 0."""
    q = qg()
    M, N = 40, 300
    Y = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((N, 16), dtype=torch.uint8, device="cuda")
    S = torch.ones((3, 1), dtype=torch.float32, device="cuda")
    Xq = torch.zeros((M, 16), dtype=torch.uint8, device="cuda")
    Sx = torch.zeros((1, 64), dtype=torch.float32, device="cuda")
    r = q.lib.qgemm_w8a8_block(Xq.data_ptr(), 16, Sx.data_ptr(), 64, W.data_ptr(), S.data_ptr(), Y.data_ptr(), N,
                               M, N, 0, None, 0, None)
    assert r == 0
    torch.cuda.synchronize()
    assert q.last_device_status() == 0
    assert torch.count_nonzero(Y.float()) == 0
