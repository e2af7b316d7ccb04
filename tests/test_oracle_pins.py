"""Pins for the CPU oracle: each test ties the oracle to something other than
itself (a library routine, a closed form, an invariant, FP64 brute force, or
numbers printed on the pages).  No GPU needed."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
U = 2.0 ** -24  # FP32 unit roundoff


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ formats
def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_float(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(ours, ref, equal_nan=True)


def test_e4m3_decode_landmarks():
    f = oracle.e4m3_to_float(np.arange(256, dtype=np.uint8))
    finite = f[np.isfinite(f)]
    # the divisor in the block scale (amax / 448) is the largest finite value
    assert finite.max() == 448.0 and finite.min() == -448.0
    assert f[0x01] == 2.0 ** -9            # smallest subnormal
    assert f[0x08] == 2.0 ** -6            # smallest normal
    assert f[0x07] == 7 * 2.0 ** -9        # largest subnormal
    assert np.isnan(f[0x7F]) and np.isnan(f[0xFF])
    assert f[0x00] == 0.0 and not np.signbit(f[0x00])
    assert f[0x80] == 0.0 and np.signbit(f[0x80])
    # positive codes are strictly increasing; negative codes mirror them
    assert np.all(np.diff(f[0:127]) > 0)
    assert np.array_equal(f[128:255], -f[0:127])
    assert np.isfinite(f).sum() == 254


def _float_samples(n, seed=7):
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 2 ** 32, size=n, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    extra = []
    # halfway points and neighbours for BF16 (low 16 bits 0x8000) and FP16 grids
    hb = (rng.integers(0, 2 ** 16, size=20000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    extra.append(hb.view(np.float32))
    extra.append((hb + 1).view(np.float32))
    extra.append((hb - 1).view(np.float32))
    h16 = rng.integers(0, 0x7C00, size=20000).astype(np.uint16).view(np.float16).astype(np.float64)
    nxt = np.nextafter(h16.astype(np.float16), np.float16(np.inf)).astype(np.float64)
    mid = ((h16 + nxt) / 2).astype(np.float32)
    extra.append(mid)
    extra.append(-mid)
    special = np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 65536.0, 6.1e-5, 5.96e-8,
                        2.98e-8, 2.99e-8, 1e-30, 3.0e38, 3.4028235e38, np.inf, -np.inf,
                        1.1754944e-38, 1e-45], dtype=np.float32)
    extra.append(special)
    return np.concatenate([f] + extra)


def test_bf16_rounding_matches_torch():
    x = _float_samples(400000)
    x = x[~np.isnan(x)]
    ours = oracle.float_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_rounding_nan_stays_nan():
    x = np.array([np.nan, -np.nan], dtype=np.float32)
    out = oracle.float_to_bf16(x)
    assert np.all((out & 0x7F80) == 0x7F80) and np.all(out & 0x7F)


def test_fp16_rounding_matches_numpy():
    x = _float_samples(400000, seed=11)
    x = x[~np.isnan(x)]
    ours = oracle.float_to_fp16(x)
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_fp16_decode_all_patterns():
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.fp16_to_float(b)
    ref = b.view(np.float16).astype(np.float32)
    assert np.array_equal(ours, ref, equal_nan=True)


# ------------------------------------------------------------------ FP8 GEMM
def _decode_problem(p):
    x = torch.from_numpy(p.X.view(np.int16)).view(torch.bfloat16).double().numpy()
    q = torch.from_numpy(p.W).view(torch.float8_e4m3fn).double().numpy()
    return x, q


def _fp64_two_level(x, q, S):
    """Exact-as-possible FP64 evaluation of the two-level sum and its absolute mass."""
    M, K = x.shape
    N = q.shape[0]
    KB = -(-K // 128)
    Y = np.zeros((M, N))
    A = np.zeros((M, N))
    for kb in range(KB):
        sl = slice(128 * kb, min(K, 128 * kb + 128))
        inner = x[:, sl] @ q[:, sl].T
        mass = np.abs(x[:, sl]) @ np.abs(q[:, sl]).T
        s = S[np.arange(N) // 128, kb].astype(np.float64)
        Y += inner * s
        A += mass * np.abs(s)
    return Y, A


def _bound(K, A):
    KB = -(-K // 128)
    return (128 + KB + 4) * U * A * 1.01


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (3, 256, 512), (2, 200, 384), (3, 130, 200),
                                   (1, 128, 16)])
def test_fp8_oracle_vs_fp64_brute_force(M, N, K):
    p = wl.make_fp8_problem(M, N, K, config_id=9)
    Yb, Yf = oracle.qgemm_fp8_block(p.X, p.W, p.S, want_f32=True)
    x, q = _decode_problem(p)
    Y64, A = _fp64_two_level(x, q, p.S)
    err = np.abs(Yf.astype(np.float64) - Y64)
    assert np.all(err <= _bound(K, A)), err.max()
    # and the BF16 output is the rounding of the FP32 value
    assert np.array_equal(Yb, torch.from_numpy(Yf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))


def test_fp8_oracle_abs_mass_matches_fp64():
    p = wl.make_fp8_problem(2, 256, 384, config_id=9)
    x, q = _decode_problem(p)
    _, A = _fp64_two_level(x, q, p.S)
    A2 = oracle.fp8_abs_mass(p.X, p.W, p.S)
    assert np.allclose(A, A2, rtol=1e-12, atol=0)


def test_fp8_unit_scales_reduce_to_matmul():
    p = wl.make_fp8_problem(3, 256, 640, config_id=10)
    S1 = np.ones_like(p.S)
    _, Yf = oracle.qgemm_fp8_block(p.X, p.W, S1, want_f32=True)
    x, q = _decode_problem(p)
    ref = np.matmul(x, q.T)
    mass = np.matmul(np.abs(x), np.abs(q).T)
    assert np.all(np.abs(Yf - ref) <= _bound(640, mass))


def test_fp8_power_of_two_scale_is_exact():
    p = wl.make_fp8_problem(3, 256, 512, config_id=11)
    S2 = np.exp2(np.round(np.log2(p.S))).astype(np.float32)
    _, Y1 = oracle.qgemm_fp8_block(p.X, p.W, S2, want_f32=True)
    _, Y2 = oracle.qgemm_fp8_block(p.X, p.W, (S2 * 2).astype(np.float32), want_f32=True)
    assert np.array_equal(Y2, Y1 * 2)


def test_fp8_linearity_in_one_block_scale():
    p = wl.make_fp8_problem(2, 384, 512, config_id=12)
    _, Y0 = oracle.qgemm_fp8_block(p.X, p.W, p.S, want_f32=True)
    S = p.S.copy()
    bn, bk = 1, 2
    delta = np.float32(3.0) * S[bn, bk]
    S[bn, bk] += delta
    _, Y1 = oracle.qgemm_fp8_block(p.X, p.W, S, want_f32=True)
    x, q = _decode_problem(p)
    rows = slice(128 * bn, 128 * bn + 128)
    ks = slice(128 * bk, 128 * bk + 128)
    inner = x[:, ks] @ q[rows, ks].T
    _, A = _fp64_two_level(x, q, S)
    pred = Y0[:, rows].astype(np.float64) + float(delta) * inner
    assert np.all(np.abs(Y1[:, rows] - pred) <= 2 * _bound(512, A[:, rows]))
    # columns outside the changed block row are untouched, bit for bit
    other = np.ones(384, dtype=bool)
    other[rows] = False
    assert np.array_equal(Y0[:, other], Y1[:, other])


def test_fp8_rows_are_independent_and_halves_match():
    p = wl.make_fp8_problem(32, 256, 512, config_id=13)
    Y = oracle.qgemm_fp8_block(p.X, p.W, p.S)
    for m in (0, 7, 31):
        assert np.array_equal(Y[m], oracle.qgemm_fp8_block(p.X[m:m + 1], p.W, p.S)[0])
    top = oracle.qgemm_fp8_block(p.X[:16], p.W, p.S)
    bot = oracle.qgemm_fp8_block(p.X[16:], p.W, p.S)
    assert np.array_equal(np.vstack([top, bot]), Y)


def test_fp8_sign_symmetry_and_block_permutation():
    p = wl.make_fp8_problem(2, 384, 256, config_id=14)
    Y = oracle.qgemm_fp8_block(p.X, p.W, p.S)
    # negating every activation flips the sign bit of every output
    Yn = oracle.qgemm_fp8_block(p.X ^ np.uint16(0x8000), p.W, p.S)
    assert np.array_equal(Yn, Y ^ np.uint16(0x8000))
    # negating every weight code does the same
    Yw = oracle.qgemm_fp8_block(p.X, p.W ^ np.uint8(0x80), p.S)
    assert np.array_equal(Yw, Y ^ np.uint16(0x8000))
    # permuting whole 128-row weight blocks (with their scale rows) permutes columns
    perm = [2, 0, 1]
    Wp = np.vstack([p.W[128 * b:128 * b + 128] for b in perm])
    Sp = p.S[perm]
    Yp = oracle.qgemm_fp8_block(p.X, Wp, Sp)
    assert np.array_equal(Yp, np.hstack([Y[:, 128 * b:128 * b + 128] for b in perm]))


def test_fp8_sampled_matches_full():
    p = wl.make_fp8_problem(5, 384, 640, config_id=15)
    Y, Yf = oracle.qgemm_fp8_block(p.X, p.W, p.S, want_f32=True)
    rng = np.random.default_rng(0)
    ms = rng.integers(0, 5, 300)
    ns = rng.integers(0, 384, 300)
    ys, yf = oracle.qgemm_fp8_block_sample(p.X, p.W, p.S, ms, ns, want_f32=True)
    assert np.array_equal(ys, Y[ms, ns]) and np.array_equal(yf, Yf[ms, ns])
    A = oracle.fp8_abs_mass(p.X, p.W, p.S)
    assert np.array_equal(oracle.fp8_abs_mass(p.X, p.W, p.S, ms, ns), A[ms, ns])


def test_quantiser_round_trip_bound():
    p = wl.make_fp8_problem(1, 256, 384, config_id=16, keep_float=True)
    deq = oracle.e4m3_to_float(p.W).astype(np.float64)
    s = np.repeat(np.repeat(p.S.astype(np.float64), 128, 0), 128, 1)[:256, :384]
    v = p.W_f32.astype(np.float64) / s
    # half an E4M3 ulp at the value's binade (subnormal quantum 2^-9 below 2^-6), plus
    # the FP32 division's own rounding
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -6)))
    half_ulp = np.exp2(e - 4)
    assert np.all(np.abs(deq - v) <= half_ulp + 1e-6 * np.abs(v) + 1e-12)
    # every block reaches the top code (its amax maps to 448)
    for i in range(2):
        for j in range(3):
            blk = deq[128 * i:128 * i + 128, 128 * j:128 * j + 128]
            assert np.abs(blk).max() == 448.0


# ------------------------------------------------------------------ criterion
def test_criterion_accepts_reassociation_and_rejects_planted_bugs():
    """The comparison rule passes a reordered FP32 sum and fails the plausible
    bugs (dropped block, wrong scale row, sign error, transposed K blocks);
    the bugs are planted in the oracle's inputs, on the CPU."""
    p = wl.make_fp8_problem(16, 512, 1024, config_id=17)
    ref = oracle.qgemm_fp8_block(p.X, p.W, p.S)
    A = oracle.fp8_abs_mass(p.X, p.W, p.S)
    # reassociated: blocks summed in descending order (still a two-level fold)
    x, q = _decode_problem(p)
    KB = 8
    xs = x.astype(np.float32)
    qs = q.astype(np.float32)
    outer = np.zeros((16, 512), dtype=np.float32)
    for kb in reversed(range(KB)):
        inner = np.zeros((16, 512), dtype=np.float32)
        for c in reversed(range(8)):            # 16-wide chunks in reverse order
            chunk = np.zeros((16, 512), dtype=np.float32)
            for k in range(128 * kb + 16 * c, 128 * kb + 16 * c + 16):
                chunk = chunk + xs[:, k:k + 1] * qs[None, :, k]
            inner = inner + chunk
        outer = outer + inner * p.S[np.arange(512) // 128, kb][None, :]
    re = torch.from_numpy(outer).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ok, rep = oracle.within_budget(re, ref, A)
    assert rep.ok, rep

    W = p.W.copy()
    W[:, 128:256] = 0                              # dropped block
    ok, rep = oracle.within_budget(oracle.qgemm_fp8_block(p.X, W, p.S), ref, A)
    assert rep.over_budget > 1000
    S = p.S[::-1].copy()                           # wrong scale row
    ok, rep = oracle.within_budget(oracle.qgemm_fp8_block(p.X, p.W, S), ref, A)
    assert rep.over_budget > 1000
    S = p.S.copy()
    S[:, 3] *= -1                                  # sign error in one block
    ok, rep = oracle.within_budget(oracle.qgemm_fp8_block(p.X, p.W, S), ref, A)
    assert rep.over_budget > 1000
    Wt = np.hstack([p.W[:, 128:256], p.W[:, 0:128], p.W[:, 256:]])  # swapped K blocks
    ok, rep = oracle.within_budget(oracle.qgemm_fp8_block(p.X, Wt, p.S), ref, A)
    assert rep.over_budget > 1000


def test_criterion_ordinals():
    assert oracle.bf16_ord(np.uint16(0x0000)) == 0
    assert oracle.bf16_ord(np.uint16(0x8000)) == 0
    assert oracle.bf16_ord(np.uint16(0x0001)) - oracle.bf16_ord(np.uint16(0x8001)) == 2
    a = np.array([0x3F80, 0x3F81, 0x3F82, 0x3F83], dtype=np.uint16)
    b = np.full(4, 0x3F80, dtype=np.uint16)
    ok, rep = oracle.within_budget(a, b, np.zeros(4))
    assert list(ok) == [True, True, True, False] and rep.max_ulp == 3


def test_page_red_cell_signature():
    """Host simulation of a tensor-core reduction order on the M=32 gate/up
    geometry (the page's red cell): a strict 2-ULP rule flags only outputs that
    cancelled to near zero, the mixed rule flags none, and nothing flips sign."""
    g = _golden("atlas_m16_tc_page.json")["red_cell"]
    M, N, K = g["M"], g["N"], g["K"]
    assert M * N == g["elements"]
    Ns = N
    p = wl.make_fp8_problem(M, Ns, K, config_id=1)
    ref, reff = oracle.qgemm_fp8_block(p.X, p.W, p.S, want_f32=True)
    A = oracle.fp8_abs_mass(p.X, p.W, p.S)
    x, q = _decode_problem(p)
    xs = x.astype(np.float32)
    qs = q.astype(np.float32)
    outer = np.zeros((M, Ns), dtype=np.float32)
    srow = np.arange(Ns) // 128
    for kb in range(K // 128):
        inner = np.zeros((M, Ns), dtype=np.float32)
        for c in range(8):
            ks = slice(128 * kb + 16 * c, 128 * kb + 16 * c + 16)
            # a 16-term chunk is reduced first (in FP64, rounded once), then added
            chunk = (x[:, ks] @ q[:, ks].T).astype(np.float32)
            inner = inner + chunk
        outer = outer + inner * p.S[srow, kb][None, :]
    sim = torch.from_numpy(outer).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ok, rep = oracle.within_budget(sim, ref, A)
    assert rep.ok and rep.sign_flips == 0, rep
    strict, srep = oracle.within_budget(sim, ref, A, margin=0.0)
    rv = oracle.bf16_to_float(ref).astype(np.float64)
    rms = np.sqrt(np.mean(rv ** 2))
    bad = ~strict
    # the strict rule does fail somewhere, and only on outputs that cancelled to
    # a tiny fraction of the RMS (the page saw |ref| / RMS of ~1e-7 .. 4e-6)
    assert bad.sum() >= 1
    assert np.all(np.abs(rv[bad]) < 1e-4 * rms)
    assert srep.sign_flips == 0 and srep.rel_rms < 1e-4
    # away from the floor every element is within one BF16 ULP
    assert rep.max_ulp_outside_floor <= 1
    assert rep.max_rel_err <= 1e-2


# ------------------------------------------------------------------ LUT3
def test_lut3_dequant_identity_and_library_product():
    qmap = wl.lut3_qmap_bits()
    one = np.float16(1.0).view(np.uint16)
    for c in range(8):
        assert oracle.lut3_dequant(c, qmap, int(one)) == int(qmap[c])
    # every FP16 scale in [0.005, 0.02], all 8 codes: one rounding of the exact product
    lo = int(np.float16(0.005).view(np.uint16))
    hi = int(np.float16(0.02).view(np.uint16))
    scales = np.arange(lo, hi + 1, dtype=np.uint16)
    codes = np.tile(np.arange(8, dtype=np.uint8), (scales.size, 16))[:, :128]
    D = oracle.lut3_dequant_matrix(codes, qmap, scales[:, None])
    qf = qmap.view(np.float16)
    ref = (qf[codes].astype(np.float32) * scales.view(np.float16)[:, None].astype(np.float32)).astype(np.float16)
    assert np.array_equal(D, ref.view(np.uint16))
    # with this distribution no dequantised value is subnormal or infinite
    Df = D.view(np.float16).astype(np.float32)
    assert np.all(np.abs(Df) >= 2.0 ** -14) and np.all(np.isfinite(Df))


def test_lut3_qmap_matches_bisection_quantiles():
    import math

    def phi(x):
        return 0.5 * (1.0 + math.erf(x / math.sqrt(2.0)))

    def inv(pv):
        lo, hi = -10.0, 10.0
        for _ in range(200):
            mid = 0.5 * (lo + hi)
            if phi(mid) < pv:
                lo = mid
            else:
                hi = mid
        return 0.5 * (lo + hi)

    ref = np.array([inv((i + 0.5) / 8) for i in range(8)], dtype=np.float32).astype(np.float16)
    q = wl.lut3_qmap_bits().view(np.float16)
    assert np.array_equal(q, ref)
    assert np.array_equal(q, -q[::-1])
    assert np.all(np.diff(q.astype(np.float32)) > 0)


def _fp64_lut3(p):
    x = p.X.view(np.float16).astype(np.float64)
    D = oracle.lut3_dequant_matrix(p.codes, p.qmap, p.scales).view(np.float16).astype(np.float64)
    return x @ D.T, np.abs(x) @ np.abs(D).T


@pytest.mark.parametrize("M,N,K", [(1, 128, 256), (4, 256, 512), (3, 200, 384)])
def test_lut3_oracle_vs_fp64_brute_force(M, N, K):
    p = wl.make_lut3_problem(M, N, K, config_id=20)
    Y, Yf = oracle.qgemm_lut3(p.X, p.codes, p.qmap, p.scales, want_f32=True)
    ref, A = _fp64_lut3(p)
    assert np.all(np.abs(Yf - ref) <= (K + 4) * U * A * 1.01)
    assert np.array_equal(Y, Yf.astype(np.float16).view(np.uint16))
    assert np.allclose(oracle.lut3_abs_mass(p.X, p.codes, p.qmap, p.scales), A, rtol=1e-12)


def test_lut3_unit_scales_reduce_to_qmap_matmul():
    p = wl.make_lut3_problem(2, 128, 256, config_id=21)
    one = np.full_like(p.scales, np.float16(1.0).view(np.uint16))
    _, Yf = oracle.qgemm_lut3(p.X, p.codes, p.qmap, one, want_f32=True)
    x = p.X.view(np.float16).astype(np.float64)
    Wq = p.qmap.view(np.float16).astype(np.float64)[p.codes]
    ref = x @ Wq.T
    assert np.all(np.abs(Yf - ref) <= (256 + 4) * U * (np.abs(x) @ np.abs(Wq).T))


def test_lut3_rows_independent_and_sampled():
    p = wl.make_lut3_problem(8, 256, 512, config_id=22)
    Y = oracle.qgemm_lut3(p.X, p.codes, p.qmap, p.scales)
    assert np.array_equal(Y[5], oracle.qgemm_lut3(p.X[5:6], p.codes, p.qmap, p.scales)[0])
    ms = np.array([0, 3, 7, 7]); ns = np.array([0, 100, 255, 17])
    assert np.array_equal(oracle.qgemm_lut3_sample(p.X, p.codes, p.qmap, p.scales, ms, ns), Y[ms, ns])


# ------------------------------------------------------------------ packing
@pytest.mark.parametrize("N,K", [(128, 256), (256, 1024), (130, 300), (1, 8), (300, 520)])
def test_oracle_pack_round_trip(N, K):
    codes = wl.uniform_codes(99, N * K).reshape(N, K)
    packed = oracle.pack_lut3(codes)
    assert packed.size == -(-N // 128) * -(-K // 256) * 16384
    assert np.array_equal(oracle.unpack_lut3(packed, N, K), codes)


def test_oracle_pack_layout_landmarks():
    """Spot checks of the documented layout: tile order, chunk/row order, word
    and nibble order, and zero padding."""
    N, K = 256, 512
    codes = np.zeros((N, K), dtype=np.uint8)
    codes[0, 0] = 1          # tile 0, chunk 0, row 0, word 0, nibble 0
    codes[0, 9] = 2          # word 1, nibble 1
    codes[5, 32] = 3         # chunk 1, row 5
    codes[130, 300] = 4      # tile (1, 1), row 2, k 44 -> chunk 1, word 1, nibble 4
    codes[255, 511] = 7      # last tile, chunk 7, row 127, word 3, nibble 7
    p = oracle.pack_lut3(codes)
    w = p.view("<u4")
    assert w[0] == 0x1
    assert w[1] == 0x2 << 4
    assert w[((1 * 128 + 5) * 16) // 4] == 0x3
    base = (1 * 2 + 1) * 16384
    assert w[(base + (1 * 128 + 2) * 16) // 4 + 1] == 0x4 << 16
    last = (1 * 2 + 1) * 16384 + (7 * 128 + 127) * 16 + 12
    assert w[last // 4] == 0x7 << 28
    assert np.count_nonzero(w) == 5
    # unpacking never sees a set top bit
    assert np.all((oracle.unpack_lut3(p, N, K) & 8) == 0)


# ------------------------------------------------------------------ page numbers
def test_page_bandwidth_arithmetic():
    """The GB/s figures printed on the atlas page are weight bytes / time in
    decimal units; the byte counting used by the benchmark reproduces them."""
    g = _golden("atlas_m16_tc_page.json")["why_table"]
    for key in ("gateup", "down"):
        row = g[key]
        wbytes = row["N"] * row["K"]
        assert abs(wbytes / 1e6 - g["weight_MB"]) < 0.2
        gbps = wbytes / (row["ms"] * 1e-3) / 1e9
        assert abs(gbps - row["GBps"]) < 1.0, (key, gbps)
    # ~30 us ideal stream at ~3,000 GB/s
    assert abs(g["weight_MB"] * 1e6 / (g["hbm3_GBps"] * 1e9) * 1e6 - g["ideal_stream_us"]) < 1.0


def test_page_grid_counts():
    g = _golden("atlas_m16_tc_page.json")["grid_table"]
    for n, ctas in g["ctas"].items():
        assert int(n) // g["n_tile"] == ctas
    assert g["sms"] * g["ctas_per_sm"] == g["resident"]


# ------------------------------------------------------------------ dense BF16 GEMM
def _bf16_decode(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (3, 200, 512), (2, 130, 1000), (4, 64, 8)])
def test_bf16_oracle_vs_fp64_brute_force(M, N, K):
    """Within the FP32 recursive-summation bound of the FP64 product, and the
    BF16 output is the rounding of the FP32 sum."""
    p = wl.make_bf16_problem(M, N, K, config_id=11)
    Yb, Yf = oracle.gemm_bf16(p.X, p.W, want_f32=True)
    x, w = _bf16_decode(p.X), _bf16_decode(p.W)
    Y64 = x @ w.T
    A = np.abs(x) @ np.abs(w).T
    err = np.abs(Yf.astype(np.float64) - Y64)
    assert np.all(err <= (K + 4) * U * A * 1.01), err.max()
    assert np.array_equal(Yb, torch.from_numpy(Yf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    assert np.allclose(oracle.bf16_abs_mass(p.X, p.W), A, rtol=1e-12, atol=0)


def test_bf16_oracle_small_integers_are_exact():
    """Small integer operands: every partial sum is an exact FP32 integer, so
    the sum is the integer matmul and only the final BF16 rounding remains."""
    rng = np.random.default_rng(12)
    M, N, K = 3, 40, 1024
    xi = rng.integers(-8, 9, size=(M, K))
    wi = rng.integers(-8, 9, size=(N, K))
    X = wl.bf16_bits_from_f32(xi.astype(np.float32))
    W = wl.bf16_bits_from_f32(wi.astype(np.float32))
    Yb, Yf = oracle.gemm_bf16(X, W, want_f32=True)
    exact = xi @ wi.T
    assert np.array_equal(Yf.astype(np.int64), exact)
    assert np.array_equal(Yb, wl.bf16_bits_from_f32(exact.astype(np.float32)))


def test_bf16_oracle_sums_in_strict_k_order():
    """x = [2^24, 1, -2^24], w = [1, 1, 1]: in strict K order 2^24 + 1 rounds to
    2^24 (tie to even) and the sum is 0; any order that adds the 1 last gives 1."""
    X = wl.bf16_bits_from_f32(np.array([[2.0 ** 24, 1.0, -(2.0 ** 24)]], dtype=np.float32))
    W = wl.bf16_bits_from_f32(np.ones((1, 3), dtype=np.float32))
    _, Yf = oracle.gemm_bf16(X, W, want_f32=True)
    assert Yf[0, 0] == 0.0
    X2 = wl.bf16_bits_from_f32(np.array([[2.0 ** 24, -(2.0 ** 24), 1.0]], dtype=np.float32))
    _, Yf2 = oracle.gemm_bf16(X2, W, want_f32=True)
    assert Yf2[0, 0] == 1.0


def test_bf16_oracle_rows_independent_and_sampled():
    p = wl.make_bf16_problem(5, 300, 640, config_id=13)
    Y = oracle.gemm_bf16(p.X, p.W)
    for m in range(5):
        assert np.array_equal(oracle.gemm_bf16(p.X[m:m + 1], p.W)[0], Y[m])
    rng = np.random.default_rng(3)
    ms = rng.integers(0, 5, 200).astype(np.int32)
    ns = rng.integers(0, 300, 200).astype(np.int32)
    assert np.array_equal(oracle.gemm_bf16_sample(p.X, p.W, ms, ns), Y[ms, ns])
    assert np.allclose(oracle.bf16_abs_mass(p.X, p.W, ms, ns), oracle.bf16_abs_mass(p.X, p.W)[ms, ns], rtol=0,
                       atol=0)


# ------------------------------------------------------------------ W8A8 (FP8 activations)
def _e4m3_grid():
    codes = np.arange(0, 0x7F, dtype=np.uint8)
    return oracle.e4m3_to_float(codes).astype(np.float64)


def test_e4m3_encoder_matches_torch():
    """Round to nearest even with saturation at 448, against torch's
    float8_e4m3fn conversion of the clamped value: random values over the
    whole range, every midpoint between neighbouring E4M3 values (ties), and
    values beyond 448."""
    rng = np.random.default_rng(31)
    x = (rng.standard_normal(20000) * np.exp2(rng.uniform(-14, 10, 20000))).astype(np.float32)
    g = _e4m3_grid()
    mids = ((g[:-1] + g[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids, np.nextafter(mids, np.float32(np.inf)),
                        np.array([448, 449, 464, 480, 1e6, -1e6, 0.0, -0.0, 2 ** -10, 3 * 2 ** -11], np.float32)])
    ours = oracle.float_to_e4m3(x)
    ref = torch.from_numpy(np.clip(x, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_activation_quantiser_rule():
    """Per (row, 128-K block): s = fl32(amax / 448), the largest |code| is
    448, every value within half an E4M3 step (times s) of x, all-zero
    blocks get s = 1 and zero codes."""
    p = wl.make_fp8_problem(4, 128, 300, config_id=32)
    X = p.X.copy()
    X[2, 128:256] = 0
    Xq, Sx = oracle.quantize_act_e4m3(X)
    x = _bf16_decode(X)
    dq = oracle.e4m3_to_float(Xq).astype(np.float64)
    for m in range(4):
        for kb in range(3):
            sl = slice(128 * kb, min(300, 128 * kb + 128))
            amax = np.float32(np.abs(x[m, sl]).max())
            if amax == 0:
                assert Sx[kb, m] == 1.0 and np.all(Xq[m, sl] & 0x7F == 0)
                continue
            assert Sx[kb, m] == np.float32(amax / np.float32(448.0))
            assert np.abs(dq[m, sl]).max() == 448.0
            s = np.float64(Sx[kb, m])
            err = np.abs(dq[m, sl] * s - x[m, sl])
            half_step = np.exp2(np.floor(np.log2(np.maximum(np.abs(dq[m, sl]), 2 ** -6))) - 4) * s
            assert np.all(err <= half_step * (1 + 2 ** -20) + 2 ** -10 * s)


def test_w8a8_with_unit_activation_scales_is_the_w8a16_oracle():
    """When the activations are E4M3 values held as BF16 and their scales are
    1, the W8A8 fold is the W8A16 fold term for term: identical bits."""
    p = wl.make_fp8_problem(3, 256, 640, config_id=33)
    rng = np.random.default_rng(33)
    Xq = rng.integers(0, 256, size=(3, 640), dtype=np.uint8)
    Xq[(Xq & 0x7F) == 0x7F] = 0x38                        # no NaN codes
    Xbf = wl.bf16_bits_from_f32(oracle.e4m3_to_float(Xq).astype(np.float32))
    Sx = np.ones((5, 3), dtype=np.float32)
    Y8, Yf8 = oracle.qgemm_w8a8_block(Xq, Sx, p.W, p.S, want_f32=True)
    Y16, Yf16 = oracle.qgemm_fp8_block(Xbf, p.W, p.S, want_f32=True)
    assert np.array_equal(Yf8.view(np.uint32), Yf16.view(np.uint32))
    assert np.array_equal(Y8, Y16)


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (3, 256, 512), (5, 130, 200)])
def test_w8a8_oracle_vs_fp64_brute_force(M, N, K):
    p = wl.make_fp8_problem(M, N, K, config_id=34)
    Xq, Sx = oracle.quantize_act_e4m3(p.X)
    Yb, Yf = oracle.qgemm_w8a8_block(Xq, Sx, p.W, p.S, want_f32=True)
    xq = oracle.e4m3_to_float(Xq).astype(np.float64)
    wq = oracle.e4m3_to_float(p.W).astype(np.float64)
    KB = -(-K // 128)
    Y64 = np.zeros((M, N))
    for kb in range(KB):
        sl = slice(128 * kb, min(K, 128 * kb + 128))
        f = Sx[kb][:, None].astype(np.float64) * p.S[np.arange(N) // 128, kb][None, :].astype(np.float64)
        Y64 += (xq[:, sl] @ wq[:, sl].T) * f
    A = oracle.w8a8_abs_mass(Xq, Sx, p.W, p.S)
    err = np.abs(Yf.astype(np.float64) - Y64)
    assert np.all(err <= (128 + KB + 6) * U * A * 1.01), err.max()
    assert np.array_equal(Yb, torch.from_numpy(Yf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))


def test_w8a8_power_of_two_activation_scale_is_exact():
    p = wl.make_fp8_problem(2, 256, 384, config_id=35)
    Xq, Sx = oracle.quantize_act_e4m3(p.X)
    _, Yf = oracle.qgemm_w8a8_block(Xq, Sx, p.W, p.S, want_f32=True)
    _, Yf2 = oracle.qgemm_w8a8_block(Xq, Sx * np.float32(4.0), p.W, p.S, want_f32=True)
    assert np.array_equal(Yf2, Yf * np.float32(4.0))
