"""The kernels' own conversions, checked value by value.

* The FP8 GEMM feeds E4M3 weights to the tensor core as stored and splits
  BF16 activations instead: per (row, 128-wide K block) an exponent e brings
  the largest |x| into [128, 256), and each x * 2^e becomes two E4M3 codes
  with x * 2^e = hi + lo / 16.  Every finite BF16 pattern is checked under
  every exponent the rule can give it.
* The LUT3 dequantiser is bit-exact against the oracle (one correct answer).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import qg, to_bits

pytestmark = pytest.mark.gpu


def _split_blocks():
    """Blocks of 128 BF16 patterns covering, for every block-maximum exponent
    E (biased, 0 = zero/subnormal .. 254), every finite pattern of magnitude
    at most that maximum, both signs; element 0 holds the maximum (negative in
    every other block).  Also one all-zero block and one all -0 block."""
    blocks, expect_e = [], []
    for E in range(255):
        mags = np.arange(0, (E + 1) << 7, dtype=np.uint32)
        pats = np.concatenate([mags, mags | 0x8000]).astype(np.uint16)
        per = 127
        nrow = -(-pats.size // per)
        pats = np.concatenate([pats, np.zeros(nrow * per - pats.size, np.uint16)])
        blk = np.empty((nrow, 128), np.uint16)
        blk[:, 0] = (E << 7) | 0x7F
        blk[1::2, 0] |= 0x8000
        blk[:, 1:] = pats.reshape(nrow, per)
        blocks.append(blk)
        expect_e.append(np.full(nrow, min(126, 134 - E), np.int32))
    blocks.append(np.zeros((1, 128), np.uint16))
    blocks.append(np.full((1, 128), 0x8000, np.uint16))
    expect_e += [np.array([126], np.int32)] * 2
    return np.concatenate(blocks), np.concatenate(expect_e)


def test_fp8_activation_split_exhaustive():
    """x * 2^e = hi + lo/16 exactly for |x * 2^e| >= 2^-6 and within 2^-14
    below; e = min(126, 134 - exponent of the block maximum)."""
    q = qg()
    X, expect_e = _split_blocks()
    Xd = torch.from_numpy(X.view(np.int16)).view(torch.bfloat16).cuda()
    hi, lo, e = q.debug_fp8_split(Xd)
    assert q.last_device_status() == 0
    hi, lo, e = hi.cpu().numpy(), lo.cpu().numpy(), e.cpu().numpy()
    np.testing.assert_array_equal(e, expect_e)
    table = oracle.e4m3_to_float(np.arange(256, dtype=np.uint8)).astype(np.float64)
    assert not np.isnan(table[hi]).any() and not np.isnan(table[lo]).any()
    x = (X.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    target = x * np.exp2(e.astype(np.float64))[:, None]
    got = table[hi] + table[lo] / 16.0
    assert np.abs(target).max() < 256.0
    exact = np.abs(target) >= 2.0 ** -6
    bad = exact & (got != target)
    assert not bad.any(), [(hex(int(X[i, j])), int(e[i]), float(target[i, j]), float(got[i, j]))
                           for i, j in zip(*np.nonzero(bad))][:8]
    err = np.abs(got - target)[~exact]
    assert err.max() <= 2.0 ** -14, float(err.max())


@pytest.mark.parametrize("N,K", [(128, 256), (200, 384), (384, 1024)])
def test_lut3_dequant_matches_oracle(N, K):
    q = qg()
    p = wl.make_lut3_problem(1, N, K, config_id=30)
    Wq = torch.from_numpy(q.pack_lut3(p.codes)).cuda()
    qm = torch.from_numpy(p.qmap.view(np.int16)).view(torch.float16).cuda()
    sc = torch.from_numpy(p.scales.view(np.int16)).view(torch.float16).cuda()
    D = q.dequant_lut3(Wq, qm, sc, N, K)
    assert q.last_device_status() == 0
    ref = oracle.lut3_dequant_matrix(p.codes, p.qmap, p.scales)
    assert np.array_equal(to_bits(D), ref)


def test_lut3_dequant_every_code_and_scale():
    """All 8 codes against every FP16 scale in [0.005, 0.02] (plus 1.0), one
    scale per 128-wide group."""
    q = qg()
    lo = int(np.float16(0.005).view(np.uint16))
    hi = int(np.float16(0.02).view(np.uint16))
    svals = np.concatenate([np.arange(lo, hi + 1, dtype=np.uint16),
                            [np.float16(1.0).view(np.uint16)]]).astype(np.uint16)
    N = 128
    G = -(-svals.size // N)
    K = 128 * G
    scales = np.resize(svals, (N, G)).astype(np.uint16)
    codes = np.tile(np.arange(8, dtype=np.uint8), (N, K // 8))
    qmap = wl.lut3_qmap_bits()
    Wq = torch.from_numpy(q.pack_lut3(codes)).cuda()
    qm = torch.from_numpy(qmap.view(np.int16)).view(torch.float16).cuda()
    sc = torch.from_numpy(scales.view(np.int16)).view(torch.float16).cuda()
    D = q.dequant_lut3(Wq, qm, sc, N, K)
    ref = oracle.lut3_dequant_matrix(codes, qmap, scales)
    assert np.array_equal(to_bits(D), ref)
