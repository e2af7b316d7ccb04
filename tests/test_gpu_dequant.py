"""The kernels' own dequantisers, checked value by value against the oracle
(bit-exact: the E4M3 -> BF16 and LUT -> FP16 conversions have one correct
answer)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import qg, to_bits

pytestmark = pytest.mark.gpu


def test_e4m3_to_bf16_all_codes_exact():
    q = qg()
    codes = np.arange(256, dtype=np.uint8)
    finite = np.array([c for c in codes if c not in (0x7F, 0xFF)], dtype=np.uint8)
    # every code, in every position of a 4-byte word, plus a ragged tail
    arr = np.concatenate([np.repeat(finite, 4), np.roll(np.repeat(finite, 4), 1),
                          np.roll(np.repeat(finite, 4), 2), finite[:3]])
    out = q.dequant_e4m3_bf16(torch.from_numpy(arr).cuda())
    assert q.last_device_status() == 0
    got = to_bits(out)
    ref = oracle.float_to_bf16(oracle.e4m3_to_float(arr))
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(hex(arr[i]), hex(got[i]), hex(ref[i])) for i in bad[:10]]


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
