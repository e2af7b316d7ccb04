"""The allocation-free FP8 entry point (for callers that cannot allocate
device memory, such as plug-ins whose host framework owns every device
buffer).  It must give the same results as qgemm_fp8_block with a caller
workspace, call after call, while using its own fixed scratch array.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import qg, to_bits

pytestmark = pytest.mark.gpu

_P = ctypes.c_void_p


def _noalloc_fn(q):
    fn = ctypes.CDLL(q.LIB_PATH).qgemm_fp8_block_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [_P, ctypes.c_int64, _P, _P, _P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P]
    return fn


@pytest.mark.parametrize("M,N,K", [(16, 5120, 5120), (32, 1024, 5120), (3, 200, 336)])
def test_noalloc_matches_workspace_entry_point(M, N, K):
    q = qg()
    fn = _noalloc_fn(q)
    p = wl.make_fp8_problem(M, N, K, config_id=60)
    X = torch.from_numpy(p.X.view(np.int16)).view(torch.bfloat16).cuda()
    W = torch.from_numpy(p.W).cuda()
    S = torch.from_numpy(p.S).cuda()
    ref = to_bits(q.qgemm_fp8_block(X, W, S, workspace=q.Workspace()))
    assert q.last_device_status() == 0
    A = oracle.fp8_abs_mass(p.X, p.W, p.S)
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):   # two calls in a row share the scratch array
        Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        Y.view(torch.int16).fill_(0x7FC1)
        r = fn(X.data_ptr(), K, W.data_ptr(), S.data_ptr(), Y.data_ptr(), N, M, N, K, stream)
        assert r == 0, q.status_string(r)
        assert q.last_device_status() == 0
        ok, rep = oracle.within_budget(to_bits(Y), ref, A)
        assert rep.ok, rep


def test_noalloc_rejects_shapes_beyond_its_scratch():
    q = qg()
    fn = _noalloc_fn(q)
    N, K = 128 * 300000, 256          # needs more than the fixed 8 MiB of scratch
    assert q.workspace_bytes(q.KIND_FP8_BLOCK, 32, N, K) > (8 << 20)
    fake = 1 << 20                    # never dereferenced: rejected before any launch
    assert fn(fake, K, fake, fake, fake, N, 32, N, K, None) == 6   # QG_ERR_WORKSPACE
