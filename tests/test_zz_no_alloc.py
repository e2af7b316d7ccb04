"""The allocation-free FP8 entry point, for callers that cannot allocate
device memory (such as plug-ins whose host framework owns every device
buffer, or servers that must not allocate while serving).  It runs the same
kernel and schedule as qgemm_fp8_block with a caller workspace, so its results
must be the same bits, call after call, while it uses its own fixed scratch
array; they are also graded against the oracle.

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


def _device_problem(M, N, K, cid):
    p = wl.make_fp8_problem(M, N, K, config_id=cid)
    X = torch.from_numpy(p.X.view(np.int16)).view(torch.bfloat16).cuda()
    W = torch.from_numpy(p.W).cuda()
    S = torch.from_numpy(p.S).cuda()
    return p, X, W, S


def _call(fn, X, W, S, M, N, K):
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    Y.view(torch.int16).fill_(0x7FC1)   # a NaN pattern: every element must be written
    r = fn(X.data_ptr(), K, W.data_ptr(), S.data_ptr(), Y.data_ptr(), N, M, N, K,
           torch.cuda.current_stream().cuda_stream)
    return r, Y


@pytest.mark.parametrize("M,N,K", [(16, 5120, 5120), (32, 1024, 5120), (3, 200, 336), (16, 17408, 5120)])
def test_noalloc_matches_workspace_entry_point(M, N, K):
    """Two calls in a row (sharing the scratch array) give exactly the bits
    of the workspace entry point, and those are within the oracle's budget."""
    q = qg()
    fn = _noalloc_fn(q)
    p, X, W, S = _device_problem(M, N, K, 60)
    ref = to_bits(q.qgemm_fp8_block(X, W, S, workspace=q.Workspace()))
    assert q.last_device_status() == 0
    for _ in range(2):
        r, Y = _call(fn, X, W, S, M, N, K)
        assert r == 0, q.status_string(r)
        assert q.last_device_status() == 0
        got = to_bits(Y)
        assert np.array_equal(got, ref), f"{int((got != ref).sum())} elements differ from qgemm_fp8_block"
    ok, rep = oracle.within_budget(got, oracle.qgemm_fp8_block(p.X, p.W, p.S), oracle.fp8_abs_mass(p.X, p.W, p.S))
    assert rep.ok, rep


def test_noalloc_recovers_after_a_timeout():
    """A call whose wait runs out (a host-side fault hook makes CTA 0 skip its
    first weight load; nothing faults) leaves arrival counters set in the
    shared scratch array; reading the timeout status clears them, and the
    next call is exact again."""
    q = qg()
    fn = _noalloc_fn(q)
    M, N, K = 32, 1024, 5120        # split over many CTAs: the counters are in use
    p, X, W, S = _device_problem(M, N, K, 61)
    ref = to_bits(q.qgemm_fp8_block(X, W, S, workspace=q.Workspace()))
    assert q.last_device_status() == 0
    q.set_wait_timeout_ns(20_000_000)
    q.set_fault_injection(0)
    try:
        r, _ = _call(fn, X, W, S, M, N, K)
        assert r == 0
        assert q.last_device_status() == 5    # QG_ERR_TIMEOUT
    finally:
        q.set_fault_injection(-1)
        q.set_wait_timeout_ns(1_000_000_000)
    for _ in range(2):
        r, Y = _call(fn, X, W, S, M, N, K)
        assert r == 0
        assert q.last_device_status() == 0
        assert np.array_equal(to_bits(Y), ref)


def test_noalloc_rejects_bad_arguments_and_oversized_shapes():
    """Argument errors come back exactly as from qgemm_fp8_block; a shape that
    needs more than the fixed 8 MiB of scratch returns QG_ERR_WORKSPACE; none
    of these enqueues anything."""
    q = qg()
    fn = _noalloc_fn(q)
    fake = 1 << 20                    # never dereferenced: rejected before any launch
    N, K = 128 * 300000, 256
    assert q.workspace_bytes(q.KIND_FP8_BLOCK, 32, N, K) > (8 << 20)
    assert fn(fake, K, fake, fake, fake, N, 32, N, K, None) == 6             # QG_ERR_WORKSPACE
    assert fn(None, K, fake, fake, fake, N, 32, N, K, None) == 1             # null X, before the size check
    assert fn(fake + 8, K, fake, fake, fake, N, 32, N, K, None) == 3         # misaligned X
    assert fn(fake, K, fake, fake, fake, N, 33, N, K, None) == 2             # M > 32
    assert fn(fake, 512, fake, fake, fake, 256, 0, 256, 512, None) == 0     # M == 0: no-op
    assert q.last_device_status() == 0
