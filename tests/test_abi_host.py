"""Host-side checks of the C ABI (no GPU): the library loads, exports every
function include/qgemm.h declares, validates arguments before touching the
device, and packs 3-bit codes bit-exactly like the oracle's independent
packer."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def qg():
    import __graft_entry__
    __graft_entry__.build_library()
    import weight_only_quantized_qgemm_gb300 as q
    return q


def _declared_functions():
    names = []
    for hdr in os.listdir(os.path.join(ROOT, "include")):
        if not hdr.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", hdr)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \*]*?\b(\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for must in ("qgemm_fp8_block", "qgemm_lut3", "pack_lut3", "qg_workspace_bytes",
                 "qg_last_device_status", "qg_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol(qg):
    handle = ctypes.CDLL(qg.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(handle, name), name


def test_status_strings(qg):
    for code in range(7):
        assert qg.status_string(code) and qg.status_string(code) != "unknown status"
    assert qg.status_string(99) == "unknown status"
    assert qg.lib.qg_version().decode().count(".") == 2


FAKE = 0x100000  # never dereferenced: every call below fails validation first


@pytest.mark.parametrize("args,expect", [
    # X, ldx, W, S, Y, ldy, M, N, K
    ((FAKE, 512, FAKE, FAKE, FAKE, 256, 0, 256, 512), 0),        # M == 0: no-op
    ((FAKE, 512, FAKE, FAKE, FAKE, 256, 4, 0, 512), 0),          # N == 0: no-op
    ((None, 512, FAKE, FAKE, FAKE, 256, 4, 256, 512), 1),        # null X
    ((FAKE, 512, None, FAKE, FAKE, 256, 4, 256, 512), 1),        # null W
    ((FAKE, 512, FAKE, None, FAKE, 256, 4, 256, 512), 1),        # null scales
    ((FAKE, 512, FAKE, FAKE, None, 256, 4, 256, 512), 1),        # null Y
    ((FAKE, 512, FAKE, FAKE, FAKE, 256, -1, 256, 512), 1),       # negative M
    ((FAKE, 512, FAKE, FAKE, FAKE, 256, 33, 256, 512), 2),       # M > 32
    ((FAKE, 520, FAKE, FAKE, FAKE, 256, 4, 256, 520), 2),        # K % 16
    ((FAKE, 256, FAKE, FAKE, FAKE, 256, 4, 256, 512), 1),        # ldx < K
    ((FAKE, 512, FAKE, FAKE, FAKE, 100, 4, 256, 512), 1),        # ldy < N
    ((FAKE + 8, 512, FAKE, FAKE, FAKE, 256, 4, 256, 512), 3),    # X not 16-byte aligned
    ((FAKE, 512, FAKE + 4, FAKE, FAKE, 256, 4, 256, 512), 3),    # W not 16-byte aligned
    ((FAKE, 516, FAKE, FAKE, FAKE, 256, 4, 256, 512), 3),        # ldx % 8
])
def test_fp8_argument_validation(qg, args, expect):
    X, ldx, W, S, Y, ldy, M, N, K = args
    assert qg.lib.qgemm_fp8_block(X, ldx, W, S, Y, ldy, M, N, K, None, 0, None) == expect


@pytest.mark.parametrize("args,expect", [
    # X_host, ldx, W, S, Y_host, ldy, M, N, K, X_stage
    ((FAKE, 512, FAKE, FAKE, FAKE, 256, 0, 256, 512, FAKE), 0),       # M == 0: no-op
    ((FAKE, 512, FAKE, FAKE, FAKE, 256, 4, 256, 512, None), 1),       # null staging buffer
    ((FAKE, 512, FAKE, FAKE, FAKE, 256, 33, 256, 512, FAKE), 2),      # M > 32
    ((FAKE, 512, FAKE, FAKE, FAKE, 256, 4, 256, 512, FAKE + 8), 3),   # staging not 16-byte aligned
    ((FAKE + 8, 512, FAKE, FAKE, FAKE, 256, 4, 256, 512, FAKE), 3),   # X not 16-byte aligned
    # pointers the runtime does not know as pinned or device memory
    ((FAKE, 512, FAKE, FAKE, FAKE, 256, 4, 256, 512, FAKE), 1),
])
def test_fp8_host_entry_argument_validation(qg, args, expect):
    X, ldx, W, S, Y, ldy, M, N, K, stage = args
    assert qg.lib.qgemm_fp8_block_host(X, ldx, W, S, Y, ldy, M, N, K, stage, None, 0, None) == expect


@pytest.mark.parametrize("args,expect", [
    # X, ldx, Wq, qmap, scales, Y, ldy, M, N, K
    ((FAKE, 512, FAKE, FAKE, FAKE, FAKE, 256, 0, 256, 512), 0),
    ((None, 512, FAKE, FAKE, FAKE, FAKE, 256, 4, 256, 512), 1),
    ((FAKE, 512, FAKE, None, FAKE, FAKE, 256, 4, 256, 512), 1),
    ((FAKE, 512, FAKE, FAKE, FAKE, FAKE, 256, 40, 256, 512), 2),
    ((FAKE, 512, FAKE, FAKE, FAKE, FAKE, 256, 4, 256, 448), 2),   # K % 128
    ((FAKE, 512, FAKE + 8, FAKE, FAKE, FAKE, 256, 4, 256, 512), 3),
    ((FAKE, 512, FAKE, FAKE + 2, FAKE, FAKE, 256, 4, 256, 512), 3),
])
def test_lut3_argument_validation(qg, args, expect):
    X, ldx, Wq, qm, sc, Y, ldy, M, N, K = args
    assert qg.lib.qgemm_lut3(X, ldx, Wq, qm, sc, Y, ldy, M, N, K, None, 0, None) == expect


def test_dequant_entry_validation(qg):
    assert qg.lib.qg_debug_fp8_split(FAKE, 0, FAKE, FAKE, FAKE, None) == 0
    assert qg.lib.qg_debug_fp8_split(None, 4, FAKE, FAKE, FAKE, None) == 1
    assert qg.lib.qg_debug_fp8_split(FAKE, -1, FAKE, FAKE, FAKE, None) == 1
    assert qg.lib.qg_debug_fp8_split(FAKE + 8, 4, FAKE, FAKE, FAKE, None) == 3
    assert qg.lib.qg_dequant_lut3(FAKE, FAKE, FAKE, FAKE, 128, 200, None) == 2
    assert qg.lib.qg_dequant_lut3(None, FAKE, FAKE, FAKE, 128, 256, None) == 1


@pytest.mark.parametrize("N,K", [(128, 256), (256, 1024), (130, 384), (1, 128), (300, 640), (28672 // 64, 8192)])
def test_pack_matches_oracle_packer(qg, N, K):
    codes = wl.uniform_codes(1234 + N + K, N * K).reshape(N, K)
    ours = qg.pack_lut3(codes)
    ref = oracle.pack_lut3(codes)
    assert ours.size == qg.lut3_packed_bytes(N, K) == ref.size == oracle.lut3_packed_bytes(N, K)
    assert np.array_equal(ours, ref)
    assert np.array_equal(qg.unpack_lut3(ours, N, K), codes)
    assert np.array_equal(oracle.unpack_lut3(ours, N, K), codes)


def test_pack_rejects_wide_codes(qg):
    codes = np.zeros((128, 256), dtype=np.uint8)
    codes[5, 17] = 8
    with pytest.raises(qg.QgemmError) as e:
        qg.pack_lut3(codes)
    assert e.value.code == 1


def test_dispatch_and_schedule_argument_validation(qg):
    """The dispatch table and the schedule probe check their arguments before
    touching a device."""
    assert qg.lib.qg_dispatch_set(7, 16, 1024, 5120, 8) == 1       # unknown kind
    assert qg.lib.qg_dispatch_set(0, 0, 1024, 5120, 8) == 1        # M < 1
    assert qg.lib.qg_dispatch_set(0, 33, 1024, 5120, 8) == 1       # M > 32
    assert qg.lib.qg_dispatch_set(0, 16, 0, 5120, 8) == 1          # N < 1
    assert qg.lib.qg_dispatch_set(0, 16, 1024, 5120, -1) == 1      # negative grid
    assert qg.lib.qg_dispatch_get(7, 16, 1024, 5120) == 0
    assert qg.lib.qg_dispatch_get(0, 40, 1024, 5120) == 0
    g = ctypes.c_int(-1)
    assert qg.lib.qg_debug_schedule(0, 16, 1024, 5120, None, None, None, 0, None) == 1   # no count pointer
    assert qg.lib.qg_debug_schedule(0, 16, 1024, 5128, ctypes.byref(g), None, None, 0, None) == 2   # K % 16
    assert qg.lib.qg_debug_schedule(1, 16, 1024, 5120 + 64, ctypes.byref(g), None, None, 0, None) == 2
    qg.dispatch_clear()


def test_multi_argument_validation(qg):
    """qgemm_fp8_block_multi checks every segment before anything is enqueued."""
    segs = (qg.Fp8Segment * 5)()
    for j in range(5):
        segs[j] = qg.Fp8Segment(FAKE, FAKE, FAKE, 256, 256)
    ptr = ctypes.cast(segs, ctypes.c_void_p)
    fn = qg.lib.qgemm_fp8_block_multi
    assert fn(FAKE, 512, ptr, 0, 4, 512, None, 0, None) == 1      # no segments
    assert fn(FAKE, 512, ptr, 5, 4, 512, None, 0, None) == 1      # more than QG_MAX_SEGMENTS
    assert fn(FAKE, 512, None, 2, 4, 512, None, 0, None) == 1     # null table
    segs[1] = qg.Fp8Segment(None, FAKE, FAKE, 256, 256)
    assert fn(FAKE, 512, ptr, 3, 4, 512, None, 0, None) == 1      # null W in segment 1
    segs[1] = qg.Fp8Segment(FAKE + 4, FAKE, FAKE, 256, 256)
    assert fn(FAKE, 512, ptr, 3, 4, 512, None, 0, None) == 3      # misaligned W in segment 1
    segs[1] = qg.Fp8Segment(FAKE, FAKE, FAKE, 100, 256)
    assert fn(FAKE, 512, ptr, 3, 4, 512, None, 0, None) == 1      # ldy < N in segment 1
    segs[1] = qg.Fp8Segment(FAKE, FAKE, FAKE, 256, 0)
    assert fn(FAKE, 512, ptr, 3, 4, 512, None, 0, None) == 1      # empty segment
    segs[1] = qg.Fp8Segment(FAKE, FAKE, FAKE, 256, 256)
    assert fn(FAKE, 512, ptr, 3, 33, 512, None, 0, None) == 2     # M > 32
    assert fn(FAKE, 512, ptr, 3, 0, 512, None, 0, None) == 0      # M == 0: no-op


def test_tuner_argument_validation(qg):
    """The tuners check their arguments before touching a device."""
    P = ctypes.c_void_p
    ptrs = (P * 1)(FAKE)
    pp = ctypes.cast(ptrs, P)
    t = qg.lib.qg_tune_fp8
    assert t(FAKE, 512, None, 1, FAKE, FAKE, 256, FAKE, 4, 256, 512, None, 0, 10, None, None, None) == 1   # no copies
    assert t(FAKE, 512, pp, 0, FAKE, FAKE, 256, FAKE, 4, 256, 512, None, 0, 10, None, None, None) == 1     # ncopies 0
    assert t(FAKE, 512, pp, 1, FAKE, FAKE, 256, None, 4, 256, 512, None, 0, 10, None, None, None) == 1     # no Y_ref
    assert t(FAKE, 512, pp, 1, FAKE, FAKE, 256, FAKE, 4, 256, 512, None, 0, 0, None, None, None) == 1      # calls 0
    assert t(FAKE, 512, pp, 1, FAKE, FAKE, 256, FAKE, 33, 256, 512, None, 0, 10, None, None, None) == 2    # M > 32
    t3 = qg.lib.qg_tune_lut3
    assert t3(FAKE, 512, None, 1, FAKE, FAKE, FAKE, 256, FAKE, 4, 256, 512, None, 0, 10, None, None, None) == 1
    assert qg.lib.qg_workspace_bytes_max(0) == 0


@pytest.mark.parametrize("args,expect", [
    # X, ldx, W, Y, ldy, M, N, K
    ((FAKE, 512, FAKE, FAKE, 256, 0, 256, 512), 0),        # M == 0: no-op
    ((None, 512, FAKE, FAKE, 256, 4, 256, 512), 1),        # null X
    ((FAKE, 512, None, FAKE, 256, 4, 256, 512), 1),        # null W
    ((FAKE, 512, FAKE, FAKE, 256, 33, 256, 512), 2),       # M > 32
    ((FAKE, 516, FAKE, FAKE, 256, 4, 256, 516), 2),        # K % 8
    ((FAKE, 256, FAKE, FAKE, 256, 4, 256, 512), 1),        # ldx < K
    ((FAKE + 8, 512, FAKE, FAKE, 256, 4, 256, 512), 3),    # X not 16-byte aligned
    ((FAKE, 512, FAKE + 2, FAKE, 256, 4, 256, 512), 3),    # W not 16-byte aligned
])
def test_bf16_argument_validation(qg, args, expect):
    X, ldx, W, Y, ldy, M, N, K = args
    assert qg.lib.qgemm_bf16(X, ldx, W, Y, ldy, M, N, K, None, 0, None) == expect


@pytest.mark.parametrize("args,expect", [
    # X, ldx, Xq, ldxq, Sx, ldsx, M, K
    ((FAKE, 512, FAKE, 512, FAKE, 64, 0, 512), 0),              # M == 0: no-op
    ((None, 512, FAKE, 512, FAKE, 64, 4, 512), 1),              # null X
    ((FAKE, 512, None, 512, FAKE, 64, 4, 512), 1),              # null Xq
    ((FAKE, 512, FAKE, 512, None, 64, 4, 512), 1),              # null scales
    ((FAKE, 520, FAKE, 520, FAKE, 64, 4, 520), 2),              # K % 16
    ((FAKE, 512, FAKE, 512, FAKE, 64, 65537, 512), 2),          # M > 65536
    ((FAKE, 256, FAKE, 512, FAKE, 64, 4, 512), 1),              # ldx < K
    ((FAKE, 512, FAKE, 256, FAKE, 64, 4, 512), 1),              # ldxq < K
    ((FAKE, 512, FAKE, 512, FAKE, 32, 33, 512), 1),             # ldsx < M rounded up to 32
    ((FAKE + 8, 512, FAKE, 512, FAKE, 64, 4, 512), 3),          # X not 16-byte aligned
    ((FAKE, 512, FAKE, 520, FAKE, 64, 4, 512), 3),              # ldxq % 16
    ((FAKE, 512, FAKE, 512, FAKE, 66, 4, 512), 3),              # ldsx % 4
    ((FAKE, 512, FAKE, 512, FAKE + 4, 64, 4, 512), 3),          # scales not 16-byte aligned
])
def test_quantize_act_argument_validation(qg, args, expect):
    X, ldx, Xq, ldxq, Sx, ldsx, M, K = args
    assert qg.lib.qg_quantize_act_e4m3(X, ldx, Xq, ldxq, Sx, ldsx, M, K, None) == expect


@pytest.mark.parametrize("args,expect", [
    # Xq, ldxq, Sx, ldsx, W, S, Y, ldy, M, N, K
    ((FAKE, 512, FAKE, 64, FAKE, FAKE, FAKE, 256, 0, 256, 512), 0),        # M == 0: no-op
    ((None, 512, FAKE, 64, FAKE, FAKE, FAKE, 256, 40, 256, 512), 1),       # null Xq
    ((FAKE, 512, None, 64, FAKE, FAKE, FAKE, 256, 40, 256, 512), 1),       # null X scales
    ((FAKE, 512, FAKE, 64, None, FAKE, FAKE, 256, 40, 256, 512), 1),       # null W
    ((FAKE, 512, FAKE, 64, FAKE, FAKE, None, 256, 40, 256, 512), 1),       # null Y
    ((FAKE, 520, FAKE, 64, FAKE, FAKE, FAKE, 256, 40, 256, 520), 2),       # K % 16
    ((FAKE, 512, FAKE, 65536, FAKE, FAKE, FAKE, 256, 65537, 256, 512), 2), # M > 65536
    ((FAKE, 512, FAKE, 32, FAKE, FAKE, FAKE, 256, 40, 256, 512), 1),       # ldsx < 64
    ((FAKE, 512, FAKE, 64, FAKE, FAKE, FAKE, 200, 40, 256, 512), 1),       # ldy < N
    ((FAKE + 16, 520, FAKE, 64, FAKE, FAKE, FAKE, 256, 40, 256, 512), 3),  # ldxq % 16
    ((FAKE, 512, FAKE + 4, 64, FAKE, FAKE, FAKE, 256, 40, 256, 512), 3),   # X scales alignment
    ((FAKE, 512, FAKE, 64, FAKE + 8, FAKE, FAKE, 256, 40, 256, 512), 3),   # W alignment
    ((FAKE, 512, FAKE, 64, FAKE, FAKE + 2, FAKE, 256, 40, 256, 512), 3),   # W scales alignment
    ((FAKE, 512, FAKE, 64, FAKE, FAKE, FAKE + 1, 256, 40, 256, 512), 3),   # Y alignment
])
def test_w8a8_argument_validation(qg, args, expect):
    Xq, ldxq, Sx, ldsx, W, S, Y, ldy, M, N, K = args
    assert qg.lib.qgemm_w8a8_block(Xq, ldxq, Sx, ldsx, W, S, Y, ldy, M, N, K, None, 0, None) == expect


def test_w8a8_dispatch_accepts_large_m(qg):
    """The W8A8 kind takes M up to 65536 in the dispatch table's checks."""
    assert qg.lib.qg_dispatch_set(qg.KIND_W8A8, 65537, 1024, 5120, 8) == 1
    assert qg.lib.qg_dispatch_set(qg.KIND_W8A8, 256, 1024, 5120, -1) == 1
    assert qg.lib.qg_dispatch_get(qg.KIND_W8A8, 0, 1024, 5120) == 0
    assert qg.lib.qg_workspace_bytes(qg.KIND_W8A8, 65537, 1024, 5120) == 0


def test_bf16_and_w8a8_tuner_argument_validation(qg):
    """The BF16 and W8A8 tuners check their arguments before touching a device."""
    P = ctypes.c_void_p
    ptrs = (P * 1)(FAKE)
    pp = ctypes.cast(ptrs, P)
    t = qg.lib.qg_tune_bf16
    assert t(FAKE, 512, None, 1, FAKE, 256, FAKE, 4, 256, 512, None, 0, 10, None, None, None) == 1   # no copies
    assert t(FAKE, 512, pp, 0, FAKE, 256, FAKE, 4, 256, 512, None, 0, 10, None, None, None) == 1     # ncopies 0
    assert t(FAKE, 512, pp, 1, FAKE, 256, None, 4, 256, 512, None, 0, 10, None, None, None) == 1     # no Y_ref
    assert t(FAKE, 512, pp, 1, FAKE, 256, FAKE, 4, 256, 512, None, 0, 0, None, None, None) == 1      # calls 0
    assert t(FAKE, 512, pp, 1, FAKE, 256, FAKE, 33, 256, 512, None, 0, 10, None, None, None) == 2    # M > 32
    w = qg.lib.qg_tune_w8a8
    assert w(FAKE, 512, FAKE, 64, None, 1, FAKE, FAKE, 256, FAKE, 40, 256, 512, None, 0, 10, None, None, None) == 1
    assert w(FAKE, 512, FAKE, 64, pp, 1, FAKE, FAKE, 256, FAKE, 40, 256, 512, None, 0, 0, None, None, None) == 1
    assert w(FAKE, 512, FAKE, 64, pp, 1, FAKE, FAKE, 256, None, 40, 256, 512, None, 0, 10, None, None, None) == 1
    assert w(FAKE, 512, FAKE, 64, pp, 1, FAKE, FAKE, 256, FAKE, 65537, 256, 512, None, 0, 10, None, None,
             None) == 2
    assert qg.lib.qg_workspace_bytes_max_w8a8(0, 256) == 0
    assert qg.lib.qg_workspace_bytes_max_w8a8(64, 0) == 0


# ------------------------------------------------------------------ dispatch rule (host only)
# The built-in rule on a 152-SM GB300 against the grids the exactness-gated
# tuner picked when it timed every candidate on the GPU (the bench's tuned
# lines): the rule was set from those measurements and should keep matching.
@pytest.mark.parametrize("kind,M,N,K,grid", [
    (0, 16, 17408, 5120, 136), (0, 1, 17408, 5120, 136),        # gate/up: one CTA per tile
    (0, 16, 5120, 17408, 120), (0, 32, 5120, 17408, 152),       # down: 3 per tile; stream-K at 32 rows
    (0, 16, 6144, 5120, 144), (0, 16, 5120, 5120, 120), (0, 16, 1024, 5120, 64),
    (1, 16, 28672, 8192, 152),                                  # LUT3: stream-K over 224 tiles
    (2, 16, 32768, 5120, 128),                                  # BF16 lm_head: two whole tiles per CTA
    (3, 64, 17408, 5120, 136), (3, 256, 17408, 5120, 136), (3, 1024, 17408, 5120, 152),
])
def test_dispatch_rule_matches_the_tuned_grids(qg, kind, M, N, K, grid):
    assert qg.dispatch_rule(kind, M, N, K, 152) == grid


def test_dispatch_rule_invariants(qg):
    """Every grid is 1 .. min(SMs, work units); with more tiles than SMs a
    grid below the SM count holds whole tiles only; with tiles <= SMs the
    grid is one CTA per tile, a whole multiple of the tiles, or one CTA per
    SM; invalid arguments give 0."""
    for kind, Ms, kmul in ((0, (1, 16, 17, 32), 16), (1, (1, 16, 32), 128), (2, (1, 32), 8), (3, (33, 64, 65, 300, 4096), 16)):
        for M in Ms:
            for N in (128, 200, 1024, 5120, 17408, 32768, 65536):
                for K in (kmul, 1024, 5120, 17408):
                    if K % kmul:
                        continue
                    rows = (64 if M <= 64 else 128) if kind == 3 else None
                    T = -(-N // 128) * (-(-M // rows) if rows else 1)
                    KU = -(-K // 256) if kind == 3 else -(-K // 128)
                    U = T * KU
                    for sms in (1, 8, 76, 148, 152, 160):
                        g = qg.dispatch_rule(kind, M, N, K, sms)
                        assert 1 <= g <= min(sms, U), (kind, M, N, K, sms, g)
                        if T > sms and g < sms:
                            assert T % g == 0, (kind, M, N, K, sms, g)
                        if T <= sms:
                            assert g == min(sms, U) or g % T == 0, (kind, M, N, K, sms, g)
    assert qg.dispatch_rule(0, 0, 128, 128, 152) == 0
    assert qg.dispatch_rule(0, 33, 128, 128, 152) == 0
    assert qg.dispatch_rule(0, 1, 128, 128, 0) == 0
    assert qg.dispatch_rule(9, 1, 128, 128, 152) == 0
