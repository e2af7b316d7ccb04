"""Python binding of libqgemm (weight-only quantized decode GEMMs for GB300).

Argument marshalling only: every step of the GEMM runs in the library's CUDA
kernels.  PyTorch provides device memory and the current stream.  If the
compiled library is missing this module raises on import; there is no
fallback implementation.

The names follow the C ABI in ``include/qgemm.h``:

* :func:`qgemm_fp8_block` -- W8A16 FP8 E4M3 weights with [128 x 128] FP32
  block scales, BF16 activations and output, two-level FP32 fold.
* :func:`qgemm_fp8_block_multi` -- several of those GEMMs sharing X (e.g. the
  Q, K and V projections) in one launch, each with its own output.
* :func:`qgemm_fp8_block_host` -- the same GEMM with X and Y in pinned host
  memory (staged in and stored out by the library's kernels).
* :func:`qgemm_lut3` -- 3-bit learned-LUT weights (see :func:`pack_lut3`),
  FP16 activations and output.
* :func:`qgemm_bf16` -- unquantised BF16 weights (e.g. an lm_head), BF16
  activations and output.
* :func:`quantize_act_e4m3` / :func:`qgemm_w8a8_block` -- the W8A8 path for
  larger batches: BF16 activations quantised to E4M3 per (row, 128-wide K
  block) with FP32 scales, then an E4M3 x E4M3 block-scaled GEMM
  (:func:`qgemm_w8a8` runs both).
* :func:`pack_lut3` / :func:`unpack_lut3` -- offline nibble packer (host).
* :func:`debug_fp8_split` / :func:`dequant_lut3` -- test aids: the FP8
  kernel's activation split and the LUT3 kernel's dequantiser on their own,
  exposed for value-by-value checks.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

__all__ = [
    "QgemmError", "LIB_PATH", "lib", "status_string", "workspace_bytes", "Workspace",
    "qgemm_fp8_block", "qgemm_fp8_block_multi", "qgemm_fp8_block_host", "Fp8Segment", "MAX_SEGMENTS", "qgemm_lut3", "pack_lut3", "unpack_lut3", "lut3_packed_bytes",
    "debug_fp8_split", "dequant_lut3", "last_device_status", "set_wait_timeout_ns",
    "set_fault_injection", "set_weight_prefetch_overlap", "dispatch_set", "dispatch_get", "dispatch_rule", "dispatch_clear",
    "debug_schedule", "tune_fp8", "tune_lut3", "workspace_bytes_max", "qgemm_bf16", "KIND_BF16", "KIND_FP8_BLOCK", "KIND_LUT3", "STATUS",
    "quantize_act_e4m3", "qgemm_w8a8_block", "qgemm_w8a8", "KIND_W8A8", "MAX_M_W8A8",
    "tune_bf16", "tune_w8a8", "workspace_bytes_max_w8a8",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqgemm.so")

KIND_FP8_BLOCK = 0
KIND_LUT3 = 1
KIND_BF16 = 2
KIND_W8A8 = 3
MAX_M_W8A8 = 65536
STATUS = {
    0: "QG_OK", 1: "QG_ERR_INVALID_ARG", 2: "QG_ERR_UNSUPPORTED_SHAPE", 3: "QG_ERR_MISALIGNED",
    4: "QG_ERR_CUDA", 5: "QG_ERR_TIMEOUT", 6: "QG_ERR_WORKSPACE",
}


class QgemmError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)} ({status_string(code)})")


if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libqgemm.so not found at {LIB_PATH}; build it first with "
        "`python -c 'import __graft_entry__ as g; g.build()'` from the repository root (needs nvcc)")

_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_int64
_S = ctypes.c_size_t

lib = ctypes.CDLL(LIB_PATH)
_SIGS = {
    "qg_workspace_bytes": (_S, [_I, _I, _I, _I]),
    "qgemm_fp8_block": (_I, [_P, _L, _P, _P, _P, _L, _I, _I, _I, _P, _S, _P]),
    "qgemm_fp8_block_multi": (_I, [_P, _L, _P, _I, _I, _I, _P, _S, _P]),
    "qgemm_fp8_block_host": (_I, [_P, _L, _P, _P, _P, _L, _I, _I, _I, _P, _P, _S, _P]),
    "qgemm_lut3": (_I, [_P, _L, _P, _P, _P, _P, _L, _I, _I, _I, _P, _S, _P]),
    "qgemm_bf16": (_I, [_P, _L, _P, _P, _L, _I, _I, _I, _P, _S, _P]),
    "qg_quantize_act_e4m3": (_I, [_P, _L, _P, _L, _P, _L, _I, _I, _P]),
    "qgemm_w8a8_block": (_I, [_P, _L, _P, _L, _P, _P, _P, _L, _I, _I, _I, _P, _S, _P]),
    "qg_lut3_packed_bytes": (_S, [_I, _I]),
    "pack_lut3": (_I, [_P, _P, _I, _I]),
    "unpack_lut3": (_I, [_P, _P, _I, _I]),
    "qg_debug_fp8_split": (_I, [_P, _L, _P, _P, _P, _P]),
    "qg_debug_schedule": (_I, [_I, _I, _I, _I, _P, _P, _P, _I, _P]),
    "qg_dispatch_set": (_I, [_I, _I, _I, _I, _I]),
    "qg_dispatch_get": (_I, [_I, _I, _I, _I]),
    "qg_dispatch_rule": (_I, [_I, _I, _I, _I, _I]),
    "qg_dispatch_clear": (None, []),
    "qg_workspace_bytes_max": (_S, [_I]),
    "qg_workspace_bytes_max_w8a8": (_S, [_I, _I]),
    "qg_tune_bf16": (_I, [_P, _L, _P, _I, _P, _L, _P, _I, _I, _I, _P, _S, _I, _P, _P, _P]),
    "qg_tune_w8a8": (_I, [_P, _L, _P, _L, _P, _I, _P, _P, _L, _P, _I, _I, _I, _P, _S, _I, _P, _P, _P]),
    "qg_tune_fp8": (_I, [_P, _L, _P, _I, _P, _P, _L, _P, _I, _I, _I, _P, _S, _I, _P, _P, _P]),
    "qg_tune_lut3": (_I, [_P, _L, _P, _I, _P, _P, _P, _L, _P, _I, _I, _I, _P, _S, _I, _P, _P, _P]),
    "qg_dequant_lut3": (_I, [_P, _P, _P, _P, _I, _I, _P]),
    "qg_last_device_status": (_I, [_P]),
    "qg_set_wait_timeout_ns": (None, [ctypes.c_uint64]),
    "qg_set_fault_injection": (None, [_I]),
    "qg_set_weight_prefetch_overlap": (None, [_I]),
    "qg_status_string": (ctypes.c_char_p, [_I]),
    "qg_version": (ctypes.c_char_p, []),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


def status_string(code: int) -> str:
    return lib.qg_status_string(int(code)).decode()


def _check(code: int, where: str) -> None:
    if code != 0:
        raise QgemmError(code, where)


def _torch():
    import torch
    return torch


def _stream_ptr(stream) -> int:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def workspace_bytes(kind: int, M: int, N: int, K: int) -> int:
    """Device workspace a call needs on the current device (may be 0)."""
    return int(lib.qg_workspace_bytes(kind, M, N, K))


class Workspace:
    """A zero-filled device byte buffer that grows on demand.  Calls leave
    its arrival counters at zero again (the partial-sum area in front of them
    is scratch), so one buffer serves any sequence of calls on one stream
    (calls that may run at the same time, on different streams, need one
    buffer each).  Growing synchronises the device, so that no call still
    uses the old buffer and the zero fill has landed before any stream uses
    the new one."""

    def __init__(self, device=None):
        self.device = device
        self.buf = None

    def get(self, nbytes: int):
        torch = _torch()
        if nbytes == 0:
            return None
        if self.buf is None or self.buf.numel() < nbytes:
            dev = self.device or torch.cuda.current_device()
            if self.buf is not None:
                torch.cuda.synchronize(dev)
            self.buf = torch.zeros(max(nbytes, 1 << 20), dtype=torch.uint8, device=dev)
            torch.cuda.synchronize(dev)
        return self.buf

    def reset(self):
        if self.buf is not None:
            self.buf.zero_()


_default_ws = {}


_ws_need = {}


def _workspace_for(kind, M, N, K, workspace, device, stream=None):
    key = (kind, M, N, K, device)
    need = _ws_need.get(key)
    if need is None:
        need = _ws_need[key] = workspace_bytes(kind, M, N, K)
    if need == 0:
        return None, 0
    if workspace is None:
        # one default buffer per device, stream (calls on different streams may
        # overlap) and layout family (the W8A8 kind's differs from the others')
        key = (device, _stream_ptr(stream), kind == KIND_W8A8)
        workspace = _default_ws.get(key)
        if workspace is None:
            workspace = _default_ws[key] = Workspace(device)
    buf = workspace.get(need) if isinstance(workspace, Workspace) else workspace
    return buf.data_ptr(), buf.numel() * buf.element_size()


def _ld(t) -> int:
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("expected a 2-D tensor with unit stride in its last dimension")
    return t.stride(0)


def qgemm_fp8_block(X, W, W_scale, Y=None, workspace=None, stream=None):
    """Y[M, N] = X[M, K] . dequant(W)[N, K]^T (BF16 out).

    X: bf16 CUDA [M, K] (row stride a multiple of 8); W: uint8 (E4M3 codes) or
    float8_e4m3fn [N, K] contiguous; W_scale: float32 [ceil(N/128), ceil(K/128)]
    contiguous.  Y (optional): bf16 [M, N] with unit column stride.
    """
    torch = _torch()
    if X.dtype != torch.bfloat16:
        raise TypeError("X must be bfloat16")
    if W.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise TypeError("W must hold E4M3 codes (uint8 or float8_e4m3fn)")
    if W_scale.dtype != torch.float32 or not W_scale.is_contiguous() or not W.is_contiguous():
        raise TypeError("W must be contiguous and W_scale contiguous float32")
    M, K = X.shape
    N = W.shape[0]
    if W.shape[1] != K or tuple(W_scale.shape) != (-(-N // 128), -(-K // 128)):
        raise ValueError("shape mismatch between X, W and W_scale")
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    ws, wsb = _workspace_for(KIND_FP8_BLOCK, M, N, K, workspace, X.device, stream)
    _check(lib.qgemm_fp8_block(X.data_ptr(), _ld(X), W.data_ptr(), W_scale.data_ptr(), Y.data_ptr(),
                               _ld(Y), M, N, K, ws, wsb, _stream_ptr(stream)), "qgemm_fp8_block")
    return Y


MAX_SEGMENTS = 4


class Fp8Segment(ctypes.Structure):
    """qg_fp8_segment of include/qgemm.h."""
    _fields_ = [("W", ctypes.c_void_p), ("W_scale", ctypes.c_void_p), ("Y", ctypes.c_void_p),
                ("ldy", ctypes.c_int64), ("N", ctypes.c_int)]


def qgemm_fp8_block_multi(X, weights, Ys=None, workspace=None, stream=None):
    """Y_j = X . dequant(W_j)^T for every (W_j, W_scale_j) in `weights`
    (1 to MAX_SEGMENTS of them, sharing X), in one launch; returns the list of
    Y_j (BF16 [M, N_j]).  Ys (optional): the output tensors, each with unit
    column stride."""
    torch = _torch()
    if X.dtype != torch.bfloat16:
        raise TypeError("X must be bfloat16")
    if not 1 <= len(weights) <= MAX_SEGMENTS:
        raise ValueError(f"between 1 and {MAX_SEGMENTS} weight matrices")
    M, K = X.shape
    segs = (Fp8Segment * len(weights))()
    outs = []
    rows = 0
    for j, (W, S) in enumerate(weights):
        if W.dtype not in (torch.uint8, torch.float8_e4m3fn) or not W.is_contiguous():
            raise TypeError("W must hold contiguous E4M3 codes (uint8 or float8_e4m3fn)")
        N = W.shape[0]
        if W.shape[1] != K or tuple(S.shape) != (-(-N // 128), -(-K // 128)) or S.dtype != torch.float32 \
                or not S.is_contiguous():
            raise ValueError(f"segment {j}: shape mismatch between X, W and W_scale")
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device) if Ys is None else Ys[j]
        outs.append(Y)
        segs[j] = Fp8Segment(W.data_ptr(), S.data_ptr(), Y.data_ptr(), _ld(Y), N)
        rows += -(-N // 128) * 128
    ws, wsb = _workspace_for(KIND_FP8_BLOCK, M, rows, K, workspace, X.device, stream)
    _check(lib.qgemm_fp8_block_multi(X.data_ptr(), _ld(X), ctypes.cast(segs, ctypes.c_void_p), len(weights), M, K,
                                     ws, wsb, _stream_ptr(stream)), "qgemm_fp8_block_multi")
    return outs


_default_stage = {}


def qgemm_fp8_block_host(X, W, W_scale, Y=None, X_stage=None, workspace=None, stream=None):
    """:func:`qgemm_fp8_block` with X and Y in pinned host memory.

    X: bf16 CPU [M, K], pinned (``tensor.pin_memory()``), row stride a
    multiple of 8; Y (optional, allocated pinned if absent): bf16 CPU [M, N],
    pinned, unit column stride.  W and W_scale are on the device as for
    :func:`qgemm_fp8_block`.  X_stage (optional): a device buffer of at least
    M*K bf16 elements that the call copies X into; a per-device buffer is
    kept when absent.  The call is asynchronous: Y is complete after the
    stream is synchronised.
    """
    torch = _torch()
    if X.dtype != torch.bfloat16:
        raise TypeError("X must be bfloat16")
    if W.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise TypeError("W must hold E4M3 codes (uint8 or float8_e4m3fn)")
    if W_scale.dtype != torch.float32 or not W_scale.is_contiguous() or not W.is_contiguous():
        raise TypeError("W must be contiguous and W_scale contiguous float32")
    if X.is_cuda or not X.is_pinned():
        raise ValueError("X must be a pinned host tensor")
    M, K = X.shape
    N = W.shape[0]
    if W.shape[1] != K or tuple(W_scale.shape) != (-(-N // 128), -(-K // 128)):
        raise ValueError("shape mismatch between X, W and W_scale")
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    elif Y.dtype != torch.bfloat16 or Y.is_cuda or not Y.is_pinned():
        raise ValueError("Y must be a pinned bfloat16 host tensor")
    if X_stage is None:
        X_stage = _default_stage.get(W.device)
        if X_stage is None or X_stage.numel() < M * K:
            X_stage = _default_stage[W.device] = torch.empty(max(M * K, 1 << 16), dtype=torch.bfloat16,
                                                             device=W.device)
    elif not X_stage.is_cuda or X_stage.numel() * X_stage.element_size() < M * K * 2:
        raise ValueError("X_stage must be a device buffer of at least M*K bfloat16 elements")
    ws, wsb = _workspace_for(KIND_FP8_BLOCK, M, N, K, workspace, W.device, stream)
    _check(lib.qgemm_fp8_block_host(X.data_ptr(), _ld(X), W.data_ptr(), W_scale.data_ptr(), Y.data_ptr(),
                                    _ld(Y), M, N, K, X_stage.data_ptr(), ws, wsb, _stream_ptr(stream)),
           "qgemm_fp8_block_host")
    return Y


def qgemm_lut3(X, Wq, qmap, scales, N: int, Y=None, workspace=None, stream=None):
    """Y[M, N] = X[M, K] . dequant(Wq)^T with the 3-bit learned-LUT format (FP16 out).

    X: fp16 CUDA [M, K]; Wq: the packed bytes from :func:`pack_lut3` on the
    device; qmap: fp16 [8]; scales: fp16 [N, K/128] contiguous.
    """
    torch = _torch()
    if X.dtype != torch.float16 or qmap.dtype != torch.float16 or scales.dtype != torch.float16:
        raise TypeError("X, qmap and scales must be float16")
    M, K = X.shape
    if tuple(scales.shape) != (N, K // 128) or not scales.is_contiguous():
        raise ValueError("scales must be a contiguous [N, K/128] tensor")
    if Wq.numel() * Wq.element_size() < lut3_packed_bytes(N, K):
        raise ValueError("packed weights are smaller than pack_lut3 produces for this shape")
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float16, device=X.device)
    ws, wsb = _workspace_for(KIND_LUT3, M, N, K, workspace, X.device, stream)
    _check(lib.qgemm_lut3(X.data_ptr(), _ld(X), Wq.data_ptr(), qmap.data_ptr(), scales.data_ptr(),
                          Y.data_ptr(), _ld(Y), M, N, K, ws, wsb, _stream_ptr(stream)), "qgemm_lut3")
    return Y


def quantize_act_e4m3(X, Xq=None, X_scale=None, stream=None):
    """E4M3 codes and FP32 scales of BF16 activations, per (row, 128-wide K
    block): scale = block max |x| / 448 (1 for a zero block), code =
    e4m3_rne_satfinite(x / scale).

    X: bf16 CUDA [M, K] (row stride a multiple of 8, K % 16 == 0).  Returns
    (Xq uint8 [M, K] (a view with row stride rounded up to 16), X_scale
    float32 [ceil(K/128), ldsx] with ldsx = M rounded up to 32; columns
    [M, ldsx) are 0).  Xq and X_scale (optional) are written in place.
    """
    torch = _torch()
    if X.dtype != torch.bfloat16:
        raise TypeError("X must be bfloat16")
    M, K = X.shape
    KB = -(-K // 128)
    if Xq is None:
        Xq = torch.empty((M, -(-K // 16) * 16), dtype=torch.uint8, device=X.device)[:, :K]
    if X_scale is None:
        X_scale = torch.empty((KB, max(32, -(-M // 32) * 32)), dtype=torch.float32, device=X.device)
    if Xq.dtype not in (torch.uint8, torch.float8_e4m3fn) or X_scale.dtype != torch.float32:
        raise TypeError("Xq must be uint8 or float8_e4m3fn, X_scale float32")
    if tuple(Xq.shape) != (M, K) or X_scale.shape[0] != KB:
        raise ValueError("shape mismatch between X, Xq and X_scale")
    _check(lib.qg_quantize_act_e4m3(X.data_ptr(), _ld(X), Xq.data_ptr(), _ld(Xq), X_scale.data_ptr(),
                                    _ld(X_scale), M, K, _stream_ptr(stream)), "qg_quantize_act_e4m3")
    return Xq, X_scale


def qgemm_w8a8_block(Xq, X_scale, W, W_scale, Y=None, workspace=None, stream=None):
    """Y[M, N] = sum over 128-wide K blocks kb of X_scale[kb, m] *
    W_scale[n/128, kb] * (Xq[m, kb] . W[n, kb]) (E4M3 x E4M3, FP32 fold, BF16
    out), with Xq, X_scale as :func:`quantize_act_e4m3` returns them."""
    torch = _torch()
    if Xq.dtype not in (torch.uint8, torch.float8_e4m3fn) or W.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise TypeError("Xq and W must hold E4M3 codes (uint8 or float8_e4m3fn)")
    if X_scale.dtype != torch.float32 or W_scale.dtype != torch.float32:
        raise TypeError("X_scale and W_scale must be float32")
    if not W.is_contiguous() or not W_scale.is_contiguous():
        raise TypeError("W and W_scale must be contiguous")
    M, K = Xq.shape
    N = W.shape[0]
    if W.shape[1] != K or tuple(W_scale.shape) != (-(-N // 128), -(-K // 128)) or X_scale.shape[0] != -(-K // 128):
        raise ValueError("shape mismatch between Xq, X_scale, W and W_scale")
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=Xq.device)
    ws, wsb = _workspace_for(KIND_W8A8, M, N, K, workspace, Xq.device, stream)
    _check(lib.qgemm_w8a8_block(Xq.data_ptr(), _ld(Xq), X_scale.data_ptr(), _ld(X_scale), W.data_ptr(),
                                W_scale.data_ptr(), Y.data_ptr(), _ld(Y), M, N, K, ws, wsb, _stream_ptr(stream)),
           "qgemm_w8a8_block")
    return Y


def qgemm_w8a8(X, W, W_scale, Y=None, workspace=None, stream=None):
    """The W8A8 path from BF16 activations: :func:`quantize_act_e4m3` then
    :func:`qgemm_w8a8_block` (two launches on one stream)."""
    Xq, X_scale = quantize_act_e4m3(X, stream=stream)
    return qgemm_w8a8_block(Xq, X_scale, W, W_scale, Y=Y, workspace=workspace, stream=stream)


def qgemm_bf16(X, W, Y=None, workspace=None, stream=None):
    """Y[M, N] = X[M, K] . W[N, K]^T with BF16 X, W and Y (FP32 sums).

    X: bf16 CUDA [M, K] (row stride a multiple of 8); W: bf16 [N, K]
    contiguous; Y (optional): bf16 [M, N] with unit column stride.
    """
    torch = _torch()
    if X.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
        raise TypeError("X and W must be bfloat16")
    if not W.is_contiguous():
        raise TypeError("W must be contiguous")
    M, K = X.shape
    N = W.shape[0]
    if W.shape[1] != K:
        raise ValueError("shape mismatch between X and W")
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    ws, wsb = _workspace_for(KIND_BF16, M, N, K, workspace, X.device, stream)
    _check(lib.qgemm_bf16(X.data_ptr(), _ld(X), W.data_ptr(), Y.data_ptr(), _ld(Y), M, N, K, ws, wsb,
                          _stream_ptr(stream)), "qgemm_bf16")
    return Y


def lut3_packed_bytes(N: int, K: int) -> int:
    return int(lib.qg_lut3_packed_bytes(N, K))


def pack_lut3(codes: np.ndarray) -> np.ndarray:
    """Pack an [N, K] uint8 matrix of 3-bit codes (host) into the kernel layout."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    N, K = c.shape
    out = np.empty(lut3_packed_bytes(N, K), dtype=np.uint8)
    _check(lib.pack_lut3(c.ctypes.data, out.ctypes.data, N, K), "pack_lut3")
    return out


def unpack_lut3(packed: np.ndarray, N: int, K: int) -> np.ndarray:
    p = np.ascontiguousarray(packed, dtype=np.uint8)
    if p.size < lut3_packed_bytes(N, K):
        raise ValueError("packed buffer too small")
    out = np.empty((N, K), dtype=np.uint8)
    _check(lib.unpack_lut3(p.ctypes.data, out.ctypes.data, N, K), "unpack_lut3")
    return out


def debug_fp8_split(X, stream=None):
    """The FP8 GEMM's activation split of BF16 X [B, 128] (one 128-wide K
    block per row): returns (hi, lo, e) with hi, lo uint8 E4M3 codes [B, 128]
    and e int32 [B], such that x * 2^e = hi + lo / 16 (see include/qgemm.h)."""
    torch = _torch()
    if X.dtype != torch.bfloat16 or X.dim() != 2 or X.shape[1] != 128 or not X.is_contiguous():
        raise ValueError("X must be a contiguous bfloat16 [B, 128] tensor")
    B = X.shape[0]
    hi = torch.empty((B, 128), dtype=torch.uint8, device=X.device)
    lo = torch.empty((B, 128), dtype=torch.uint8, device=X.device)
    e = torch.empty((B,), dtype=torch.int32, device=X.device)
    _check(lib.qg_debug_fp8_split(X.data_ptr(), B, hi.data_ptr(), lo.data_ptr(), e.data_ptr(), _stream_ptr(stream)),
           "qg_debug_fp8_split")
    return hi, lo, e


def dequant_lut3(Wq, qmap, scales, N: int, K: int, out=None, stream=None):
    """Packed LUT3 weights -> FP16 [N, K], with the LUT3 GEMM's own dequantiser."""
    torch = _torch()
    if out is None:
        out = torch.empty((N, K), dtype=torch.float16, device=Wq.device)
    _check(lib.qg_dequant_lut3(Wq.data_ptr(), qmap.data_ptr(), scales.data_ptr(), out.data_ptr(), N, K,
                               _stream_ptr(stream)), "qg_dequant_lut3")
    return out


def last_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the kernels' status code."""
    return int(lib.qg_last_device_status(_stream_ptr(stream)))


def set_wait_timeout_ns(ns: int) -> None:
    lib.qg_set_wait_timeout_ns(int(ns))


def set_fault_injection(unit: int) -> None:
    lib.qg_set_fault_injection(int(unit))


def set_weight_prefetch_overlap(enable: bool) -> None:
    """Let consecutive GEMMs on a stream overlap (weights stream early); see
    include/qgemm.h for the condition under which this is safe."""
    lib.qg_set_weight_prefetch_overlap(1 if enable else 0)


def dispatch_set(kind: int, M: int, N: int, K: int, ctas: int) -> None:
    """Set (ctas > 0) or remove (ctas == 0) the dispatch-table grid of a shape."""
    _check(lib.qg_dispatch_set(kind, M, N, K, ctas), "qg_dispatch_set")
    _ws_need.clear()   # a shape's workspace need follows its grid


def dispatch_get(kind: int, M: int, N: int, K: int) -> int:
    """The grid (CTA count) the next call of this shape launches."""
    return int(lib.qg_dispatch_get(kind, M, N, K))


def dispatch_rule(kind: int, M: int, N: int, K: int, sms: int) -> int:
    """The grid the built-in cost rule picks for this shape on a device with
    `sms` SMs, ignoring the dispatch table (host only; 0 for invalid
    arguments)."""
    return int(lib.qg_dispatch_rule(kind, M, N, K, sms))


def dispatch_clear() -> None:
    lib.qg_dispatch_clear()
    _ws_need.clear()


def debug_schedule(kind: int, M: int, N: int, K: int, stream=None):
    """The device's work split of a shape: (ranges int64 [G, 2], info int32
    [G, 6]) as numpy arrays (see include/qgemm.h)."""
    torch = _torch()
    g = ctypes.c_int(0)
    _check(lib.qg_debug_schedule(kind, M, N, K, ctypes.byref(g), None, None, 0, None), "qg_debug_schedule")
    G = g.value
    ranges = torch.empty((G, 2), dtype=torch.int64, device="cuda")
    info = torch.empty((G, 6), dtype=torch.int32, device="cuda")
    _check(lib.qg_debug_schedule(kind, M, N, K, ctypes.byref(g), ranges.data_ptr(), info.data_ptr(), G,
                                 _stream_ptr(stream)), "qg_debug_schedule")
    torch.cuda.synchronize()
    return ranges.cpu().numpy(), info.cpu().numpy()


def workspace_bytes_max(N: int) -> int:
    """The workspace any grid of a shape with N output rows may need."""
    return int(lib.qg_workspace_bytes_max(N))


def _tune_common(M, N, X, Y_ref, workspace, nbytes=None):
    if workspace is None:
        workspace = Workspace(X.device)
    need = workspace_bytes_max(N) if nbytes is None else nbytes
    buf = workspace.get(need) if isinstance(workspace, Workspace) else workspace
    return buf, (buf.numel() * buf.element_size() if buf is not None else 0)


def tune_fp8(X, W_copies, W_scale, calls: int = 200, workspace=None, stream=None):
    """Exactness-gated tuning of the dispatch table for the shape of X and W
    (see qg_tune_fp8 in include/qgemm.h).  W_copies: equal E4M3 weight
    tensors the timed calls rotate over.  Returns (grid, us per call)."""
    torch = _torch()
    M, K = X.shape
    N = W_copies[0].shape[0]
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    Y_ref = torch.empty_like(Y)
    buf, nb = _tune_common(M, N, X, Y_ref, workspace)
    ptrs = (ctypes.c_void_p * len(W_copies))(*[w.data_ptr() for w in W_copies])
    g, us = ctypes.c_int(0), ctypes.c_float(0)
    _check(lib.qg_tune_fp8(X.data_ptr(), _ld(X), ctypes.cast(ptrs, ctypes.c_void_p), len(W_copies),
                           W_scale.data_ptr(), Y.data_ptr(), N, Y_ref.data_ptr(), M, N, K,
                           buf.data_ptr() if buf is not None else None, nb, calls, ctypes.byref(g), ctypes.byref(us),
                           _stream_ptr(stream)), "qg_tune_fp8")
    _ws_need.clear()
    return g.value, us.value


def workspace_bytes_max_w8a8(M: int, N: int) -> int:
    """The largest workspace any grid of a W8A8 shape with M activation rows
    and N output rows may need on the current device."""
    return int(lib.qg_workspace_bytes_max_w8a8(M, N))


def tune_bf16(X, W_copies, calls: int = 200, workspace=None, stream=None):
    """As tune_fp8 for the dense BF16 GEMM (W_copies: equal BF16 weights)."""
    torch = _torch()
    M, K = X.shape
    N = W_copies[0].shape[0]
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    Y_ref = torch.empty_like(Y)
    buf, nb = _tune_common(M, N, X, Y_ref, workspace)
    ptrs = (ctypes.c_void_p * len(W_copies))(*[w.data_ptr() for w in W_copies])
    g, us = ctypes.c_int(0), ctypes.c_float(0)
    _check(lib.qg_tune_bf16(X.data_ptr(), _ld(X), ctypes.cast(ptrs, ctypes.c_void_p), len(W_copies), Y.data_ptr(),
                            N, Y_ref.data_ptr(), M, N, K, buf.data_ptr() if buf is not None else None, nb, calls,
                            ctypes.byref(g), ctypes.byref(us), _stream_ptr(stream)), "qg_tune_bf16")
    _ws_need.clear()
    return g.value, us.value


def tune_w8a8(Xq, X_scale, W_copies, W_scale, calls: int = 100, workspace=None, stream=None):
    """As tune_fp8 for the W8A8 GEMM on quantised activations (Xq, X_scale as
    quantize_act_e4m3 returns them; W_copies: equal E4M3 weights)."""
    torch = _torch()
    M, K = Xq.shape
    N = W_copies[0].shape[0]
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=Xq.device)
    Y_ref = torch.empty_like(Y)
    buf, nb = _tune_common(M, N, Xq, Y_ref, workspace, workspace_bytes_max_w8a8(M, N))
    ptrs = (ctypes.c_void_p * len(W_copies))(*[w.data_ptr() for w in W_copies])
    g, us = ctypes.c_int(0), ctypes.c_float(0)
    _check(lib.qg_tune_w8a8(Xq.data_ptr(), _ld(Xq), X_scale.data_ptr(), _ld(X_scale),
                            ctypes.cast(ptrs, ctypes.c_void_p), len(W_copies), W_scale.data_ptr(), Y.data_ptr(), N,
                            Y_ref.data_ptr(), M, N, K, buf.data_ptr() if buf is not None else None, nb, calls,
                            ctypes.byref(g), ctypes.byref(us), _stream_ptr(stream)), "qg_tune_w8a8")
    _ws_need.clear()
    return g.value, us.value


def tune_lut3(X, Wq_copies, qmap, scales, N: int, calls: int = 200, workspace=None, stream=None):
    """As tune_fp8 for the 3-bit LUT GEMM (Wq_copies: equal packed weights)."""
    torch = _torch()
    M, K = X.shape
    Y = torch.empty((M, N), dtype=torch.float16, device=X.device)
    Y_ref = torch.empty_like(Y)
    buf, nb = _tune_common(M, N, X, Y_ref, workspace)
    ptrs = (ctypes.c_void_p * len(Wq_copies))(*[w.data_ptr() for w in Wq_copies])
    g, us = ctypes.c_int(0), ctypes.c_float(0)
    _check(lib.qg_tune_lut3(X.data_ptr(), _ld(X), ctypes.cast(ptrs, ctypes.c_void_p), len(Wq_copies),
                            qmap.data_ptr(), scales.data_ptr(), Y.data_ptr(), N, Y_ref.data_ptr(), M, N, K,
                            buf.data_ptr() if buf is not None else None, nb, calls, ctypes.byref(g),
                            ctypes.byref(us), _stream_ptr(stream)), "qg_tune_lut3")
    _ws_need.clear()
    return g.value, us.value
