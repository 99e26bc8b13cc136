"""Python binding of libfp8moe.so (the C ABI in include/fp8moe.h).

Argument marshalling only: it checks dtypes/devices/contiguity, allocates the
outputs (and, when the caller passes none, the workspace) with torch, and passes
raw device pointers, sizes and the current CUDA stream to the library. Every
step of the computation runs in the library's CUDA kernels; if the library is
missing or fails to load, every call raises.

Function names follow the C ABI without the ``fp8moe_`` prefix.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

OK = 0
ERRORS = {-1: "EINVAL", -2: "EALIGN", -3: "EWORKSPACE", -4: "ECUDA", -5: "EUNSUPPORTED"}

OP_GMM_FP8_FWD = 1
OP_GMM_SILU_FP8_FWD = 2
OP_GMM_DLHS_FP8 = 3
OP_TGMM_DRHS_QUANT = 4
OP_GMM_BF16_FWD = 5
OP_GMM_FP8_FWD_BLOCK = 7

STATUS_NEGATIVE_GROUP = 0x1
STATUS_GROUPS_EXCEED_M = 0x2
STATUS_WAIT_TIMEOUT = 0x4

# every symbol include/fp8moe.h declares
EXPORTS = [
    "fp8moe_workspace_size", "fp8moe_gmm_fp8_fwd", "fp8moe_gmm_silu_fp8_fwd",
    "fp8moe_gmm_dlhs_fp8", "fp8moe_gmm_dlhs_fp8_path", "fp8moe_tgmm_drhs_quant",
    "fp8moe_dequantize_fp8_codes", "fp8moe_gmm_bf16_fwd", "fp8moe_quantize_rows",
    "fp8moe_tgmm_quantize_tiles", "fp8moe_read_status", "fp8moe_status_string",
    "fp8moe_last_cuda_error", "fp8moe_num_sms", "fp8moe_gmm_silu_fp8_fwd_noalloc",
    "fp8moe_gmm_dlhs_dswiglu_fp8", "fp8moe_gmm_dlhs_dswiglu_fp8_path",
    "fp8moe_tgmm_drhs_quant_fmt", "fp8moe_tgmm_quantize_tiles_fmt",
    "fp8moe_gmm_fp8_fwd_block", "fp8moe_quantize_rows_block", "fp8moe_selftest_wait_timeout",
    "fp8moe_selftest_cast_f32",
]

FMT = {"e4m3": 0, "e5m2": 1}

_lock = threading.Lock()
_lib = None


class Fp8MoeError(RuntimeError):
    pass


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load (building first if needed) the shared library and declare the ABI."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise Fp8MoeError(f"libfp8moe.so not built ({path})")
            _build.build()
        L = ctypes.CDLL(path)
        P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
        sig = {
            "fp8moe_workspace_size": ([I32, I64, I64, I64, I32], SZ),
            "fp8moe_gmm_fp8_fwd": ([P, I64, I64, P, P, I32, I64, P, P, P, SZ, P], I32),
            "fp8moe_gmm_silu_fp8_fwd": ([P, I64, I64, P, P, I32, I64, P, P, P, SZ, P], I32),
            "fp8moe_gmm_dlhs_fp8": ([P, I64, I64, P, P, I32, I64, P, P, P, SZ, P], I32),
            "fp8moe_gmm_dlhs_fp8_path": ([P, I64, I64, P, P, I32, I64, P, P, I32, P], I32),
            "fp8moe_tgmm_drhs_quant": ([P, P, I64, I64, I64, I32, P, P, P, SZ, P], I32),
            "fp8moe_dequantize_fp8_codes": ([P, P, I32, I64, I64, P, P], I32),
            "fp8moe_gmm_bf16_fwd": ([P, I64, I64, P, I32, I64, P, I32, P, P], I32),
            "fp8moe_quantize_rows": ([P, I64, I64, P, I32, P, P, P], I32),
            "fp8moe_tgmm_quantize_tiles": ([P, P, I64, I64, I64, I32, P, P, P, P, P, P], I32),
            "fp8moe_read_status": ([P, ctypes.POINTER(ctypes.c_uint32)], I32),
            "fp8moe_status_string": ([I32], ctypes.c_char_p),
            "fp8moe_last_cuda_error": ([], I32),
            "fp8moe_num_sms": ([], I32),
            "fp8moe_gmm_silu_fp8_fwd_noalloc": ([P, I64, I64, P, P, I32, I64, P, P, P], I32),
            "fp8moe_gmm_dlhs_dswiglu_fp8": ([P, I64, I64, P, P, I32, I64, P, P, P, P, SZ, P], I32),
            "fp8moe_gmm_dlhs_dswiglu_fp8_path": ([P, I64, I64, P, P, I32, I64, P, P, P, I32, P],
                                                 I32),
            "fp8moe_tgmm_drhs_quant_fmt": ([P, P, I64, I64, I64, I32, P, P, P, SZ, I32, P], I32),
            "fp8moe_tgmm_quantize_tiles_fmt": ([P, P, I64, I64, I64, I32, P, P, P, P, P, I32, P],
                                               I32),
            "fp8moe_gmm_fp8_fwd_block": ([P, I64, I64, P, P, I32, I64, P, P, P, SZ, I32, I32, P],
                                         I32),
            "fp8moe_quantize_rows_block": ([P, I64, I64, P, I32, I32, P, P, P], I32),
            "fp8moe_selftest_wait_timeout": ([ctypes.c_uint32, P], I32),
            "fp8moe_selftest_cast_f32": ([P, I64, I32, P, P], I32),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
        return _lib


def _check(rc: int, what: str):
    if rc != OK:
        L = load()
        msg = L.fp8moe_status_string(rc).decode()
        extra = ""
        if rc == -4:
            extra = f" (cudaError {L.fp8moe_last_cuda_error()})"
        raise Fp8MoeError(f"{what}: {ERRORS.get(rc, rc)} -- {msg}{extra}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _req(t: torch.Tensor, dtype, name: str, ndim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def workspace_size(op: int, M: int, K: int, N: int, E: int) -> int:
    return int(load().fp8moe_workspace_size(op, M, K, N, E))


def _workspace(op, M, K, N, E, device, workspace):
    need = workspace_size(op, M, K, N, E)
    if workspace is None:
        if need == 0:
            return None, 0
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    return workspace, workspace.numel() * workspace.element_size()


def _fwd(lhs, codes, scale, group_sizes, out, workspace, silu: bool):
    L = load()
    _req(lhs, torch.bfloat16, "lhs", 2)
    _req(codes, torch.uint8, "codes", 3)
    _req(scale, torch.float32, "scale", 2)
    _req(group_sizes, torch.int32, "group_sizes", 1)
    M, K = lhs.shape
    E, K2, N = codes.shape
    if K2 != K or scale.shape != (E, N) or group_sizes.numel() != E:
        raise ValueError("shape mismatch")
    Nout = N // 2 if silu else N
    if out is None:
        out = torch.empty(M, Nout, dtype=torch.bfloat16, device=lhs.device)
    else:
        _req(out, torch.bfloat16, "out", 2)
        if out.shape != (M, Nout):
            raise ValueError("out shape")
    op = OP_GMM_SILU_FP8_FWD if silu else OP_GMM_FP8_FWD
    ws, wsb = _workspace(op, M, K, N, E, lhs.device, workspace)
    fn = L.fp8moe_gmm_silu_fp8_fwd if silu else L.fp8moe_gmm_fp8_fwd
    _check(fn(_ptr(lhs), M, K, _ptr(codes), _ptr(scale), E, N, _ptr(group_sizes), _ptr(out),
              _ptr(ws), wsb, _stream(lhs.device)), fn.__name__)
    return out


def gmm_fp8_fwd(lhs, codes, scale, group_sizes, out=None, workspace=None):
    """wo forward: bf16 [M, N] (see fp8moe_gmm_fp8_fwd)."""
    return _fwd(lhs, codes, scale, group_sizes, out, workspace, silu=False)


def gmm_silu_fp8_fwd(lhs, codes, scale, group_sizes, out=None, workspace=None):
    """wi forward with fused SwiGLU: bf16 [M, N/2] (see fp8moe_gmm_silu_fp8_fwd)."""
    return _fwd(lhs, codes, scale, group_sizes, out, workspace, silu=True)


def gmm_fp8_fwd_block(lhs, codes, scale, group_sizes, swiglu: bool, out=None, workspace=None,
                      block: int = 512):
    """Forward GMM with per-512-column block activation scales and bf16
    accumulation across blocks (see fp8moe_gmm_fp8_fwd_block)."""
    L = load()
    _req(lhs, torch.bfloat16, "lhs", 2)
    _req(codes, torch.uint8, "codes", 3)
    _req(scale, torch.float32, "scale", 2)
    _req(group_sizes, torch.int32, "group_sizes", 1)
    M, K = lhs.shape
    E, K2, N = codes.shape
    if K2 != K or scale.shape != (E, N) or group_sizes.numel() != E:
        raise ValueError("shape mismatch")
    Nout = N // 2 if swiglu else N
    if out is None:
        out = torch.empty(M, Nout, dtype=torch.bfloat16, device=lhs.device)
    else:
        _req(out, torch.bfloat16, "out", 2)
    ws, wsb = _workspace(OP_GMM_FP8_FWD_BLOCK, M, K, N, E, lhs.device, workspace)
    _check(L.fp8moe_gmm_fp8_fwd_block(_ptr(lhs), M, K, _ptr(codes), _ptr(scale), E, N,
                                      _ptr(group_sizes), _ptr(out), _ptr(ws), wsb, block,
                                      1 if swiglu else 0, _stream(lhs.device)),
           "fp8moe_gmm_fp8_fwd_block")
    return out


def quantize_rows_block(lhs, group_sizes, block: int = 512):
    """Parity export of the per-block activation quantization: codes u8 [M, K]
    and bf16-valued f32 scales [M, ceil(K / block)]."""
    L = load()
    _req(lhs, torch.bfloat16, "lhs", 2)
    _req(group_sizes, torch.int32, "group_sizes", 1)
    M, K = lhs.shape
    nb = (K + block - 1) // block
    q = torch.zeros(M, K, dtype=torch.uint8, device=lhs.device)
    sb = torch.full((M, nb), float("nan"), dtype=torch.float32, device=lhs.device)
    _check(L.fp8moe_quantize_rows_block(_ptr(lhs), M, K, _ptr(group_sizes), group_sizes.numel(),
                                        block, _ptr(q), _ptr(sb), _stream(lhs.device)),
           "fp8moe_quantize_rows_block")
    return q, sb


NOALLOC_SCRATCH_BYTES = 32 << 20


def gmm_silu_fp8_fwd_noalloc(lhs, codes, scale, group_sizes, out):
    """wi forward without a caller workspace: the library's fixed 32 MiB device
    array stands in for it (see fp8moe_gmm_silu_fp8_fwd_noalloc). ``out`` must be
    given; this call allocates nothing."""
    L = load()
    _req(lhs, torch.bfloat16, "lhs", 2)
    _req(codes, torch.uint8, "codes", 3)
    _req(scale, torch.float32, "scale", 2)
    _req(group_sizes, torch.int32, "group_sizes", 1)
    _req(out, torch.bfloat16, "out", 2)
    M, K = lhs.shape
    E, _, N = codes.shape
    _check(L.fp8moe_gmm_silu_fp8_fwd_noalloc(_ptr(lhs), M, K, _ptr(codes), _ptr(scale), E, N,
                                             _ptr(group_sizes), _ptr(out), _stream(lhs.device)),
           "fp8moe_gmm_silu_fp8_fwd_noalloc")
    return out


def gmm_dlhs_fp8(dout, codes, scale, group_sizes, out=None, path: Optional[int] = None):
    """dLHS: bf16 [M, K] (see fp8moe_gmm_dlhs_fp8; path forces 0 streaming /
    1 cached / 2 CTA pairs with the weight in tensor memory)."""
    L = load()
    _req(dout, torch.bfloat16, "dout", 2)
    _req(codes, torch.uint8, "codes", 3)
    _req(scale, torch.float32, "scale", 2)
    _req(group_sizes, torch.int32, "group_sizes", 1)
    M, N = dout.shape
    E, K, N2 = codes.shape
    if N2 != N or scale.shape != (E, N) or group_sizes.numel() != E:
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty(M, K, dtype=torch.bfloat16, device=dout.device)
    else:
        _req(out, torch.bfloat16, "out", 2)
    st = _stream(dout.device)
    if path is None:
        rc = L.fp8moe_gmm_dlhs_fp8(_ptr(dout), M, N, _ptr(codes), _ptr(scale), E, K,
                                   _ptr(group_sizes), _ptr(out), None, 0, st)
    else:
        rc = L.fp8moe_gmm_dlhs_fp8_path(_ptr(dout), M, N, _ptr(codes), _ptr(scale), E, K,
                                        _ptr(group_sizes), _ptr(out), int(path), st)
    _check(rc, "fp8moe_gmm_dlhs_fp8")
    return out


def gmm_dlhs_dswiglu_fp8(dout, codes, scale, gu, group_sizes, out=None,
                         path: Optional[int] = None):
    """wo dLHS + SwiGLU backward: dgu bf16 [M, 2F] from dout [M, N], the wo
    codes [E, F, N] and the wi output gu [M, 2F] (see fp8moe_gmm_dlhs_dswiglu_fp8;
    path forces 0 streaming / 1 cached / 2 CTA pairs)."""
    L = load()
    _req(dout, torch.bfloat16, "dout", 2)
    _req(codes, torch.uint8, "codes", 3)
    _req(scale, torch.float32, "scale", 2)
    _req(gu, torch.bfloat16, "gu", 2)
    _req(group_sizes, torch.int32, "group_sizes", 1)
    M, N = dout.shape
    E, F, N2 = codes.shape
    if N2 != N or scale.shape != (E, N) or group_sizes.numel() != E or gu.shape != (M, 2 * F):
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty(M, 2 * F, dtype=torch.bfloat16, device=dout.device)
    else:
        _req(out, torch.bfloat16, "out", 2)
    st = _stream(dout.device)
    if path is None:
        rc = L.fp8moe_gmm_dlhs_dswiglu_fp8(_ptr(dout), M, N, _ptr(codes), _ptr(scale), E, F,
                                           _ptr(gu), _ptr(group_sizes), _ptr(out), None, 0, st)
    else:
        rc = L.fp8moe_gmm_dlhs_dswiglu_fp8_path(_ptr(dout), M, N, _ptr(codes), _ptr(scale), E,
                                                F, _ptr(gu), _ptr(group_sizes), _ptr(out),
                                                int(path), st)
    _check(rc, "fp8moe_gmm_dlhs_dswiglu_fp8")
    return out


def tgmm_drhs_quant(lhs, dout, group_sizes, out=None, workspace=None, dout_fmt: str = "e4m3"):
    """Weight gradient f32 [E, K, N] (see fp8moe_tgmm_drhs_quant; dout_fmt
    "e5m2" quantizes the gradient operand to e5m2, fp8moe_tgmm_drhs_quant_fmt)."""
    L = load()
    _req(lhs, torch.bfloat16, "lhs", 2)
    _req(dout, torch.bfloat16, "dout", 2)
    _req(group_sizes, torch.int32, "group_sizes", 1)
    M, K = lhs.shape
    M2, N = dout.shape
    if M2 != M:
        raise ValueError("shape mismatch")
    E = group_sizes.numel()
    if out is None:
        out = torch.empty(E, K, N, dtype=torch.float32, device=lhs.device)
    else:
        _req(out, torch.float32, "out", 3)
    ws, wsb = _workspace(OP_TGMM_DRHS_QUANT, M, K, N, E, lhs.device, workspace)
    if dout_fmt == "e4m3":
        rc = L.fp8moe_tgmm_drhs_quant(_ptr(lhs), _ptr(dout), M, K, N, E, _ptr(group_sizes),
                                      _ptr(out), _ptr(ws), wsb, _stream(lhs.device))
    else:
        rc = L.fp8moe_tgmm_drhs_quant_fmt(_ptr(lhs), _ptr(dout), M, K, N, E, _ptr(group_sizes),
                                          _ptr(out), _ptr(ws), wsb, FMT[dout_fmt],
                                          _stream(lhs.device))
    _check(rc, "fp8moe_tgmm_drhs_quant")
    return out


def dequantize_fp8_codes(codes, scale, out=None):
    """bf16 [E, K, N] = bf16(code * scale) (see fp8moe_dequantize_fp8_codes)."""
    L = load()
    _req(codes, torch.uint8, "codes", 3)
    _req(scale, torch.float32, "scale", 2)
    E, K, N = codes.shape
    if out is None:
        out = torch.empty(E, K, N, dtype=torch.bfloat16, device=codes.device)
    _check(L.fp8moe_dequantize_fp8_codes(_ptr(codes), _ptr(scale), E, K, N, _ptr(out),
                                         _stream(codes.device)), "fp8moe_dequantize_fp8_codes")
    return out


def gmm_bf16_fwd(lhs, w, group_sizes, swiglu: bool, out=None):
    """BF16 comparison GMM (see fp8moe_gmm_bf16_fwd)."""
    L = load()
    _req(lhs, torch.bfloat16, "lhs", 2)
    _req(w, torch.bfloat16, "w", 3)
    _req(group_sizes, torch.int32, "group_sizes", 1)
    M, K = lhs.shape
    E, K2, N = w.shape
    if K2 != K:
        raise ValueError("shape mismatch")
    Nout = N // 2 if swiglu else N
    if out is None:
        out = torch.empty(M, Nout, dtype=torch.bfloat16, device=lhs.device)
    _check(L.fp8moe_gmm_bf16_fwd(_ptr(lhs), M, K, _ptr(w), E, N, _ptr(group_sizes),
                                 int(bool(swiglu)), _ptr(out), _stream(lhs.device)),
           "fp8moe_gmm_bf16_fwd")
    return out


def quantize_rows(lhs, group_sizes, q=None, sx=None):
    """Parity export: codes u8 [M, K] and scales f32 [M] for rows < T."""
    L = load()
    _req(lhs, torch.bfloat16, "lhs", 2)
    _req(group_sizes, torch.int32, "group_sizes", 1)
    M, K = lhs.shape
    if q is None:
        q = torch.zeros(M, K, dtype=torch.uint8, device=lhs.device)
    if sx is None:
        sx = torch.full((M,), float("nan"), dtype=torch.float32, device=lhs.device)
    _check(L.fp8moe_quantize_rows(_ptr(lhs), M, K, _ptr(group_sizes), group_sizes.numel(),
                                  _ptr(q), _ptr(sx), _stream(lhs.device)), "fp8moe_quantize_rows")
    return q, sx


def segment_bound(M: int, E: int) -> int:
    return (M + 127) // 128 + E


def tgmm_quantize_tiles(lhs, dout, group_sizes, dout_fmt: str = "e4m3"):
    """Parity export of the tgmm operand quantization (slot layout)."""
    L = load()
    _req(lhs, torch.bfloat16, "lhs", 2)
    _req(dout, torch.bfloat16, "dout", 2)
    _req(group_sizes, torch.int32, "group_sizes", 1)
    M, K = lhs.shape
    _, N = dout.shape
    E = group_sizes.numel()
    S = segment_bound(M, E)
    dev = lhs.device
    qx = torch.zeros(S, 128, K, dtype=torch.uint8, device=dev)
    sx = torch.full((S, K), float("nan"), dtype=torch.float32, device=dev)
    qd = torch.zeros(S, 128, N, dtype=torch.uint8, device=dev)
    sd = torch.full((S, N), float("nan"), dtype=torch.float32, device=dev)
    _check(L.fp8moe_tgmm_quantize_tiles_fmt(_ptr(lhs), _ptr(dout), M, K, N, E, _ptr(group_sizes),
                                            _ptr(qx), _ptr(sx), _ptr(qd), _ptr(sd), FMT[dout_fmt],
                                            _stream(dev)),
           "fp8moe_tgmm_quantize_tiles")
    return qx, sx, qd, sd


def selftest_wait_timeout(limit_us: int, device=None) -> None:
    """Enqueue the bounded-wait failure self-test (see fp8moe_selftest_wait_timeout)."""
    _check(load().fp8moe_selftest_wait_timeout(int(limit_us), _stream(device)),
           "fp8moe_selftest_wait_timeout")


def selftest_cast_f32(x, fmt: str = "e4m3", codes=None):
    """The quantizers' f32 -> fp8 cast on arbitrary f32 values (a device tensor):
    codes u8 of x's shape (see fp8moe_selftest_cast_f32)."""
    _req(x, torch.float32, "x", x.dim())
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    _check(load().fp8moe_selftest_cast_f32(_ptr(x), x.numel(), FMT[fmt], _ptr(codes),
                                           _stream(x.device)), "fp8moe_selftest_cast_f32")
    return codes


def read_status(device=None) -> int:
    """Synchronize the current stream and return (and clear) the status bits."""
    L = load()
    flags = ctypes.c_uint32(0)
    _check(L.fp8moe_read_status(_stream(device), ctypes.byref(flags)), "fp8moe_read_status")
    return int(flags.value)


def num_sms() -> int:
    return int(load().fp8moe_num_sms())
