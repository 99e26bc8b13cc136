"""ctypes front end of the CPU oracle (oracle/fp8moe_oracle.cpp).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg use this module; the library and its Python binding never do.

Every function takes and returns torch CPU tensors (bf16 as torch.bfloat16,
codes as torch.uint8) and returns, next to its results, the number of reads of
rows at or past T = sum(group_sizes) that the oracle's guarded accessor saw.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "fp8moe_oracle.cpp")
LIB = os.path.join(HERE, "_build", "libfp8moe_oracle.so")

# Plain C++17 + OpenMP. -ffp-contract=off: no fused multiply-add may merge the
# f32 roundings the pages' definitions take one at a time (GCC contracts by
# default on aarch64).
CXXFLAGS = ["-O2", "-std=c++17", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
            "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", *CXXFLAGS, SRC, "-o", tmp])
        os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P, I64, I32, U32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32
            L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_decode.restype = ctypes.c_double
            L.orc_e4m3_encode_f32.argtypes = [P, I64, P]
            L.orc_e4m3_encode_bits.argtypes = [U32, I64, P]
            L.orc_f64_to_bf16.argtypes = [P, I64, P]
            L.orc_num_threads.restype = ctypes.c_int
            L.orc_quantize_rows.argtypes = [P, I64, I64, P, I32, P, P]
            L.orc_quantize_rows.restype = I64
            L.orc_gmm_fwd.argtypes = [P, I64, I64, P, P, I32, I64, P, I32, P, I64, P, P]
            L.orc_gmm_fwd.restype = I64
            L.orc_dequantize.argtypes = [P, P, I32, I64, I64, P]
            L.orc_gmm_dlhs.argtypes = [P, I64, I64, P, P, I32, I64, P, P, I64, P, P]
            L.orc_dswiglu.argtypes = [P, P, I64, I64, P, I64, P, P]
            L.orc_quantize_rows_block.argtypes = [P, I64, I64, I64, P, I32, P, P]
            L.orc_quantize_rows_block.restype = I64
            L.orc_gmm_fwd_block.argtypes = [P, I64, I64, I64, P, P, I32, I64, P, I32, P, I64,
                                            P, P, P]
            L.orc_gmm_fwd_block.restype = I64
            L.orc_dswiglu.restype = None
            L.orc_gmm_dlhs.restype = I64
            L.orc_tgmm_quantize_tiles.argtypes = [P, P, I64, I64, I64, I32, P, I64,
                                                  P, P, P, P, P, I32]
            L.orc_tgmm_quantize_tiles.restype = I64
            L.orc_tgmm.argtypes = [P, P, I64, I64, I64, I32, P, P, I32,
                                   I64, I64, I64, I64, P, I32]
            L.orc_e5m2_decode.argtypes = [ctypes.c_uint8]
            L.orc_e5m2_decode.restype = ctypes.c_double
            L.orc_e5m2_encode_f32.argtypes = [P, I64, P]
            L.orc_e5m2_encode_f32.restype = None
            L.orc_tgmm.restype = I64
            _lib = L
    return _lib


def _p(t):
    if t is None:
        return None
    assert t.device.type == "cpu" and t.is_contiguous()
    return ctypes.c_void_p(t.data_ptr())


def num_threads() -> int:
    return lib().orc_num_threads()


def e4m3_decode(code: int) -> float:
    return lib().orc_e4m3_decode(code)


FMT = {"e4m3": 0, "e5m2": 1}


def e5m2_decode(code: int) -> float:
    return lib().orc_e5m2_decode(code)


def e5m2_encode(x: torch.Tensor) -> torch.Tensor:
    x = x.to(torch.float32).contiguous()
    out = torch.empty(x.shape, dtype=torch.uint8)
    lib().orc_e5m2_encode_f32(_p(x), x.numel(), _p(out))
    return out


def e4m3_decode_all() -> torch.Tensor:
    return torch.tensor([e4m3_decode(c) for c in range(256)], dtype=torch.float64)


def e4m3_encode(x: torch.Tensor) -> torch.Tensor:
    x = x.to(torch.float32).contiguous()
    out = torch.empty(x.shape, dtype=torch.uint8)
    lib().orc_e4m3_encode_f32(_p(x), x.numel(), _p(out))
    return out


def e4m3_encode_bits(lo: int, n: int) -> torch.Tensor:
    out = torch.empty(n, dtype=torch.uint8)
    lib().orc_e4m3_encode_bits(lo, n, _p(out))
    return out


def f64_to_bf16(x: torch.Tensor) -> torch.Tensor:
    x = x.to(torch.float64).contiguous()
    out = torch.empty(x.shape, dtype=torch.int16)
    lib().orc_f64_to_bf16(_p(x), x.numel(), _p(out))
    return out.view(torch.bfloat16)


def _gs(gs):
    return gs.to(torch.int32).contiguous()


def quantize_rows(lhs: torch.Tensor, gs: torch.Tensor, fill_q=0, fill_s=float("nan")):
    """a1: per-row full-K codes and f32 scales for rows < T. Rows >= T keep the
    fill values. Returns (q uint8 [M,K], sx f32 [M], bad_reads)."""
    M, K = lhs.shape
    lhs = lhs.contiguous()
    q = torch.full((M, K), fill_q, dtype=torch.uint8)
    sx = torch.full((M,), fill_s, dtype=torch.float32)
    gs = _gs(gs)
    bad = lib().orc_quantize_rows(_p(lhs), M, K, _p(gs), gs.numel(), _p(q), _p(sx))
    return q, sx, bad


def gmm_fwd(lhs, codes, scale, gs, silu: bool, rows=None, fill=None, want_f64=False):
    """a2-a4: ragged FP8 GMM (+SwiGLU). Returns (out bf16 [M, Nout], out_f64 or
    None, bad_reads). Entries not computed keep ``fill`` (bf16 bit pattern as
    int16, default 0)."""
    M, K = lhs.shape
    E, K2, N = codes.shape
    assert K2 == K
    Nout = N // 2 if silu else N
    out = torch.full((M, Nout), 0 if fill is None else fill, dtype=torch.int16)
    out64 = torch.full((M, Nout), float("nan"), dtype=torch.float64) if want_f64 else None
    gs = _gs(gs)
    r = None if rows is None else rows.to(torch.int64).contiguous()
    bad = lib().orc_gmm_fwd(_p(lhs.contiguous()), M, K, _p(codes.contiguous()),
                            _p(scale.contiguous()), E, N, _p(gs), int(silu),
                            _p(r), 0 if r is None else r.numel(), _p(out), _p(out64))
    return out.view(torch.bfloat16), out64, bad


def dequantize(codes, scale) -> torch.Tensor:
    """a5: bf16 [E, K, N] = bf16(f32(code) * scale[e, n])."""
    E, K, N = codes.shape
    out = torch.empty(E, K, N, dtype=torch.int16)
    lib().orc_dequantize(_p(codes.contiguous()), _p(scale.contiguous()), E, K, N, _p(out))
    return out.view(torch.bfloat16)


def gmm_dlhs(dout, codes, scale, gs, rows=None, fill=None, want_f64=False):
    """a6: dlhs bf16 [M, K] = dout [M, N] x dequant(codes)[e]^T per group."""
    M, N = dout.shape
    E, K, N2 = codes.shape
    assert N2 == N
    out = torch.full((M, K), 0 if fill is None else fill, dtype=torch.int16)
    out64 = torch.full((M, K), float("nan"), dtype=torch.float64) if want_f64 else None
    gs = _gs(gs)
    r = None if rows is None else rows.to(torch.int64).contiguous()
    bad = lib().orc_gmm_dlhs(_p(dout.contiguous()), M, N, _p(codes.contiguous()),
                             _p(scale.contiguous()), E, K, _p(gs), _p(r),
                             0 if r is None else r.numel(), _p(out), _p(out64))
    return out.view(torch.bfloat16), out64, bad


def quantize_rows_block(lhs, gs, block=512, fill_q=0, fill_s=float("nan")):
    """Per-512-column block quantization: codes u8 [M, K], bf16-valued f32
    scales [M, ceil(K / block)] for rows < T (others keep the fill)."""
    M, K = lhs.shape
    nb = (K + block - 1) // block
    q = torch.full((M, K), fill_q, dtype=torch.uint8)
    sb = torch.full((M, nb), fill_s, dtype=torch.float32)
    gs = _gs(gs)
    bad = lib().orc_quantize_rows_block(_p(lhs.contiguous()), M, K, block, _p(gs), gs.numel(),
                                        _p(q), _p(sb))
    return q, sb, bad


def gmm_fwd_block(lhs, codes, scale, gs, silu: bool, block=512, rows=None, fill=None,
                  want_f64=False, want_acc_max=False):
    """Forward GMM with per-block bf16 activation scales and bf16 accumulation
    across blocks. Returns (out, out_f64, acc_max, bad)."""
    M, K = lhs.shape
    E, K2, N = codes.shape
    assert K2 == K
    Nout = N // 2 if silu else N
    out = torch.full((M, Nout), 0 if fill is None else fill, dtype=torch.int16)
    out64 = torch.full((M, Nout), float("nan"), dtype=torch.float64) if want_f64 else None
    amx = torch.full((M, N), float("nan"), dtype=torch.float64) if want_acc_max else None
    gs = _gs(gs)
    r = None if rows is None else rows.to(torch.int64).contiguous()
    bad = lib().orc_gmm_fwd_block(_p(lhs.contiguous()), M, K, block, _p(codes.contiguous()),
                                  _p(scale.contiguous()), E, N, _p(gs), 1 if silu else 0, _p(r),
                                  0 if r is None else r.numel(), _p(out), _p(out64), _p(amx))
    return out.view(torch.bfloat16), out64, amx, bad


def dswiglu(dh_f64, gu, rows=None, fill=None, want_f64=False):
    """SwiGLU backward: dgu bf16 [M, 2F] from the unrounded upstream gradient
    dh (float64 [M, F]) and the wi output gu (bf16 [M, 2F], gate | up)."""
    M, F = dh_f64.shape
    assert gu.shape == (M, 2 * F)
    out = torch.full((M, 2 * F), 0 if fill is None else fill, dtype=torch.int16)
    out64 = torch.full((M, 2 * F), float("nan"), dtype=torch.float64) if want_f64 else None
    r = None if rows is None else rows.to(torch.int64).contiguous()
    lib().orc_dswiglu(_p(dh_f64.contiguous()), _p(gu.contiguous()), M, F, _p(r),
                      0 if r is None else r.numel(), _p(out), _p(out64))
    return out.view(torch.bfloat16), out64


def gmm_dlhs_dswiglu(dout, codes, scale, gu, gs, rows=None, fill=None, want_f64=False):
    """wo dLHS followed by the SwiGLU backward: dgu bf16 [M, 2F] where
    dh = dout [M, N] x dequant(codes)[e]^T ([E, F, N] codes) is kept unrounded."""
    M, N = dout.shape
    E, F, N2 = codes.shape
    assert N2 == N and gu.shape == (M, 2 * F)
    _, dh64, bad = gmm_dlhs(dout, codes, scale, gs, rows=rows, want_f64=True)
    dh64 = torch.nan_to_num(dh64, nan=0.0)      # rows the dLHS did not compute
    if rows is None:
        T = int(_gs(gs).clamp_min(0).sum().clamp_max(M))
        rows = torch.arange(T, dtype=torch.int64)
    out, out64 = dswiglu(dh64, gu, rows=rows, fill=fill, want_f64=want_f64)
    return out, out64, bad


def segment_bound(M: int, E: int) -> int:
    """Upper bound on the number of (gm tile, group) segments: ceil(M/128) + E."""
    return (M + 127) // 128 + E


def tgmm_quantize_tiles(lhs, dout, gs, Smax=None, dout_fmt="e4m3"):
    """a7: per-segment per-channel codes and scales (slot layout, see the C
    source). Returns (qx, sx, qd, sd, nseg, bad_reads)."""
    M, K = lhs.shape
    M2, N = dout.shape
    assert M2 == M
    gs = _gs(gs)
    E = gs.numel()
    if Smax is None:
        Smax = segment_bound(M, E)
    qx = torch.zeros(Smax, 128, K, dtype=torch.uint8)
    sx = torch.full((Smax, K), float("nan"), dtype=torch.float32)
    qd = torch.zeros(Smax, 128, N, dtype=torch.uint8)
    sd = torch.full((Smax, N), float("nan"), dtype=torch.float32)
    nseg = ctypes.c_int64(0)
    bad = lib().orc_tgmm_quantize_tiles(_p(lhs.contiguous()), _p(dout.contiguous()),
                                        M, K, N, E, _p(gs), Smax, _p(qx), _p(sx),
                                        _p(qd), _p(sd), ctypes.byref(nseg), FMT[dout_fmt])
    return qx, sx, qd, sd, nseg.value, bad


def tgmm(lhs, dout, gs, experts=None, k_range=None, n_range=None, dout_fmt="e4m3"):
    """a8: dW f32 [len(experts) or E, k1 - k0, n1 - n0] for the selected experts
    and block (default: all of it). Returns (dW, bad_reads)."""
    M, K = lhs.shape
    _, N = dout.shape
    gs = _gs(gs)
    E = gs.numel()
    k0, k1 = k_range if k_range else (0, K)
    n0, n1 = n_range if n_range else (0, N)
    ex = None if experts is None else torch.tensor(list(experts), dtype=torch.int32)
    nex = E if ex is None else ex.numel()
    dW = torch.full((nex, k1 - k0, n1 - n0), float("nan"), dtype=torch.float32)
    bad = lib().orc_tgmm(_p(lhs.contiguous()), _p(dout.contiguous()), M, K, N, E, _p(gs),
                         _p(ex), 0 if ex is None else ex.numel(), k0, k1, n0, n1, _p(dW),
                         FMT[dout_fmt])
    return dW, bad
