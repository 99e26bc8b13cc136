"""The C-ABI library builds, loads without a GPU, and exports every symbol the
header declares; host-side argument checks reject bad calls before any launch."""
import ctypes
import os
import re

import pytest

from fp8_moe_routed_gb300 import binding as fb
from fp8_moe_routed_gb300 import build as fbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "fp8moe.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_what_the_binding_exports():
    assert declared_functions() == sorted(fb.EXPORTS)


def test_library_loads_and_exports_every_symbol():
    L = fb.load()
    for name in declared_functions():
        assert hasattr(L, name), name
    assert L.fp8moe_status_string(0).decode() == "ok"


def test_workspace_sizes():
    # activation codes (M*K) + row scales (M*4), each rounded to 256 bytes
    assert fb.workspace_size(fb.OP_GMM_SILU_FP8_FWD, 32768, 7168, 4096, 32) == 32768 * 7168 + 32768 * 4
    assert fb.workspace_size(fb.OP_GMM_DLHS_FP8, 100, 256, 256, 4) == 0
    S = (65536 + 127) // 128 + 32
    want = S * 128 * 7168 + S * 128 * 2048 + S * 7168 * 4 + S * 2048 * 4
    assert fb.workspace_size(fb.OP_TGMM_DRHS_QUANT, 65536, 7168, 2048, 32) == want


def _call_fwd(L, M=128, K=256, N=256, E=4, lhs=16, codes=16, ws=256, wsb=10 ** 9):
    P = ctypes.c_void_p
    return L.fp8moe_gmm_silu_fp8_fwd(P(lhs), M, K, P(codes), P(16), E, N, P(16), P(16),
                                     P(ws), wsb, None)


def test_argument_checks_run_before_any_device_call():
    L = fb.load()
    assert _call_fwd(L, K=250) == -2                  # K not a multiple of 16
    assert _call_fwd(L, N=250) == -2
    assert _call_fwd(L, N=304) == -2                  # SwiGLU up half not 16-byte aligned
    assert _call_fwd(L, E=0) == -1
    assert _call_fwd(L, E=2000) == -1
    assert _call_fwd(L, M=-1) == -1
    assert _call_fwd(L, lhs=8) == -2                  # misaligned pointer
    assert _call_fwd(L, ws=128) == -2                 # workspace not 256-aligned
    assert _call_fwd(L, wsb=16) == -3                 # workspace too small
    assert _call_fwd(L, ws=0) == -3                   # no workspace
    assert _call_fwd(L, M=0) == 0                     # empty: nothing to launch
    P = ctypes.c_void_p
    assert L.fp8moe_gmm_dlhs_fp8_path(P(16), 64, 512, P(16), P(16), 4, 256, P(16), P(16), 1,
                                      None) == -1     # cached path needs N <= 256
    assert L.fp8moe_gmm_dlhs_fp8_path(P(16), 64, 512, P(16), P(16), 4, 256, P(16), P(16), 3,
                                      None) == -1     # paths are 0, 1, 2
    assert L.fp8moe_dequantize_fp8_codes(P(16), P(16), 4, 256, 8, P(16), None) == -2
    # argument checks of the entry points added for the next steps of the path
    assert L.fp8moe_selftest_wait_timeout(0, None) == -1              # limit must be > 0
    assert L.fp8moe_selftest_wait_timeout(3000000, None) == -1        # and <= 2 s
    assert L.fp8moe_selftest_cast_f32(P(16), -1, 0, P(16), None) == -1  # n >= 0
    assert L.fp8moe_selftest_cast_f32(P(16), 8, 7, P(16), None) == -1   # unknown format
    assert L.fp8moe_selftest_cast_f32(None, 8, 0, P(16), None) == -1    # null input
    assert L.fp8moe_selftest_cast_f32(P(18), 8, 1, P(16), None) == -2   # x not 4-byte aligned
    assert L.fp8moe_selftest_cast_f32(None, 0, 0, None, None) == 0      # empty: nothing to do
    assert L.fp8moe_gmm_fp8_fwd_block(P(16), 128, 512, P(16), P(16), 2, 256, P(16), P(16),
                                      P(256), 10 ** 9, 256, 0, None) == -1   # block must be 512
    assert L.fp8moe_tgmm_drhs_quant_fmt(P(16), P(16), 128, 64, 64, 1, P(16), P(16), P(256),
                                        10 ** 9, 7, None) == -1       # unknown dout format
    assert L.fp8moe_gmm_dlhs_dswiglu_fp8(P(16), 128, 256, P(16), P(16), 2, 64, None, P(16),
                                         P(16), None, 0, None) == -1  # gu missing


def test_build_is_up_to_date():
    assert os.path.exists(fbuild.build())
