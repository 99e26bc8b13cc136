"""The allocation-free wi forward (fp8moe_gmm_silu_fp8_fwd_noalloc).

Callers that cannot allocate device memory (a plugin inside a framework whose
caching allocator holds nearly all of it, or a runtime that forbids allocations
after start-up) get the wi forward with its workspace taken from a fixed device
array inside the library. This checks, through the C ABI, that two calls in a row
on different inputs give what the regular entry point gives with a caller
workspace (so nothing left in the shared array from one call leaks into the
next), and that a size whose workspace would not fit is refused.

Kept in its own file, named to be collected last, so that a stop-at-first-failure
run has already run every other test if this one fails.
"""
import ctypes

import pytest
import torch

from fp8_moe_routed_gb300 import binding as fb
from fp8_moe_routed_gb300 import workloads as W
from parity_util import check_bf16

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _call_noalloc(L, x, codes, scale, gs, out):
    M, K = x.shape
    E, _, N = codes.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return L.fp8moe_gmm_silu_fp8_fwd_noalloc(_p(x), M, K, _p(codes), _p(scale), E, N, _p(gs),
                                             _p(out), stream)


def _case(M, K, N, E, gs, seed):
    gs = torch.tensor(gs, dtype=torch.int32)
    x = W.fill_tail_garbage(W.activations(M, K, seed, outlier_frac=0.01), int(gs.sum()))
    codes, scale = W.fp8_weights(E, K, N, 0.02, seed + 1)
    return [t.cuda() for t in (x, codes, scale, gs)]


def test_noalloc_matches_regular_entry_point_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L = fb.load()
    cases = [
        _case(1024, 2048, 512, 4, [300, 0, 500, 200], seed=11),      # T = 1000 of 1024
        _case(640, 1024, 768, 3, [130, 257, 200], seed=23),          # different shapes
    ]
    for x, codes, scale, gs in cases:
        M, N = x.shape[0], codes.shape[2]
        T = int(gs.sum())
        ref = fb.gmm_silu_fp8_fwd(x, codes, scale, gs)
        out = torch.full((M, N // 2), 7.0, dtype=torch.bfloat16, device="cuda")
        rc = _call_noalloc(L, x, codes, scale, gs, out)
        assert rc == 0, L.fp8moe_status_string(rc).decode()
        torch.cuda.synchronize()
        check_bf16(out[:T], ref[:T].float(), what="noalloc vs regular")
        assert torch.equal(out[:T], ref[:T])
        assert (out[T:].float() == 7.0).all()
    assert fb.read_status() == 0


def test_noalloc_rejects_sizes_past_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L = fb.load()
    M, K, N, E = 8192, 7168, 256, 2          # 58.7 MB of activation codes > 32 MiB
    assert fb.workspace_size(fb.OP_GMM_SILU_FP8_FWD, M, K, N, E) > fb.NOALLOC_SCRATCH_BYTES
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    P = ctypes.c_void_p
    rc = L.fp8moe_gmm_silu_fp8_fwd_noalloc(P(256), M, K, P(256), P(256), E, N, P(256), P(256),
                                           stream)
    assert rc == -3   # FP8MOE_EWORKSPACE, nothing launched


def test_noalloc_at_exactly_the_scratch_size_through_the_binding():
    """A problem whose workspace is exactly the 32 MiB array (the activation
    codes and the row scales end at its last byte), through the Python binding:
    the same bits as the regular entry point."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    M, K, N, E = 16352, 2048, 256, 4
    assert fb.workspace_size(fb.OP_GMM_SILU_FP8_FWD, M, K, N, E) == fb.NOALLOC_SCRATCH_BYTES
    x, codes, scale, gs = _case(M, K, N, E, [4000, 5000, 0, 7352], seed=31)
    ref = fb.gmm_silu_fp8_fwd(x, codes, scale, gs)
    out = torch.empty(M, N // 2, dtype=torch.bfloat16, device="cuda")
    fb.gmm_silu_fp8_fwd_noalloc(x, codes, scale, gs, out)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert fb.read_status() == 0


def test_noalloc_checks_arguments_before_the_size():
    """A bad argument gets the regular entry point's code even when the size
    would not fit either (nothing is launched in any of these calls)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L = fb.load()
    M, K, N, E = 8192, 7168, 256, 2
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    P = ctypes.c_void_p
    # lhs not 16-byte aligned: FP8MOE_EALIGN
    assert L.fp8moe_gmm_silu_fp8_fwd_noalloc(P(258), M, K, P(256), P(256), E, N, P(256), P(256),
                                             stream) == -2
    # null output: FP8MOE_EINVAL
    assert L.fp8moe_gmm_silu_fp8_fwd_noalloc(P(256), M, K, P(256), P(256), E, N, P(256), None,
                                             stream) == -1
    # N not a multiple of 32 for SwiGLU: FP8MOE_EALIGN
    assert L.fp8moe_gmm_silu_fp8_fwd_noalloc(P(256), M, K, P(256), P(256), E, 272, P(256),
                                             P(256), stream) == -2
