"""GPU parity: every entry point of the C ABI against the CPU oracle on the same
seeded inputs, at sizes that span several tiles and ragged tails, plus the edge
cases (empty groups, all groups empty, tail garbage, sizes that are not tile
multiples)."""
import pytest
import torch

from fp8_moe_routed_gb300 import binding as fb
from fp8_moe_routed_gb300 import workloads as W
from parity_util import bf16_ulp, bits16, check_bf16, check_f32_rel

pytestmark = pytest.mark.gpu

DEV = "cuda"


def cuda(*ts):
    return [t.to(DEV) for t in ts]


@pytest.fixture(autouse=True, scope="module")
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fb.load()
    yield
    torch.cuda.synchronize()


@pytest.fixture(autouse=True)
def _status_clean():
    fb.read_status()
    yield
    assert fb.read_status() == 0


# ------------------------------------------------------------------ dequant
def test_dequantize_all_codes_bit_exact(orc):
    E, K, N = 3, 512, 256
    g = torch.Generator().manual_seed(5)
    codes = (torch.arange(E * K * N) * 7 + 3).remainder(256).to(torch.uint8).view(E, K, N)
    codes[(codes & 0x7F) == 0x7F] = 0x11       # NaN codes are not weights
    scale = torch.exp(torch.randn(E, N, generator=g) * 3).float()
    out = fb.dequantize_fp8_codes(*cuda(codes, scale))
    ref = orc.dequantize(codes, scale)
    assert torch.equal(bits16(out), bits16(ref))


@pytest.mark.parametrize("E,K,N", [(4, 256, 256), (2, 7168, 64), (5, 48, 4096)])
def test_dequantize_shapes(orc, E, K, N):
    codes, scale = W.fp8_weights(E, K, N, 0.01, seed=E + K)
    out = fb.dequantize_fp8_codes(*cuda(codes, scale))
    assert torch.equal(bits16(out), bits16(orc.dequantize(codes, scale)))


# ------------------------------------------------------------- row quantize
@pytest.mark.parametrize("M,K,gs", [
    (512, 256, None), (300, 2048, [100, 0, 150, 20]), (200, 7168, [64, 64, 0, 60]),
    (64, 9216, [40, 24]), (130, 16, [129, 1]),
])
def test_quantize_rows_bit_exact(orc, M, K, gs):
    gs = W.group_sizes("tiny", seed=1, M=M) if gs is None else torch.tensor(gs, dtype=torch.int32)
    x = W.activations(M, K, seed=K, outlier_frac=0.05)
    T = int(gs.sum())
    x = W.fill_tail_garbage(x, T)
    x[0, :] = 0                         # zero row -> scale 1e-12/448
    q, sx = fb.quantize_rows(*cuda(x, gs))
    q_ref, sx_ref, bad = orc.quantize_rows(x, gs)
    assert bad == 0
    assert torch.equal(q.cpu()[:T], q_ref[:T])
    assert torch.equal(sx.cpu()[:T], sx_ref[:T])
    assert (q.cpu()[T:] == 0).all() and torch.isnan(sx.cpu()[T:]).all()   # untouched


# ------------------------------------------------------------ forward GMM
def fwd_case(M, K, N, E, gs, seed, outliers=0.0, tail_garbage=True):
    gs = torch.tensor(gs, dtype=torch.int32) if isinstance(gs, list) else gs
    x = W.activations(M, K, seed, outlier_frac=outliers)
    if tail_garbage:
        x = W.fill_tail_garbage(x, int(gs.sum()))
    codes, scale = W.fp8_weights(E, K, N, 0.02, seed + 1)
    return x, codes, scale, gs


FWD_CASES = [
    # M, K, N, E, group sizes
    (512, 256, 256, 4, "tiny"),
    (700, 512, 512, 5, [300, 0, 129, 1, 200]),      # T=630 < M: ragged tail
    (384, 1024, 768, 3, [0, 384, 0]),               # one group owns everything
    (256, 256, 352, 2, [100, 100]),                 # N not a multiple of 256 (silu: 176)
    (300, 336, 224, 3, [120, 0, 150]),              # K not a multiple of the 128-wide k step
]


@pytest.mark.parametrize("silu", [True, False])
@pytest.mark.parametrize("M,K,N,E,gs", FWD_CASES)
def test_gmm_fwd_vs_oracle(orc, M, K, N, E, gs, silu):
    if gs == "tiny":
        gs = W.group_sizes("tiny", seed=0, M=M, E=E)
    x, codes, scale, gs = fwd_case(M, K, N, E, gs, seed=M + N, outliers=0.01)
    T = int(gs.sum())
    Nout = N // 2 if silu else N
    out = torch.full((M, Nout), 7.0, dtype=torch.bfloat16, device=DEV)   # sentinel
    fn = fb.gmm_silu_fp8_fwd if silu else fb.gmm_fp8_fwd
    fn(*cuda(x, codes, scale, gs), out=out)
    ref, _, bad = orc.gmm_fwd(x, codes, scale, gs, silu=silu)
    assert bad == 0
    check_bf16(out[:T], ref[:T], what=f"fwd silu={silu}")
    assert (out[T:].float() == 7.0).all(), "rows >= T were written"


@pytest.mark.parametrize("silu", [True, False])
@pytest.mark.parametrize("M,K,N,gs", [
    (512, 256, 256, "tiny"), (700, 512, 512, [300, 0, 129, 1, 200]),
    (200, 7168, 256, [64, 64, 0, 60]), (64, 9216, 64, [40, 24]), (130, 64, 64, [129, 1]),
    (2048, 2048, 256, [1000, 0, 1000, 47]),
])
def test_gmm_fwd_workspace_codes_and_scales_bit_exact(orc, M, K, N, gs, silu):
    """The codes and row scales the forward GMM consumed are left in its
    workspace (codes [M, K], then the row scales [M]): after the call they are
    bit-exact against the oracle's quantization for every row < T, and the
    output is within tolerance."""
    gs = W.group_sizes("tiny", seed=2, M=M) if gs == "tiny" else torch.tensor(gs, dtype=torch.int32)
    E = gs.numel()
    T = int(gs.sum())
    x = W.fill_tail_garbage(W.activations(M, K, seed=K + M, outlier_frac=0.05), T)
    x[0, :] = 0
    codes, scale = W.fp8_weights(E, K, N, 0.02, seed=7)
    op = fb.OP_GMM_SILU_FP8_FWD if silu else fb.OP_GMM_FP8_FWD
    ws = torch.zeros(fb.workspace_size(op, M, K, N, E), dtype=torch.uint8, device=DEV)
    fn = fb.gmm_silu_fp8_fwd if silu else fb.gmm_fp8_fwd
    out = fn(*cuda(x, codes, scale, gs), workspace=ws)
    q = ws[:M * K].view(M, K).cpu()
    off = (M * K + 255) // 256 * 256
    sx = ws[off:off + 4 * M].view(torch.float32).cpu()
    q_ref, sx_ref, bad = orc.quantize_rows(x, gs)
    assert bad == 0
    assert torch.equal(sx[:T], sx_ref[:T])
    assert torch.equal(q[:T], q_ref[:T])
    ref, _, bad = orc.gmm_fwd(x, codes, scale, gs, silu=silu)
    assert bad == 0
    check_bf16(out[:T], ref[:T], what="fwd with in-kernel quantization")


def test_gmm_fwd_all_groups_empty():
    M, K, N, E = 256, 256, 256, 4
    x, codes, scale, gs = fwd_case(M, K, N, E, [0, 0, 0, 0], seed=3)
    out = torch.full((M, N // 2), 7.0, dtype=torch.bfloat16, device=DEV)
    fb.gmm_silu_fp8_fwd(*cuda(x, codes, scale, gs), out=out)
    assert (out.float() == 7.0).all()


def test_gmm_fwd_lossless_rows_equal_plain_matmul():
    """Rows on the e4m3 grid with amax 448: quantization is exact, the FP8 GMM
    equals the float64 matmul with the dequantized weight (to one rounding)."""
    M, K, N, E = 256, 512, 256, 2
    g = torch.Generator().manual_seed(4)
    cx = torch.randint(0, 256, (M, K), generator=g, dtype=torch.uint8)
    cx[(cx & 0x7F) == 0x7F] = 0x30
    cx[:, 0] = 0x7E
    x = cx.view(torch.float8_e4m3fn).to(torch.bfloat16)
    codes, scale = W.fp8_weights(E, K, N, 0.05, 9)
    gs = torch.tensor([100, 156], dtype=torch.int32)
    out = fb.gmm_fp8_fwd(*cuda(x, codes, scale, gs))
    w = codes.view(torch.float8_e4m3fn).double() * scale.double()[:, None, :]
    ref = torch.cat([x[:100].double() @ w[0], x[100:].double() @ w[1]])
    check_bf16(out, ref, what="lossless")


# ------------------------------------------------------------------- dLHS
DLHS_CASES = [
    (512, 256, 256, 4, "tiny"),                      # contraction 256: cached path
    (700, 512, 512, 5, [300, 0, 129, 1, 200]),       # streaming
    (300, 2048, 256, 3, [0, 280, 20]),
    (260, 512, 1088, 2, [130, 100]),                 # K-out not a multiple of 256
]


@pytest.mark.parametrize("M,N,K,E,gs", DLHS_CASES)
def test_dlhs_vs_oracle_and_paths_identical(orc, M, N, K, E, gs):
    if gs == "tiny":
        gs = W.group_sizes("tiny", seed=0, M=M, E=E)
    gs = torch.tensor(gs, dtype=torch.int32) if isinstance(gs, list) else gs
    T = int(gs.sum())
    dout = W.fill_tail_garbage(W.cotangent(M, N, seed=N), T)
    codes, scale = W.fp8_weights(E, K, N, 0.02, seed=K)
    args = cuda(dout, codes, scale, gs)
    out0 = torch.full((M, K), 7.0, dtype=torch.bfloat16, device=DEV)
    fb.gmm_dlhs_fp8(*args, out=out0, path=0)
    ref, _, bad = orc.gmm_dlhs(dout, codes, scale, gs)
    assert bad == 0
    check_bf16(out0[:T], ref[:T], what="dlhs")
    assert (out0[T:].float() == 7.0).all()
    if N <= 256:
        out1 = torch.full((M, K), 7.0, dtype=torch.bfloat16, device=DEV)
        fb.gmm_dlhs_fp8(*args, out=out1, path=1)
        assert torch.equal(bits16(out1), bits16(out0)), "cached and streaming paths differ"
    # CTA pairs with the dequantized weight in tensor memory: the same bits
    out2 = torch.full((M, K), 7.0, dtype=torch.bfloat16, device=DEV)
    fb.gmm_dlhs_fp8(*args, out=out2, path=2)
    assert torch.equal(bits16(out2), bits16(out0)), "pair and streaming paths differ"


PAIR_CASES = [
    (800, 320, 384, 3, [130, 0, 300]),                # k tile of 128 past K = 384
    (600, 176, 272, 2, [100, 200]),                   # N % 64 = 48, K % 256 = 16
    (1100, 4096, 512, 4, [1, 255, 257, 512]),         # one-row group, 257 = 256 + 1
]


@pytest.mark.parametrize("M,N,K,E,gs", PAIR_CASES)
def test_dlhs_pair_path_edges(orc, M, N, K, E, gs):
    """The CTA-pair path (256 weight rows x 256 token rows per unit) on the
    shapes where its tiling is ragged: against the oracle and bit for bit
    against the streaming path; rows past T untouched."""
    gs = torch.tensor(gs, dtype=torch.int32)
    T = int(gs.sum())
    dout = W.fill_tail_garbage(W.cotangent(M, N, seed=N + 7), T)
    codes, scale = W.fp8_weights(E, K, N, 0.02, seed=K + 7)
    args = cuda(dout, codes, scale, gs)
    out2 = torch.full((M, K), 7.0, dtype=torch.bfloat16, device=DEV)
    fb.gmm_dlhs_fp8(*args, out=out2, path=2)
    ref, _, bad = orc.gmm_dlhs(dout, codes, scale, gs)
    assert bad == 0
    check_bf16(out2[:T], ref[:T], what="dlhs pair path")
    assert (out2[T:].float() == 7.0).all(), "rows >= T were written"
    out0 = torch.full((M, K), 7.0, dtype=torch.bfloat16, device=DEV)
    fb.gmm_dlhs_fp8(*args, out=out0, path=0)
    assert torch.equal(bits16(out2), bits16(out0)), "pair and streaming paths differ"


def test_dlhs_all_groups_empty_every_path():
    """No rows at all (every group empty, M > 0): each dLHS path launches, finds
    no work unit, writes nothing and leaves the status word clean."""
    M, N, K, E = 96, 320, 256, 3
    gs = torch.zeros(E, dtype=torch.int32, device=DEV)
    dout = torch.randn(M, N, device=DEV).to(torch.bfloat16)
    codes, scale = W.fp8_weights(E, K, N, 0.02, seed=9, device=DEV)
    for path in (0, 2):
        out = torch.full((M, K), 7.0, dtype=torch.bfloat16, device=DEV)
        fb.gmm_dlhs_fp8(dout, codes, scale, gs, out=out, path=path)
        torch.cuda.synchronize()
        assert (out.float() == 7.0).all(), f"path {path} wrote rows of empty groups"
    c1, s1 = W.fp8_weights(E, K, 256, 0.02, seed=10, device=DEV)
    out = torch.full((M, K), 7.0, dtype=torch.bfloat16, device=DEV)
    fb.gmm_dlhs_fp8(dout[:, :256].contiguous(), c1, s1, gs, out=out, path=1)
    torch.cuda.synchronize()
    assert (out.float() == 7.0).all(), "path 1 wrote rows of empty groups"


# ---------------------------------------------------- wo dLHS + dSwiGLU
DSWIGLU_CASES = [
    (512, 256, 128, 4, "tiny"),                       # N <= 256: all three paths
    (1024, 512, 272, 3, [300, 0, 500]),               # F = 272: partial column chunk
    (640, 160, 64, 2, [0, 600]),                      # first expert empty, all three paths
]


@pytest.mark.parametrize("M,N,F,E,gs", DSWIGLU_CASES)
def test_dlhs_dswiglu_vs_oracle_and_paths_identical(orc, M, N, F, E, gs):
    if gs == "tiny":
        gs = W.group_sizes("tiny", seed=5, M=M, E=E)
    gs = torch.tensor(gs, dtype=torch.int32) if isinstance(gs, list) else gs
    T = int(gs.sum())
    d = W.fill_tail_garbage(W.cotangent(M, N, seed=N + 1), T)
    gu = W.fill_tail_garbage(W.activations(M, 2 * F, seed=F + 2), T)
    codes, scale = W.fp8_weights(E, F, N, 0.05, seed=E + 3)
    dg, gug, cg, sg, gsg = cuda(d, gu, codes, scale, gs)
    out0 = torch.full((M, 2 * F), 7.0, dtype=torch.bfloat16, device=DEV)
    fb.gmm_dlhs_dswiglu_fp8(dg, cg, sg, gug, gsg, out=out0, path=0)
    ref, _, bad = orc.gmm_dlhs_dswiglu(d, codes, scale, gu, gs)
    assert bad == 0
    check_bf16(out0[:T], ref[:T], what="dlhs+dswiglu streaming")
    assert (out0[T:] == 7.0).all(), "rows >= T were written"
    if N <= 256:
        out1 = torch.full((M, 2 * F), 7.0, dtype=torch.bfloat16, device=DEV)
        fb.gmm_dlhs_dswiglu_fp8(dg, cg, sg, gug, gsg, out=out1, path=1)
        assert torch.equal(bits16(out1), bits16(out0)), "cached and streaming paths differ"
    out3 = torch.full((M, 2 * F), 7.0, dtype=torch.bfloat16, device=DEV)
    fb.gmm_dlhs_dswiglu_fp8(dg, cg, sg, gug, gsg, out=out3, path=2)
    assert torch.equal(bits16(out3), bits16(out0)), "pair and streaming paths differ"
    # the default entry point picks one of the paths
    out2 = fb.gmm_dlhs_dswiglu_fp8(dg, cg, sg, gug, gsg)
    assert torch.equal(bits16(out2[:T]), bits16(out0[:T]))


def test_dlhs_dswiglu_rejects_missing_gu_and_misalignment():
    M, N, F, E = 128, 256, 64, 2
    gs = torch.tensor([64, 64], dtype=torch.int32, device=DEV)
    d = torch.zeros(M, N, dtype=torch.bfloat16, device=DEV)
    codes = torch.zeros(E, F, N, dtype=torch.uint8, device=DEV)
    scale = torch.ones(E, N, dtype=torch.float32, device=DEV)
    out = torch.empty(M, 2 * F, dtype=torch.bfloat16, device=DEV)
    L = fb.load()
    st = fb._stream(d.device)
    rc = L.fp8moe_gmm_dlhs_dswiglu_fp8(fb._ptr(d), M, N, fb._ptr(codes), fb._ptr(scale), E, F,
                                       None, fb._ptr(gs), fb._ptr(out), None, 0, st)
    assert rc == -1
    gu = torch.zeros(M * 2 * F + 8, dtype=torch.bfloat16, device=DEV)[1:1 + M * 2 * F]
    rc = L.fp8moe_gmm_dlhs_dswiglu_fp8(fb._ptr(d), M, N, fb._ptr(codes), fb._ptr(scale), E, F,
                                       fb._ptr(gu), fb._ptr(gs), fb._ptr(out), None, 0, st)
    assert rc == -2


# ------------------------------------------------------------------- tgmm
TGMM_CASES = [
    (512, 256, 256, 4, "tiny"),
    (1024, 512, 512, 6, [300, 0, 129, 1, 200, 0]),   # T=630, tail garbage, straddles
    (384, 256, 768, 3, [0, 0, 0]),                   # all empty: dW = 0
]


@pytest.mark.parametrize("M,K,N,E,gs", TGMM_CASES)
def test_tgmm_vs_oracle(orc, M, K, N, E, gs):
    if gs == "tiny":
        gs = W.group_sizes("tiny", seed=2, M=M, E=E)
    gs = torch.tensor(gs, dtype=torch.int32) if isinstance(gs, list) else gs
    T = int(gs.sum())
    x = W.fill_tail_garbage(W.activations(M, K, seed=K), T)
    d = W.fill_tail_garbage(W.cotangent(M, N, seed=N), T)
    dw = fb.tgmm_drhs_quant(*cuda(x, d, gs))
    ref, bad = orc.tgmm(x, d, gs)
    assert bad == 0
    assert torch.isfinite(dw).all()
    if T == 0:
        assert (dw == 0).all()
    else:
        check_f32_rel(dw, ref, what="tgmm")
        for e in range(E):
            if int(gs[e]) == 0:
                assert (dw[e] == 0).all()


def test_tgmm_odd_segments_ragged_tiles_and_16b_aligned_out(orc):
    """Experts with an odd number of 128-row segments (a pipeline stage then
    carries one live segment), k and n tiles cut by K = 272 and N = 144, and a dW
    that is 16- but not 32-byte aligned (the kernel's narrower store path); the
    same call on an aligned dW must give the same bits."""
    M, K, N = 1280, 272, 144
    gs = torch.tensor([300, 400, 0, 400], dtype=torch.int32)   # 3, 4, 0, 4 segments
    T = int(gs.sum())
    x = W.fill_tail_garbage(W.activations(M, K, seed=31), T)
    d = W.fill_tail_garbage(W.cotangent(M, N, seed=32), T)
    xg, dg, gsg = cuda(x, d, gs)
    E = gs.numel()
    buf = torch.full((E * K * N + 4,), 5.0, dtype=torch.float32, device=DEV)
    out = buf[4:].view(E, K, N)
    assert out.data_ptr() % 32 == 16
    dw = fb.tgmm_drhs_quant(xg, dg, gsg, out=out)
    ref, bad = orc.tgmm(x, d, gs)
    assert bad == 0
    check_f32_rel(dw, ref, what="tgmm odd/ragged")
    assert (dw[2] == 0).all()
    assert (buf[:4] == 5.0).all()
    dw2 = fb.tgmm_drhs_quant(xg, dg, gsg)
    assert dw2.data_ptr() % 32 == 0
    assert torch.equal(dw2, dw)


def test_tgmm_quantize_tiles_bit_exact(orc):
    M, K, N = 1024, 512, 256
    gs = torch.tensor([300, 0, 129, 1, 200, 0], dtype=torch.int32)
    T = int(gs.sum())
    x = W.fill_tail_garbage(W.activations(M, K, seed=1), T)
    d = W.fill_tail_garbage(W.cotangent(M, N, seed=2), T)
    qx, sx, qd, sd = fb.tgmm_quantize_tiles(*cuda(x, d, gs))
    rqx, rsx, rqd, rsd, nseg, bad = orc.tgmm_quantize_tiles(x, d, gs)
    assert bad == 0
    assert torch.equal(qx.cpu()[:nseg], rqx[:nseg]) and torch.equal(qd.cpu()[:nseg], rqd[:nseg])
    assert torch.equal(sx.cpu()[:nseg], rsx[:nseg]) and torch.equal(sd.cpu()[:nseg], rsd[:nseg])


# -------------------------------------------- e5m2 gradient operand (tgmm)
@pytest.mark.parametrize("M,K,N,E,gs", TGMM_CASES)
def test_tgmm_e5m2_vs_oracle(orc, M, K, N, E, gs):
    """The gradient fp8 dtype e5m2 ("MoE fp8 backward ...", What): dout codes
    e5m2 with max 57344, lhs codes e4m3, e4m3 x e5m2 MMA."""
    if gs == "tiny":
        gs = W.group_sizes("tiny", seed=2, M=M, E=E)
    gs = torch.tensor(gs, dtype=torch.int32) if isinstance(gs, list) else gs
    T = int(gs.sum())
    x = W.fill_tail_garbage(W.activations(M, K, seed=K + 5), T)
    d = W.fill_tail_garbage(W.cotangent(M, N, seed=N + 6), T)
    dw = fb.tgmm_drhs_quant(*cuda(x, d, gs), dout_fmt="e5m2")
    ref, bad = orc.tgmm(x, d, gs, dout_fmt="e5m2")
    assert bad == 0
    assert torch.isfinite(dw).all()
    if T == 0:
        assert (dw == 0).all()
    else:
        check_f32_rel(dw, ref, what="tgmm e5m2")
        # e5m2 and e4m3 dout give different (coarser) results: the format is live
        dw4 = fb.tgmm_drhs_quant(*cuda(x, d, gs))
        assert not torch.equal(dw4, dw)


def test_tgmm_quantize_tiles_e5m2_bit_exact(orc):
    M, K, N = 1024, 512, 256
    gs = torch.tensor([300, 0, 129, 1, 200, 0], dtype=torch.int32)
    T = int(gs.sum())
    x = W.fill_tail_garbage(W.activations(M, K, seed=7), T)
    d = W.fill_tail_garbage(W.cotangent(M, N, seed=8), T)
    qx, sx, qd, sd = fb.tgmm_quantize_tiles(*cuda(x, d, gs), dout_fmt="e5m2")
    rqx, rsx, rqd, rsd, nseg, bad = orc.tgmm_quantize_tiles(x, d, gs, dout_fmt="e5m2")
    assert bad == 0
    assert torch.equal(qx.cpu()[:nseg], rqx[:nseg]) and torch.equal(qd.cpu()[:nseg], rqd[:nseg])
    assert torch.equal(sx.cpu()[:nseg], rsx[:nseg]) and torch.equal(sd.cpu()[:nseg], rsd[:nseg])


def _e5m2_stress_cols(n_cols=64, seed=19):
    """Column c holds every bf16 magnitude of the 31 binades below a random amax,
    both signs, shuffled down 8192 rows: per 128-row segment x / scale sweeps the
    e5m2 rounding boundaries down into its subnormal range."""
    g = torch.Generator().manual_seed(seed)
    cols = []
    for c in range(n_cols):
        e = int(torch.randint(-20, 20, (1,), generator=g))
        mant = int(torch.randint(0, 128, (1,), generator=g))
        hi_bits = ((e + 127) << 7) | mant
        lo_bits = (e - 31 + 127) << 7
        mags = torch.arange(lo_bits, hi_bits + 1, dtype=torch.int32)
        vals = torch.cat([mags, mags | 0x8000]).to(torch.int16)
        col = torch.zeros(8192, dtype=torch.int16)
        col[:vals.numel()] = vals[torch.randperm(vals.numel(), generator=g)]
        cols.append(col)
    return torch.stack(cols, dim=1).contiguous().view(torch.bfloat16)


def test_tgmm_quantize_e5m2_quotient_stress_bit_exact(orc):
    d = _e5m2_stress_cols()
    M = d.shape[0]
    lhs = W.activations(M, 32, 4)
    gs = torch.tensor([4000, 4192], dtype=torch.int32)
    qx, sx, qd, sd = fb.tgmm_quantize_tiles(*cuda(lhs, d, gs), dout_fmt="e5m2")
    rqx, rsx, rqd, rsd, nseg, bad = orc.tgmm_quantize_tiles(lhs, d, gs, dout_fmt="e5m2")
    assert bad == 0
    assert torch.equal(sd.cpu()[:nseg], rsd[:nseg]) and torch.equal(qd.cpu()[:nseg], rqd[:nseg])
    assert torch.equal(sx.cpu()[:nseg], rsx[:nseg]) and torch.equal(qx.cpu()[:nseg], rqx[:nseg])
    # the sweep reaches the e5m2 subnormal codes (exponent field 0, nonzero)
    sub = ((rqd[:nseg] & 0x7C) == 0) & ((rqd[:nseg] & 0x03) != 0)
    assert int(sub.sum()) > 100


def test_tgmm_rejects_unknown_dout_format():
    x = torch.zeros(128, 64, dtype=torch.bfloat16, device=DEV)
    d = torch.zeros(128, 64, dtype=torch.bfloat16, device=DEV)
    gs = torch.tensor([128], dtype=torch.int32, device=DEV)
    out = torch.empty(1, 64, 64, dtype=torch.float32, device=DEV)
    L = fb.load()
    ws = torch.empty(fb.workspace_size(fb.OP_TGMM_DRHS_QUANT, 128, 64, 64, 1), dtype=torch.uint8,
                     device=DEV)
    rc = L.fp8moe_tgmm_drhs_quant_fmt(fb._ptr(x), fb._ptr(d), 128, 64, 64, 1, fb._ptr(gs),
                                      fb._ptr(out), fb._ptr(ws), ws.numel(), 2, fb._stream(x.device))
    assert rc == -1


# ---------------------------------- per-512 block quantization (NEXT-3)
BLOCK_CASES = [
    (512, 1024, 256, 4, "tiny"),
    (1024, 1280, 384, 3, [300, 0, 500]),     # K = 1280: partial last block; tail garbage
    (640, 7168, 512, 2, [0, 600]),            # 14 blocks, first expert empty
]


def _block_case(M, K, E, gs, seed):
    if gs == "tiny":
        gs = W.group_sizes("tiny", seed=seed, M=M, E=E)
    gs = torch.tensor(gs, dtype=torch.int32) if isinstance(gs, list) else gs
    T = int(gs.sum())
    x = W.fill_tail_garbage(W.activations(M, K, seed=K + seed), T)
    return gs, T, x


@pytest.mark.parametrize("M,K,N,E,gs", BLOCK_CASES)
def test_quantize_rows_block_bit_exact(orc, M, K, N, E, gs):
    gs, T, x = _block_case(M, K, E, gs, 1)
    q, sb = fb.quantize_rows_block(*cuda(x, gs))
    rq, rsb, bad = orc.quantize_rows_block(x, gs)
    assert bad == 0
    assert torch.equal(sb.cpu()[:T], rsb[:T]) and torch.equal(q.cpu()[:T], rq[:T])


@pytest.mark.parametrize("M,K,N,E,gs", BLOCK_CASES)
def test_gmm_fwd_block_vs_oracle(orc, M, K, N, E, gs):
    """Tolerance from the arithmetic: GPU and oracle take the same bf16
    rounding steps; the f32 block product (summation order) and the fused
    multiply-add before the bf16 rounding can flip a step by one bf16 ulp of the
    running sum, so |gpu - ref| <= nblk * ulp(max |acc|) * |sw| + 1 ulp(ref);
    and almost every element is bit-identical."""
    gs, T, x = _block_case(M, K, E, gs, 2)
    codes, scale = W.fp8_weights(E, K, N, 0.05, seed=E + 7)
    out = fb.gmm_fp8_fwd_block(*cuda(x, codes, scale, gs), False)
    ref, _, amx, bad = orc.gmm_fwd_block(x, codes, scale, gs, silu=False, want_acc_max=True)
    assert bad == 0
    nblk = (K + 511) // 512
    g, r = out.cpu()[:T].double(), ref[:T].double()
    assert torch.isfinite(g).all()
    sw = torch.zeros(T, N, dtype=torch.float64)
    off = 0
    for e, n in enumerate(gs.tolist()):
        sw[off:off + n] = scale[e].double()
        off += n
    bound = nblk * bf16_ulp(amx[:T]) * sw.abs() + bf16_ulp(r)
    assert ((g - r).abs() <= bound).all()
    same = (out.cpu()[:T].view(torch.int16) == ref[:T].view(torch.int16)).float().mean().item()
    assert same > 0.95, same


@pytest.mark.parametrize("M,K,N,E,gs", BLOCK_CASES)
def test_gmm_fwd_block_swiglu_vs_oracle(orc, M, K, N, E, gs):
    """The bound of the plain block forward carried through h = silu(g) * u.

    Both sides take the same bf16 rounding steps, so g and u (the scaled
    accumulators of the gate and up columns) differ from the oracle's by at most
        dg = nblk * ulp(max |acc_g|) * |sw_g|,   du = nblk * ulp(max |acc_u|) * |sw_u|
    (test above). By the mean value theorem, with L = sup |silu'| < 1.1,
        |silu(g') u' - silu(g) u| <= L dg (|u| + du) + |silu(g)| du.
    The kernel evaluates silu(g) * u in f32 (exponential, add, divide, multiply):
    a relative error below 2^-20 of |silu(g) u|. Rounding both results to bf16
    adds at most one bf16 ulp of the larger of the two."""
    gs, T, x = _block_case(M, K, E, gs, 3)
    codes, scale = W.fp8_weights(E, K, N, 0.05, seed=E + 8)
    out = fb.gmm_fp8_fwd_block(*cuda(x, codes, scale, gs), True)
    ref, _, _, bad = orc.gmm_fwd_block(x, codes, scale, gs, silu=True)
    assert bad == 0
    # g and u unrounded (double) and the accumulator magnitudes, from the same
    # oracle without the SwiGLU step
    _, y64, amx, bad = orc.gmm_fwd_block(x, codes, scale, gs, silu=False, want_f64=True,
                                         want_acc_max=True)
    assert bad == 0
    F = N // 2
    nblk = (K + 511) // 512
    sw = torch.zeros(T, N, dtype=torch.float64)
    off = 0
    for e, n in enumerate(gs.tolist()):
        sw[off:off + n] = scale[e].double()
        off += n
    dy = nblk * bf16_ulp(amx[:T]) * sw.abs()
    gg, uu = y64[:T, :F], y64[:T, F:]
    dg, du = dy[:, :F], dy[:, F:]
    sg = torch.nn.functional.silu(gg)
    g, r = out.cpu()[:T].double(), ref[:T].double()
    assert torch.isfinite(g).all()
    bound = (1.1 * dg * (uu.abs() + du) + sg.abs() * du + 2.0 ** -20 * (sg * uu).abs()
             + bf16_ulp(torch.maximum(g.abs(), r.abs())))
    err = (g - r).abs()
    assert (err <= bound).all(), (err - bound).max().item()


def test_gmm_fwd_block_rejects_other_block_sizes():
    x = torch.zeros(128, 512, dtype=torch.bfloat16, device=DEV)
    codes = torch.zeros(1, 512, 64, dtype=torch.uint8, device=DEV)
    scale = torch.ones(1, 64, device=DEV)
    gs = torch.tensor([128], dtype=torch.int32, device=DEV)
    with pytest.raises(fb.Fp8MoeError):
        fb.gmm_fp8_fwd_block(x, codes, scale, gs, False, block=256)


# --------------------------------------------------------- BF16 comparison
@pytest.mark.parametrize("swiglu", [True, False])
def test_bf16_gmm_vs_float64(orc, swiglu):
    M, K, N, E = 640, 512, 512, 4
    gs = torch.tensor([200, 0, 300, 100], dtype=torch.int32)
    T = 600
    x = W.fill_tail_garbage(W.activations(M, K, seed=8), T)
    codes, scale = W.fp8_weights(E, K, N, 0.02, seed=9)
    w = orc.dequantize(codes, scale)
    out = fb.gmm_bf16_fwd(*cuda(x, w, gs), swiglu=swiglu)
    xd, wd = x.double(), w.double()
    ref = torch.zeros(M, N, dtype=torch.float64)
    off = 0
    for e, g in enumerate(gs.tolist()):
        ref[off:off + g] = xd[off:off + g] @ wd[e]
        off += g
    if swiglu:
        ref = torch.nn.functional.silu(ref[:, :N // 2]) * ref[:, N // 2:]
    check_bf16(out[:T], ref[:T], what="bf16 gmm")


def _quotient_stress_rows(n_rows=2048, seed=17):
    """Row r holds every bf16 value within 12 binades below a random amax (both
    signs), so x / scale sweeps every e4m3 rounding boundary for 2048 scales."""
    g = torch.Generator().manual_seed(seed)
    rows = []
    for r in range(n_rows):
        e = int(torch.randint(-20, 20, (1,), generator=g))
        mant = int(torch.randint(0, 128, (1,), generator=g))
        amax_bits = ((e + 127) << 7) | mant
        lo_bits = ((e - 12 + 127) << 7)
        mags = torch.arange(lo_bits, amax_bits + 1, dtype=torch.int32)
        vals = torch.cat([mags, mags | 0x8000]).to(torch.int16)
        rows.append(vals)
    K = max(v.numel() for v in rows)
    K = (K + 15) // 16 * 16
    out = torch.zeros(n_rows, K, dtype=torch.int16)
    for r, v in enumerate(rows):
        out[r, :v.numel()] = v[torch.randperm(v.numel(), generator=g)]
    return out.view(torch.bfloat16)


def test_quantize_quotient_stress_bit_exact(orc):
    x = _quotient_stress_rows()
    M, K = x.shape
    gs = torch.tensor([M], dtype=torch.int32)
    q, sx = fb.quantize_rows(*cuda(x, gs))
    q_ref, sx_ref, bad = orc.quantize_rows(x, gs)
    assert bad == 0
    assert torch.equal(sx.cpu(), sx_ref)
    assert torch.equal(q.cpu(), q_ref)


def test_tgmm_quantize_quotient_stress_bit_exact(orc):
    """The same values laid out down the columns of 128-row tiles."""
    x = _quotient_stress_rows(n_rows=256, seed=18)          # [256, K]
    cols = x.view(torch.int16)[:, :1024].reshape(256, 1024)
    lhs = cols.t().contiguous().view(torch.bfloat16)        # [1024 rows, 256 cols]
    lhs = lhs[:, :256].contiguous()
    M = lhs.shape[0]
    dout = W.cotangent(M, 64, 3)
    gs = torch.tensor([300, 500, 224], dtype=torch.int32)
    qx, sxt, qd, sd = fb.tgmm_quantize_tiles(*cuda(lhs, dout, gs))
    rqx, rsx, rqd, rsd, nseg, bad = orc.tgmm_quantize_tiles(lhs, dout, gs)
    assert bad == 0
    assert torch.equal(sxt.cpu()[:nseg], rsx[:nseg]) and torch.equal(qx.cpu()[:nseg], rqx[:nseg])
    assert torch.equal(sd.cpu()[:nseg], rsd[:nseg]) and torch.equal(qd.cpu()[:nseg], rqd[:nseg])


# ------------------------------------------------- failure detection (GPU)
def test_bounded_wait_times_out_records_status_and_context_survives(orc):
    """A wait that nothing completes gives up after its limit, records the
    timeout (where = 6) in the status word, and the next call works: the
    failure path of every pipeline wait, made to run out on purpose."""
    import time
    t0 = time.time()
    fb.selftest_wait_timeout(20000)                  # 20 ms
    st = fb.read_status()
    assert time.time() - t0 < 5.0
    assert st & fb.STATUS_WAIT_TIMEOUT
    assert (st >> 8) & 0xFF == 6
    assert fb.read_status() == 0                     # read clears
    codes, scale = W.fp8_weights(2, 64, 32, 0.05, 9, device=DEV)
    out = fb.dequantize_fp8_codes(codes, scale)
    ref = orc.dequantize(codes.cpu(), scale.cpu())
    assert torch.equal(bits16(out), bits16(ref))
