"""GPU parity at the workloads' full sizes, in the launch configuration bench.py
times: the kernels run on the whole problem, the oracle recomputes sampled rows
(or blocks) one by one, and properties that hold at any size are checked on all
of the output (finite values, untouched rows past T, tail invariance).

Workloads: balanced DeepSeek-V3-like layer (E=32, K=7168, F=2048, M=32768),
skewed Zipf routing with empty experts, the dropless tgmm buffer (M=65536 with
NaN/Inf/1e30 tail), and the E=128 tile-dispatch sweep."""
import pytest
import torch

from fp8_moe_routed_gb300 import binding as fb
from fp8_moe_routed_gb300 import workloads as W
from parity_util import bits16, check_bf16, check_f32_rel

pytestmark = pytest.mark.gpu

DEV = "cuda"


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


def sample_rows(gs: torch.Tensor, n_per_group: int, seed: int, extra=()):
    """Sampled rows: first and last row of every non-empty group plus random ones."""
    g = torch.Generator().manual_seed(seed)
    rows, off = [], 0
    for s in gs.tolist():
        if s > 0:
            rows += [off, off + s - 1]
            rows += (off + torch.randint(0, s, (n_per_group,), generator=g)).tolist()
        off += s
    rows += list(extra)
    return torch.tensor(sorted(set(rows)), dtype=torch.int64)


def layer_inputs(kind: str, seed: int):
    E, K, F, M = 32, 7168, 2048, 32768
    gs = W.group_sizes(kind, seed=seed, E=E, M=M)
    x = W.activations(M, K, seed, outlier_frac=0.001, device=DEV)
    wi_c, wi_s = W.fp8_weights(E, K, 2 * F, 0.006, seed + 1, device=DEV)
    wo_c, wo_s = W.fp8_weights(E, F, K, 0.006, seed + 2, device=DEV)
    return E, K, F, M, gs, x, wi_c, wi_s, wo_c, wo_s


@pytest.mark.parametrize("kind", ["balanced", "skewed"])
def test_layer_forward_and_dlhs_sampled(orc, kind):
    E, K, F, M, gs, x, wi_c, wi_s, wo_c, wo_s = layer_inputs(kind, seed=1)
    gsd = gs.to(DEV)
    T = int(gs.sum())
    # wi forward (+SwiGLU) and wo forward, exactly as the benchmark step runs them
    h = fb.gmm_silu_fp8_fwd(x, wi_c, wi_s, gsd)
    y = fb.gmm_fp8_fwd(h, wo_c, wo_s, gsd)
    # activation codes and scales of the whole wi input: bit-exact
    q, sx = fb.quantize_rows(x, gsd)
    xc = x.cpu()
    q_ref, sx_ref, bad = orc.quantize_rows(xc, gs)
    assert bad == 0
    assert torch.equal(sx.cpu()[:T], sx_ref[:T])
    assert torch.equal(q.cpu()[:T], q_ref[:T])
    del q, q_ref
    rows = sample_rows(gs, 2, seed=7)
    wi_cc, wi_sc, wo_cc, wo_sc = wi_c.cpu(), wi_s.cpu(), wo_c.cpu(), wo_s.cpu()
    ref_h, _, bad = orc.gmm_fwd(xc, wi_cc, wi_sc, gs, silu=True, rows=rows)
    assert bad == 0
    check_bf16(h.cpu()[rows], ref_h[rows], what=f"{kind} wi fwd")
    hc = h.cpu()
    ref_y, _, bad = orc.gmm_fwd(hc, wo_cc, wo_sc, gs, silu=False, rows=rows)
    assert bad == 0
    check_bf16(y.cpu()[rows], ref_y[rows], what=f"{kind} wo fwd")
    assert torch.isfinite(h[:T].float()).all() and torch.isfinite(y[:T].float()).all()
    # dLHS of both GMMs (dout N(0,1)), sampled rows
    dy = W.cotangent(M, K, 4, device=DEV)
    dgu = W.cotangent(M, 2 * F, 5, device=DEV)
    dh = fb.gmm_dlhs_fp8(dy, wo_c, wo_s, gsd)
    dx = fb.gmm_dlhs_fp8(dgu, wi_c, wi_s, gsd)
    rows_b = rows[:: max(1, len(rows) // 24)]
    ref_dh, _, bad = orc.gmm_dlhs(dy.cpu(), wo_cc, wo_sc, gs, rows=rows_b)
    assert bad == 0
    check_bf16(dh.cpu()[rows_b], ref_dh[rows_b], what=f"{kind} wo dlhs")
    ref_dx, _, bad = orc.gmm_dlhs(dgu.cpu(), wi_cc, wi_sc, gs, rows=rows_b)
    assert bad == 0
    check_bf16(dx.cpu()[rows_b], ref_dx[rows_b], what=f"{kind} wi dlhs")


def test_dequantize_full_wi_weight_bit_exact(orc):
    codes, scale = W.fp8_weights(8, 7168, 4096, 0.006, 3, device=DEV)
    out = fb.dequantize_fp8_codes(codes, scale)
    ref = orc.dequantize(codes.cpu(), scale.cpu())
    assert torch.equal(bits16(out), bits16(ref))


def test_dropless_tgmm_blocks_finite_and_tail_blind(orc):
    E, K, N, M = 32, 7168, 2048, 65536
    gs = W.group_sizes("dropless", seed=2, E=E)
    T = int(gs.sum())
    assert T == 32768
    x = W.fill_tail_garbage(W.activations(M, K, 11, device=DEV), T)
    d = W.fill_tail_garbage(W.cotangent(M, N, 12, device=DEV), T)
    gsd = gs.to(DEV)
    dw = fb.tgmm_drhs_quant(x, d, gsd)
    assert torch.isfinite(dw).all()
    empty = (gs == 0).nonzero().flatten().tolist()
    assert len(empty) == 4
    for e in empty:
        assert (dw[e] == 0).all()
    # a different garbage tail gives bit-identical dW
    x2, d2 = x.clone(), d.clone()
    x2[T:] = 3.0e38
    d2[T:] = float("nan")
    dw2 = fb.tgmm_drhs_quant(x2, d2, gsd)
    assert torch.equal(dw2, dw)
    del dw2, x2, d2
    # oracle blocks: the largest expert, a small one, straddling tiles
    order = torch.argsort(gs, descending=True).tolist()
    xc, dc = x.cpu(), d.cpu()
    for e, kr, nr in [(order[0], (0, 128), (0, 128)), (order[0], (7040, 7168), (1920, 2048)),
                      (order[27], (1024, 1152), (512, 640))]:
        ref, bad = orc.tgmm(xc, dc, gs, experts=[e], k_range=kr, n_range=nr)
        assert bad == 0
        check_f32_rel(dw[e, kr[0]:kr[1], nr[0]:nr[1]], ref[0], what=f"tgmm e={e}")


@pytest.mark.parametrize("M", [8192, 16384, 32768, 65536, 131072])
def test_sweep_forward_and_dlhs_paths(orc, M):
    """E=128, K=4096, F=1536 at every swept M: FP8 wi forward (+SwiGLU) and wo
    forward (K=1536, N=4096) vs the oracle on sampled rows and vs the BF16
    comparison GMM on the same inputs; dLHS with the pair and streaming paths
    (contraction 3072) and the cached path (contraction 256, forward N=256)."""
    E, K, F = 128, 4096, 1536
    gs = W.group_sizes("sweep", seed=3, E=E, M=M)
    gsd = gs.to(DEV)
    x = W.activations(M, K, 21, device=DEV)
    wi_c, wi_s = W.fp8_weights(E, K, 2 * F, 0.02, 22, device=DEV)
    h = fb.gmm_silu_fp8_fwd(x, wi_c, wi_s, gsd)
    rows = sample_rows(gs, 0, seed=5)[::7]
    ref, _, bad = orc.gmm_fwd(x.cpu(), wi_c.cpu(), wi_s.cpu(), gs, silu=True, rows=rows)
    assert bad == 0
    check_bf16(h.cpu()[rows], ref[rows], what="sweep wi fwd")
    # the BF16 arm on the dequantized weight agrees to FP8 quantization error
    w_bf = fb.dequantize_fp8_codes(wi_c, wi_s)
    hb = fb.gmm_bf16_fwd(x, w_bf, gsd, True)
    rel = ((hb.float() - h.float()).norm() / hb.float().norm()).item()
    assert rel < 0.1, rel
    del w_bf, hb
    # wo forward on the wi output: K = 1536, N = 4096
    wo_c, wo_s = W.fp8_weights(E, F, K, 0.02, 26, device=DEV)
    y = fb.gmm_fp8_fwd(h, wo_c, wo_s, gsd)
    ref_y, _, bad = orc.gmm_fwd(h.cpu(), wo_c.cpu(), wo_s.cpu(), gs, silu=False, rows=rows)
    assert bad == 0
    check_bf16(y.cpu()[rows], ref_y[rows], what="sweep wo fwd")
    wo_bf = fb.dequantize_fp8_codes(wo_c, wo_s)
    yb = fb.gmm_bf16_fwd(h, wo_bf, gsd, False)
    rel = ((yb.float() - y.float()).norm() / yb.float().norm()).item()
    assert rel < 0.1, rel
    del wo_c, wo_bf, y, yb
    # dLHS, contraction N = 3072: the default (CTA-pair) path against the oracle
    # on sampled rows and bit for bit against the streaming path
    dgu = W.cotangent(M, 2 * F, 23, device=DEV)
    dx = fb.gmm_dlhs_fp8(dgu, wi_c, wi_s, gsd)
    rows_b = rows[:: max(1, len(rows) // 12)]
    ref_dx, _, bad = orc.gmm_dlhs(dgu.cpu(), wi_c.cpu(), wi_s.cpu(), gs, rows=rows_b)
    assert bad == 0
    check_bf16(dx.cpu()[rows_b], ref_dx[rows_b], what="sweep dlhs pair")
    T = int(gs.sum())
    dx0 = fb.gmm_dlhs_fp8(dgu, wi_c, wi_s, gsd, path=0)
    assert torch.equal(bits16(dx[:T]), bits16(dx0[:T])), "pair and streaming paths differ"
    del dx0
    # dLHS cached (contraction 256) equals streaming bit for bit, and the oracle
    c2, s2 = W.fp8_weights(E, K, 256, 0.02, 24, device=DEV)
    d2 = W.cotangent(M, 256, 25, device=DEV)
    a = fb.gmm_dlhs_fp8(d2, c2, s2, gsd, path=1)
    b = fb.gmm_dlhs_fp8(d2, c2, s2, gsd, path=0)
    assert torch.equal(bits16(a[:T]), bits16(b[:T]))
    ref_a, _, bad = orc.gmm_dlhs(d2.cpu(), c2.cpu(), s2.cpu(), gs, rows=rows_b)
    assert bad == 0
    check_bf16(a.cpu()[rows_b], ref_a[rows_b], what="sweep dlhs cached")


def test_microbench_shape_forward_and_dlhs_sampled(orc):
    """The pages' kernel microbenchmark shape (64 experts at full fill, 225,280
    rows, hidden 4096, moe intermediate 1024; every expert ends in a partial
    128-row tile): wi forward + SwiGLU and wo forward on sampled rows, both dLHS
    GMMs on fewer rows."""
    mb = W.MICROBENCH
    gs = W.group_sizes(mb.routing, E=mb.E, M=mb.M)
    gsd = gs.to(DEV)
    x = W.activations(mb.M, mb.K, 51, device=DEV)
    wi_c, wi_s = W.fp8_weights(mb.E, mb.K, 2 * mb.F, mb.sigma_wi, 52, device=DEV)
    wo_c, wo_s = W.fp8_weights(mb.E, mb.F, mb.K, mb.sigma_wo, 53, device=DEV)
    h = fb.gmm_silu_fp8_fwd(x, wi_c, wi_s, gsd)
    y = fb.gmm_fp8_fwd(h, wo_c, wo_s, gsd)
    rows = sample_rows(gs, 0, seed=9)[::3]
    wi_cc, wi_sc, wo_cc, wo_sc = wi_c.cpu(), wi_s.cpu(), wo_c.cpu(), wo_s.cpu()
    ref_h, _, bad = orc.gmm_fwd(x.cpu(), wi_cc, wi_sc, gs, silu=True, rows=rows)
    assert bad == 0
    check_bf16(h.cpu()[rows], ref_h[rows], what="microbench wi fwd")
    ref_y, _, bad = orc.gmm_fwd(h.cpu(), wo_cc, wo_sc, gs, silu=False, rows=rows)
    assert bad == 0
    check_bf16(y.cpu()[rows], ref_y[rows], what="microbench wo fwd")
    del x, y
    dy = W.cotangent(mb.M, mb.K, 54, device=DEV)
    dgu = W.cotangent(mb.M, 2 * mb.F, 55, device=DEV)
    dh = fb.gmm_dlhs_fp8(dy, wo_c, wo_s, gsd)
    dx = fb.gmm_dlhs_fp8(dgu, wi_c, wi_s, gsd)
    rows_b = rows[:: max(1, len(rows) // 16)]
    ref_dh, _, bad = orc.gmm_dlhs(dy.cpu(), wo_cc, wo_sc, gs, rows=rows_b)
    assert bad == 0
    check_bf16(dh.cpu()[rows_b], ref_dh[rows_b], what="microbench wo dlhs")
    ref_dx, _, bad = orc.gmm_dlhs(dgu.cpu(), wi_cc, wi_sc, gs, rows=rows_b)
    assert bad == 0
    check_bf16(dx.cpu()[rows_b], ref_dx[rows_b], what="microbench wi dlhs")


def test_balanced_wo_dlhs_dswiglu_sampled(orc):
    """wo dLHS with the SwiGLU backward fused (balanced layer): gu is the wi
    forward output before SwiGLU, dout ~ N(0, 1); sampled rows vs the oracle."""
    E, K, F, M = 32, 7168, 2048, 32768
    gs = W.group_sizes("balanced", E=E, M=M)
    gsd = gs.to(DEV)
    x = W.activations(M, K, 61, outlier_frac=0.001, device=DEV)
    wi_c, wi_s = W.fp8_weights(E, K, 2 * F, 0.006, 62, device=DEV)
    wo_c, wo_s = W.fp8_weights(E, F, K, 0.006, 63, device=DEV)
    gu = fb.gmm_fp8_fwd(x, wi_c, wi_s, gsd)             # [M, 2F], gate | up
    del x, wi_c
    dy = W.cotangent(M, K, 64, device=DEV)
    dgu = fb.gmm_dlhs_dswiglu_fp8(dy, wo_c, wo_s, gu, gsd)
    assert torch.isfinite(dgu.float()).all()
    rows = sample_rows(gs, 1, seed=11)[::2]
    ref, _, bad = orc.gmm_dlhs_dswiglu(dy.cpu(), wo_c.cpu(), wo_s.cpu(), gu.cpu(), gs, rows=rows)
    assert bad == 0
    check_bf16(dgu.cpu()[rows], ref[rows], what="balanced wo dlhs+dswiglu")


def test_dropless_tgmm_e5m2_blocks_finite_and_tail_blind(orc):
    """The dropless tgmm with the e5m2 gradient dtype: finite, tail-blind, empty
    experts zero, oracle blocks of the largest expert and a small one."""
    E, K, N, M = 32, 7168, 2048, 65536
    gs = W.group_sizes("dropless", seed=2, E=E)
    T = int(gs.sum())
    x = W.fill_tail_garbage(W.activations(M, K, 13, device=DEV), T)
    d = W.fill_tail_garbage(W.cotangent(M, N, 14, device=DEV), T)
    gsd = gs.to(DEV)
    dw = fb.tgmm_drhs_quant(x, d, gsd, dout_fmt="e5m2")
    assert torch.isfinite(dw).all()
    for e in (gs == 0).nonzero().flatten().tolist():
        assert (dw[e] == 0).all()
    x[T:] = float("nan")
    d[T:] = -3.0e38
    dw2 = fb.tgmm_drhs_quant(x, d, gsd, dout_fmt="e5m2")
    assert torch.equal(dw2, dw)
    del dw2
    order = torch.argsort(gs, descending=True).tolist()
    xc, dc = x.cpu(), d.cpu()
    for e, kr, nr in [(order[0], (128, 256), (1024, 1152)), (order[20], (7040, 7168), (0, 128))]:
        ref, bad = orc.tgmm(xc, dc, gs, experts=[e], k_range=kr, n_range=nr, dout_fmt="e5m2")
        assert bad == 0
        check_f32_rel(dw[e, kr[0]:kr[1], nr[0]:nr[1]], ref[0], what=f"tgmm e5m2 e={e}")
