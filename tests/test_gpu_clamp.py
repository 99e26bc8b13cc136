"""GPU parity on the data-dependent part of the group-size contract.

The host cannot see group_sizes without a synchronization, so every entry point
takes them as they are and fixes two kinds of bad input on the device: a
negative size counts as 0, and sizes that add up past the static buffer of M
rows are clipped at M (a group that starts at or past M is empty, the one that
crosses M loses its rows from M on). Each fix sets a bit of the status word
(FP8MOE_STATUS_NEGATIVE_GROUP, FP8MOE_STATUS_GROUPS_EXCEED_M). The oracle clamps
the same way, so the outputs are compared with it at the usual tolerances.

The bad sizes are made here on the host; they are the documented input of every
call, not a fault."""
import pytest
import torch

from fp8_moe_routed_gb300 import binding as fb
from fp8_moe_routed_gb300 import workloads as W
from parity_util import bits16, check_bf16, check_f32_rel

pytestmark = pytest.mark.gpu

DEV = "cuda"
NEG, EXC = fb.STATUS_NEGATIVE_GROUP, fb.STATUS_GROUPS_EXCEED_M
M = 640

# group sizes, status bits expected, and the effective row ranges they clamp to
CASES = {
    # T = 500: expert 1 counts as empty
    "negative": ([200, -50, 160, 140], NEG),
    # sum 900 > 640: expert 2 keeps 130 of its 300 rows, expert 3 starts past M
    "exceed": ([250, 260, 300, 90], EXC),
    # both at once: expert 0 negative, expert 2 crosses M
    "both": ([-7, 400, 300, 0], NEG | EXC),
}


def effective(gs):
    """(begin, end) of every expert after the clamp, and T."""
    out, off = [], 0
    for g in gs:
        g = max(g, 0)
        out.append((min(off, M), min(off + g, M)))
        off += g
    return out, min(off, M)


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


def _gs(name):
    sizes, bits = CASES[name]
    return torch.tensor(sizes, dtype=torch.int32), bits, effective(sizes)[1]


def _expect(bits, what):
    st = fb.read_status()
    assert st == bits, f"{what}: status {st:#x}, expected {bits:#x}"


def test_effective_ranges_are_what_the_cases_say():
    assert effective(CASES["negative"][0]) == ([(0, 200), (200, 200), (200, 360), (360, 500)], 500)
    assert effective(CASES["exceed"][0]) == ([(0, 250), (250, 510), (510, 640), (640, 640)], 640)
    assert effective(CASES["both"][0]) == ([(0, 0), (0, 400), (400, 640), (640, 640)], 640)


@pytest.mark.parametrize("name", list(CASES))
def test_quantizers_clamp(orc, name):
    gs, bits, T = _gs(name)
    K = 1024
    x = W.fill_tail_garbage(W.activations(M, K, 3, outlier_frac=0.02), T)
    q, sx = fb.quantize_rows(x.to(DEV), gs.to(DEV))
    _expect(bits, "quantize_rows")
    rq, rsx, bad = orc.quantize_rows(x, gs)
    assert bad == 0
    assert torch.equal(q.cpu()[:T], rq[:T]) and torch.equal(sx.cpu()[:T], rsx[:T])
    assert torch.isnan(sx.cpu()[T:]).all()
    qb, sb = fb.quantize_rows_block(x.to(DEV), gs.to(DEV))
    _expect(bits, "quantize_rows_block")
    rqb, rsb, bad = orc.quantize_rows_block(x, gs)
    assert bad == 0
    assert torch.equal(qb.cpu()[:T], rqb[:T]) and torch.equal(sb.cpu()[:T], rsb[:T])


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("silu", [True, False])
def test_forward_clamp(orc, name, silu):
    gs, bits, T = _gs(name)
    K, N, E = 512, 512, 4
    x = W.fill_tail_garbage(W.activations(M, K, 5, outlier_frac=0.01), T)
    codes, scale = W.fp8_weights(E, K, N, 0.02, 6)
    Nout = N // 2 if silu else N
    out = torch.full((M, Nout), 7.0, dtype=torch.bfloat16, device=DEV)
    fn = fb.gmm_silu_fp8_fwd if silu else fb.gmm_fp8_fwd
    fn(x.to(DEV), codes.to(DEV), scale.to(DEV), gs.to(DEV), out=out)
    _expect(bits, "forward")
    ref, _, bad = orc.gmm_fwd(x, codes, scale, gs, silu=silu)
    assert bad == 0
    check_bf16(out[:T], ref[:T], what=f"clamp {name} fwd silu={silu}")
    assert (out[T:].float() == 7.0).all()
    # the BF16 comparison GMM on the same clamp
    w = orc.dequantize(codes, scale)
    outb = torch.full((M, Nout), 7.0, dtype=torch.bfloat16, device=DEV)
    fb.gmm_bf16_fwd(x.to(DEV), w.to(DEV), gs.to(DEV), silu, out=outb)
    _expect(bits, "bf16 forward")
    assert (outb[T:].float() == 7.0).all()
    assert torch.isfinite(outb[:T].float()).all()


@pytest.mark.parametrize("name", list(CASES))
def test_block_forward_clamp(orc, name):
    gs, bits, T = _gs(name)
    K, N, E = 1024, 256, 4
    x = W.fill_tail_garbage(W.activations(M, K, 7), T)
    codes, scale = W.fp8_weights(E, K, N, 0.05, 8)
    out = torch.full((M, N), 7.0, dtype=torch.bfloat16, device=DEV)
    fb.gmm_fp8_fwd_block(x.to(DEV), codes.to(DEV), scale.to(DEV), gs.to(DEV), False, out=out)
    _expect(bits, "block forward")
    ref, _, _, bad = orc.gmm_fwd_block(x, codes, scale, gs, silu=False)
    assert bad == 0
    assert (out[T:].float() == 7.0).all()
    same = (bits16(out[:T]) == bits16(ref[:T])).float().mean().item()
    assert same > 0.95, same


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("N,path", [(512, 0), (512, 2), (256, 1)])
def test_dlhs_clamp(orc, name, N, path):
    gs, bits, T = _gs(name)
    K, E = 384, 4
    d = W.fill_tail_garbage(W.cotangent(M, N, 9), T)
    codes, scale = W.fp8_weights(E, K, N, 0.02, 10)
    out = torch.full((M, K), 7.0, dtype=torch.bfloat16, device=DEV)
    fb.gmm_dlhs_fp8(d.to(DEV), codes.to(DEV), scale.to(DEV), gs.to(DEV), out=out, path=path)
    _expect(bits, f"dlhs path {path}")
    ref, _, bad = orc.gmm_dlhs(d, codes, scale, gs)
    assert bad == 0
    check_bf16(out[:T], ref[:T], what=f"clamp {name} dlhs path {path}")
    assert (out[T:].float() == 7.0).all()


@pytest.mark.parametrize("name", list(CASES))
def test_dlhs_dswiglu_clamp(orc, name):
    gs, bits, T = _gs(name)
    F, N, E = 256, 512, 4
    d = W.fill_tail_garbage(W.cotangent(M, N, 11), T)
    gu = W.fill_tail_garbage(W.activations(M, 2 * F, 12), T)
    codes, scale = W.fp8_weights(E, F, N, 0.02, 13)
    out = torch.full((M, 2 * F), 7.0, dtype=torch.bfloat16, device=DEV)
    fb.gmm_dlhs_dswiglu_fp8(d.to(DEV), codes.to(DEV), scale.to(DEV), gu.to(DEV), gs.to(DEV),
                            out=out)
    _expect(bits, "dlhs dswiglu")
    ref, _, bad = orc.gmm_dlhs_dswiglu(d, codes, scale, gu, gs)
    assert bad == 0
    check_bf16(out[:T], ref[:T], what=f"clamp {name} dlhs dswiglu")
    assert (out[T:].float() == 7.0).all()


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_tgmm_clamp(orc, name, fmt):
    gs, bits, T = _gs(name)
    K, N = 256, 384
    x = W.fill_tail_garbage(W.activations(M, K, 14, outlier_frac=0.02), T)
    d = W.fill_tail_garbage(W.cotangent(M, N, 15), T)
    qx, sx, qd, sd = fb.tgmm_quantize_tiles(x.to(DEV), d.to(DEV), gs.to(DEV), dout_fmt=fmt)
    _expect(bits, "tgmm_quantize_tiles")
    rqx, rsx, rqd, rsd, nseg, bad = orc.tgmm_quantize_tiles(x, d, gs, dout_fmt=fmt)
    assert bad == 0
    assert torch.equal(qx.cpu()[:nseg], rqx[:nseg]) and torch.equal(sx.cpu()[:nseg], rsx[:nseg])
    assert torch.equal(qd.cpu()[:nseg], rqd[:nseg]) and torch.equal(sd.cpu()[:nseg], rsd[:nseg])
    dw = fb.tgmm_drhs_quant(x.to(DEV), d.to(DEV), gs.to(DEV), dout_fmt=fmt)
    _expect(bits, "tgmm_drhs_quant")
    ref, bad = orc.tgmm(x, d, gs, dout_fmt=fmt)
    assert bad == 0
    rng, _ = effective(CASES[name][0])
    for e, (b, en) in enumerate(rng):
        if b == en:
            assert (dw[e] == 0).all(), f"expert {e} has no rows after the clamp"
        else:
            check_f32_rel(dw[e], ref[e], what=f"clamp {name} tgmm {fmt} e={e}")


@pytest.mark.parametrize("name", ["negative", "exceed"])
def test_noalloc_forward_clamp(name):
    gs, bits, T = _gs(name)
    K, N, E = 512, 512, 4
    x = W.fill_tail_garbage(W.activations(M, K, 16), T).to(DEV)
    codes, scale = W.fp8_weights(E, K, N, 0.02, 17, device=DEV)
    a = torch.full((M, N // 2), 7.0, dtype=torch.bfloat16, device=DEV)
    b = torch.full((M, N // 2), 7.0, dtype=torch.bfloat16, device=DEV)
    fb.gmm_silu_fp8_fwd(x, codes, scale, gs.to(DEV), out=a)
    _expect(bits, "forward")
    fb.gmm_silu_fp8_fwd_noalloc(x, codes, scale, gs.to(DEV), b)
    _expect(bits, "noalloc forward")
    assert torch.equal(bits16(a), bits16(b))
