"""Pins of the oracle's path functions against things other than itself.

* row quantization: closed forms (power-of-two amax gives an exact scale),
  power-of-two invariance, the amax element maps to +-448, torch's float8 cast
  reproduces the codes given the scale, tail rows never read;
* forward GMM: equal to a dense float64 matmul with a block-diagonal expert mask
  (torch.matmul), SwiGLU equal to torch.nn.functional.silu, a lossless special
  case that reduces to the plain matmul, zero-size groups write nothing, locality;
* dequantization: bit-identical to torch's codes x scale -> bf16;
* dLHS: float64 torch matmul per group with the dequantized weights;
* dSwiGLU (the SwiGLU backward fused into the wo dLHS): torch autograd of
  silu(g) * u in float64, exact special values, and the fused op equal to a
  per-group float64 matmul followed by autograd;
* tgmm: a lossless special case equal to X_e^T D_e (textbook), brute force in
  plain Python on a tiny case, tail invariance, locality, empty experts.

Page references: "MoE: native FP8 QAT for routed-expert GMMs" (Description,
Implementation, Tests) and "MoE fp8 backward: in-kernel drhs operand
quantization" (What).
"""
import math

import numpy as np
import pytest
import torch

from fp8_moe_routed_gb300 import workloads as W

F8 = torch.float8_e4m3fn


def dec(codes):
    return codes.view(F8).to(torch.float64)


def small_case(M=96, K=64, N=48, E=3, gs=(30, 0, 50), seed=0, wsig=0.05):
    gs = torch.tensor(gs, dtype=torch.int32)
    x = W.activations(M, K, seed)
    codes, scale = W.fp8_weights(E, K, N, wsig, seed + 1)
    return x, codes, scale, gs


def expert_of_rows(gs, M):
    e_of = torch.full((M,), -1, dtype=torch.long)
    off = 0
    for e, g in enumerate(gs.tolist()):
        e_of[off:off + g] = e
        off += g
    return e_of, off


# ---------------------------------------------------------------- a1 row quant
def test_row_scale_power_of_two_closed_form(orc):
    K = 40
    rows = []
    for j in range(-6, 7):
        r = torch.linspace(-1, 1, K) * 448.0 * 2.0 ** j * 0.5
        r[3] = 448.0 * 2.0 ** j          # amax exactly 448 * 2^j
        rows.append(r)
    x = torch.stack(rows).to(torch.bfloat16)
    gs = torch.tensor([x.shape[0]], dtype=torch.int32)
    q, sx, bad = orc.quantize_rows(x, gs)
    assert bad == 0
    assert sx.tolist() == [2.0 ** j for j in range(-6, 7)]
    assert (q[:, 3] == 0x7E).all()


def test_row_quant_power_of_two_invariance(orc):
    x = W.activations(64, 256, seed=5)
    gs = torch.tensor([64], dtype=torch.int32)
    q0, s0, _ = orc.quantize_rows(x, gs)
    for j in (-8, -1, 1, 3, 10):
        q1, s1, _ = orc.quantize_rows((x.float() * 2.0 ** j).to(torch.bfloat16), gs)
        assert torch.equal(q0, q1)
        assert torch.equal(s1, s0 * 2.0 ** j)


def test_row_quant_amax_maps_to_448_and_codes_match_torch_cast(orc):
    x = W.activations(200, 384, seed=11, outlier_frac=0.05)
    gs = torch.tensor([120, 80], dtype=torch.int32)
    q, sx, bad = orc.quantize_rows(x, gs)
    assert bad == 0
    xf = x.float()
    amax = xf.abs().amax(dim=1)
    assert torch.equal(sx, torch.maximum(amax, torch.tensor(1e-12, dtype=torch.float32)) / 448.0)
    ref = (xf / sx[:, None]).clamp(-448, 448).to(F8).view(torch.uint8)
    assert torch.equal(q, ref)
    arg = xf.abs().argmax(dim=1)
    top = q[torch.arange(200), arg]
    assert bool(((top == 0x7E) | (top == 0xFE)).all())


def test_row_quant_zero_row_and_tail(orc):
    x = W.activations(10, 32, seed=2)
    x[1] = 0
    x = W.fill_tail_garbage(x, 6)
    gs = torch.tensor([2, 0, 4], dtype=torch.int32)  # T = 6
    q, sx, bad = orc.quantize_rows(x, gs, fill_q=0xAB)
    assert bad == 0
    assert (q[1] == 0).all() and sx[1].item() > 0 and sx[1].item() < 1e-14
    assert (q[6:] == 0xAB).all() and torch.isnan(sx[6:]).all()
    assert torch.isfinite(sx[:6]).all()


# ----------------------------------------------------------- a2-a4 forward GMM
def dense_block_diag_reference(x, codes, scale, gs, q=None, sx=None):
    """sum_e mask_e * (Xdeq @ W_e) in float64 with torch's own float8 cast."""
    M, K = x.shape
    xf = x.float()
    if sx is None:
        amax = xf.abs().amax(dim=1)
        sx = torch.maximum(amax, torch.tensor(1e-12)) / 448.0
    qx = (xf / sx[:, None]).clamp(-448, 448).to(F8)
    xdeq = qx.to(torch.float64) * sx.double()[:, None]
    e_of, T = expert_of_rows(gs, M)
    out = torch.zeros(M, codes.shape[2], dtype=torch.float64)
    for e in range(codes.shape[0]):
        we = dec(codes[e]) * scale[e].double()[None, :]
        mask = (e_of == e).double()[:, None]
        out += mask * (xdeq @ we)
    return out, T


def test_gmm_fwd_equals_block_diagonal_dense_matmul(orc):
    x, codes, scale, gs = small_case()
    out, out64, bad = orc.gmm_fwd(x, codes, scale, gs, silu=False, want_f64=True)
    assert bad == 0
    ref, T = dense_block_diag_reference(x, codes, scale, gs)
    assert torch.allclose(out64[:T], ref[:T], rtol=1e-12, atol=1e-300)
    assert torch.equal(out[:T].view(torch.int16), orc.f64_to_bf16(out64[:T]).view(torch.int16))


def test_gmm_fwd_swiglu_matches_torch_silu(orc):
    x, codes, scale, gs = small_case(N=64)
    out, out64, bad = orc.gmm_fwd(x, codes, scale, gs, silu=True, want_f64=True)
    assert bad == 0
    ref, T = dense_block_diag_reference(x, codes, scale, gs)
    g, u = ref[:, :32], ref[:, 32:]
    sw = torch.nn.functional.silu(g) * u
    assert torch.allclose(out64[:T], sw[:T], rtol=1e-11, atol=1e-300)
    assert out.shape == (x.shape[0], 32)


def test_gmm_fwd_lossless_case_is_plain_matmul(orc):
    """Rows on the e4m3 grid with amax 448: the scale is 1 and the codes are the
    values, so the GMM is the plain matmul with the dequantized weight."""
    M, K, N, E = 64, 96, 40, 2
    g = torch.Generator().manual_seed(9)
    codes_x = torch.randint(0, 256, (M, K), generator=g, dtype=torch.uint8)
    codes_x[(codes_x & 0x7F) == 0x7F] = 0x10
    codes_x[:, 5] = 0x7E
    x = codes_x.view(F8).to(torch.bfloat16)           # exact: e4m3 values fit bf16
    codes, scale = W.fp8_weights(E, K, N, 0.1, 4)
    gs = torch.tensor([20, 44], dtype=torch.int32)
    _, out64, bad = orc.gmm_fwd(x, codes, scale, gs, silu=False, want_f64=True)
    assert bad == 0
    xs = x.double()
    for e, (a, b) in enumerate([(0, 20), (20, 64)]):
        ref = xs[a:b] @ (dec(codes[e]) * scale[e].double()[None, :])
        assert torch.allclose(out64[a:b], ref, rtol=1e-13, atol=0)


def test_gmm_fwd_zero_groups_and_tail_write_nothing(orc):
    M, K, N = 80, 64, 32
    x = W.activations(M, K, 1)
    x = W.fill_tail_garbage(x, 50)
    codes, scale = W.fp8_weights(4, K, N, 0.05, 2)
    gs = torch.tensor([0, 30, 0, 20], dtype=torch.int32)    # T = 50
    sentinel = 0x7BCD
    out, _, bad = orc.gmm_fwd(x, codes, scale, gs, silu=False, fill=sentinel)
    assert bad == 0
    o = out.view(torch.int16)
    assert (o[50:] == sentinel).all()
    assert (o[:50] != sentinel).all() and torch.isfinite(out[:50].float()).all()


def test_gmm_fwd_locality_and_tail_invariance(orc):
    x, codes, scale, gs = small_case(M=100, gs=(30, 10, 40))   # T = 80
    base, _, _ = orc.gmm_fwd(x, codes, scale, gs, silu=False)
    x2 = x.clone()
    x2[35] *= 3                                                 # a row of group 1
    x2 = W.fill_tail_garbage(x2, 80)
    pert, _, bad = orc.gmm_fwd(x2, codes, scale, gs, silu=False)
    assert bad == 0
    changed = (pert.view(torch.int16) != base.view(torch.int16)).any(dim=1)
    assert changed.nonzero().flatten().tolist() == [35]


def test_gmm_fwd_sampled_rows_equal_full(orc):
    x, codes, scale, gs = small_case()
    full, _, _ = orc.gmm_fwd(x, codes, scale, gs, silu=True)
    rows = torch.tensor([0, 29, 30, 79])
    part, _, bad = orc.gmm_fwd(x, codes, scale, gs, silu=True, rows=rows)
    assert bad == 0
    assert torch.equal(part[rows].view(torch.int16), full[rows].view(torch.int16))
    _, _, bad = orc.gmm_fwd(x, codes, scale, gs, silu=True, rows=torch.tensor([80, 95]))
    assert bad == 2    # rows past T are refused and counted


# ------------------------------------------------------------- a5 dequantize
def test_dequantize_bit_identical_to_codes_times_scale(orc):
    E, K, N = 3, 256, 64
    g = torch.Generator().manual_seed(1)
    codes = torch.arange(E * K * N, dtype=torch.int64).remainder(256).to(torch.uint8)
    codes = codes.view(E, K, N)
    scale = torch.exp(torch.randn(E, N, generator=g) * 4).float()
    out = orc.dequantize(codes, scale)
    ref = (codes.view(F8).float() * scale[:, None, :]).to(torch.bfloat16)
    o, r = out.float(), ref.float()
    nan = torch.isnan(r)
    assert torch.equal(torch.isnan(o), nan)
    assert torch.equal(out.view(torch.int16)[~nan], ref.view(torch.int16)[~nan])


# ------------------------------------------------------------------- a6 dLHS
def test_dlhs_matches_float64_matmul_per_group(orc):
    M, N, K, E = 90, 64, 48, 3
    gs = torch.tensor([25, 0, 55], dtype=torch.int32)
    d = W.cotangent(M, N, 3)
    d = W.fill_tail_garbage(d, 80)
    codes, scale = W.fp8_weights(E, K, N, 0.05, 6)
    out, out64, bad = orc.gmm_dlhs(d, codes, scale, gs, want_f64=True, fill=0x7BCD)
    assert bad == 0
    wb = (codes.view(F8).float() * scale[:, None, :]).to(torch.bfloat16).double()
    for e, (a, b) in enumerate([(0, 25), (25, 25), (25, 80)]):
        if b > a:
            ref = d[a:b].double() @ wb[e].T
            assert torch.allclose(out64[a:b], ref, rtol=1e-12, atol=1e-300)
    assert (out.view(torch.int16)[80:] == 0x7BCD).all()


# ----------------------------------- per-512 block quantization (NEXT-3)
def test_block_quant_scales_and_codes_match_torch(orc):
    """s[m, b] = bf16(max(amax over the block, 1e-12) / 448) in f32 then bf16 (torch),
    codes = torch's float8_e4m3fn cast of x / s; K = 1280 has a partial last block."""
    M, K = 24, 1280
    x = W.activations(M, K, 41)
    x[3, 512:1024] = 0.0                                     # an all-zero block
    gs = torch.tensor([10, 14], dtype=torch.int32)
    q, sb, bad = orc.quantize_rows_block(x, gs)
    assert bad == 0 and sb.shape == (M, 3)
    xf = x.float()
    for b, (k0, k1) in enumerate([(0, 512), (512, 1024), (1024, 1280)]):
        amax = xf[:, k0:k1].abs().amax(dim=1)
        s = (torch.clamp(amax, min=1e-12) / 448.0).to(torch.bfloat16).float()
        assert torch.equal(sb[:, b], s)
        ref = (xf[:, k0:k1] / s[:, None]).to(F8).view(torch.uint8)
        assert torch.equal(q[:, k0:k1], ref)
    assert sb[3, 1].item() == torch.tensor(1e-12 / 448.0).to(torch.bfloat16).float().item()


def test_block_quant_blocks_are_independent(orc):
    M, K = 8, 1536
    x = W.activations(M, K, 42)
    gs = torch.tensor([M], dtype=torch.int32)
    q, sb, _ = orc.quantize_rows_block(x, gs)
    x2 = x.clone()
    x2[:, 600:700] *= 37.0                                   # only block 1 changes
    q2, sb2, _ = orc.quantize_rows_block(x2, gs)
    assert torch.equal(q[:, :512], q2[:, :512]) and torch.equal(q[:, 1024:], q2[:, 1024:])
    assert torch.equal(sb[:, [0, 2]], sb2[:, [0, 2]]) and not torch.equal(sb[:, 1], sb2[:, 1])


def test_gmm_fwd_block_restated_in_python(orc):
    """Plain-Python restatement on a tiny case (K = 1280: blocks 512, 512, 256):
    the exact block product rounded to f32, acc = bf16(acc + d * s) with one
    rounding (the oracle's pinned f64 -> bf16), then * sw and one last rounding."""
    M, K, N, E = 6, 1280, 8, 2
    gs = torch.tensor([2, 4], dtype=torch.int32)
    x = W.activations(M, K, 43)
    codes, scale = W.fp8_weights(E, K, N, 0.05, 44)
    out, out64, amx, bad = orc.gmm_fwd_block(x, codes, scale, gs, silu=False, want_f64=True,
                                             want_acc_max=True)
    assert bad == 0
    q, sb, _ = orc.quantize_rows_block(x, gs)
    qd = q.view(F8).double().numpy()
    wd = codes.view(F8).double().numpy()
    for m in range(M):
        e = 0 if m < 2 else 1
        for n in range(N):
            acc = 0.0
            for b, (k0, k1) in enumerate([(0, 512), (512, 1024), (1024, 1280)]):
                d = float(np.float32(np.dot(qd[m, k0:k1], wd[e, k0:k1, n])))
                v = acc + d * float(sb[m, b])
                acc = float(orc.f64_to_bf16(torch.tensor([v], dtype=torch.float64)).float())
            y = acc * float(scale[e, n])
            assert out64[m, n].item() == y
            assert out[m, n].view(torch.int16) == orc.f64_to_bf16(torch.tensor([y])).view(torch.int16)[0]


def test_gmm_fwd_block_lossless_case_is_integer_matmul(orc):
    """Every block of every row holds one 448 (on a weight row of zeros) and
    small integers elsewhere; weights are 0 / +-1 with channel scale 1: every
    block scale is 1, codes and block products are exact integers below 256 and
    the bf16 accumulation is exact, so the result equals the integer matmul."""
    M, K, N, E = 16, 1536, 12, 1
    g = torch.Generator().manual_seed(45)
    x = torch.zeros(M, K)
    nz = torch.rand(M, K, generator=g) < 0.02
    x[nz] = torch.randint(-2, 3, (int(nz.sum()),), generator=g).float()
    for b in range(3):
        x[:, 512 * b + 7] = 448.0
    w = torch.randint(-1, 2, (K, N), generator=g).float()
    for b in range(3):
        w[512 * b + 7] = 0.0
    codes = w.to(F8).view(torch.uint8)[None].contiguous()
    scale = torch.ones(E, N)
    gs = torch.tensor([M], dtype=torch.int32)
    out, out64, _, bad = orc.gmm_fwd_block(x.to(torch.bfloat16), codes, scale, gs, silu=False,
                                           want_f64=True)
    assert bad == 0
    ref = x.double() @ w.double()
    assert ref.abs().max() < 256
    assert torch.equal(out64, ref)
    full, _, _ = orc.gmm_fwd(x.to(torch.bfloat16), codes, scale, gs, silu=False)
    assert torch.equal(out.view(torch.int16), full.view(torch.int16))


# ------------------------------------------------------ dSwiGLU (wo backward)
def _autograd_dswiglu(dh64, gu):
    """Gradients of sum(dh * silu(g) * u) w.r.t. g and u, float64 autograd."""
    F = dh64.shape[1]
    g = gu[:, :F].double().clone().requires_grad_(True)
    u = gu[:, F:].double().clone().requires_grad_(True)
    (torch.nn.functional.silu(g) * u).backward(dh64)
    return g.grad, u.grad


def test_dswiglu_matches_float64_autograd(orc):
    M, F = 40, 24
    gen = torch.Generator().manual_seed(3)
    dh = torch.randn(M, F, generator=gen, dtype=torch.float64) * 3
    gu = (torch.randn(M, 2 * F, generator=gen) * 4).to(torch.bfloat16)
    out, out64 = orc.dswiglu(dh, gu, want_f64=True)
    dg, du = _autograd_dswiglu(dh, gu)
    assert torch.allclose(out64[:, :F], dg, rtol=1e-12, atol=1e-300)
    assert torch.allclose(out64[:, F:], du, rtol=1e-12, atol=1e-300)
    # one rounding to bf16 of the exact value
    assert torch.equal(out.view(torch.int16), orc.f64_to_bf16(out64).view(torch.int16))


def test_dswiglu_special_values(orc):
    # g = 0: silu(0) = 0 and silu'(0) = 1/2 -> du = 0, dg = dh * u / 2 (exact)
    # large |g|: sig -> 1 (silu' -> 1, silu -> g) or sig -> 0 (both -> 0)
    F = 4
    gu = torch.tensor([[0.0, 0.0, 60.0, -80.0, 2.0, -3.0, 1.5, 0.25]], dtype=torch.bfloat16)
    dh = torch.tensor([[1.5, -0.75, 2.0, 5.0]], dtype=torch.float64)
    _, out64 = orc.dswiglu(dh, gu, want_f64=True)
    assert out64[0, 0].item() == 1.5 * 2.0 / 2 and out64[0, 1].item() == -0.75 * -3.0 / 2
    assert out64[0, F + 0].item() == 0.0 and out64[0, F + 1].item() == 0.0
    assert abs(out64[0, 2].item() - 2.0 * 1.5) < 1e-20          # silu'(60) = 1 - O(60 e^-60)
    assert abs(out64[0, F + 2].item() - 2.0 * 60.0) < 1e-20
    assert abs(out64[0, 3].item()) < 1e-30 and abs(out64[0, F + 3].item()) < 1e-30


def test_gmm_dlhs_dswiglu_is_matmul_then_autograd(orc):
    M, N, F, E = 90, 64, 40, 3
    gs = torch.tensor([25, 0, 55], dtype=torch.int32)
    d = W.fill_tail_garbage(W.cotangent(M, N, 13), 80)
    gu = W.fill_tail_garbage(W.activations(M, 2 * F, 14), 80)
    codes, scale = W.fp8_weights(E, F, N, 0.05, 15)
    out, out64, bad = orc.gmm_dlhs_dswiglu(d, codes, scale, gu, gs, want_f64=True, fill=0x7BCD)
    assert bad == 0
    wb = (codes.view(F8).float() * scale[:, None, :]).to(torch.bfloat16).double()
    for e, (a, b) in enumerate([(0, 25), (25, 25), (25, 80)]):
        if b > a:
            dh = d[a:b].double() @ wb[e].T
            dg, du = _autograd_dswiglu(dh, gu[a:b])
            assert torch.allclose(out64[a:b, :F], dg, rtol=1e-9, atol=1e-12)
            assert torch.allclose(out64[a:b, F:], du, rtol=1e-9, atol=1e-12)
    assert (out.view(torch.int16)[80:] == 0x7BCD).all()


# ------------------------------------------------------------------- a7-a8 tgmm
def test_tgmm_lossless_case_is_textbook_xt_d(orc):
    """Every channel of every segment on the e4m3 grid with amax 448 -> all
    scales are 1 -> dW_e = X_e^T D_e exactly (rounded to f32)."""
    M, K, N = 300, 24, 20
    gs = torch.tensor([100, 150, 0, 40], dtype=torch.int32)    # T = 290, straddles
    g = torch.Generator().manual_seed(2)

    def grid(rows, cols):
        c = torch.randint(0, 256, (rows, cols), generator=g, dtype=torch.uint8)
        c[(c & 0x7F) == 0x7F] = 0x20
        return c.view(F8).to(torch.float32)

    x = grid(M, K)
    d = grid(M, N)
    # put +-448 in every column of every segment
    bounds = [(0, 100), (100, 250), (250, 290)]
    for a, b in bounds:
        for t in range(a // 128, (b - 1) // 128 + 1):
            r = max(a, 128 * t)
            x[r] = 448.0
            d[r] = -448.0
    x, d = x.to(torch.bfloat16), d.to(torch.bfloat16)
    x = W.fill_tail_garbage(x, 290)
    d = W.fill_tail_garbage(d, 290)
    dW, bad = orc.tgmm(x, d, gs)
    assert bad == 0
    for e, (a, b) in zip([0, 1, 3], bounds):
        ref = (x[a:b].double().T @ d[a:b].double()).float()
        assert torch.equal(dW[e], ref)
    assert (dW[2] == 0).all()


def test_tgmm_bruteforce_tiny(orc):
    """Plain Python restatement on a tiny case: segments, per-channel scales in
    f32 (numpy), codes by torch's float8 cast, double dot products."""
    M, K, N = 260, 3, 2
    gs = [70, 100, 0, 60]             # T = 230; tile 0 holds groups 0,1; tile 1 holds 1,3
    x = W.activations(M, K, 21)
    d = W.cotangent(M, N, 22)
    x = W.fill_tail_garbage(x, 230)
    dW, bad = orc.tgmm(x, d, torch.tensor(gs, dtype=torch.int32))
    assert bad == 0
    xf = x.float().numpy()
    df = d.float().numpy()
    off = 0
    for e, g in enumerate(gs):
        ref = np.zeros((K, N))
        a, b = off, off + g
        off += g
        if g == 0:
            assert (dW[e] == 0).all()
            continue
        for t in range(a // 128, (b - 1) // 128 + 1):
            r0, r1 = max(a, 128 * t), min(b, 128 * t + 128)
            def quant(col):
                amax = np.float32(np.abs(col).max())
                s = np.float32(max(amax, np.float32(1e-12))) / np.float32(448.0)
                q = torch.from_numpy((col / s).astype(np.float32)).to(F8).double().numpy()
                return s, q
            for k in range(K):
                sk, qk = quant(xf[r0:r1, k])
                for n in range(N):
                    sn, qn = quant(df[r0:r1, n])
                    ref[k, n] += float(sk) * float(sn) * float(np.dot(qk, qn))
        assert np.array_equal(dW[e].numpy(), ref.astype(np.float32))


F8E5 = torch.float8_e5m2


def test_tgmm_e5m2_lossless_case_is_textbook_xt_d(orc):
    """e5m2 gradient operand ("MoE fp8 backward ...", What: configurable gradient
    dtype): x channels on the e4m3 grid with amax 448 and dout channels on the
    e5m2 grid with amax 57344 in every segment -> all scales are 1 -> dW_e =
    X_e^T D_e exactly. dout codes keep |v| >= 2^-6 so every double sum is exact."""
    M, K, N = 300, 20, 24
    gs = torch.tensor([100, 150, 0, 40], dtype=torch.int32)
    g = torch.Generator().manual_seed(4)
    c = torch.randint(0, 256, (M, K), generator=g, dtype=torch.uint8)
    c[(c & 0x7F) == 0x7F] = 0x20
    x = c.view(F8).to(torch.float32)
    e = torch.randint(0x0C, 0x7C, (M, N), generator=g, dtype=torch.uint8)   # 2^-6 .. 57344
    e |= (torch.randint(0, 2, (M, N), generator=g, dtype=torch.uint8) << 7)
    d = e.view(F8E5).to(torch.float32)
    bounds = [(0, 100), (100, 250), (250, 290)]
    for a, b in bounds:
        for t in range(a // 128, (b - 1) // 128 + 1):
            r = max(a, 128 * t)
            x[r] = -448.0
            d[r] = 57344.0
    x = W.fill_tail_garbage(x.to(torch.bfloat16), 290)
    d = W.fill_tail_garbage(d.to(torch.bfloat16), 290)
    dW, bad = orc.tgmm(x, d, gs, dout_fmt="e5m2")
    assert bad == 0
    for ex, (a, b) in zip([0, 1, 3], bounds):
        ref = (x[a:b].double().T @ d[a:b].double()).float()
        assert torch.equal(dW[ex], ref)
    assert (dW[2] == 0).all()
    _, sx, _, sd, nseg, bad = orc.tgmm_quantize_tiles(x, d, gs, dout_fmt="e5m2")
    assert bad == 0 and (sx[:nseg] == 1.0).all() and (sd[:nseg] == 1.0).all()


def test_tgmm_e5m2_bruteforce_tiny(orc):
    """Plain Python restatement with an e5m2 dout operand: segments, f32
    per-channel scales max(amax, 1e-12)/57344 (numpy), codes by torch's
    float8_e5m2 cast, double dot products."""
    M, K, N = 260, 3, 2
    gs = [70, 100, 0, 60]
    x = W.fill_tail_garbage(W.activations(M, K, 23), 230)
    d = W.cotangent(M, N, 24) * 1000
    dW, bad = orc.tgmm(x, d, torch.tensor(gs, dtype=torch.int32), dout_fmt="e5m2")
    assert bad == 0
    xf, df = x.float().numpy(), d.float().numpy()

    def quant(col, fmax, dt):
        amax = np.float32(np.abs(col).max())
        s = np.float32(max(amax, np.float32(1e-12))) / np.float32(fmax)
        return s, torch.from_numpy((col / s).astype(np.float32)).to(dt).double().numpy()

    off = 0
    for e, g in enumerate(gs):
        ref = np.zeros((K, N))
        a, b = off, off + g
        off += g
        if g == 0:
            assert (dW[e] == 0).all()
            continue
        for t in range(a // 128, (b - 1) // 128 + 1):
            r0, r1 = max(a, 128 * t), min(b, 128 * t + 128)
            for k in range(K):
                sk, qk = quant(xf[r0:r1, k], 448.0, F8)
                for n in range(N):
                    sn, qn = quant(df[r0:r1, n], 57344.0, F8E5)
                    ref[k, n] += float(sk) * float(sn) * float(np.dot(qk, qn))
        assert np.array_equal(dW[e].numpy(), ref.astype(np.float32))


def test_tgmm_tail_invariance_locality_empty(orc):
    M, K, N = 512, 32, 16
    gs = torch.tensor([0, 130, 77, 0, 90], dtype=torch.int32)   # T = 297
    x = W.activations(M, K, 31)
    d = W.cotangent(M, N, 32)
    base, bad = orc.tgmm(x, d, gs)
    assert bad == 0
    x2, d2 = W.fill_tail_garbage(x.clone(), 297), W.fill_tail_garbage(d.clone(), 297)
    tail, bad = orc.tgmm(x2, d2, gs)
    assert bad == 0 and torch.equal(tail, base) and torch.isfinite(tail).all()
    assert (base[0] == 0).all() and (base[3] == 0).all()
    x3 = x.clone()
    x3[140] *= 2          # group 1 covers rows [0, 130) ... group 2 covers [130, 207)
    pert, _ = orc.tgmm(x3, d, gs)
    diff = [(pert[e] != base[e]).any().item() for e in range(5)]
    assert diff == [False, False, True, False, False]


def test_tgmm_quantize_tiles_layout(orc):
    M, K, N = 400, 40, 24
    gs = torch.tensor([100, 0, 200, 60], dtype=torch.int32)     # T = 360
    x = W.fill_tail_garbage(W.activations(M, K, 41), 360)
    d = W.fill_tail_garbage(W.cotangent(M, N, 42), 360)
    qx, sx, qd, sd, nseg, bad = orc.tgmm_quantize_tiles(x, d, gs)
    assert bad == 0
    # segments: e0 tile0 [0,100); e2 tiles 0,1,2 -> [100,128),[128,256),[256,300);
    # e3 tiles 2 -> [300,360)
    segs = [(0, 0, 100), (0, 100, 128), (1, 128, 256), (2, 256, 300), (2, 300, 360)]
    assert nseg == len(segs)
    for q, (t, r0, r1) in enumerate(segs):
        for src, qq, ss in ((x, qx, sx), (d, qd, sd)):
            rows = src[r0:r1].float()
            s = torch.maximum(rows.abs().amax(dim=0), torch.tensor(1e-12)) / 448.0
            assert torch.equal(ss[q], s)
            ref = (rows / s[None, :]).clamp(-448, 448).to(F8).view(torch.uint8)
            slot = qq[q]
            assert torch.equal(slot[r0 - 128 * t:r1 - 128 * t], ref)
            assert (slot[:r0 - 128 * t] == 0).all() and (slot[r1 - 128 * t:] == 0).all()


def test_tgmm_block_selection_equals_full(orc):
    M, K, N = 300, 48, 40
    gs = torch.tensor([120, 180], dtype=torch.int32)
    x = W.activations(M, K, 51)
    d = W.cotangent(M, N, 52)
    full, _ = orc.tgmm(x, d, gs)
    blk, bad = orc.tgmm(x, d, gs, experts=[1], k_range=(8, 40), n_range=(16, 40))
    assert bad == 0
    assert torch.equal(blk[0], full[1, 8:40, 16:40])
