"""Comparison helpers for the GPU-vs-oracle parity tests.

Tolerances:
  * codes, scales, dequantized weights: bit-exact (integer work, and the same
    f32 operations in the same order on both sides);
  * forward outputs and dLHS (bf16): per element
        |gpu - ref| <= max(1 bf16 ulp of ref, 2e-3 * rms(ref))
    The oracle rounds its exact (float64) result once to bf16. The kernels sum
    f32 products in a different order and round once, so they may land one bf16
    step away; where an output is far below the typical magnitude, the f32
    summation error of the row (about K * 2^-24 of rms-sized partial sums) can
    exceed an ulp of that small value, and 2e-3 * rms bounds it;
  * tgmm (f32): max |gpu - ref| <= 1e-2 * rms(ref) and every value finite. The
    per-segment rescale adds one f32 multiply and one f32 fused multiply-add
    per segment and element, in a different order than the float64 oracle.
"""
import torch


def bf16_ulp(x: torch.Tensor) -> torch.Tensor:
    """Spacing of the bf16 grid at |x| (float64)."""
    a = x.abs().double().clamp_min(2.0 ** -126)
    e = torch.floor(torch.log2(a))
    return torch.pow(2.0, e - 7)


def check_bf16(gpu: torch.Tensor, ref: torch.Tensor, rel: float = 2e-3, what: str = ""):
    g = gpu.detach().float().cpu().double()
    r = ref.detach().float().cpu().double()
    assert g.shape == r.shape, (g.shape, r.shape)
    assert torch.isfinite(r).all(), f"{what}: oracle produced non-finite values"
    assert torch.isfinite(g).all(), f"{what}: non-finite GPU output"
    rms = r.pow(2).mean().sqrt().item() if r.numel() else 0.0
    err = (g - r).abs()
    bound = torch.maximum(bf16_ulp(r), torch.full_like(r, rel * rms))
    bad = err > bound
    if bad.any():
        i = int(bad.flatten().nonzero()[0])
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {r.numel()} elements out of tolerance; first at "
            f"{i}: gpu={g.flatten()[i].item()} ref={r.flatten()[i].item()} rms={rms} "
            f"max_err={err.max().item()}")
    return {"max_err_over_rms": (err.max().item() / rms) if rms else 0.0,
            "ulp_gt1": int((err > bf16_ulp(r)).sum())}


def check_f32_rel(gpu: torch.Tensor, ref: torch.Tensor, rel: float = 1e-2, what: str = ""):
    g = gpu.detach().cpu().double()
    r = ref.detach().cpu().double()
    assert torch.isfinite(g).all(), f"{what}: non-finite GPU values"
    rms = r.pow(2).mean().sqrt().item() if r.numel() else 0.0
    err = (g - r).abs().max().item() if r.numel() else 0.0
    assert err <= rel * rms or err == 0.0, f"{what}: max_err={err} rms={rms}"
    return err / rms if rms else 0.0


def bits16(t: torch.Tensor) -> torch.Tensor:
    return t.detach().cpu().contiguous().view(torch.int16)
