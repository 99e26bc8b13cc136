"""Pins of the oracle's number formats against things other than itself.

e4m3fn (OCP float8, the forward dtype named on "Fix fp8 MoE on the sparse_matmul
path", section Fix) is checked against torch's own float8_e4m3fn type (a library
routine, independent of the oracle), against values that follow from the format
definition (special codes, round trips, midpoints) and by brute force over whole
binades. bf16 rounding is checked against torch's float32 -> bfloat16 cast and
closed-form double-rounding cases.
"""
import math

import numpy as np
import pytest
import torch

F8 = torch.float8_e4m3fn


def torch_decode(codes: torch.Tensor) -> torch.Tensor:
    return codes.to(torch.uint8).view(F8).to(torch.float64)


def torch_encode(x: torch.Tensor) -> torch.Tensor:
    """torch's RNE cast; it saturates below 464 only, so callers keep |x| < 464."""
    return x.to(torch.float32).to(F8).view(torch.uint8)


def test_decode_all_codes_match_torch(orc):
    ours = orc.e4m3_decode_all()
    ref = torch_decode(torch.arange(256, dtype=torch.uint8))
    nan = torch.isnan(ref)
    assert torch.equal(torch.isnan(ours), nan)
    assert nan.sum() == 2 and bool(nan[0x7F]) and bool(nan[0xFF])
    assert torch.equal(ours[~nan], ref[~nan])
    # signed zero is kept
    assert math.copysign(1.0, float(ours[0x80])) == -1.0


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6),
    (0x38, 1.0), (0x39, 1.125), (0x40, 2.0), (0x7E, 448.0), (0xFE, -448.0),
    (0xB8, -1.0), (0x77, 240.0),
])
def test_decode_special_values(orc, code, value):
    assert orc.e4m3_decode(code) == value


def test_encode_roundtrip_all_finite_codes(orc):
    codes = torch.tensor([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=torch.uint8)
    vals = orc.e4m3_decode_all()[codes.long()].to(torch.float32)
    assert torch.equal(orc.e4m3_encode(vals), codes)


def test_encode_midpoints_round_to_even_code(orc):
    v = orc.e4m3_decode_all()[:127]          # ascending non-negative finite values
    mids = ((v[:-1] + v[1:]) / 2)             # exact in f32: <= 5 significant bits
    mids32 = mids.to(torch.float32)
    assert torch.equal(mids32.double(), mids)
    got = orc.e4m3_encode(mids32).long()
    lo = torch.arange(126)
    want = torch.where(lo % 2 == 0, lo, lo + 1)
    assert torch.equal(got, want)
    # one f32 ulp either side of the midpoint picks the nearer code
    below = torch.nextafter(mids32, torch.zeros_like(mids32))
    above = torch.nextafter(mids32, torch.full_like(mids32, 1e9))
    assert torch.equal(orc.e4m3_encode(below).long(), lo)
    assert torch.equal(orc.e4m3_encode(above).long(), lo + 1)
    # negative side mirrors
    assert torch.equal(orc.e4m3_encode(-mids32).long(), want + 128)


def test_encode_saturates_and_nan(orc):
    x = torch.tensor([448.0, 448.5, 463.99, 464.0, 480.0, 1e6, float("inf"),
                      -449.0, -1e30, float("-inf")], dtype=torch.float32)
    got = orc.e4m3_encode(x).tolist()
    assert got == [0x7E] * 7 + [0xFE] * 3
    assert orc.e4m3_encode(torch.tensor([float("nan")])).item() == 0x7F


def test_encode_signed_zero_and_underflow(orc):
    x = torch.tensor([0.0, -0.0, 2.0 ** -11, -2.0 ** -11, 2.0 ** -10, 2.0 ** -10 * 1.0001,
                      -(2.0 ** -10) * 1.0001], dtype=torch.float32)
    # 2^-10 is the midpoint between 0 and 2^-9: ties to the even code 0
    assert orc.e4m3_encode(x).tolist() == [0x00, 0x80, 0x00, 0x80, 0x00, 0x01, 0x81]


@pytest.mark.parametrize("scale", [1e-4, 0.01, 1.0, 30.0, 200.0])
def test_encode_matches_torch_on_random_values(orc, scale):
    g = torch.Generator().manual_seed(7)
    x = (torch.randn(400_000, generator=g) * scale).clamp(-463.0, 463.0)
    assert torch.equal(orc.e4m3_encode(x), torch_encode(x))


@pytest.mark.parametrize("lo_exp", [-12, -9, -7, 0, 5, 8])
def test_encode_bruteforce_binade_vs_torch(orc, lo_exp):
    """Every f32 in the binade [2^lo_exp, 2^(lo_exp+1)) (8 Mi patterns), both signs."""
    lo_bits = int(np.array([2.0 ** lo_exp], dtype=np.float32).view(np.uint32)[0])
    n = 1 << 23
    ours = orc.e4m3_encode_bits(lo_bits, n)
    bits = torch.arange(lo_bits, lo_bits + n, dtype=torch.int64).to(torch.int32)
    x = bits.view(torch.float32)
    if lo_exp == 8:   # [256, 512): torch turns >= 480 into NaN, the format saturates
        keep = x < 464.0
        assert bool((ours[~keep] == 0x7E).all())
        ours, x = ours[keep], x[keep]
    assert torch.equal(ours, torch_encode(x))
    neg = orc.e4m3_encode(-x)
    assert torch.equal(neg, torch_encode(-x))


def test_bf16_rounding_matches_torch_from_f32(orc):
    g = torch.Generator().manual_seed(3)
    x = torch.randn(1_000_000, generator=g, dtype=torch.float32) * 10.0 ** torch.randint(
        -30, 30, (1_000_000,), generator=g).float()
    x = torch.cat([x, torch.tensor([0.0, -0.0, 1e-40, -1e-40, 3.3e38, -3.3e38])])
    ours = orc.f64_to_bf16(x.double()).view(torch.int16)
    ref = x.to(torch.bfloat16).view(torch.int16)
    assert torch.equal(ours, ref)


def test_bf16_single_rounding_from_double(orc):
    # 1 + 2^-8 is the midpoint between 1 and 1 + 2^-7 (ties to even -> 1); a hair
    # above it must go up, which a detour through f32 would lose.
    d = torch.tensor([1 + 2.0 ** -8, 1 + 2.0 ** -8 + 2.0 ** -40, 1 + 3 * 2.0 ** -8,
                      1 + 2.0 ** -8 - 2.0 ** -40], dtype=torch.float64)
    got = orc.f64_to_bf16(d).to(torch.float64).tolist()
    assert got == [1.0, 1 + 2.0 ** -7, 1 + 2 * 2.0 ** -7, 1.0]
    big = orc.f64_to_bf16(torch.tensor([3.4e38, float("nan")], dtype=torch.float64))
    assert math.isinf(float(big[0])) and math.isnan(float(big[1]))


# --------------------------------------------------------------------- e5m2
# The tgmm's gradient operand may be e5m2 ("MoE fp8 backward: in-kernel drhs
# operand quantization + configurable gradient dtype", What). OCP e5m2: bias 15,
# 2 mantissa bits, subnormals m * 2^-16, exponent 31 = Inf / NaN, max 57344.
F8E5 = torch.float8_e5m2


def e5m2_formula(c: int) -> float:
    s = -1.0 if c & 0x80 else 1.0
    e, m = (c >> 2) & 0x1F, c & 0x3
    if e == 31:
        return s * math.inf if m == 0 else math.nan
    if e == 0:
        return s * m * 2.0 ** -16
    return s * (1.0 + m / 4.0) * 2.0 ** (e - 15)


def test_e5m2_decode_all_codes_match_torch_and_formula(orc):
    ours = torch.tensor([orc.e5m2_decode(c) for c in range(256)], dtype=torch.float64)
    theirs = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(F8E5).to(torch.float64)
    form = torch.tensor([e5m2_formula(c) for c in range(256)], dtype=torch.float64)
    for ref in (theirs, form):
        nan = torch.isnan(ref)
        assert torch.equal(torch.isnan(ours), nan)
        assert torch.equal(ours[~nan], ref[~nan])
    assert orc.e5m2_decode(0x7B) == 57344.0 and orc.e5m2_decode(0x01) == 2.0 ** -16
    assert math.isinf(orc.e5m2_decode(0x7C))


def test_e5m2_encode_roundtrip_all_finite_codes(orc):
    codes = [c for c in range(256) if (c & 0x7F) < 0x7C]
    vals = torch.tensor([orc.e5m2_decode(c) for c in codes], dtype=torch.float32)
    got = orc.e5m2_encode(vals)
    # +0 and -0 both keep their sign
    assert got.tolist() == codes


def test_e5m2_encode_midpoints_round_to_even_code(orc):
    mids, want = [], []
    for c in range(0, 0x7B):
        a, b = orc.e5m2_decode(c), orc.e5m2_decode(c + 1)
        mids.append((a + b) / 2)            # exact in f32: 3 significant bits
        want.append(c if c % 2 == 0 else c + 1)
    got = orc.e5m2_encode(torch.tensor(mids, dtype=torch.float32))
    assert got.tolist() == want
    neg = orc.e5m2_encode(-torch.tensor(mids, dtype=torch.float32))
    assert neg.tolist() == [w | 0x80 for w in want]


def test_e5m2_encode_saturates_and_nan(orc):
    x = torch.tensor([57344.0, 61440.0, 65535.0, 1e30, math.inf, -math.inf, -61440.0],
                     dtype=torch.float32)
    assert orc.e5m2_encode(x).tolist() == [0x7B] * 5 + [0xFB, 0xFB]
    n = orc.e5m2_encode(torch.tensor([math.nan], dtype=torch.float32))
    assert (int(n[0]) & 0x7F) > 0x7C               # a NaN code


@pytest.mark.parametrize("scale", [1e-6, 1e-3, 1.0, 300.0, 40000.0])
def test_e5m2_encode_matches_torch_on_random_values(orc, scale):
    g = torch.Generator().manual_seed(int(scale * 7) + 3)
    x = (torch.randn(200000, generator=g) * scale).to(torch.float32)
    x = x.clamp(-57344.0, 57344.0)                 # torch overflows to Inf past the max
    ours = orc.e5m2_encode(x)
    theirs = x.to(F8E5).view(torch.uint8)
    assert torch.equal(ours, theirs)
