"""The quantizers' f32 -> fp8 cast against the oracle's encoder over whole
binades of f32 bit patterns.

Every quantizer of the library ends in the same step: a correctly rounded f32
quotient cast to e4m3 ("MoE: native FP8 QAT for routed-expert GMMs",
Implementation) or, for the weight gradient's dout operand, e5m2 ("MoE fp8
backward: in-kernel drhs operand quantization", What), round to nearest even and
saturating. fp8moe_selftest_cast_f32 runs that cast, through the kernels' own
helpers, on arbitrary f32 inputs; here it is compared bit for bit with the
oracle's encoder (itself pinned against torch's float8 types in
test_oracle_codec.py) on every f32 of a set of binades: the subnormal range of
each format, the values that underflow to zero, ordinary binades, and the
saturation region, both signs.
"""
import numpy as np
import pytest
import torch

from fp8_moe_routed_gb300 import binding as fb

pytestmark = pytest.mark.gpu

N23 = 1 << 23


@pytest.fixture(autouse=True, scope="module")
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fb.load()
    yield
    torch.cuda.synchronize()


def binade(lo_exp: int) -> torch.Tensor:
    """All 2^23 f32 values in [2^lo_exp, 2^(lo_exp + 1))."""
    lo = int(np.array([2.0 ** lo_exp], dtype=np.float32).view(np.uint32)[0])
    bits = torch.arange(lo, lo + N23, dtype=torch.int64).to(torch.int32)
    return bits.view(torch.float32)


def gpu_cast(x: torch.Tensor, fmt: str) -> torch.Tensor:
    return fb.selftest_cast_f32(x.cuda(), fmt).cpu()


# e4m3: subnormals from 2^-9, smallest normal 2^-6, max 448 (binade [256, 512)
# holds the saturation region); 2^-12 and 2^-11 round to zero or the smallest code
E4M3_BINADES = [-12, -11, -10, -9, -8, -7, -6, -1, 0, 3, 7, 8, 9]
# e5m2: subnormals from 2^-16, smallest normal 2^-14, max 57344 (in [2^15, 2^16))
E5M2_BINADES = [-19, -18, -17, -16, -15, -14, -1, 0, 9, 14, 15, 16]


@pytest.mark.parametrize("lo_exp", E4M3_BINADES)
def test_e4m3_cast_whole_binade_bit_exact(orc, lo_exp):
    x = binade(lo_exp)
    for v in (x, -x):
        assert torch.equal(gpu_cast(v, "e4m3"), orc.e4m3_encode(v)), f"binade 2^{lo_exp}"


@pytest.mark.parametrize("lo_exp", E5M2_BINADES)
def test_e5m2_cast_whole_binade_bit_exact(orc, lo_exp):
    x = binade(lo_exp)
    for v in (x, -x):
        assert torch.equal(gpu_cast(v, "e5m2"), orc.e5m2_encode(v)), f"binade 2^{lo_exp}"


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_cast_special_values_and_odd_length(orc, fmt):
    x = torch.tensor([0.0, -0.0, float("inf"), -float("inf"), float("nan"), 3.4e38, -3.4e38,
                      1e-45, -1e-45, 448.0, 464.0, -464.0, 57344.0, 61440.0, 1.0],
                     dtype=torch.float32)   # 15 values: the last one converts beside a zero
    enc = orc.e4m3_encode if fmt == "e4m3" else orc.e5m2_encode
    assert torch.equal(gpu_cast(x, fmt), enc(x))
    one = torch.tensor([-2.5], dtype=torch.float32)
    assert torch.equal(gpu_cast(one, fmt), enc(one))
