"""Seeded synthetic inputs for the FP8 MoE grouped-matmul path.

This module only draws inputs: group sizes, activations, cotangents, garbage
tails and the FP8 weight codes with their per-channel scales. It holds none of
the arithmetic of the path under test (activation quantization, the grouped
matmuls, SwiGLU, dequantization, the per-tile quantization of the weight
gradient). Both the CUDA library and the CPU oracle receive the very same bytes
from here.

Weight codes are an *input* of every kernel. They are made the way the pages
describe the trainer's FP8 weights (per-output-channel absmax scale over K, codes
in float8_e4m3fn): a Gaussian weight is divided by its channel scale and cast
with torch's own float8_e4m3fn conversion. That weight quantizer is input
preparation, not a step of the path.

Workload recipes (sizes follow the DeepSeek-V3-like per-device MoE shapes and the
dropless buffer described on "MoE fp8 backward: in-kernel drhs operand
quantization", section What/Repro; the pages' own data is a trainer run and is
not available, these synthetic draws stand in for it):

* ``tiny``: E=4, K=256, N=128 (wi 2N=256), M=512, multinomial routing with one
  group forced to zero.
* ``balanced``: E=32, K=7168, moe intermediate 2048, M=32768, 1024 rows each.
* ``skewed``: balanced shapes, Zipf(1.2) routing over 28 experts + 4 empty.
* ``dropless``: M=65536 static rows, the skewed sizes (T=32768), NaN/+-Inf/1e30
  in the tail rows.
* ``sweep``: E=128, K=4096, N=1536 (wi 3072), M in {8192 .. 131072}, sizes
  uniform in [0, 2M/128] then adjusted by +-1 to sum to M.
* ``microbench``: the kernel microbenchmark shape of "MoE: native FP8 QAT for
  routed-expert GMMs", section Tests (one call at full fill, 64 experts,
  225,280 rows, the Qwen3.5-397B-A17B per-device MLP: hidden 4096, moe
  intermediate 1024, so wi is [64, 4096, 2048] and wo [64, 1024, 4096]);
  full fill read as 225,280 / 64 = 3520 rows per expert.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

# Zipf(s=1.2) sizes over 28 non-empty experts, largest-remainder rounding of
# rank^-1.2 to a total of 32768 (max 10804 > 8192); 4 more experts get 0 rows.
ZIPF_28 = [10804, 4703, 2891, 2047, 1566, 1258, 1046, 891, 773, 682, 608, 548,
           497, 455, 419, 388, 361, 337, 315, 297, 280, 265, 251, 238, 227, 216,
           207, 198]

E4M3_MAX = 448.0


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def zipf_sizes(total: int = 32768, n_nonzero: int = 28, n_experts: int = 32,
               s: float = 1.2) -> list:
    """Largest-remainder rounding of rank^-s to ``total`` (rank 1 first)."""
    w = [r ** (-s) for r in range(1, n_nonzero + 1)]
    tot = sum(w)
    raw = [total * x / tot for x in w]
    base = [int(x) for x in raw]
    rem = total - sum(base)
    order = sorted(range(n_nonzero), key=lambda i: -(raw[i] - base[i]))
    for i in order[:rem]:
        base[i] += 1
    return base + [0] * (n_experts - n_nonzero)


def group_sizes(kind: str, seed: int = 0, E: Optional[int] = None,
                M: Optional[int] = None) -> torch.Tensor:
    """int32 [E] group sizes for the named routing recipe."""
    g = _gen(seed)
    if kind == "tiny":
        E = E or 4
        M = M or 512
        probs = torch.full((E,), 1.0 / E)
        idx = torch.multinomial(probs, M, replacement=True, generator=g)
        gs = torch.bincount(idx, minlength=E).to(torch.int64)
        z = int(torch.randint(0, E, (1,), generator=g))
        gs[(z + 1) % E] += gs[z]
        gs[z] = 0
        return gs.to(torch.int32)
    if kind == "balanced":
        E = E or 32
        M = M or 32768
        assert M % E == 0
        return torch.full((E,), M // E, dtype=torch.int32)
    if kind == "full_fill":
        E = E or 64
        M = M or 225280
        assert M % E == 0
        return torch.full((E,), M // E, dtype=torch.int32)
    if kind in ("skewed", "dropless"):
        E = E or 32
        sizes = torch.tensor(zipf_sizes(32768, 28, E), dtype=torch.int32)
        perm = torch.randperm(E, generator=g)
        return sizes[perm].contiguous()
    if kind == "sweep":
        E = E or 128
        assert M is not None
        hi = 2 * M // E
        gs = torch.randint(0, hi + 1, (E,), generator=g).to(torch.int64)
        # +-1 adjustments on random in-range groups until the sum is M
        diff = int(gs.sum()) - M
        while diff != 0:
            e = int(torch.randint(0, E, (1,), generator=g))
            if diff > 0 and gs[e] > 0:
                gs[e] -= 1
                diff -= 1
            elif diff < 0 and gs[e] < hi:
                gs[e] += 1
                diff += 1
        return gs.to(torch.int32)
    raise ValueError(f"unknown routing recipe {kind!r}")


def activations(M: int, K: int, seed: int, outlier_frac: float = 0.0,
                outlier_scale: float = 50.0, device="cpu") -> torch.Tensor:
    """bf16 [M, K] ~ N(0, 1); a seeded fraction of rows is scaled by
    ``outlier_scale`` (0.1 % rows x50 in the balanced recipe)."""
    g = _gen(seed, device)
    x = torch.randn(M, K, generator=g, device=device, dtype=torch.float32)
    n_out = int(round(outlier_frac * M))
    if n_out:
        rows = torch.randperm(M, generator=g, device=device)[:n_out]
        x[rows] *= outlier_scale
    return x.to(torch.bfloat16)


def fill_tail_garbage(x: torch.Tensor, T: int) -> torch.Tensor:
    """Rows [T, M) of a bf16 buffer cycle through NaN, +Inf, -Inf, 1e30
    (dropless buffer tails, "MoE fp8 backward ...", section What)."""
    vals = torch.tensor([float("nan"), float("inf"), float("-inf"), 1e30],
                        dtype=torch.float32)
    M = x.shape[0]
    if T < M:
        n = M - T
        cyc = vals[torch.arange(n) % 4].to(torch.bfloat16).to(x.device)
        x[T:] = cyc[:, None].expand(n, x.shape[1])
    return x


def fp8_weights(E: int, K: int, N: int, sigma: float, seed: int,
                device="cpu", chunk_experts: int = 4):
    """FP8 weight codes uint8 [E, K, N] (float8_e4m3fn bit patterns) and f32
    per-output-channel scales [E, N] = amax_k |w| / 448, from w ~ N(0, sigma).

    The cast to float8_e4m3fn is torch's (round to nearest even); the scaled
    values are clamped to +-448 first so that a division that rounds up past
    448 stays finite."""
    g = _gen(seed, device)
    codes = torch.empty(E, K, N, dtype=torch.uint8, device=device)
    scale = torch.empty(E, N, dtype=torch.float32, device=device)
    for e0 in range(0, E, chunk_experts):
        e1 = min(E, e0 + chunk_experts)
        w = torch.randn(e1 - e0, K, N, generator=g, device=device,
                        dtype=torch.float32) * sigma
        s = w.abs().amax(dim=1) / E4M3_MAX            # [e, N]
        q = (w / s[:, None, :]).clamp_(-E4M3_MAX, E4M3_MAX)
        codes[e0:e1] = q.to(torch.float8_e4m3fn).view(torch.uint8)
        scale[e0:e1] = s
        del w, q
    return codes, scale


def cotangent(M: int, N: int, seed: int, device="cpu") -> torch.Tensor:
    """bf16 [M, N] ~ N(0, 1) (dout)."""
    g = _gen(seed, device)
    return torch.randn(M, N, generator=g, device=device,
                       dtype=torch.float32).to(torch.bfloat16)


@dataclasses.dataclass
class Shapes:
    """One routed-expert MLP: wi is [E, K, 2 * F] (gate | up), wo is [E, F, K]."""
    name: str
    E: int
    K: int        # hidden (model) dim
    F: int        # moe intermediate dim; wi produces 2F columns
    M: int        # static rows of the ragged buffer
    routing: str
    outlier_frac: float = 0.0
    sigma_wi: float = 0.02
    sigma_wo: float = 0.02


TINY = Shapes("tiny", E=4, K=256, F=128, M=512, routing="tiny")
BALANCED = Shapes("balanced", E=32, K=7168, F=2048, M=32768, routing="balanced",
                  outlier_frac=0.001, sigma_wi=0.006, sigma_wo=0.006)
SKEWED = Shapes("skewed", E=32, K=7168, F=2048, M=32768, routing="skewed",
                sigma_wi=0.006, sigma_wo=0.006)
DROPLESS = Shapes("dropless", E=32, K=7168, F=1024, M=65536, routing="dropless",
                  sigma_wi=0.006, sigma_wo=0.006)


MICROBENCH = Shapes("microbench", E=64, K=4096, F=1024, M=225280, routing="full_fill",
                    sigma_wi=0.02, sigma_wo=0.02)


def sweep_shapes(M: int) -> Shapes:
    return Shapes(f"sweep_M{M}", E=128, K=4096, F=1536, M=M, routing="sweep",
                  sigma_wi=0.02, sigma_wo=0.02)


@dataclasses.dataclass(frozen=True)
class ExpertShard:
    """One rank's part of an expert-parallel split of the ragged buffer: the
    experts [e0, e1) and the rows [row0, row1) their groups cover."""
    rank: int
    world: int
    e0: int
    e1: int
    row0: int
    row1: int

    def take(self, gs: torch.Tensor, rows=(), experts=()):
        """This rank's slice of group_sizes, of every row-indexed tensor in
        ``rows`` (leading dim = the buffer's rows) and of every expert-indexed
        tensor in ``experts`` (leading dim = E)."""
        return (gs[self.e0:self.e1].contiguous(),
                [t[self.row0:self.row1] for t in rows],
                [t[self.e0:self.e1] for t in experts])


def expert_shard(gs: torch.Tensor, rank: int, world: int, M: Optional[int] = None) -> ExpertShard:
    """Expert parallelism (each rank owns a contiguous block of the experts, as
    equal in count as possible, with the rows of their groups). Group sizes are
    read the way the kernels read them: a negative size counts as 0 and row
    ranges are clipped at M (default: the sum of the sizes)."""
    E = gs.numel()
    if not 0 <= rank < world or world > E:
        raise ValueError(f"rank {rank} of {world} for {E} experts")
    e0 = rank * E // world
    e1 = (rank + 1) * E // world
    sizes = gs.to(torch.int64).clamp_min(0)
    off = torch.cat([torch.zeros(1, dtype=torch.int64), sizes.cumsum(0)])
    total = int(off[-1])
    M = total if M is None else M
    row0 = min(int(off[e0]), M)
    row1 = min(int(off[e1]), M)
    return ExpertShard(rank, world, e0, e1, row0, row1)
