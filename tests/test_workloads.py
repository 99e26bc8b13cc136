"""The seeded input recipes produce the shapes and routing the workloads name."""
import torch

from fp8_moe_routed_gb300 import workloads as W


def test_zipf_sizes_match_recipe():
    s = W.zipf_sizes()
    assert s[:28] == W.ZIPF_28 and sum(s) == 32768 and s[28:] == [0] * 4
    assert max(s) > 8192


def test_group_size_recipes():
    t = W.group_sizes("tiny", seed=0)
    assert t.numel() == 4 and int(t.sum()) == 512 and (t == 0).sum() >= 1
    b = W.group_sizes("balanced")
    assert (b == 1024).all() and b.numel() == 32
    z = W.group_sizes("skewed", seed=3)
    assert sorted(z.tolist()) == sorted(W.zipf_sizes()) and (z == 0).sum() == 4
    for M in (8192, 131072):
        s = W.group_sizes("sweep", seed=1, M=M)
        assert int(s.sum()) == M and s.min() >= 0 and s.max() <= 2 * M // 128
        assert (s % 128 != 0).any()
    assert torch.equal(W.group_sizes("sweep", seed=1, M=8192), W.group_sizes("sweep", seed=1, M=8192))
    ff = W.group_sizes("full_fill")
    assert ff.numel() == 64 and int(ff.sum()) == 225280 and (ff == 3520).all()
    assert 3520 % 128 != 0          # every expert ends in a partial 128-row tile
    mb = W.MICROBENCH
    assert (mb.E, mb.K, mb.F, mb.M) == (64, 4096, 1024, 225280)


def test_weights_are_valid_e4m3_with_channel_max():
    codes, scale = W.fp8_weights(3, 64, 32, 0.02, seed=1)
    assert codes.dtype == torch.uint8 and scale.shape == (3, 32)
    assert not ((codes & 0x7F) == 0x7F).any()          # no NaN codes
    mag = (codes & 0x7F).amax(dim=1)
    assert (mag == 0x7E).all()                           # every channel reaches 448
    assert (scale > 0).all()


def test_tail_garbage():
    x = W.fill_tail_garbage(W.activations(10, 4, 0), 6)
    v = x.float()
    assert torch.isnan(v[6]).all() and (v[7] == float("inf")).all()
    assert (v[8] == float("-inf")).all() and (v[9] > 9e29).all()
    assert torch.isfinite(v[:6]).all()
