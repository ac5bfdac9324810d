"""CPU checks that the seeded input generators follow the stated recipe: the
outlier channel counts per K, their x20 gain, the weight and activation
spreads, the size of one policy update, and seed determinism."""
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from precision_rl_rollout_gb300 import synth  # noqa: E402


def test_outlier_channel_counts():
    # round(0.01 K) distinct channels: 36 / 51 / 189 / 276 for the Qwen2.5 widths
    for K, n in ((3584, 36), (5120, 51), (18944, 189), (27648, 276), (256, 3), (128, 1)):
        ch = synth.outlier_channels(K, 1234)
        assert ch.numel() == n
        assert len(set(ch.tolist())) == n and int(ch.min()) >= 0 and int(ch.max()) < K


def test_activation_outliers_are_x20_and_shared_by_every_token():
    M, K, seed = 4096, 512, synth.seed_for(2, 1)
    X = synth.activation(M, K, seed).float()
    ch = synth.outlier_channels(K, seed)
    mask = torch.zeros(K, dtype=torch.bool)
    mask[ch] = True
    s_out = X[:, mask].std().item()
    s_in = X[:, ~mask].std().item()
    assert abs(s_in - 1.0) < 0.02
    assert abs(s_out / s_in - 20.0) < 1.0
    # the tiny layer's reading: the first two channels of the set only
    X2 = synth.activation(M, K, seed, n_outliers=2).float()
    big = (X2.abs() > 8).float().mean(dim=0) > 0.3
    assert int(big.sum()) == 2 and bool(big[ch[:2]].all())


def test_weight_spread_and_policy_update_size():
    W = synth.weight(512, 1024, synth.seed_for(2, 0))
    assert W.dtype == torch.bfloat16
    assert abs(W.float().std().item() - 0.02) < 0.0005
    W0 = W.clone()
    synth.policy_update_(W, synth.seed_for(2, 5))
    d = (W.float() - W0.float())
    # N(0, 1e-4) added in fp32 then rounded to bf16: most changes are 0 or one
    # bf16 step, and their spread stays on the order of 1e-4
    assert 0.3e-4 < d.std().item() < 3e-4
    assert d.abs().max().item() < 2e-3


def test_seeded_draws_are_deterministic():
    a = synth.activation(8, 256, 99)
    b = synth.activation(8, 256, 99)
    c = synth.activation(8, 256, 100)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert not torch.equal(a.view(torch.int16), c.view(torch.int16))
    assert synth.seed_for(3, 7) == 1234 + 300 + 7
