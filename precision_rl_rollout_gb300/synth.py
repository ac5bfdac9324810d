"""Seeded synthetic inputs for the 8-bit rollout linear layer.

This module builds inputs only; it holds none of the method's arithmetic (no
scale, no rounding to 8 bits, no GEMM), so that the CUDA library and the CPU
oracle can both consume its output without sharing any of the method.

Recipe (the pages measure on real models and datasets that are not available
here, so Qwen2.5-shaped synthetic layers stand in for them):

* weights ``W ~ N(0, 0.02)`` drawn in fp32 and rounded to bf16 (0.02 is the
  usual initialisation standard deviation);
* activations ``X ~ N(0, 1)`` with ``round(0.01 * K)`` outlier channels (at
  least one; 2 of 256 for the tiny layer) multiplied by 20 before rounding to
  bf16; the channel set is drawn once per seed and shared by every token;
* one policy update before each requant, ``W <- bf16(fp32(W) + N(0, 1e-4))``
  (the policy changes every RL step: FP8-RL, Abstract; FlashRL write-up,
  online quantization).

``seed = 1234 + 100 * config + tensor_id`` names every tensor.  Draws use a
torch generator on the requested device (Philox on CUDA, the CPU generator on
the host); a test that compares the GPU with the oracle generates once and
hands the same bytes to both sides.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

W_STD = 0.02
X_STD = 1.0
UPDATE_STD = 1e-4
OUTLIER_FRAC = 0.01
OUTLIER_GAIN = 20.0


def seed_for(config: int, tensor_id: int) -> int:
    return 1234 + 100 * config + tensor_id


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def weight(N: int, K: int, seed: int, device="cpu", std: float = W_STD) -> torch.Tensor:
    """bf16 [N, K] ~ N(0, std)."""
    g = _gen(seed, device)
    w = torch.empty((N, K), dtype=torch.float32, device=device)
    w.normal_(0.0, std, generator=g)
    return w.to(torch.bfloat16)


def weight_bf16_direct(N: int, K: int, seed: int, device="cuda", std: float = W_STD) -> torch.Tensor:
    """bf16 [N, K] ~ N(0, std) drawn straight into a bf16 tensor (no fp32 copy),
    for full-model weight sets that would not fit twice in memory."""
    g = _gen(seed, device)
    w = torch.empty((N, K), dtype=torch.bfloat16, device=device)
    w.normal_(0.0, std, generator=g)
    return w


def outlier_channels(K: int, seed: int) -> torch.Tensor:
    n = max(1, int(round(OUTLIER_FRAC * K)))
    g = _gen(seed + 7, "cpu")
    return torch.randperm(K, generator=g)[:n]


def activation(M: int, K: int, seed: int, device="cpu", n_outliers: int | None = None) -> torch.Tensor:
    """bf16 [M, K] ~ N(0, 1) with outlier channels x20."""
    g = _gen(seed, device)
    x = torch.empty((M, K), dtype=torch.float32, device=device)
    x.normal_(0.0, X_STD, generator=g)
    ch = outlier_channels(K, seed)
    if n_outliers is not None:
        ch = ch[:n_outliers]
    x[:, ch.to(device)] *= OUTLIER_GAIN
    return x.to(torch.bfloat16)


def policy_update_(W: torch.Tensor, seed: int) -> torch.Tensor:
    """In place: W <- bf16(fp32(W) + N(0, 1e-4)); done row-slab by row-slab so a
    multi-GB weight never needs a full fp32 copy."""
    g = _gen(seed, W.device)
    rows = max(1, (64 << 20) // max(1, W.shape[1]))
    for r0 in range(0, W.shape[0], rows):
        sl = W[r0:r0 + rows]
        d = torch.empty(sl.shape, dtype=torch.float32, device=W.device)
        d.normal_(0.0, UPDATE_STD, generator=g)
        sl.copy_((sl.float() + d).to(torch.bfloat16))
    return W


def edge_case_weight(N: int, K: int, seed: int) -> torch.Tensor:
    """bf16 [N, K] (N, K multiples of 128, at least 3x3 blocks) of ordinary
    N(0, 0.02) values with planted blocks: all zero; all -0.0; one non-zero
    element; huge values (1e30); bf16 subnormals; all equal; exact powers of two
    on E4M3 ties; a mix of both signs at the same magnitude."""
    W = weight(N, K, seed)
    B = 128
    f = torch.float32
    W[0:B, 0:B] = 0
    W[0:B, B:2 * B] = torch.tensor(-0.0, dtype=f)
    blk = torch.zeros(B, B, dtype=f)
    blk[37, 91] = -3.0
    W[0:B, 2 * B:3 * B] = blk
    W[B:2 * B, 0:B] = (torch.randn(B, B, generator=_gen(seed + 1, "cpu")) * 1e30)
    W[B:2 * B, B:2 * B] = (torch.randn(B, B, generator=_gen(seed + 2, "cpu")) * 1e-39)
    W[B:2 * B, 2 * B:3 * B] = 0.75
    ties = torch.tensor([448.0, 17.0, 18.0, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10, 1.5, 0.4375,
                         336.0, -336.0, 208.0, -232.0, 9.0, 11.0, 13.0, -15.0], dtype=f)
    W[2 * B:3 * B, 0:B] = ties.repeat(B * B // ties.numel()).reshape(B, B)
    signs = torch.where(torch.rand(B, B, generator=_gen(seed + 3, "cpu")) < 0.5, -1.0, 1.0)
    W[2 * B:3 * B, B:2 * B] = signs * 0.0625
    return W.to(torch.bfloat16)


def edge_case_activation(M: int, K: int, seed: int) -> torch.Tensor:
    """bf16 [M, K] (M >= 6) with planted rows: all zero, all -0.0, a single
    non-zero, huge, bf16 subnormal, E4M3 ties."""
    X = activation(M, K, seed).float()
    X[0] = 0
    X[1] = -0.0
    X[2] = 0
    X[2, K // 2 + 3] = 5.0
    X[3] = torch.randn(K, generator=_gen(seed + 1, "cpu")) * 1e30
    X[4] = torch.randn(K, generator=_gen(seed + 2, "cpu")) * 1e-39
    ties = torch.tensor([448.0, 17.0, -18.0, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10, 1.5, -0.4375],
                        dtype=torch.float32)
    X[5] = ties.repeat(K // ties.numel() + 1)[:K]
    return X.to(torch.bfloat16)


def bf16_bits(t: torch.Tensor):
    """Host numpy uint16 view of a bf16 tensor's bits."""
    import numpy as np
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


@dataclass(frozen=True)
class LinearShape:
    name: str
    K: int
    N: int

    @property
    def elems(self) -> int:
        return self.N * self.K


# Qwen2.5-7B: hidden 3584, 28 q heads / 4 kv heads of 128 -> qkv 4608, MLP 18944.
QWEN25_7B = (LinearShape("qkv", 3584, 4608), LinearShape("o_proj", 3584, 3584),
             LinearShape("gate_up", 3584, 37888), LinearShape("down", 18944, 3584))
# Qwen2.5-32B: hidden 5120, 40 q heads / 8 kv heads of 128 -> qkv 7168, MLP 27648.
QWEN25_32B = (LinearShape("qkv", 5120, 7168), LinearShape("o_proj", 5120, 5120),
              LinearShape("gate_up", 5120, 55296), LinearShape("down", 27648, 5120))
QWEN25_32B_LAYERS = 64
TINY = LinearShape("tiny", 256, 512)
TINY_M = 16
DECODE_M_SWEEP = (1, 8, 32, 128, 256)
INT8_M_SWEEP = (32, 256, 4096)
PREFILL_M = 8192
