"""Helpers shared by the GPU parity tests: seeded inputs, host<->device moves and
cached oracle quantizations (so that GEMM inputs always come from the oracle or
the generator, never from the CUDA path)."""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
from precision_rl_rollout_gb300 import synth


def dev(a: np.ndarray, dtype=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def host(t: torch.Tensor) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bits_u32(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


@functools.lru_cache(maxsize=None)
def weight_cpu(N: int, K: int, seed: int, update: bool = True) -> torch.Tensor:
    """Seeded bf16 weight on the host, after one policy update."""
    W = synth.weight(N, K, seed)
    if update:
        synth.policy_update_(W, seed + 50)
    return W


@functools.lru_cache(maxsize=None)
def act_cpu(M: int, K: int, seed: int, n_outliers=None) -> torch.Tensor:
    return synth.activation(M, K, seed, n_outliers=n_outliers)


@functools.lru_cache(maxsize=None)
def oracle_fp8_weight(N: int, K: int, seed: int):
    return oracle.fp8_quant_weight_block(synth.bf16_bits(weight_cpu(N, K, seed)))


@functools.lru_cache(maxsize=None)
def oracle_fp8_act(M: int, K: int, seed: int):
    return oracle.fp8_quant_act_group(synth.bf16_bits(act_cpu(M, K, seed)))


@functools.lru_cache(maxsize=None)
def oracle_int8_weight(N: int, K: int, seed: int):
    return oracle.int8_quant_rows(synth.bf16_bits(weight_cpu(N, K, seed)))


@functools.lru_cache(maxsize=None)
def oracle_int8_act(M: int, K: int, seed: int):
    return oracle.int8_quant_rows(synth.bf16_bits(act_cpu(M, K, seed)))


def sample_rows(M: int, n: int, seed: int) -> np.ndarray:
    """First, last and n-2 seeded rows in between (sorted, unique)."""
    if M <= n:
        return np.arange(M)
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(1, M - 1), size=n - 2, replace=False)
    return np.unique(np.concatenate([[0, M - 1], mid]))


def sample_blocks(NB: int, KB: int, n: int, seed: int):
    rng = np.random.default_rng(seed)
    pairs = {(0, 0), (NB - 1, KB - 1), (NB - 1, 0), (0, KB - 1)}
    while len(pairs) < min(n, NB * KB):
        pairs.add((int(rng.integers(NB)), int(rng.integers(KB))))
    return sorted(pairs)


def assert_fp8_gemm_close(y_gpu_bits: np.ndarray, y_ref: np.ndarray, what: str, rms_ref=None):
    """|y - y_ref| <= 2^-7 |y_ref| + 1e-3 rms(y_ref) element by element."""
    y = oracle.bf16_to_f32(y_gpu_bits).astype(np.float64)
    rms = float(np.sqrt(np.mean(np.square(y_ref)))) if rms_ref is None else rms_ref
    tol = np.abs(y_ref) * 2.0 ** -7 + 1e-3 * rms
    err = np.abs(y - y_ref)
    bad = np.argwhere(err > tol)
    assert bad.size == 0, (f"{what}: {len(bad)} of {y.size} outside tolerance; first {bad[:4].tolist()} "
                           f"y={y[tuple(bad[0])]} ref={y_ref[tuple(bad[0])]} tol={tol[tuple(bad[0])]}")
    return float((err / np.maximum(tol, 1e-300)).max())
