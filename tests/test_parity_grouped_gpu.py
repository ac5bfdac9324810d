"""GPU parity of the grouped (mixture-of-experts) FP8 GEMM against the oracle.

Token rows are grouped by expert with seeded counts (some experts empty); every
computed row must lie within |y - y_ref| <= 2^-7 |y_ref| + 1e-3 rms(y_ref) of
the oracle's per-expert fp64 dequant-matmul, and rows the kernel must not touch
keep their sentinel.  Operands are quantized by the oracle."""
import numpy as np
import pytest
import torch

import oracle
from precision_rl_rollout_gb300 import binding as fb
from precision_rl_rollout_gb300 import synth
from parity_util import assert_fp8_gemm_close, dev, host

pytestmark = pytest.mark.gpu


def _experts(E, N, K, seed):
    Wq, Ws = [], []
    for e in range(E):
        W = synth.weight(N, K, seed + e)
        q, s = oracle.fp8_quant_weight_block(synth.bf16_bits(W))
        Wq.append(q)
        Ws.append(s)
    return np.stack(Wq), np.stack(Ws)


def _routed_tokens(counts, K, seed):
    T = int(np.sum(counts))
    X = synth.activation(T, K, seed)
    Xq, Xs = oracle.fp8_quant_act_group(synth.bf16_bits(X))
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return Xq, Xs, offsets


def _grouped_case(counts, N, K, seed, bound=None, what=""):
    E = len(counts)
    Wq, Ws = _experts(E, N, K, seed)
    Xq, Xs, offsets = _routed_tokens(counts, K, seed + 1000)
    T = Xq.shape[0]
    Y = torch.full((T, N), 5.0, dtype=torch.bfloat16, device="cuda")
    fb.fp8rl_gemm_w8a8_block_grouped(dev(Xq), dev(Xs), dev(Wq), dev(Ws), dev(offsets),
                                     max_tokens_per_expert=bound, Y=Y)
    ref = oracle.fp8_gemm_grouped(Xq, Xs, Wq, Ws, offsets)
    assert_fp8_gemm_close(host(Y), ref, what or f"counts={list(counts)} N={N} K={K}")
    assert fb.fp8rl_check_device_error() == 0


@pytest.mark.parametrize("counts,N,K", [([3, 0, 17, 5], 256, 512), ([1], 128, 128), ([0, 0, 2], 384, 256),
                                        ([16, 16, 33], 128, 640), ([70, 1, 0, 130], 256, 384),
                                        ([5, 9, 0, 0, 12, 3, 1, 7], 640, 1280)])
def test_grouped_small_full(cuda_lib, counts, N, K):
    _grouped_case(np.array(counts), N, K, seed=sum(counts) + N + K)


@pytest.mark.parametrize("bound", [None, "max"])
def test_grouped_seeded_routing(cuda_lib, bound):
    rng = np.random.default_rng(17)
    counts = rng.multinomial(96, rng.dirichlet(np.ones(12) * 0.5))
    b = None if bound is None else int(counts.max())
    _grouped_case(counts, 256, 1024, seed=23, bound=b, what=f"routing {counts.tolist()} bound={b}")


def test_grouped_moe_decode_shape(cuda_lib):
    # 64 decode tokens, top-8 of 32 experts with the gate_up shape of a
    # hidden-2048 / expert-FFN-768 MoE layer (N = 1536, K = 2048)
    rng = np.random.default_rng(31)
    E = 32
    picks = np.array([rng.choice(E, size=8, replace=False) for _ in range(64)])
    counts = np.bincount(picks.ravel(), minlength=E)
    _grouped_case(counts, 1536, 2048, seed=41, bound=int(counts.max()), what="MoE gate_up shape")


def test_grouped_rows_beyond_the_bound_are_reported_not_written(cuda_lib):
    # expert 0 has 40 tokens but the caller promised at most 4: the grid covers
    # one 16-row token tile per expert, so rows 16..39 are not computed, keep
    # their sentinel, and the device reports the broken bound
    counts = np.array([40, 2])
    N, K = 128, 256
    Wq, Ws = _experts(2, N, K, 51)
    Xq, Xs, offsets = _routed_tokens(counts, K, 52)
    Y = torch.full((42, N), 5.0, dtype=torch.bfloat16, device="cuda")
    fb.fp8rl_gemm_w8a8_block_grouped(dev(Xq), dev(Xs), dev(Wq), dev(Ws), dev(offsets),
                                     max_tokens_per_expert=4, Y=Y)
    word = fb.fp8rl_check_device_error()
    assert word != 0 and (word & 0xFFFF) == 2, hex(word)
    ref = oracle.fp8_gemm_grouped(Xq, Xs, Wq, Ws, offsets)
    Yh = host(Y)
    done = np.r_[0:16, 40:42]
    assert_fp8_gemm_close(Yh[done], ref[done], "covered rows")
    assert np.all(oracle.bf16_to_f32(Yh[16:40]) == 5.0), "rows beyond the bound were written"
    assert fb.fp8rl_check_device_error() == 0, "the device word is cleared by the check"


def test_grouped_persistent_many_items_skewed_routing(cuda_lib):
    # 64 experts x 16 weight slabs = 1024 (expert, slab) items, more than the
    # GPU holds at once, K = 768 not split: persistent CTAs take the items in
    # turn.  Skewed routing leaves some experts empty (items skipped by every
    # role) and gives others up to a few dozen tokens (one 32- or 64-row tile)
    rng = np.random.default_rng(71)
    counts = rng.multinomial(256, rng.dirichlet(np.ones(64) * 0.3))
    assert (counts == 0).any() and counts.max() > 16
    _grouped_case(counts, 2048, 768, seed=73, bound=int(counts.max()),
                  what=f"persistent, routing {counts.tolist()}")


def test_grouped_persistent_two_token_tiles(cuda_lib):
    # bound 150 -> 128-row token tiles, two per expert: 8 experts x 10 slabs x
    # 2 tiles = 160 items over one CTA per SM; item w is token tile w % 2 of
    # slab w / 2, and the second tile of an expert with <= 128 tokens is empty
    counts = np.array([150, 0, 3, 129, 1, 0, 40, 77])
    _grouped_case(counts, 1280, 512, seed=79, bound=150, what="persistent, two token tiles")


def test_grouped_persistent_rows_beyond_the_bound(cuda_lib):
    # 40 experts x 8 slabs = 320 items (persistent); expert 0 has 40 tokens
    # but the caller promised at most 4: rows 16..39 keep their sentinel and
    # the device reports the broken bound
    counts = np.array([40] + [1] * 39)
    N, K = 1024, 256
    Wq, Ws = _experts(40, N, K, 81)
    Xq, Xs, offsets = _routed_tokens(counts, K, 82)
    T = int(counts.sum())
    Y = torch.full((T, N), 5.0, dtype=torch.bfloat16, device="cuda")
    fb.fp8rl_gemm_w8a8_block_grouped(dev(Xq), dev(Xs), dev(Wq), dev(Ws), dev(offsets),
                                     max_tokens_per_expert=4, Y=Y)
    word = fb.fp8rl_check_device_error()
    assert word != 0 and (word & 0xFFFF) == 2, hex(word)
    ref = oracle.fp8_gemm_grouped(Xq, Xs, Wq, Ws, offsets)
    Yh = host(Y)
    done = np.r_[0:16, 40:T]
    assert_fp8_gemm_close(Yh[done], ref[done], "covered rows")
    assert np.all(oracle.bf16_to_f32(Yh[16:40]) == 5.0), "rows beyond the bound were written"
    assert fb.fp8rl_check_device_error() == 0
