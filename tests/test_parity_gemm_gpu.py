"""GPU parity of the GEMMs against the CPU oracle.

FP8: |y - y_ref| <= 2^-7 |y_ref| + 1e-3 rms(y_ref) element by element, y_ref
the oracle's fp64 dequant-matmul of the same codes (rms over the compared
rows).  INT8: accumulators and bf16 outputs bit-exact.  Operands are always
quantized by the oracle (or drawn by the generator), never by the CUDA path."""
import numpy as np
import pytest
import torch

import oracle
from precision_rl_rollout_gb300 import binding as fb
from precision_rl_rollout_gb300 import synth
from parity_util import (assert_fp8_gemm_close, dev, host, oracle_fp8_act, oracle_fp8_weight,
                         oracle_int8_act, oracle_int8_weight, sample_rows)

pytestmark = pytest.mark.gpu


def _fp8_case(M, N, K, seed_w, seed_x, rows=None, what=""):
    Wq, Ws = oracle_fp8_weight(N, K, seed_w)
    Xq, Xs = oracle_fp8_act(M, K, seed_x)
    Y = fb.fp8rl_gemm_w8a8_block(dev(Xq), dev(Xs), dev(Wq), dev(Ws))
    Yh = host(Y)
    if rows is None:
        rows = np.arange(M)
    ref = oracle.fp8_gemm(Xq[rows], Xs[:, rows], Wq, Ws)
    return assert_fp8_gemm_close(Yh[rows], ref, what or f"M={M} N={N} K={K}")


@pytest.mark.parametrize("M,N,K", [(16, 512, 256), (1, 128, 128), (5, 256, 384), (37, 384, 640),
                                   (64, 256, 1024), (129, 128, 256), (256, 640, 512), (257, 384, 128),
                                   (300, 384, 384), (1000, 768, 1280), (512, 256, 128), (700, 640, 384),
                                   (1537, 1152, 640),
                                   # few tiles, long K: split-K with the fp32 partials in the workspace
                                   (300, 256, 4096), (520, 512, 8192), (260, 384, 2048)])
def test_fp8_gemm_small_full(cuda_lib, M, N, K):
    _fp8_case(M, N, K, 100 + N + K, 200 + M + K)


def test_fp8_gemm_split_k_without_workspace_matches(cuda_lib):
    # a split-K shape run with and without the workspace it asks for: both
    # within tolerance of the oracle (the call without it gives up the split)
    M, N, K = 300, 256, 4096
    assert fb.fp8rl_gemm_workspace_bytes(M, N, K) > 0
    Wq, Ws = oracle_fp8_weight(N, K, 91)
    Xq, Xs = oracle_fp8_act(M, K, 92)
    ref = oracle.fp8_gemm(Xq, Xs, Wq, Ws)
    Y1 = fb.fp8rl_gemm_w8a8_block(dev(Xq), dev(Xs), dev(Wq), dev(Ws))
    Y2 = fb.fp8rl_gemm_w8a8_block(dev(Xq), dev(Xs), dev(Wq), dev(Ws),
                                  workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert_fp8_gemm_close(host(Y1), ref, "split-K")
    assert_fp8_gemm_close(host(Y2), ref, "no split")


@pytest.mark.parametrize("M,N,K", [(16, 4608, 3584), (9, 3584, 18944), (32, 5120, 5120)])
def test_fp8_decode_exchange_with_and_without_workspace(cuda_lib, M, N, K):
    # decode shapes whose split CTAs exchange partials through the workspace
    # (in a cluster after one barrier for 16-32 token tiles) and, with no
    # workspace, through distributed shared memory (kept to token tiles of up
    # to 32): both within tolerance of the oracle on the sampled rows
    assert fb.fp8rl_gemm_workspace_bytes(M, N, K) > 0
    Wq, Ws = oracle_fp8_weight(N, K, 95 + M)
    Xq, Xs = oracle_fp8_act(M, K, 96 + M)
    rows = sample_rows(M, 6, seed=M)
    ref = oracle.fp8_gemm(Xq[rows], Xs[:, rows], Wq, Ws)
    Y1 = fb.fp8rl_gemm_w8a8_block(dev(Xq), dev(Xs), dev(Wq), dev(Ws))
    Y2 = fb.fp8rl_gemm_w8a8_block(dev(Xq), dev(Xs), dev(Wq), dev(Ws),
                                  workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert_fp8_gemm_close(host(Y1)[rows], ref, "through memory")
    assert_fp8_gemm_close(host(Y2)[rows], ref, "on chip")


@pytest.mark.parametrize("M,N,K", [(64, 1024, 8192), (100, 768, 6144)])
def test_fp8_wide_token_tile_without_workspace(cuda_lib, M, N, K):
    # 64- and 128-token tiles with a K longer than one CTA's 32 blocks: with the
    # workspace the split CTAs exchange through memory; without it the call
    # goes to the 128 x 256 tile kernel (no exchange through distributed shared
    # memory for these tiles); both within tolerance on every row
    Wq, Ws = oracle_fp8_weight(N, K, 81 + M)
    Xq, Xs = oracle_fp8_act(M, K, 82 + M)
    ref = oracle.fp8_gemm(Xq, Xs, Wq, Ws)
    Y1 = fb.fp8rl_gemm_w8a8_block(dev(Xq), dev(Xs), dev(Wq), dev(Ws))
    Y2 = fb.fp8rl_gemm_w8a8_block(dev(Xq), dev(Xs), dev(Wq), dev(Ws),
                                  workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert_fp8_gemm_close(host(Y1), ref, "with workspace")
    assert_fp8_gemm_close(host(Y2), ref, "without workspace")


@pytest.mark.parametrize("M", [1, 8, 40])
def test_fp8_gemm_k_beyond_decode_limit(cuda_lib, M):
    # K = 33024 (258 blocks) is beyond the decode kernel's 8 x 32 blocks: every
    # M goes to the 128 x 256 tile kernel (split into K ranges through the
    # workspace, or whole without it); both within tolerance on every row
    N, K = 256, 33024
    Wq, Ws = oracle_fp8_weight(N, K, 83)
    Xq, Xs = oracle_fp8_act(M, K, 84 + M)
    ref = oracle.fp8_gemm(Xq, Xs, Wq, Ws)
    assert fb.fp8rl_gemm_workspace_bytes(M, N, K) > 0
    Y1 = fb.fp8rl_gemm_w8a8_block(dev(Xq), dev(Xs), dev(Wq), dev(Ws))
    Y2 = fb.fp8rl_gemm_w8a8_block(dev(Xq), dev(Xs), dev(Wq), dev(Ws),
                                  workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert_fp8_gemm_close(host(Y1), ref, f"split K, M={M}")
    assert_fp8_gemm_close(host(Y2), ref, f"whole K, M={M}")


def test_fp8_gemm_prefill_tail_split_sampled(cuda_lib):
    # 3 x 54 = 162 tiles of 128 x 256: one full wave on 152 SMs and 10 tiles
    # after it, which are split into K ranges through the workspace; sampled
    # rows cover every row tile and, with all columns, the split tiles too.
    # Also run without the workspace (no split): both within tolerance.
    M, N, K = 384, 13824, 8192
    Wq, Ws = oracle_fp8_weight(N, K, 93)
    Xq, Xs = oracle_fp8_act(M, K, 94)
    rows = np.array([0, 127, 128, 200, 255, 256, 300, 383])
    ref = oracle.fp8_gemm(Xq[rows], Xs[:, rows], Wq, Ws)
    Y1 = fb.fp8rl_gemm_w8a8_block(dev(Xq), dev(Xs), dev(Wq), dev(Ws))
    Y2 = fb.fp8rl_gemm_w8a8_block(dev(Xq), dev(Xs), dev(Wq), dev(Ws),
                                  workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert_fp8_gemm_close(host(Y1)[rows], ref, "tail split")
    assert_fp8_gemm_close(host(Y2)[rows], ref, "no split")


@pytest.mark.parametrize("N", [768, 13824])
def test_fp8_gemm_prefill_grouped_tile_order(cuda_lib, N):
    # activations above 48 MB (2560 x 20480): the 128 x 256 tile kernel walks
    # groups of 16 token tiles (here 16 + a last group of 4); N = 768 splits
    # every tile in K (reduced by a second launch), N = 13824 splits none.
    # One sampled row in every token tile, all columns.
    M, K = 2560, 20480
    Wq, Ws = oracle_fp8_weight(N, K, 77)
    Xq, Xs = oracle_fp8_act(M, K, 78)
    rows = _rows_in_distinct_tiles(M, 20, seed=N)
    ref = oracle.fp8_gemm(Xq[rows], Xs[:, rows], Wq, Ws)
    Y = fb.fp8rl_gemm_w8a8_block(dev(Xq), dev(Xs), dev(Wq), dev(Ws))
    assert_fp8_gemm_close(host(Y)[rows], ref, f"grouped order N={N}")


def test_fp8_gemm_tiny_config(cuda_lib):
    Wq, Ws = oracle_fp8_weight(synth.TINY.N, synth.TINY.K, synth.seed_for(1, 0))
    from parity_util import act_cpu
    X = act_cpu(synth.TINY_M, synth.TINY.K, synth.seed_for(1, 1), n_outliers=2)
    Xq, Xs = oracle.fp8_quant_act_group(synth.bf16_bits(X))
    Y = fb.fp8rl_gemm_w8a8_block(dev(Xq), dev(Xs), dev(Wq), dev(Ws))
    assert_fp8_gemm_close(host(Y), oracle.fp8_gemm(Xq, Xs, Wq, Ws), "tiny")


def test_fp8_gemm_empty_batch_and_strided_output(cuda_lib):
    Wq, Ws = oracle_fp8_weight(256, 256, 5)
    Y0 = fb.fp8rl_gemm_w8a8_block(torch.empty(0, 256, dtype=torch.uint8, device="cuda"),
                                  torch.empty(2, 0, device="cuda"), dev(Wq), dev(Ws))
    assert Y0.shape == (0, 256)
    Xq, Xs = oracle_fp8_act(9, 256, 6)
    big = torch.full((9, 264), 7.0, dtype=torch.bfloat16, device="cuda")
    fb.fp8rl_gemm_w8a8_block(dev(Xq), dev(Xs), dev(Wq), dev(Ws), Y=big[:, :256])
    assert_fp8_gemm_close(host(big[:, :256]), oracle.fp8_gemm(Xq, Xs, Wq, Ws), "strided Y")
    assert bool((big[:, 256:] == 7.0).all()), "GEMM wrote outside Y"


@pytest.mark.parametrize("shape", synth.QWEN25_7B, ids=lambda s: s.name)
def test_fp8_gemm_qwen7b_decode_m64_sampled(cuda_lib, shape):
    _fp8_case(64, shape.N, shape.K, synth.seed_for(2, 0), synth.seed_for(2, 1),
              rows=sample_rows(64, 6, seed=shape.N), what=f"7B {shape.name}")


@pytest.mark.parametrize("M", synth.DECODE_M_SWEEP)
@pytest.mark.parametrize("shape", synth.QWEN25_32B, ids=lambda s: s.name)
def test_fp8_gemm_qwen32b_decode_sweep_sampled(cuda_lib, shape, M):
    _fp8_case(M, shape.N, shape.K, synth.seed_for(3, 0), synth.seed_for(3, 1),
              rows=sample_rows(M, 3, seed=M), what=f"32B {shape.name} M={M}")


def _rows_in_distinct_tiles(M, n, seed, tile=128):
    """n rows, each in its own `tile`-row tile: the first and last tiles and n-2
    seeded ones between them, one seeded row inside each."""
    rng = np.random.default_rng(seed)
    tiles = (M + tile - 1) // tile
    pick = np.concatenate([[0, tiles - 1], rng.choice(np.arange(1, tiles - 1), size=n - 2, replace=False)])
    rows = [min(M - 1, t * tile + int(rng.integers(tile))) for t in sorted(pick)]
    return np.array(rows)


@pytest.mark.parametrize("shape", synth.QWEN25_32B, ids=lambda s: s.name)
def test_fp8_gemm_qwen32b_prefill_sampled(cuda_lib, shape):
    # M = 8192 (64 token tiles of the persistent 128 x 256 schedule): 16 rows,
    # each in a different token tile, against every output column
    rows = _rows_in_distinct_tiles(synth.PREFILL_M, 16, seed=shape.K + shape.N)
    assert len(set(r // 128 for r in rows)) == 16
    _fp8_case(synth.PREFILL_M, shape.N, shape.K, synth.seed_for(4, 0), synth.seed_for(4, 1),
              rows=rows, what=f"prefill {shape.name}")


def _int8_case(M, N, K, seed_w, seed_x, rows=None):
    Wq, Ws = oracle_int8_weight(N, K, seed_w)
    Xq, Xs = oracle_int8_act(M, K, seed_x)
    Y, acc = fb.int8rl_gemm_w8a8(dev(Xq), dev(Xs), dev(Wq), dev(Ws), want_acc=True)
    if rows is None:
        rows = np.arange(M)
    want_acc, want_y = oracle.int8_gemm(Xq[rows], Xs[rows], Wq, Ws)
    got_acc, got_y = host(acc)[rows], host(Y)[rows]
    assert np.array_equal(got_acc, want_acc), f"acc differs at {np.argwhere(got_acc != want_acc)[:4].tolist()}"
    assert np.array_equal(got_y, want_y), f"Y differs at {np.argwhere(got_y != want_y)[:4].tolist()}"


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (16, 512, 256), (37, 384, 640), (300, 256, 384),
                                   (513, 256, 640), (1000, 384, 128)])
def test_int8_gemm_small_full(cuda_lib, M, N, K):
    _int8_case(M, N, K, 300 + N, 400 + M)


def test_int8_gemm_extreme_codes_exact(cuda_lib):
    M, N, K = 3, 128, 27648
    Xq = np.full((M, K), 127, np.int8)
    Xq[1] = -127
    Xq[2, ::2] = -127
    Wq = np.full((N, K), 127, np.int8)
    Xs = np.array([1.0, 0.5, 3.0], np.float32)
    Ws = np.linspace(0.001, 2.0, N).astype(np.float32)
    Y, acc = fb.int8rl_gemm_w8a8(dev(Xq), dev(Xs), dev(Wq), dev(Ws), want_acc=True)
    want_acc, want_y = oracle.int8_gemm(Xq, Xs, Wq, Ws)
    assert np.array_equal(host(acc), want_acc) and int(want_acc[0, 0]) == 127 * 127 * K
    assert np.array_equal(host(Y), want_y)


def test_int8_gemm_large_batch_path_ragged(cuda_lib):
    # 3 x 51 = 153 tiles of 128 x 256: the large-batch path (fp16 copies in the
    # workspace).  M = 300 leaves a partial token tile, N = 12928 a last tile
    # with one 128-column half beyond N, K = 1152 a last TMEM group of 2 of 8
    # stages.  The same call without the workspace runs the small-batch kernel;
    # both are bit-exact on the sampled rows.
    M, N, K = 300, 12928, 1152
    assert fb.int8rl_gemm_workspace_bytes(M, N, K) == (M + N) * K * 2
    Wq, Ws = oracle_int8_weight(N, K, 97)
    Xq, Xs = oracle_int8_act(M, K, 98)
    rows = np.array([0, 1, 127, 128, 255, 256, 290, 299])
    want_acc, want_y = oracle.int8_gemm(Xq[rows], Xs[rows], Wq, Ws)
    for ws in (None, torch.empty(16, dtype=torch.uint8, device="cuda")):
        Y, acc = fb.int8rl_gemm_w8a8(dev(Xq), dev(Xs), dev(Wq), dev(Ws), want_acc=True, workspace=ws)
        got_acc, got_y = host(acc)[rows], host(Y)[rows]
        assert np.array_equal(got_acc, want_acc), f"acc differs at {np.argwhere(got_acc != want_acc)[:4].tolist()}"
        assert np.array_equal(got_y, want_y), f"Y differs at {np.argwhere(got_y != want_y)[:4].tolist()}"


def test_int8_gemm_large_batch_split_k_ragged(cuda_lib):
    # 3 x 11 = 33 tiles, too few for the GPU: each tile's K (4096) is split in
    # 4 ranges of 16 stages, whose int32 partials a second launch adds; M = 300
    # leaves a partial token tile and N = 2688 a last tile with one half beyond N
    M, N, K = 300, 2688, 4096
    need = fb.int8rl_gemm_workspace_bytes(M, N, K)
    assert need > (M + N) * K * 2                      # fp16 copies + int32 partials
    Wq, Ws = oracle_int8_weight(N, K, 99)
    Xq, Xs = oracle_int8_act(M, K, 100)
    rows = np.array([0, 1, 127, 128, 255, 256, 290, 299])
    want_acc, want_y = oracle.int8_gemm(Xq[rows], Xs[rows], Wq, Ws)
    Y, acc = fb.int8rl_gemm_w8a8(dev(Xq), dev(Xs), dev(Wq), dev(Ws), want_acc=True)
    got_acc, got_y = host(acc)[rows], host(Y)[rows]
    assert np.array_equal(got_acc, want_acc), f"acc differs at {np.argwhere(got_acc != want_acc)[:4].tolist()}"
    assert np.array_equal(got_y, want_y), f"Y differs at {np.argwhere(got_y != want_y)[:4].tolist()}"


def test_int8_gemm_large_batch_extreme_codes_exact(cuda_lib):
    # every code at +-127 over K = 8192 (16 exact TMEM groups of 512) on the
    # large-batch path: |acc| = 127^2 K
    M, N, K = 256, 19456, 8192
    assert fb.int8rl_gemm_workspace_bytes(M, N, K) > 0
    Xq = np.full((M, K), 127, np.int8)
    Xq[1::2] = -127
    Xq[2, ::2] = -127
    Wq = np.full((N, K), 127, np.int8)
    Wq[N // 2:] = -127
    Xs = np.linspace(0.5, 3.0, M).astype(np.float32)
    Ws = np.linspace(0.001, 2.0, N).astype(np.float32)
    Y, acc = fb.int8rl_gemm_w8a8(dev(Xq), dev(Xs), dev(Wq), dev(Ws), want_acc=True)
    rows = np.array([0, 1, 2, 255])
    want_acc, want_y = oracle.int8_gemm(Xq[rows], Xs[rows], Wq, Ws)
    assert int(want_acc[0, 0]) == 127 * 127 * K and int(want_acc[1, 0]) == -127 * 127 * K
    assert np.array_equal(host(acc)[rows], want_acc)
    assert np.array_equal(host(Y)[rows], want_y)


@pytest.mark.parametrize("M,N,K", [(65, 384, 640), (129, 256, 1152), (200, 384, 2048), (256, 128, 128),
                                   (256, 1280, 3840), (128, 128, 128), (100, 512, 256), (96, 256, 1152),
                                   (128, 768, 4096)])
def test_int8_gemm_256_token_path(cuda_lib, M, N, K):
    # 65 .. 256 tokens: weight blocks in TMEM against 256-token tiles of an fp16
    # copy of X (in the workspace).  Few weight slabs split K: the int32
    # partials of the ranges go to the workspace and a second launch adds them.
    # K = 128 is one exact group of one block; K = 1152 ends on a group of one.
    # Up to 128 tokens the two MMA threads take alternate blocks for the same
    # 128 tokens (M = 128, K = 128: the second has none; K = 256: one each).
    need = fb.int8rl_gemm_workspace_bytes(M, N, K)
    assert need >= M * K * 2
    assert fb.int8rl_gemm_kernel_count(M, N, K, need) in (2, 3)
    _int8_case(M, N, K, 500 + N + K, 600 + M + K)


@pytest.mark.parametrize("K", [640, 1152])
def test_int8_small_batch_persistent_many_items(cuda_lib, K):
    # the small-batch kernel without a workspace: 200 tokens are four 64-token
    # tiles, 19456 rows 152 slabs, so 608 work items over a persistent grid of
    # one CTA per SM (four each, token tile fastest).  K = 640 is 5 blocks: a
    # last promotion group of one block, where the second MMA issuer has no
    # block and only keeps its barrier phases in step, item after item.
    M, N = 200, 19456
    Wq, Ws = oracle_int8_weight(N, K, 71 + K)
    Xq, Xs = oracle_int8_act(M, K, 72 + K)
    Y, acc = fb.int8rl_gemm_w8a8(dev(Xq), dev(Xs), dev(Wq), dev(Ws), want_acc=True,
                                 workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    rows = np.array([0, 63, 64, 127, 130, 191, 192, 199])
    want_acc, want_y = oracle.int8_gemm(Xq[rows], Xs[rows], Wq, Ws)
    assert np.array_equal(host(acc)[rows], want_acc), f"acc differs at {np.argwhere(host(acc)[rows] != want_acc)[:4].tolist()}"
    assert np.array_equal(host(Y)[rows], want_y), f"Y differs at {np.argwhere(host(Y)[rows] != want_y)[:4].tolist()}"


def test_int8_gemm_256_token_path_splits_and_ragged_second_tile(cuda_lib):
    # 300 tokens on a layer of 2^27 weights: two 256-token tiles, the second
    # with 44 live rows; checked on rows of both tiles.  Seeded random codes
    # and scales (the quantizer is not under test here).
    M, N, K = 300, 16384, 8192
    assert N * K >= 1 << 27 and fb.int8rl_gemm_workspace_bytes(M, N, K) >= M * K * 2
    rng = np.random.default_rng(77)
    Wq = rng.integers(-127, 128, size=(N, K), dtype=np.int8)
    Xq = rng.integers(-127, 128, size=(M, K), dtype=np.int8)
    Ws = (rng.random(N) * 1e-3 + 1e-5).astype(np.float32)
    Xs = (rng.random(M) * 1e-2 + 1e-4).astype(np.float32)
    Y, acc = fb.int8rl_gemm_w8a8(dev(Xq), dev(Xs), dev(Wq), dev(Ws), want_acc=True)
    rows = np.array([0, 1, 130, 255, 256, 280, 299])
    want_acc, want_y = oracle.int8_gemm(Xq[rows], Xs[rows], Wq, Ws)
    assert np.array_equal(host(acc)[rows], want_acc), "acc differs"
    assert np.array_equal(host(Y)[rows], want_y), "Y differs"


@pytest.mark.parametrize("M", [200, 128])
def test_int8_gemm_256_token_path_extreme_codes_exact(cuda_lib, M):
    # every code at +-127 over K = 8192 on the 256-token path with a K split
    # (two weight slabs): each exact TMEM group of two K blocks reaches
    # 256 * 127^2, the top of its range, and |acc| = 127^2 K (M = 128: the
    # one-half form, whose two accumulators are added at the end)
    N, K = 256, 8192
    ws = fb.int8rl_gemm_workspace_bytes(M, N, K)
    assert fb.int8rl_gemm_kernel_count(M, N, K, ws) == 3            # conversion, GEMM, split reduction
    Xq = np.full((M, K), 127, np.int8)
    Xq[1::2] = -127
    Xq[2, ::2] = -127
    Wq = np.full((N, K), 127, np.int8)
    Wq[N // 2:] = -127
    Xs = np.linspace(0.5, 3.0, M).astype(np.float32)
    Ws = np.linspace(0.001, 2.0, N).astype(np.float32)
    Y, acc = fb.int8rl_gemm_w8a8(dev(Xq), dev(Xs), dev(Wq), dev(Ws), want_acc=True)
    want_acc, want_y = oracle.int8_gemm(Xq, Xs, Wq, Ws)
    assert int(want_acc[0, 0]) == 127 * 127 * K and int(want_acc[1, 0]) == -127 * 127 * K
    assert np.array_equal(host(acc), want_acc)
    assert np.array_equal(host(Y), want_y)


def test_int8_gemm_256_token_shape_without_workspace(cuda_lib):
    # the same batch with too little workspace runs the small-batch kernel: also exact
    M, N, K = 200, 384, 2048
    Wq, Ws = oracle_int8_weight(N, K, 81)
    Xq, Xs = oracle_int8_act(M, K, 82)
    want_acc, want_y = oracle.int8_gemm(Xq, Xs, Wq, Ws)
    Y, acc = fb.int8rl_gemm_w8a8(dev(Xq), dev(Xs), dev(Wq), dev(Ws), want_acc=True,
                                 workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert np.array_equal(host(acc), want_acc) and np.array_equal(host(Y), want_y)


@pytest.mark.parametrize("M", synth.INT8_M_SWEEP)
@pytest.mark.parametrize("shape", synth.QWEN25_32B, ids=lambda s: s.name)
def test_int8_gemm_qwen32b_sampled(cuda_lib, shape, M):
    _int8_case(M, shape.N, shape.K, synth.seed_for(5, 0), synth.seed_for(5, 1),
               rows=sample_rows(M, 3, seed=M + shape.N))


@pytest.mark.parametrize("M,N,K", [(1, 4608, 3584), (16, 3584, 18944), (32, 5120, 5120), (64, 3584, 3584),
                                   (64, 3584, 18944), (256, 5120, 27648), (300, 256, 4096)])
def test_fp8_gemm_is_deterministic(cuda_lib, M, N, K):
    # every split-K exchange adds the partials in a fixed order: repeated calls,
    # with the workspace reused, give the same bits (each path of the plan:
    # cluster shared memory / cluster L2 / second launch / prefill split)
    g = torch.Generator(device="cuda").manual_seed(M + N + K)
    Xq = torch.randint(0, 0x7e, (M, K), dtype=torch.uint8, device="cuda", generator=g)
    Wq = torch.randint(0, 0x7e, (N, K), dtype=torch.uint8, device="cuda", generator=g)
    Xs = torch.rand((K // 128, M), device="cuda", generator=g)
    Ws = torch.rand((N // 128, K // 128), device="cuda", generator=g)
    ws = torch.empty(max(16, fb.fp8rl_gemm_workspace_bytes(M, N, K)), dtype=torch.uint8, device="cuda")
    Y0 = fb.fp8rl_gemm_w8a8_block(Xq, Xs, Wq, Ws, workspace=ws)
    for _ in range(3):
        assert torch.equal(fb.fp8rl_gemm_w8a8_block(Xq, Xs, Wq, Ws, workspace=ws), Y0)


@pytest.mark.parametrize("M", [1, 8, 32, 64, 200])
@pytest.mark.parametrize("shape", [synth.QWEN25_7B[0], synth.QWEN25_7B[1], synth.QWEN25_32B[0],
                                   synth.QWEN25_32B[1], synth.QWEN25_7B[3]], ids=lambda s: s.name + str(s.K))
def test_fp8_gemm_weights_stable_flag_back_to_back(cuda_lib, shape, M):
    # FP8RL_GEMM_WEIGHTS_STABLE: weight tiles are loaded before the dependency
    # wait (shapes of at most 48 MB); a chain of calls on different weights
    # and inputs, each right after the previous GEMM, every output checked
    seeds = [(61, 62), (63, 64), (65, 66)]
    cases = [(oracle_fp8_weight(shape.N, shape.K, sw), oracle_fp8_act(M, shape.K, sx)) for sw, sx in seeds]
    dev_cases = [(dev(wq), dev(ws), dev(xq), dev(xs)) for (wq, ws), (xq, xs) in cases]
    Ys = [torch.empty(M, shape.N, dtype=torch.bfloat16, device="cuda") for _ in seeds]
    torch.cuda.synchronize()
    for (wq, ws, xq, xs), Y in zip(dev_cases, Ys):
        fb.fp8rl_gemm_w8a8_block(xq, xs, wq, ws, Y=Y, weights_stable=True)
    rows = sample_rows(M, 4, seed=M + shape.N)
    for ((wq, ws), (xq, xs)), Y in zip(cases, Ys):
        ref = oracle.fp8_gemm(xq[rows], xs[:, rows], wq, ws)
        assert_fp8_gemm_close(host(Y)[rows], ref, f"stable weights {shape.name} M={M}")


def test_no_device_error_after_gemms(cuda_lib):
    assert fb.fp8rl_check_device_error() == 0


def test_requant_then_gemm_back_to_back_same_buffers(cuda_lib):
    """Kernels are launched with programmatic dependent launch; a GEMM issued right
    after a requant that rewrites its weight buffers must see the new codes."""
    from parity_util import weight_cpu
    N, K = 1024, 768
    seeds = (72, 73, 74)
    Wd = [weight_cpu(N, K, seed).cuda() for seed in seeds]
    for M in (8, 300):
        Xq, Xs = oracle_fp8_act(M, K, 71)
        Xqd, Xsd = dev(Xq), dev(Xs)
        Wq = torch.empty(N, K, dtype=torch.uint8, device="cuda")
        Ws = torch.empty(N // 128, K // 128, dtype=torch.float32, device="cuda")
        Ys = [torch.empty(M, N, dtype=torch.bfloat16, device="cuda") for _ in seeds]
        torch.cuda.synchronize()
        for W, Y in zip(Wd, Ys):                          # requant, GEMM, requant, GEMM, ... back to back
            fb.fp8rl_quant_weight_block(W, Wq, Ws)        # same weight buffers every time
            fb.fp8rl_gemm_w8a8_block(Xqd, Xsd, Wq, Ws, Y=Y)
        for seed, Y in zip(seeds, Ys):
            wq, ws = oracle_fp8_weight(N, K, seed)
            assert_fp8_gemm_close(host(Y), oracle.fp8_gemm(Xq, Xs, wq, ws), f"seed {seed} M={M}")
