"""GPU parity of the whole 8-bit linear layer from bf16 activations
(fp8rl_linear_w8a8_block: the activation quantizer, then the GEMM).

The activation codes and scales the call reports are compared bit for bit with
the oracle's 1x128 quantizer; Y is compared with the oracle's fp64
dequant-matmul of those codes within |y - y_ref| <= 2^-7 |y_ref| + 1e-3
rms(y_ref), the GEMM's tolerance.  Weights are quantized by the oracle."""
import numpy as np
import pytest
import torch

import oracle
from precision_rl_rollout_gb300 import binding as fb
from precision_rl_rollout_gb300 import synth
from parity_util import (act_cpu, assert_fp8_gemm_close, dev, host, oracle_fp8_weight, sample_rows)

pytestmark = pytest.mark.gpu


def _linear_case(X_cpu, N, K, seed_w, rows=None, what="", ldx_pad=0, ldy_pad=0):
    M = X_cpu.shape[0]
    Wq, Ws = oracle_fp8_weight(N, K, seed_w)
    bits = synth.bf16_bits(X_cpu)
    Xq_ref, Xs_ref = oracle.fp8_quant_act_group(bits)
    Xd = dev(bits, torch.bfloat16)
    if ldx_pad:
        big = torch.zeros((M, K + ldx_pad), dtype=torch.bfloat16, device="cuda")
        big[:, :K] = Xd
        Xd = big[:, :K]
    Ybuf = None
    if ldy_pad:
        Ybuf = torch.full((M, N + ldy_pad), 3.0, dtype=torch.bfloat16, device="cuda")
    Y, Xq, Xs = fb.fp8rl_linear_w8a8_block(Xd, dev(Wq), dev(Ws), Y=None if Ybuf is None else Ybuf[:, :N],
                                           want_codes=True)
    Xq_h, Xs_h = host(Xq), host(Xs)
    assert np.array_equal(Xq_h, Xq_ref), f"{what}: codes differ at {np.argwhere(Xq_h != Xq_ref)[:4].tolist()}"
    assert np.array_equal(Xs_h.view(np.uint32), Xs_ref.view(np.uint32)), f"{what}: scales differ"
    if Ybuf is not None:
        assert bool((Ybuf[:, N:] == 3.0).all()), f"{what}: wrote outside Y"
    if rows is None:
        rows = np.arange(M)
    ref = oracle.fp8_gemm(Xq_ref[rows], Xs_ref[:, rows], Wq, Ws)
    return assert_fp8_gemm_close(host(Y)[rows], ref, what)


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (5, 256, 384), (16, 512, 256), (17, 384, 640),
                                   (32, 256, 1280), (33, 128, 1024), (48, 640, 512), (64, 256, 4352),
                                   (65, 256, 256), (200, 384, 384)])
def test_linear_small_full(cuda_lib, M, N, K):
    _linear_case(act_cpu(M, K, 300 + M + K), N, K, 400 + N + K, what=f"M={M} N={N} K={K}")


def test_linear_edge_rows_and_strides(cuda_lib):
    # planted rows (all zero, all -0, one non-zero, huge, subnormal, E4M3 ties),
    # padded X and Y rows
    X = synth.edge_case_activation(24, 768, 71)
    _linear_case(X, 384, 768, 72, what="edge rows", ldx_pad=64, ldy_pad=8)
    X = synth.edge_case_activation(64, 512, 73)
    _linear_case(X, 256, 512, 74, what="edge rows M=64", ldx_pad=8)


def test_linear_without_codes_matches_with_codes(cuda_lib):
    X = dev(synth.bf16_bits(act_cpu(40, 1024, 81)), torch.bfloat16)
    Wq, Ws = oracle_fp8_weight(512, 1024, 82)
    Y1 = fb.fp8rl_linear_w8a8_block(X, dev(Wq), dev(Ws))
    Y2, _, _ = fb.fp8rl_linear_w8a8_block(X, dev(Wq), dev(Ws), want_codes=True)
    Y3 = fb.fp8rl_linear_w8a8_block(X, dev(Wq), dev(Ws))
    assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))
    assert torch.equal(Y1.view(torch.int16), Y3.view(torch.int16)), "two calls in a row differ"


def test_linear_empty_batch(cuda_lib):
    Wq, Ws = oracle_fp8_weight(256, 256, 5)
    Y = fb.fp8rl_linear_w8a8_block(torch.empty(0, 256, dtype=torch.bfloat16, device="cuda"), dev(Wq), dev(Ws))
    assert Y.shape == (0, 256)


@pytest.mark.parametrize("shape", synth.QWEN25_7B, ids=lambda s: s.name)
def test_linear_qwen7b_decode_m64_sampled(cuda_lib, shape):
    X = act_cpu(64, shape.K, synth.seed_for(2, 1))
    _linear_case(X, shape.N, shape.K, synth.seed_for(2, 0), rows=sample_rows(64, 6, seed=shape.N),
                 what=f"7B {shape.name}")


@pytest.mark.parametrize("M", (1, 8, 32, 128))
@pytest.mark.parametrize("shape", synth.QWEN25_32B, ids=lambda s: s.name)
def test_linear_qwen32b_decode_sampled(cuda_lib, shape, M):
    X = act_cpu(M, shape.K, synth.seed_for(3, 1))
    _linear_case(X, shape.N, shape.K, synth.seed_for(3, 0), rows=sample_rows(M, 3, seed=M),
                 what=f"32B {shape.name} M={M}")


def test_no_device_error_after_linear(cuda_lib):
    w = fb.fp8rl_check_device_error()
    assert w == 0, f"a bounded wait ran out: {w:#x}"
