"""The workspace-free KV-cache quantizer (fp8rl_quant_kv_tensor_noalloc).

It exists for callers that cannot allocate device memory for a workspace --
an engine that has reserved nearly all GPU memory for its KV-cache pool, or a
serving loop that must not call cudaMalloc/cudaFree because they synchronize
the device.  It keeps its scratch in a fixed library-owned device array.

This file is collected last on purpose, so that a run that stops at the first
failure has run every other test first.  It must also pass on its own in a
fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from precision_rl_rollout_gb300 import synth

pytestmark = pytest.mark.gpu


def _call_noalloc(lib, X, KVq, scale):
    R, C = X.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.fp8rl_quant_kv_tensor_noalloc(ctypes.c_void_p(X.data_ptr()), R, C, X.stride(0),
                                             ctypes.c_void_p(KVq.data_ptr()),
                                             ctypes.c_void_p(scale.data_ptr()), stream)


def _call_workspace(lib, X):
    R, C = X.shape
    KVq = torch.empty(R, C, dtype=torch.uint8, device="cuda")
    scale = torch.empty(1, dtype=torch.float32, device="cuda")
    need = lib.fp8rl_kv_workspace_bytes(R, C)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.fp8rl_quant_kv_tensor(ctypes.c_void_p(X.data_ptr()), R, C, X.stride(0),
                                   ctypes.c_void_p(KVq.data_ptr()), ctypes.c_void_p(scale.data_ptr()),
                                   ctypes.c_void_p(ws.data_ptr()), need, stream)
    assert rc == 0
    return KVq, scale


def test_noalloc_kv_quant_matches_workspace_version_on_two_calls_in_a_row(cuda_lib):
    lib = cuda_lib
    # two different tensors, the second larger than the first, through the same
    # shared scratch array back to back; outputs must equal the workspace
    # entry point's bit for bit (the quantizer's parity tolerance is exact)
    shapes = [(3000, 1024, 7), (8192 + 37, 1024, 8)]
    outs = []
    for R, C, seed in shapes:
        X = synth.activation(R, C, synth.seed_for(6, seed), device="cuda")
        KVq = torch.empty(R, C, dtype=torch.uint8, device="cuda")
        scale = torch.empty(1, dtype=torch.float32, device="cuda")
        assert _call_noalloc(lib, X, KVq, scale) == 0
        outs.append((X, KVq, scale))
    torch.cuda.synchronize()
    for X, KVq, scale in outs:
        ref_q, ref_s = _call_workspace(lib, X)
        torch.cuda.synchronize()
        assert torch.equal(scale.view(torch.int32), ref_s.view(torch.int32))
        assert torch.equal(KVq, ref_q)


def test_noalloc_kv_quant_rejects_tensors_above_its_limit(cuda_lib):
    lib = cuda_lib
    A = 0x10000   # never dereferenced: the size check comes before any CUDA call
    rc = lib.fp8rl_quant_kv_tensor_noalloc(A, 16384 + 1, 16384, 16384, A, A, None)
    assert rc == 6  # FP8RL_ERR_UNSUPPORTED
    rc = lib.fp8rl_quant_kv_tensor_noalloc(A, 16384, 16384 + 8, 16384 + 8, A, A, None)
    assert rc == 6


def _check_error_word(lib):
    word = ctypes.c_uint32(0)
    rc = lib.fp8rl_check_device_error(ctypes.byref(word))
    assert rc == 0 and word.value == 0, f"device error word {word.value:#x} (status {rc})"


def test_noalloc_kv_quant_paths_in_turn_match_oracle(cuda_lib):
    lib = cuda_lib
    # 16384 x 1024 is 1024 slices: too many for one pass.  With a row pitch its
    # partials go through the shared array in three launches; contiguous, one
    # CTA per SM publishes tagged slots there.  The calls after each find the
    # earlier call's words in the same array and must not mistake them for
    # their own slots.  Every output is compared with the oracle, bit for bit.
    for R, C, ld, seed in [(16384, 1024, 1032, 11), (3000, 1024, 1024, 12), (16384, 1024, 1024, 13),
                           (16384, 1024, 1032, 16), (8229, 1024, 1024, 14), (16384, 1024, 1024, 17)]:
        wide = synth.activation(R, ld, synth.seed_for(6, seed), device="cuda")
        X = wide[:, :C]
        KVq = torch.empty(R, C, dtype=torch.uint8, device="cuda")
        scale = torch.empty(1, dtype=torch.float32, device="cuda")
        assert _call_noalloc(lib, X, KVq, scale) == 0
        torch.cuda.synchronize()
        want_q, want_s = oracle.fp8_quant_tensor(synth.bf16_bits(X.cpu()))
        assert scale.cpu().view(torch.int32).item() == int(np.float32(want_s).view(np.int32))
        assert np.array_equal(KVq.cpu().numpy(), want_q)
    _check_error_word(lib)


def test_noalloc_kv_quant_at_its_size_limit(cuda_lib):
    lib = cuda_lib
    # 16384 x 16384 values, the documented maximum (16384 partials filling the
    # array): equal to the workspace entry point bit for bit, its scale equal
    # to fl32(amax / 448) of the whole tensor, and sampled rows equal to the
    # oracle's codes under that scale
    R = C = 16384
    X = synth.activation(R, C, synth.seed_for(6, 15), device="cuda")
    X[R - 1, C - 1] = -777.0                       # the amax in the last slice
    KVq = torch.empty(R, C, dtype=torch.uint8, device="cuda")
    scale = torch.empty(1, dtype=torch.float32, device="cuda")
    assert _call_noalloc(lib, X, KVq, scale) == 0
    ref_q, ref_s = _call_workspace(lib, X)
    torch.cuda.synchronize()
    assert torch.equal(scale.view(torch.int32), ref_s.view(torch.int32))
    assert torch.equal(KVq, ref_q)
    amax = np.float32(abs(X.float()).max().item())
    assert scale.cpu().numpy()[0] == np.float32(amax / np.float32(448.0))
    rows = np.array([0, 1, 8191, R - 2, R - 1])
    want = oracle.fp8_quant_with_scale(synth.bf16_bits(X[rows].cpu()), float(scale.cpu().numpy()[0]))
    assert np.array_equal(KVq[rows].cpu().numpy(), want)
    del X, KVq, ref_q
    _check_error_word(lib)
