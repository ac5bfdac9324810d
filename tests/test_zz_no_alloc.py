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
