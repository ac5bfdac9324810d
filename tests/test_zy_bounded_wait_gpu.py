"""Failure detection without a fault: the bounded mbarrier wait used by every
tcgen05 kernel gives up on a barrier that nothing completes, within its limit,
and the context stays usable (a library call after it still runs and passes
its own device check).  The test kernel is built here from the library's
header; it waits on a barrier of its own, not on another rank or kernel."""
import ctypes
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import torch

from precision_rl_rollout_gb300 import binding as fb

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "precision_rl_rollout_gb300", "csrc")


@pytest.fixture(scope="module")
def selftest_lib():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    d = tempfile.mkdtemp(prefix="fp8rl_selftest_")
    so = os.path.join(d, "libbounded_wait.so")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared",
                    "-Xcompiler", "-fPIC", "-I", CSRC, "-o", so,
                    os.path.join(HERE, "cuda", "bounded_wait_selftest.cu")], check=True)
    lib = ctypes.CDLL(so)
    lib.run_bounded_wait.argtypes = [ctypes.c_ulonglong, ctypes.c_void_p]
    lib.run_bounded_wait.restype = ctypes.c_int
    yield lib
    shutil.rmtree(d, ignore_errors=True)


def test_bounded_wait_gives_up_and_context_survives(cuda_lib, selftest_lib):
    limit_ns = 20_000_000                                      # 20 ms
    out = torch.zeros(3, dtype=torch.int64, device="cuda")
    assert selftest_lib.run_bounded_wait(limit_ns, ctypes.c_void_p(out.data_ptr())) == 0
    torch.cuda.synchronize()
    ok, t_wait, t_drain = (int(v) for v in out.cpu())
    assert ok == 0, "a wait on a barrier nothing completes reported success"
    assert limit_ns <= t_wait < 50 * limit_ns, t_wait
    assert limit_ns <= t_drain < 50 * limit_ns, t_drain
    # the context is still usable: a library call runs and passes its own check
    X = torch.randn(16, 256, device="cuda").to(torch.bfloat16)
    Xq, Xs = fb.fp8rl_quant_act_group(X)
    torch.cuda.synchronize()
    assert fb.fp8rl_check_device_error() == 0
    assert np.isfinite(Xs.cpu().numpy()).all()
