"""GPU parity of the token-level TIS/MIS rollout correction against the CPU
oracle: clipped/masked and valid counts exact, weights within 4 ulp of the
fp64 exp, sums within fp32 accumulation error."""
import math

import numpy as np
import pytest
import torch

import oracle
from parity_util import host
from precision_rl_rollout_gb300 import binding as fb

pytestmark = pytest.mark.gpu


def _inputs(n, seed, sigma=0.3):
    g = torch.Generator().manual_seed(seed)
    lt = torch.randn(n, generator=g) * 1.5 - 2.0
    lr = lt + torch.randn(n, generator=g) * sigma
    mask = (torch.rand(n, generator=g) < 0.9).to(torch.uint8)
    return lt.float(), lr.float(), mask


@pytest.mark.parametrize("n", [0, 1, 7, 4096, 4097, 100003, 1 << 20])
@pytest.mark.parametrize("mode", [0, 1])
def test_rollout_is_matches_oracle(cuda_lib, n, mode):
    lt, lr, mask = _inputs(n, 100 + n)
    log_clip = float(np.float32(math.log(2.0)))
    w, stats = fb.fp8rl_rollout_is_weights(lt.cuda(), lr.cuda(), mask.cuda(), log_clip, mode)
    want_w, want_st = oracle.rollout_is(lt.numpy(), lr.numpy(), mask.numpy(), log_clip, mode)
    got_w, got_st = host(w).astype(np.float64), host(stats)
    assert got_st[0] == want_st[0] and got_st[1] == want_st[1]      # exact counts
    assert np.all(np.abs(got_w - want_w) <= 4 * 2.0 ** -23 * np.abs(want_w))
    tol = 1e-6 * max(1.0, float(np.sum(np.abs(want_w))))
    assert abs(got_st[2] - want_st[2]) <= tol
    d = np.abs(lt.numpy() - lr.numpy()).astype(np.float64)
    assert abs(got_st[3] - want_st[3]) <= 1e-6 * max(1.0, float(np.sum(d)))


def test_rollout_is_no_mask_and_deterministic(cuda_lib):
    n = 3 * 4096 + 5
    lt, lr, _ = _inputs(n, 9, sigma=1.0)
    runs = [fb.fp8rl_rollout_is_weights(lt.cuda(), lr.cuda(), None, 0.0, 0) for _ in range(2)]
    want_w, want_st = oracle.rollout_is(lt.numpy(), lr.numpy(), np.ones(n, np.uint8), 0.0, 0)
    assert host(runs[0][1])[0] == n and host(runs[0][1])[1] == want_st[1]
    assert np.array_equal(host(runs[0][1]), host(runs[1][1]))        # same bits run to run
    assert np.all(host(runs[0][0]) <= 1.0)                           # C = 1 truncates to <= 1


def test_rollout_is_shared_workspace_across_calls_and_graph_replays(cuda_lib):
    # One workspace, filled with garbage first, serves calls of different sizes:
    # a large call leaves tagged records that a later smaller call must not
    # take, and every call derives its tag from the one the previous left.
    # Then a CUDA graph replays one call on new inputs: each replay gets a new
    # tag from the header word, so its statistics are its own.
    big = 1 << 20
    ws = torch.full((fb.fp8rl_rollout_is_workspace_bytes(big),), 0xFF, dtype=torch.uint8, device="cuda")
    log_clip = float(np.float32(math.log(2.0)))
    for k, n in enumerate([big, 5000, big, 77, 4096 * 3]):
        lt, lr, mask = _inputs(n, 300 + k)
        w = torch.empty(n, dtype=torch.float32, device="cuda")
        st = torch.empty(4, dtype=torch.float64, device="cuda")
        fb.fp8rl_rollout_is_weights(lt.cuda(), lr.cuda(), mask.cuda(), log_clip, k % 2, w, st, ws)
        want_w, want_st = oracle.rollout_is(lt.numpy(), lr.numpy(), mask.numpy(), log_clip, k % 2)
        got = host(st)
        assert got[0] == want_st[0] and got[1] == want_st[1], (n, got, want_st)
        assert abs(got[2] - want_st[2]) <= 1e-6 * max(1.0, float(np.sum(np.abs(want_w))))
    n = 100003
    lt_d = torch.empty(n, device="cuda")
    lr_d = torch.empty(n, device="cuda")
    mask_d = torch.empty(n, dtype=torch.uint8, device="cuda")
    w = torch.empty(n, dtype=torch.float32, device="cuda")
    st = torch.empty(4, dtype=torch.float64, device="cuda")
    lt, lr, mask = _inputs(n, 400)
    lt_d.copy_(lt), lr_d.copy_(lr), mask_d.copy_(mask)
    fb.fp8rl_rollout_is_weights(lt_d, lr_d, mask_d, log_clip, 0, w, st, ws)     # warm up before capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fb.fp8rl_rollout_is_weights(lt_d, lr_d, mask_d, log_clip, 0, w, st, ws)
    for r in range(3):
        lt, lr, mask = _inputs(n, 500 + r)
        lt_d.copy_(lt), lr_d.copy_(lr), mask_d.copy_(mask)
        g.replay()
        want_w, want_st = oracle.rollout_is(lt.numpy(), lr.numpy(), mask.numpy(), log_clip, 0)
        got = host(st)
        assert got[0] == want_st[0] and got[1] == want_st[1], (r, got, want_st)
        assert np.all(np.abs(host(w).astype(np.float64) - want_w) <= 4 * 2.0 ** -23 * np.abs(want_w))
    assert fb.fp8rl_check_device_error() == 0


@pytest.mark.parametrize("mode", [0, 1])
def test_rollout_is_unaligned_inputs_take_the_scalar_path(cuda_lib, mode):
    # log-prob views that start one element into their buffers (4-byte but not
    # 16-byte aligned) and a mask that starts one byte in: the kernel's scalar
    # path, with the same one-launch statistics; over several CTAs' ranges
    n = 3 * 4096 * 7 + 13
    lt, lr, mask = _inputs(n + 1, 900 + mode)
    lt_d, lr_d, mask_d = lt.cuda()[1:], lr.cuda()[1:], mask.cuda()[1:]
    assert lt_d.data_ptr() % 16 != 0 and mask_d.data_ptr() % 4 != 0
    log_clip = float(np.float32(math.log(2.0)))
    w, stats = fb.fp8rl_rollout_is_weights(lt_d, lr_d, mask_d, log_clip, mode)
    want_w, want_st = oracle.rollout_is(lt.numpy()[1:], lr.numpy()[1:], mask.numpy()[1:], log_clip, mode)
    got_w, got_st = host(w).astype(np.float64), host(stats)
    assert got_st[0] == want_st[0] and got_st[1] == want_st[1]
    assert np.all(np.abs(got_w - want_w) <= 4 * 2.0 ** -23 * np.abs(want_w))
    assert abs(got_st[2] - want_st[2]) <= 1e-6 * max(1.0, float(np.sum(np.abs(want_w))))
    assert fb.fp8rl_check_device_error() == 0
