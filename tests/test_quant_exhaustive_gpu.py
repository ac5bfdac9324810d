"""Exhaustive-domain parity of the quantizers against the CPU oracle.

A block's codes depend only on its amax A (a bf16 value) and on each element x
with |x| <= A.  For every positive finite bf16 amax (32639 bit patterns) these
tests build a block / group / row holding A and the 2561 bf16 magnitudes just
below it (down to ~20 binades under A, i.e. every quotient x/s from 448 down
past the E4M3 underflow boundary 2^-10 and every INT8 half-integer boundary),
each with both signs, and require the GPU codes and scales to equal the
oracle's bit for bit.  This covers the whole input domain of the division and
rounding steps of the quantizers (their fast reciprocal-based division is
exact on it), not a random sample."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import bits_u32, host
from precision_rl_rollout_gb300 import binding as fb

pytestmark = pytest.mark.gpu

N_AMAX = 0x7F7F          # positive finite bf16 patterns 0x0001 .. 0x7F7F
SPAN = 2561              # magnitudes A, A-1, ..., A-2560 (clamped at 0)


def _value_lists():
    """[N_AMAX, 2*SPAN] uint16: for amax pattern A the values +-(A - j)."""
    A = np.arange(1, N_AMAX + 1, dtype=np.int64)[:, None]
    mag = np.maximum(A - np.arange(SPAN, dtype=np.int64)[None, :], 0).astype(np.uint16)
    return np.concatenate([mag, mag | 0x8000], axis=1), A[:, 0].astype(np.uint16)


def _fill(lists, amax, width):
    """Rows of `width`: amax first, then the row's value list cycled."""
    reps = -(-(width - 1) // lists.shape[1])
    body = np.tile(lists, (1, reps))[:, :width - 1]
    return np.concatenate([amax[:, None], body], axis=1)


def test_fp8_weight_block_quant_exhaustive_domain(cuda_lib):
    lists, amax = _value_lists()
    blocks = _fill(lists, amax, 128 * 128)                   # [N_AMAX, 16384]
    side = int(np.ceil(np.sqrt(N_AMAX)))                      # 181 x 181 blocks
    pad = side * side - N_AMAX
    blocks = np.concatenate([blocks, np.tile(blocks[-1:], (pad, 1))])
    W = blocks.reshape(side, side, 128, 128).transpose(0, 2, 1, 3).reshape(side * 128, side * 128)
    W = np.ascontiguousarray(W)
    Wq, Ws = fb.fp8rl_quant_weight_block(torch.from_numpy(W.view(np.int16)).view(torch.bfloat16).cuda())
    want_q, want_s = oracle.fp8_quant_weight_block(W)
    assert np.array_equal(bits_u32(host(Ws)), bits_u32(want_s))
    got = host(Wq)
    bad = np.argwhere(got != want_q)
    assert bad.size == 0, f"{len(bad)} codes differ, first {bad[:4].tolist()}"


def _row_domain():
    lists, amax = _value_lists()
    groups_per_row = -(-lists.shape[1] // 127)               # 41 groups of 128
    return lists, amax, groups_per_row


def test_fp8_act_group_quant_exhaustive_domain(cuda_lib):
    lists, amax, G = _row_domain()
    # group g of row A: amax A first, then values g*127 .. g*127+126 of A's list (cycled)
    idx = (np.arange(G)[:, None] * 127 + np.arange(127)[None, :]) % lists.shape[1]
    body = lists[:, idx]                                       # [N_AMAX, G, 127]
    X = np.concatenate([np.broadcast_to(amax[:, None, None], (N_AMAX, G, 1)), body], axis=2)
    X = np.ascontiguousarray(X.reshape(N_AMAX, G * 128))
    Xq, Xs = fb.fp8rl_quant_act_group(torch.from_numpy(X.view(np.int16)).view(torch.bfloat16).cuda())
    want_q, want_s = oracle.fp8_quant_act_group(X)
    assert np.array_equal(bits_u32(host(Xs)), bits_u32(want_s))
    got = host(Xq)
    bad = np.argwhere(got != want_q)
    assert bad.size == 0, f"{len(bad)} codes differ, first {bad[:4].tolist()}"


def test_int8_row_quant_exhaustive_domain(cuda_lib):
    lists, amax, G = _row_domain()
    A = np.ascontiguousarray(_fill(lists, amax, G * 128))      # [N_AMAX, 5248]
    At = torch.from_numpy(A.view(np.int16)).view(torch.bfloat16).cuda()
    want_q, want_s = oracle.int8_quant_rows(A)
    for fn in (fb.int8rl_quant_weight_channel, fb.int8rl_quant_act_token):
        Q, S = fn(At)
        assert np.array_equal(bits_u32(host(S)), bits_u32(want_s))
        got = host(Q)
        bad = np.argwhere(got != want_q)
        assert bad.size == 0, f"{len(bad)} codes differ, first {bad[:4].tolist()}"
