"""Readers and checks of the hand-worked quantizer examples in tests/golden/.

Each check takes the quantizer under test as a callable, so that the same
golden values pin both the oracle (tests/test_oracle_pins.py) and deliberately
broken copies of it (tests/test_oracle_mutants.py)."""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def exact_value(tok: str) -> float:
    """A golden value written as an integer, a fraction p/q or -0 (all exact in bf16)."""
    if tok == "-0":
        return -0.0
    return float(Fraction(tok))


def bf16_bits_exact(a: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns of float32 values that are exact in bf16."""
    t = torch.from_numpy(np.ascontiguousarray(a, np.float32))
    b = t.to(torch.bfloat16)
    assert torch.equal(b.float(), t) and torch.equal(torch.signbit(b), torch.signbit(t)), \
        "golden values must be exact in bf16"
    return b.view(torch.int16).numpy().view(np.uint16)


def read_weight_block_golden(name="e4m3_weight_block_256x256.txt"):
    """-> (W float32 [256,256], {(nb, kb): scale bits}, {(row, col): code})."""
    W = np.zeros((256, 256), np.float32)
    scales, codes = {}, {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            tok = line.split()
            if not tok or tok[0].startswith("#"):
                continue
            if tok[0] == "block":
                scales[(int(tok[1]), int(tok[2]))] = int(tok[4], 16)
            elif tok[0] == "w":
                r, c = int(tok[1]), int(tok[2])
                W[r, c] = exact_value(tok[3])
                codes[(r, c)] = int(tok[4], 16)
    return W, scales, codes


def check_weight_block_golden(quant) -> None:
    """quant(W uint16 [N,K]) -> (Wq uint8 [N,K], Ws float32 [N/128, K/128])."""
    W, scales, codes = read_weight_block_golden()
    Wq, Ws = quant(bf16_bits_exact(W))
    assert Ws.shape == (2, 2)
    for (nb, kb), bits in scales.items():
        got = int(np.asarray(Ws[nb, kb], np.float32).view(np.uint32))
        assert got == bits, f"block ({nb},{kb}) scale {got:08x}, expected {bits:08x}"
    want = np.zeros((256, 256), np.uint8)
    for (r, c), code in codes.items():
        want[r, c] = code
    bad = np.argwhere(Wq != want)
    assert bad.size == 0, (f"{len(bad)} codes differ; first at {bad[0].tolist()}: "
                           f"{Wq[tuple(bad[0])]:02x}, expected {want[tuple(bad[0])]:02x}")


def read_int8_rows_golden(name="int8_rows_4x128.txt"):
    """-> (A float32 [R,128], [scale bits per row], int8 codes [3,128])."""
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            tok = line.split()
            if not tok or tok[0].startswith("#"):
                continue
            rows.setdefault(int(tok[1]), {})[tok[2]] = tok[3:]
    R = len(rows)
    A = np.zeros((R, 128), np.float32)
    Q = np.zeros((R, 128), np.int8)
    S = []
    for r in range(R):
        for j, t in enumerate(rows[r]["values"]):
            A[r, j] = exact_value(t)
        for j, t in enumerate(rows[r]["codes"]):
            Q[r, j] = int(t)
        S.append(int(rows[r]["scale"][0], 16))
    return A, S, Q


def check_int8_rows_golden(quant) -> None:
    """quant(A uint16 [R,K]) -> (Q int8 [R,K], S float32 [R])."""
    A, S_bits, Q_want = read_int8_rows_golden()
    Q, S = quant(bf16_bits_exact(A))
    for r, bits in enumerate(S_bits):
        got = int(np.asarray(S[r], np.float32).view(np.uint32))
        assert got == bits, f"row {r} scale {got:08x}, expected {bits:08x}"
    bad = np.argwhere(Q != Q_want)
    assert bad.size == 0, (f"{len(bad)} codes differ; first at {bad[0].tolist()}: "
                           f"{int(Q[tuple(bad[0])])}, expected {int(Q_want[tuple(bad[0])])}")
