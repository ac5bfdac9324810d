"""Pins for the CPU oracle: each check ties the oracle to something other than
itself (the E4M3FN format definition by brute force, a hand-worked example,
library routines, closed forms and derived error bounds), chosen so that a
dropped term, a wrong sign or index or a transposed operand fails one of them.

These run on the CPU (no GPU marker)."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import golden_pins
import oracle
from precision_rl_rollout_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ E4M3FN format

def _finite_e4m3_table():
    """(codes, values) of every finite E4M3FN code, read through torch's
    float8_e4m3fn dtype (a library decoder, independent of the oracle)."""
    codes = torch.arange(256, dtype=torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    keep = ~np.isnan(vals)
    return codes.numpy()[keep], vals[keep]


def test_e4m3_decode_matches_library_and_format_facts():
    dec = oracle.e4m3_decode_table()
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    both_nan = np.isnan(dec) & np.isnan(lib)
    assert np.array_equal(np.isnan(dec), np.isnan(lib))
    assert np.all((dec == lib) | both_nan)
    # format facts of OCP E4M3FN
    assert np.isnan(dec[0x7F]) and np.isnan(dec[0xFF]) and np.sum(np.isnan(dec)) == 2
    assert dec[0x7E] == 448.0 and dec[0xFE] == -448.0
    assert dec[0x01] == 2.0 ** -9 and dec[0x08] == 2.0 ** -6 and dec[0x38] == 1.0
    pos = dec[:0x7F]
    assert np.all(np.diff(pos) > 0), "positive codes must be strictly increasing"
    assert np.array_equal(dec[0x80:0xFF], -pos) or np.all(dec[0x80:0xFF] == -pos)


def _bruteforce_e4m3(v: np.ndarray) -> np.ndarray:
    """Nearest finite E4M3FN value by exhaustive search; ties to the even
    mantissa; values beyond 448 land on 448 because nothing finite lies
    above it; the sign bit follows the input (so -0 -> 0x80)."""
    codes, vals = _finite_e4m3_table()
    pos = vals >= 0
    pc, pv = codes[pos & (codes < 0x80)], vals[pos & (codes < 0x80)]
    a = np.abs(v.astype(np.float64))
    d = np.abs(a[:, None] - pv[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    # among tied candidates keep the one with an even mantissa bit
    even = (pc & 1) == 0
    pick_even = cand & even[None, :]
    has_even = pick_even.any(axis=1)
    idx = np.where(has_even, pick_even.argmax(axis=1), cand.argmax(axis=1))
    # float64 distances are exact except for huge inputs: search those with exact rationals
    for i in np.nonzero(a > 2.0 ** 20)[0]:
        fa = Fraction(float(a[i]))
        dist = [abs(fa - Fraction(float(x))) for x in pv]
        dmin = min(dist)
        ties = [j for j, dj in enumerate(dist) if dj == dmin]
        evens = [j for j in ties if pc[j] % 2 == 0]
        idx[i] = (evens or ties)[0]
    out = pc[idx].astype(np.uint8)
    neg = np.signbit(v)
    out[neg] |= 0x80
    return out


def _sweep_inputs() -> np.ndarray:
    codes, vals = _finite_e4m3_table()
    pv = np.unique(vals[vals >= 0]).astype(np.float32)
    mids = ((pv[:-1].astype(np.float64) + pv[1:]) / 2).astype(np.float32)
    assert np.all(mids.astype(np.float64) == (pv[:-1].astype(np.float64) + pv[1:]) / 2)
    up = np.nextafter(mids, np.float32(np.inf))
    dn = np.nextafter(mids, np.float32(-np.inf))
    specials = np.array([0.0, 448.0, 448.0001, 449.0, 460.0, 463.99997, 464.0, 464.00003, 479.0,
                         480.0, 500.0, 1e6, 3e38, 2.0 ** -10, 2.0 ** -11, 1e-30, 1e-45,
                         np.nextafter(np.float32(2.0 ** -10), np.float32(1))], np.float32)
    rng = np.random.default_rng(20250101)
    r1 = rng.uniform(-470, 470, 20000).astype(np.float32)
    r2 = (rng.choice([-1, 1], 20000) * 2.0 ** rng.uniform(-14, 9, 20000)).astype(np.float32)
    base = np.concatenate([pv, mids, up, dn, specials, r1, r2]).astype(np.float32)
    return np.concatenate([base, -base, np.array([-0.0], np.float32)])


def test_e4m3_encoder_bruteforce():
    v = _sweep_inputs()
    got = oracle.e4m3_encode(v)
    want = _bruteforce_e4m3(v)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} mismatches, e.g. v={v[bad[:5]]} got={got[bad[:5]]} want={want[bad[:5]]}"


def test_e4m3_encoder_matches_library_cast_inside_range():
    # torch's fp32 -> float8_e4m3fn cast rounds to nearest even; it does not
    # saturate, so compare only on |v| <= 448.
    v = _sweep_inputs()
    v = v[np.abs(v) <= 448]
    lib = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(v)
    assert np.array_equal(got, lib)


def test_e4m3_encoder_never_emits_nan_codes():
    v = _sweep_inputs()
    got = oracle.e4m3_encode(v)
    assert not np.any((got == 0x7F) | (got == 0xFF))
    assert np.all(got[np.abs(v) >= 448] & 0x7F == 0x7E)


# ------------------------------------------------------------------ bf16 rounding

def test_f32_to_bf16_matches_library():
    rng = np.random.default_rng(7)
    v = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 1e3,
                        (rng.standard_normal(2000) * 1e-38).astype(np.float32),
                        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 0.0, -0.0,
                                  3.3895e38, 65504.0, 2 ** 24 + 1], np.float32)])
    got = oracle.f32_to_bf16_rn(v)
    lib = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, lib)


# ------------------------------------------------------------------ hand-worked example

def _parse_golden(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            _, r, kind, *rest = line.split()
            rows.setdefault(int(r), {})[kind] = rest
    return rows


def _golden_value(tok: str) -> float:
    if tok == "-0":
        return -0.0
    if "^" in tok:
        mul = 1.0
        if "*" in tok:
            a, tok = tok.split("*")
            mul = float(a)
        base, exp = tok.split("^")
        return mul * float(base) ** int(exp)
    return float(tok)


def test_act_quant_hand_worked_example():
    rows = _parse_golden("e4m3_act_group_2x128.txt")
    M, K = len(rows), 128
    X = np.zeros((M, K), np.float32)
    for r, d in rows.items():
        for j, tok in enumerate(d["values"]):
            X[r, j] = _golden_value(tok)
    Xb = torch.from_numpy(X).to(torch.bfloat16)
    assert torch.equal(Xb.float(), torch.from_numpy(X)), "example values must be exact in bf16"
    Xq, Xs = oracle.fp8_quant_act_group(synth.bf16_bits(Xb))
    for r, d in rows.items():
        want_codes = np.zeros(K, np.uint8)
        for j, tok in enumerate(d["codes"]):
            want_codes[j] = int(tok, 16)
        assert np.array_equal(Xq[r], want_codes), f"row {r}: {Xq[r][:12]}"
        want_scale = np.array([int(d["scale"][0], 16)], np.uint32).view(np.float32)[0]
        assert Xs[0, r].view(np.uint32) == want_scale.view(np.uint32), f"row {r} scale"


def test_weight_block_quant_hand_worked_example():
    # 2 x 2 blocks: an inexact scale (amax 4: 3c124925) with a tie at -336, an exact
    # non-power-of-two scale (amax 49: 7/64) whose quotients all land on E4M3
    # midpoints, a block of zeros and negative zeros, and a fourth block whose
    # scale (1/896) shares the first one's mantissa; each amax away from row 0 and
    # column 0 of its block (tests/golden/e4m3_weight_block_256x256.txt)
    golden_pins.check_weight_block_golden(oracle.fp8_quant_weight_block)


def test_int8_row_quant_hand_worked_example():
    # an inexact scale with amax 19/32 (3b993265, derived bit by bit) whose x/s
    # lands exactly on 63.5, an exact scale (1/32) with ties at 64.5, 80.5, 66.5,
    # 0.5, 1.5, 2.5 (to even), a zero row, and amax 9/32 (3b112245) whose x = amax/2
    # falls just below 63.5 (tests/golden/int8_rows_4x128.txt)
    golden_pins.check_int8_rows_golden(oracle.int8_quant_rows)


# ------------------------------------------------------------------ quantizer invariants

def _ulp_e4m3(v):
    a = np.abs(v)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    return 2.0 ** (e - 3)


def _weight_with_block_magnitudes(N, K, seed):
    g = torch.Generator().manual_seed(seed)
    W = torch.randn(N, K, generator=g) * 0.02
    mag = 10.0 ** (torch.rand(N // 128, K // 128, generator=g) * 6 - 3)
    W = W * mag.repeat_interleave(128, 0).repeat_interleave(128, 1)
    return W.to(torch.bfloat16)


@pytest.mark.parametrize("seed", [1, 2])
def test_weight_block_quant_invariants(seed):
    N, K = 384, 640
    Wb = _weight_with_block_magnitudes(N, K, seed)
    Wq, Ws = oracle.fp8_quant_weight_block(synth.bf16_bits(Wb))
    W = Wb.float().numpy().astype(np.float64)
    dq = oracle.e4m3_decode_table()[Wq]
    assert Ws.shape == (N // 128, K // 128)
    assert not np.any((Wq == 0x7F) | (Wq == 0xFF))
    for nb in range(N // 128):
        for kb in range(K // 128):
            blk = W[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            qb = dq[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            s = float(Ws[nb, kb])
            amax = np.abs(blk).max()
            # the scale stored at [nb, kb] belongs to block (nb, kb): s * 448 == amax within 1 ulp
            assert abs(s * 448.0 - amax) <= amax * 2.0 ** -23
            # the block's largest magnitude encodes to exactly 448
            assert np.abs(qb).max() == 448.0
            # round-trip within half an E4M3 ulp (of the larger of input and result) plus fp32 division rounding
            v = blk / s
            err = np.abs(v - qb)
            bound = 0.5 * _ulp_e4m3(np.maximum(np.abs(v), np.abs(qb))) + np.abs(v) * 2.0 ** -23
            assert np.all(err <= bound)


def test_weight_block_quant_edge_cases():
    N, K = 384, 384
    Wb = synth.edge_case_weight(N, K, seed=5)
    Wq, Ws = oracle.fp8_quant_weight_block(synth.bf16_bits(Wb))
    B = 128
    assert Ws[0, 0] == 1.0 and np.all(Wq[:B, :B] == 0x00)          # all zero
    assert Ws[0, 1] == 1.0 and np.all(Wq[:B, B:2 * B] == 0x80)     # all -0.0 keeps the sign
    blk = Wq[:B, 2 * B:3 * B]
    assert blk[37, 91] == 0xFE and np.sum(blk != 0) == 1            # lone -3 -> -448
    assert Ws[0, 2] == np.float32(3.0) / np.float32(448.0)
    assert np.all(Wq[B:2 * B, 2 * B:3 * B] == 0x7E)                 # all equal -> 448
    dq = oracle.e4m3_decode_table()[Wq]
    for nb, kb in [(1, 0), (1, 1), (2, 0), (2, 1)]:                   # huge, subnormal, ties, signs
        assert np.abs(dq[nb * B:(nb + 1) * B, kb * B:(kb + 1) * B]).max() == 448.0
    assert not np.any((Wq == 0x7F) | (Wq == 0xFF))


def _bruteforce_int8(v32: np.ndarray) -> np.ndarray:
    """Nearest integer in [-127, 127] by exhaustive search, ties to even."""
    cand = np.arange(-127, 128, dtype=np.float64)
    d = np.abs(v32.astype(np.float64)[:, None] - cand[None, :])
    best = d.min(axis=1, keepdims=True)
    tie = (d == best)
    even = (np.arange(-127, 128) % 2 == 0)
    pick = np.where((tie & even).any(axis=1), (tie & even).argmax(axis=1), tie.argmax(axis=1))
    return (pick - 127).astype(np.int8)


def test_int8_row_quant_bruteforce_and_invariants():
    R, K = 40, 384
    Ab = synth.edge_case_activation(R, K, seed=11)
    Q, S = oracle.int8_quant_rows(synth.bf16_bits(Ab))
    A = Ab.float().numpy()
    for r in range(R):
        amax = np.float32(np.abs(A[r]).max())
        s = np.float32(1.0) if amax == 0 else amax / np.float32(127.0)
        assert S[r].view(np.uint32) == np.float32(s).view(np.uint32)
        v = (A[r].astype(np.float32) / s).astype(np.float32)
        assert np.array_equal(Q[r], _bruteforce_int8(v)), f"row {r}"
        if amax > 0:
            assert np.abs(Q[r].astype(int)).max() == 127
    assert np.all(Q >= -127)


# ------------------------------------------------------------------ INT8 GEMM

def test_int8_gemm_exact_against_library_matmul():
    rng = np.random.default_rng(3)
    M, N, K = 7, 256, 384
    Xq = rng.integers(-127, 128, (M, K)).astype(np.int8)
    Wq = rng.integers(-127, 128, (N, K)).astype(np.int8)
    Xq[0] = 127
    Wq[0] = 127
    Wq[1] = -127
    Xs = np.ones(M, np.float32)
    Ws = np.ones(N, np.float32)
    acc, _ = oracle.int8_gemm(Xq, Xs, Wq, Ws)
    ref = Xq.astype(np.int64) @ Wq.astype(np.int64).T
    assert np.array_equal(acc.astype(np.int64), ref)
    assert acc[0, 0] == 127 * 127 * K and acc[0, 1] == -127 * 127 * K


def test_int8_gemm_epilogue_power_of_two_scales():
    rng = np.random.default_rng(4)
    M, N, K = 6, 128, 256
    Xq = rng.integers(-127, 128, (M, K)).astype(np.int8)
    Wq = rng.integers(-127, 128, (N, K)).astype(np.int8)
    ex = rng.integers(-6, 6, M)
    ew = rng.integers(-6, 6, N)
    Xs = (2.0 ** ex).astype(np.float32)
    Ws = (2.0 ** ew).astype(np.float32)
    acc, Y = oracle.int8_gemm(Xq, Xs, Wq, Ws)
    exact = acc.astype(np.float64) * 2.0 ** (ex[:, None] + ew[None, :])   # exact; |acc| < 2^24
    lib = torch.from_numpy(exact).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(Y, lib)
    # row/column placement: the row scale follows the token, the column scale the channel
    Xs2 = Xs.copy()
    Xs2[2] *= 2
    _, Y2 = oracle.int8_gemm(Xq, Xs2, Wq, Ws)
    f = oracle.bf16_to_f32
    assert np.array_equal(f(Y2[2]), 2 * f(Y[2])) and np.array_equal(Y2[[0, 1, 3, 4, 5]], Y[[0, 1, 3, 4, 5]])


def test_int8_gemm_reports_int32_overflow():
    K = 140000  # 127^2 * K > 2^31
    Xq = np.full((1, K), 127, np.int8)
    Wq = np.full((1, K), 127, np.int8)
    with pytest.raises(ValueError):
        oracle.int8_gemm(Xq, np.ones(1, np.float32), Wq, np.ones(1, np.float32))


# ------------------------------------------------------------------ FP8 GEMM

def _int_codes(shape, rng):
    ints = rng.integers(-16, 17, shape)
    codes = torch.from_numpy(ints.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return ints, codes


def test_fp8_gemm_integer_special_case_is_exact():
    rng = np.random.default_rng(5)
    M, N, K = 5, 256, 384
    xi, Xq = _int_codes((M, K), rng)
    wi, Wq = _int_codes((N, K), rng)
    Y = oracle.fp8_gemm(Xq, np.ones((K // 128, M), np.float32), Wq, np.ones((N // 128, K // 128), np.float32))
    assert np.array_equal(Y, (xi @ wi.T).astype(np.float64))


def test_fp8_gemm_scale_placement_power_of_two():
    rng = np.random.default_rng(6)
    M, N, K = 3, 384, 512
    xi, Xq = _int_codes((M, K), rng)
    wi, Wq = _int_codes((N, K), rng)
    ex = rng.integers(-4, 5, (K // 128, M))
    ew = rng.integers(-4, 5, (N // 128, K // 128))
    Y = oracle.fp8_gemm(Xq, (2.0 ** ex).astype(np.float32), Wq, (2.0 ** ew).astype(np.float32))
    # expand every scale to element granularity and use the library matmul
    xs_full = np.repeat(2.0 ** ex.T, 128, axis=1)                       # [M, K]
    ws_full = np.repeat(np.repeat(2.0 ** ew, 128, axis=0), 128, axis=1)  # [N, K]
    ref = (xi * xs_full) @ (wi * ws_full).T
    assert np.array_equal(Y, ref)


def test_fp8_gemm_single_term_closed_form():
    M, N, K = 1, 256, 256
    Xq = np.zeros((M, K), np.uint8)
    Wq = np.zeros((N, K), np.uint8)
    Xq[0, 200] = 0x3C                      # 1.5
    Wq[130, 200] = 0xFA                    # -320
    Xs = np.array([[0.25], [3.0]], np.float32)
    Ws = np.array([[1.0, 1.0], [1.0, 0.5]], np.float32)
    Y = oracle.fp8_gemm(Xq, Xs, Wq, Ws)
    want = np.zeros((M, N))
    want[0, 130] = 1.5 * 3.0 * -320 * 0.5
    assert np.array_equal(Y, want)


def test_fp8_gemm_within_quantization_bound_of_unquantized_matmul():
    # Quantize bf16 operands with blocks of very different magnitude, then bound
    # |y_q - y_true| by the E4M3 half-ulp error of each operand: a transposed
    # scale index or operand would leave this bound by orders of magnitude.
    M, N, K = 9, 384, 640
    Wb = _weight_with_block_magnitudes(N, K, 21)
    g = torch.Generator().manual_seed(22)
    Xf = torch.randn(M, K, generator=g) * (10.0 ** (torch.rand(M, K // 128, generator=g) * 4 - 2)).repeat_interleave(128, 1)
    Xb = Xf.to(torch.bfloat16)
    Wq, Ws = oracle.fp8_quant_weight_block(synth.bf16_bits(Wb))
    Xq, Xs = oracle.fp8_quant_act_group(synth.bf16_bits(Xb))
    Y = oracle.fp8_gemm(Xq, Xs, Wq, Ws)
    X = Xb.double().numpy()
    W = Wb.double().numpy()
    Ytrue = X @ W.T                                                    # library fp64 matmul
    sx = np.repeat(Xs.T.astype(np.float64), 128, axis=1)
    sw = np.repeat(np.repeat(Ws.astype(np.float64), 128, 0), 128, 1)
    ex = 2.0 ** -4 * np.abs(X) + 2.0 ** -10 * sx                      # per-element E4M3 error bound
    ew = 2.0 ** -4 * np.abs(W) + 2.0 ** -10 * sw
    bound = np.abs(X) @ ew.T + ex @ (np.abs(W) + ew).T
    assert np.all(np.abs(Y - Ytrue) <= bound * (1 + 1e-9) + 1e-300)
    # and the bound is not vacuous: the error is well below the signal
    assert np.abs(Y - Ytrue).max() < 0.2 * np.abs(Ytrue).max()


def _e4m3_code(v: float) -> int:
    return int(torch.tensor([v]).to(torch.float8_e4m3fn).view(torch.uint8)[0])


def test_fp8_gemm_grouped_routes_each_token_to_its_expert():
    # Expert e's weights are all the E4M3 value (e+1) with scale 2^-kb on K block
    # kb; activations are small integers with unit scales.  So for a token t of
    # expert e, y[t, n] = (e+1) * sum_kb 2^-kb * sum_{k in kb} x[t, k] for every n:
    # a token sent to the wrong expert, a wrong expert's scale row or a shifted
    # token range changes the multiplier.
    E, N, K = 4, 256, 384
    KB = K // 128
    rng = np.random.default_rng(5)
    offsets = np.array([0, 3, 3, 8, 9])                     # expert 1 has no tokens
    T = offsets[-1]
    xv = rng.integers(-3, 4, size=(T, K)).astype(np.float64)
    Xq = np.array([[_e4m3_code(v) for v in row] for row in xv], np.uint8)
    Xs = np.ones((KB, T), np.float32)
    Wq = np.stack([np.full((N, K), _e4m3_code(e + 1.0), np.uint8) for e in range(E)])
    Ws = np.stack([np.tile((2.0 ** -np.arange(KB)).astype(np.float32), (N // 128, 1)) for _ in range(E)])
    Y = oracle.fp8_gemm_grouped(Xq, Xs, Wq, Ws, offsets)
    blk = (xv.reshape(T, KB, 128).sum(axis=2) * 2.0 ** -np.arange(KB)).sum(axis=1)
    expert_of = np.repeat(np.arange(E), np.diff(offsets))
    want = ((expert_of + 1) * blk)[:, None] * np.ones((1, N))
    assert np.array_equal(Y, want)


def test_fp8_gemm_grouped_all_tokens_in_one_expert_is_the_dense_gemm_of_that_expert():
    # closed form again: one expert holds every token; the others (empty) must not
    # contribute, and the result is the single-term dequantized product
    E, N, K, T = 3, 128, 256, 5
    Xq = np.full((T, K), _e4m3_code(2.0), np.uint8)
    Xs = np.full((K // 128, T), 0.5, np.float32)
    Wq = np.stack([np.full((N, K), _e4m3_code(v), np.uint8) for v in (1.0, 3.0, 5.0)])
    Ws = np.full((E, N // 128, K // 128), 0.25, np.float32)
    Y = oracle.fp8_gemm_grouped(Xq, Xs, Wq, Ws, [0, 0, T, T])
    assert np.array_equal(Y, np.full((T, N), K * (2.0 * 0.5) * (3.0 * 0.25)))


def test_bf16_matmul_f64_matches_library():
    g = torch.Generator().manual_seed(9)
    X = torch.randn(4, 256, generator=g).to(torch.bfloat16)
    W = torch.randn(128, 256, generator=g).to(torch.bfloat16)
    Y = oracle.bf16_matmul_f64(synth.bf16_bits(X), synth.bf16_bits(W))
    assert np.allclose(Y, X.double().numpy() @ W.double().numpy().T, rtol=1e-12, atol=1e-12)


def test_tiny_config_inputs_have_requested_structure():
    X = synth.activation(synth.TINY_M, synth.TINY.K, synth.seed_for(1, 1), n_outliers=2)
    amax_per_ch = X.float().abs().amax(0)
    assert int((amax_per_ch > 10).sum()) == 2
    W = synth.weight(synth.TINY.N, synth.TINY.K, synth.seed_for(1, 0))
    assert abs(float(W.float().std()) - 0.02) < 0.002


# ------------------------------------------------------------------ KV-cache per-tensor quant

def test_per_tensor_quant_reduces_to_single_block_quant():
    # a 128x128 tensor is one weight block: the per-tensor quantizer must agree
    # with the (pinned) block quantizer on codes and scale
    Wb = _weight_with_block_magnitudes(128, 128, 31)
    q1, s1 = oracle.fp8_quant_tensor(synth.bf16_bits(Wb))
    q2, s2 = oracle.fp8_quant_weight_block(synth.bf16_bits(Wb))
    assert np.array_equal(q1, q2) and s1.view(np.uint32) == s2[0, 0].view(np.uint32)


def test_per_tensor_quant_uses_the_global_amax():
    g = torch.Generator().manual_seed(41)
    X = torch.randn(300, 1024, generator=g) * 0.1
    X[217, 901] = -7.5                                   # the tensor's amax, far from row/column 0
    Xb = X.to(torch.bfloat16)
    q, s = oracle.fp8_quant_tensor(synth.bf16_bits(Xb))
    assert s.view(np.uint32) == (np.float32(7.5) / np.float32(448)).view(np.uint32)
    assert q[217, 901] == 0xFE and np.sum((q & 0x7F) == 0x7E) == 1
    dq = oracle.e4m3_decode_table()[q]
    v = Xb.double().numpy() / float(s)
    bound = 0.5 * _ulp_e4m3(np.maximum(np.abs(v), np.abs(dq))) + np.abs(v) * 2.0 ** -23
    assert np.all(np.abs(v - dq) <= bound)
    # with that scale given explicitly, the with-scale quantizer gives the same codes
    assert np.array_equal(oracle.fp8_quant_with_scale(synth.bf16_bits(Xb), float(s)), q)


def test_per_tensor_quant_zero_tensor():
    q, s = oracle.fp8_quant_tensor(np.zeros((3, 16), np.uint16))
    assert s == 1.0 and not q.any()


# ------------------------------------------------------------------ TIS / MIS rollout correction

def test_rollout_is_closed_forms():
    lt = np.array([-1.0, -2.0, -0.5, -3.0, -1.0, -7.0], np.float32)
    lr = np.array([-1.0, -2.0 - np.log(2.0), -0.5 + np.log(4.0), -1.0, -1.0, -7.0], np.float32)
    mask = np.array([1, 1, 1, 1, 0, 1], np.uint8)
    log_clip = np.float32(np.log(3.0))
    d = lt - lr                                           # 0, ln2, -ln4, -2, (masked), 0
    w, st = oracle.rollout_is(lt, lr, mask, log_clip, 0)
    assert w[0] == 1.0 and abs(w[1] - 2.0) < 1e-6 and abs(w[2] - 0.25) < 1e-6
    assert abs(w[3] - np.exp(-2.0)) < 1e-7 and w[4] == 0.0 and w[5] == 1.0
    assert st[0] == 5 and st[1] == 0
    assert abs(st[3] - float(np.sum(d[mask == 1].astype(np.float64)))) < 1e-12
    # a ratio above the threshold: TIS truncates it to C, MIS drops it
    lt2 = np.array([0.0, -0.1], np.float32)
    lr2 = np.array([-2.0, -0.1], np.float32)              # ratio e^2 > 3, and 1
    w2, st2 = oracle.rollout_is(lt2, lr2, np.ones(2, np.uint8), log_clip, 0)
    assert abs(w2[0] - 3.0) < 1e-6 and w2[1] == 1.0 and st2[1] == 1 and abs(st2[2] - 4.0) < 1e-6
    w3, st3 = oracle.rollout_is(lt2, lr2, np.ones(2, np.uint8), log_clip, 1)
    assert w3[0] == 0.0 and w3[1] == 1.0 and st3[1] == 1 and st3[2] == 1.0


def test_rollout_is_matches_library_exp_and_counts():
    rng = np.random.default_rng(12)
    lt = rng.normal(-2.0, 1.0, 5000).astype(np.float32)
    lr = (lt + rng.normal(0.0, 0.3, 5000)).astype(np.float32)
    mask = (rng.random(5000) < 0.9).astype(np.uint8)
    log_clip = np.float32(np.log(2.0))
    d = (lt - lr).astype(np.float32)
    for mode in (0, 1):
        w, st = oracle.rollout_is(lt, lr, mask, log_clip, mode)
        clipped = (d > log_clip) & (mask == 1)
        keep = np.exp(d.astype(np.float64))
        want = np.where(mask == 0, 0.0, np.where(clipped, np.exp(float(log_clip)) if mode == 0 else 0.0, keep))
        assert np.allclose(w, want, rtol=1e-12, atol=0)
        assert st[0] == mask.sum() and st[1] == clipped.sum()


# ------------------------------------------------------------------ mismatch KL

def _bf16(v):
    return oracle.f32_to_bf16_rn(np.asarray(v, np.float32))


def test_logits_kl_two_symbol_closed_form():
    # V = 2: the softmax is a Bernoulli with p = sigmoid(a0 - a1), so the KL is
    # p log(p/q) + (1-p) log((1-p)/(1-q)); the inputs are exact in bf16
    a = np.array([[1.5, -0.25], [0.0, 0.0], [3.0, 1.0]], np.float32)
    b = np.array([[0.5, 0.5], [2.0, -1.0], [-1.0, 4.0]], np.float32)
    kl = oracle.logits_kl(_bf16(a), _bf16(b))
    for m in range(3):
        p = 1.0 / (1.0 + math.exp(-(float(a[m, 0]) - float(a[m, 1]))))
        q = 1.0 / (1.0 + math.exp(-(float(b[m, 0]) - float(b[m, 1]))))
        want = p * math.log(p / q) + (1 - p) * math.log((1 - p) / (1 - q))
        assert abs(kl[m] - want) <= 1e-14 * max(1.0, abs(want))


def test_logits_kl_uniform_against_one_raised_logit_closed_form():
    # p uniform over V; q puts logit c on symbol 0 and 0 elsewhere:
    # KL = -log V - (1/V) [log q0 + (V-1) log q1], q0 = e^c / Z, q1 = 1 / Z, Z = e^c + V - 1
    V, c = 1000, 2.5
    a = np.zeros((1, V), np.float32)
    b = np.zeros((1, V), np.float32)
    b[0, 0] = c
    Z = math.exp(c) + V - 1
    want = -math.log(V) - (math.log(math.exp(c) / Z) + (V - 1) * math.log(1 / Z)) / V
    kl = oracle.logits_kl(_bf16(a), _bf16(b))
    assert abs(kl[0] - want) <= 1e-12


def test_logits_kl_zero_for_equal_rows_positive_otherwise_and_shift_invariant():
    rng = np.random.default_rng(3)
    a = _bf16(rng.normal(0, 2, size=(4, 513)))
    assert np.all(np.abs(oracle.logits_kl(a, a)) <= 1e-14)
    b = _bf16(oracle.bf16_to_f32(a) + rng.normal(0, 0.05, size=a.shape).astype(np.float32))
    kl = oracle.logits_kl(a, b)
    assert np.all(kl > 0)
    # a shift by a power of two keeps small integers exact in bf16, and the
    # softmax does not see a constant added to every logit of a row
    ai = _bf16(rng.integers(-8, 9, size=(3, 257)).astype(np.float32))
    bi = _bf16(rng.integers(-8, 9, size=(3, 257)).astype(np.float32))
    shifted = _bf16(oracle.bf16_to_f32(bi) + np.float32(16.0))
    assert np.allclose(oracle.logits_kl(ai, bi), oracle.logits_kl(ai, shifted), rtol=1e-12, atol=1e-14)
