"""Planted mistakes in copies of the CPU oracle must fail its pins.

Each case copies oracle/oracle.c, changes one step of one quantizer the way a
plausible slip would (multiplying by a reciprocal instead of dividing by the
stored scale, taking the amax over one row of the block, rounding ties away
from zero), compiles the copy with gcc into a temporary directory and checks
that the hand-worked golden examples reject it.  The oracle itself is never
modified; an unchanged copy built the same way must pass.  CPU only."""
import ctypes
import os
import re
import shutil
import subprocess

import numpy as np
import pytest

import golden_pins

ORACLE_C = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "oracle.c")
CFLAGS = ["-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-shared", "-fPIC"]


def _function_span(src: str, name: str):
    """(start, end) of the body of the C function `name` (from its signature to
    the closing brace at column 0)."""
    m = re.search(r"^\w[^\n]*\b" + re.escape(name) + r"\(", src, re.M)
    assert m, name
    end = src.index("\n}\n", m.start()) + 3
    return m.start(), end


def _mutate(src: str, func: str, old: str, new: str, count: int = 1) -> str:
    a, b = _function_span(src, func)
    body = src[a:b]
    assert body.count(old) >= count, f"{old!r} not in {func}"
    return src[:a] + body.replace(old, new, count) + src[b:]


def _build(tmp_path, src: str):
    c = tmp_path / "oracle_copy.c"
    so = tmp_path / "liboracle_copy.so"
    c.write_text(src)
    subprocess.check_call([shutil.which("gcc") or "gcc", *CFLAGS, str(c), "-o", str(so), "-lm"])
    lib = ctypes.CDLL(str(so))
    P, I = ctypes.c_void_p, ctypes.c_int64
    for fn in (lib.oracle_fp8_quant_weight_block, lib.oracle_int8_quant_rows):
        fn.restype = ctypes.c_int
        fn.argtypes = [P, I, I, I, P, P]
    return lib


def _weight_quant(lib):
    def q(W):
        W = np.ascontiguousarray(W, np.uint16)
        N, K = W.shape
        Wq = np.empty((N, K), np.uint8)
        Ws = np.empty((N // 128, K // 128), np.float32)
        assert lib.oracle_fp8_quant_weight_block(W.ctypes.data, N, K, K, Wq.ctypes.data, Ws.ctypes.data) == 0
        return Wq, Ws
    return q


def _int8_quant(lib):
    def q(A):
        A = np.ascontiguousarray(A, np.uint16)
        R, K = A.shape
        Q = np.empty((R, K), np.int8)
        S = np.empty((R,), np.float32)
        assert lib.oracle_int8_quant_rows(A.ctypes.data, R, K, K, Q.ctypes.data, S.ctypes.data) == 0
        return Q, S
    return q


def _source():
    with open(ORACLE_C) as f:
        return f.read()


def test_unchanged_copy_passes_the_golden_pins(tmp_path):
    lib = _build(tmp_path, _source())
    golden_pins.check_weight_block_golden(_weight_quant(lib))
    golden_pins.check_int8_rows_golden(_int8_quant(lib))


WEIGHT_MUTANTS = {
    # codes from w * (1/s) instead of w / s
    "reciprocal_multiply": ("oracle_fp8_quant_weight_block", "oracle_e4m3_encode(x / s)",
                            "oracle_e4m3_encode(x * (1.0f / s))"),
    # the block amax taken over the block's first row only
    "amax_of_first_row": ("oracle_fp8_quant_weight_block", "for (int64_t i = 0; i < QBLK; ++i)",
                          "for (int64_t i = 0; i < 1; ++i)"),
    # the block amax taken over the block's first column only
    "amax_of_first_column": ("oracle_fp8_quant_weight_block", "for (int64_t j = 0; j < QBLK; ++j) {",
                             "for (int64_t j = 0; j < 1; ++j) {"),
}

INT8_MUTANTS = {
    "reciprocal_multiply": ("oracle_int8_quant_rows", "bf16_to_f32(A[r * lda + k]) / s",
                            "bf16_to_f32(A[r * lda + k]) * (1.0f / s)"),
    "ties_away_from_zero": ("oracle_int8_quant_rows", "nearbyintf(v)", "roundf(v)"),
    "truncation": ("oracle_int8_quant_rows", "nearbyintf(v)", "truncf(v)"),
}


@pytest.mark.parametrize("name", sorted(WEIGHT_MUTANTS))
def test_weight_block_mutant_fails_the_golden_pin(tmp_path, name):
    func, old, new = WEIGHT_MUTANTS[name]
    lib = _build(tmp_path, _mutate(_source(), func, old, new))
    with pytest.raises(AssertionError):
        golden_pins.check_weight_block_golden(_weight_quant(lib))


@pytest.mark.parametrize("name", sorted(INT8_MUTANTS))
def test_int8_rows_mutant_fails_the_golden_pin(tmp_path, name):
    func, old, new = INT8_MUTANTS[name]
    lib = _build(tmp_path, _mutate(_source(), func, old, new))
    with pytest.raises(AssertionError):
        golden_pins.check_int8_rows_golden(_int8_quant(lib))


def test_scale_by_reciprocal_constant_fails_a_golden_pin(tmp_path):
    # fl32(amax * fl32(1/448)) and fl32(amax * fl32(1/127)) in place of the
    # divisions: the exact scale 7/64 of the amax-49 block and the bit-by-bit
    # derived 3b993265 of the amax-19/32 row both move
    src = _source().replace("amax / 448.0f", "amax * (1.0f / 448.0f)").replace(
        "amax / 127.0f", "amax * (1.0f / 127.0f)")
    lib = _build(tmp_path, src)
    with pytest.raises(AssertionError):
        golden_pins.check_weight_block_golden(_weight_quant(lib))
    with pytest.raises(AssertionError):
        golden_pins.check_int8_rows_golden(_int8_quant(lib))
