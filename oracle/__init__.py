"""CPU oracle for the 8-bit rollout linear layer (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The product library never does:
it must fail loudly when its CUDA extension is missing, never fall back here.

The arithmetic lives in ``oracle.c`` (plain C, IEEE fp32 quantizers, fp64
dequant-matmul, int64 INT8 GEMM).  This module only compiles it with gcc and
marshals numpy arrays.  bf16 tensors travel as ``uint16`` bit patterns.

Functions whose result is pinned by ``tests/test_oracle_pins.py``:
``e4m3_encode``/``e4m3_decode`` (brute force over all 256 codes),
``fp8_quant_act_group`` (hand-worked example: two worked rows and a zero row), the quantizers (round-trip
and saturation invariants), ``int8_gemm`` (int64 library matmul) and
``fp8_gemm`` (exact integer special case, quantization error bound).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_CFLAGS = ["-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-shared", "-fPIC"]
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, a second or two)."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I = ctypes.c_int64
            lib.oracle_e4m3_decode.restype = ctypes.c_double
            lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            lib.oracle_e4m3_encode_array.argtypes = [P, I, P]
            lib.oracle_f32_to_bf16_rn.restype = ctypes.c_uint16
            lib.oracle_f32_to_bf16_rn.argtypes = [ctypes.c_float]
            lib.oracle_bf16_to_f32.restype = ctypes.c_float
            lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
            for name, nargs in [("oracle_fp8_quant_weight_block", 6),
                                ("oracle_fp8_quant_act_group", 6),
                                ("oracle_int8_quant_rows", 6),
                                ("oracle_fp8_gemm", 8),
                                ("oracle_bf16_matmul_f64", 8),
                                ("oracle_int8_gemm", 9)]:
                fn = getattr(lib, name)
                fn.restype = ctypes.c_int
            lib.oracle_fp8_quant_weight_block.argtypes = [P, I, I, I, P, P]
            lib.oracle_fp8_quant_act_group.argtypes = [P, I, I, I, P, P]
            lib.oracle_int8_quant_rows.argtypes = [P, I, I, I, P, P]
            lib.oracle_fp8_gemm.argtypes = [P, P, P, P, I, I, I, P]
            lib.oracle_bf16_matmul_f64.argtypes = [P, I, P, I, I, I, I, P]
            lib.oracle_int8_gemm.argtypes = [P, P, P, P, I, I, I, P, P]
            lib.oracle_fp8_quant_tensor.restype = ctypes.c_int
            lib.oracle_fp8_quant_tensor.argtypes = [P, I, I, I, P, P]
            lib.oracle_fp8_quant_with_scale.restype = ctypes.c_int
            lib.oracle_fp8_quant_with_scale.argtypes = [P, I, I, I, ctypes.c_float, P]
            lib.oracle_logits_kl.restype = ctypes.c_int
            lib.oracle_logits_kl.argtypes = [P, I, P, I, I, I, P]
            lib.oracle_rollout_is.restype = ctypes.c_int
            lib.oracle_rollout_is.argtypes = [P, P, P, I, ctypes.c_float, ctypes.c_int, P, P]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _bits16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, "bf16 operands are passed as uint16 bit patterns"
    return a


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what}: rc={rc}")


# ---------------------------------------------------------------- formats

def e4m3_decode(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.oracle_e4m3_decode(int(x)) for x in c.ravel()],
                    dtype=np.float64).reshape(c.shape)


def e4m3_decode_table() -> np.ndarray:
    return e4m3_decode(np.arange(256, dtype=np.uint8))


def e4m3_encode(v) -> np.ndarray:
    lib = _load()
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float32))
    out = np.empty(v.shape, dtype=np.uint8)
    lib.oracle_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def f32_to_bf16_rn(v) -> np.ndarray:
    lib = _load()
    v = np.asarray(v, dtype=np.float32)
    return np.array([lib.oracle_f32_to_bf16_rn(float(x)) for x in v.ravel()],
                    dtype=np.uint16).reshape(v.shape)


def bf16_to_f32(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- quantizers

def fp8_quant_weight_block(W: np.ndarray):
    """W uint16 [N,K] -> (Wq uint8 [N,K], Ws float32 [N/128, K/128])."""
    W = _bits16(W)
    N, K = W.shape
    Wq = np.empty((N, K), np.uint8)
    Ws = np.empty((N // 128, K // 128), np.float32)
    _check(_load().oracle_fp8_quant_weight_block(_ptr(W), N, K, K, _ptr(Wq), _ptr(Ws)),
           "fp8_quant_weight_block")
    return Wq, Ws


def fp8_quant_act_group(X: np.ndarray):
    """X uint16 [M,K] -> (Xq uint8 [M,K], Xs float32 [K/128, M])."""
    X = _bits16(X)
    M, K = X.shape
    Xq = np.empty((M, K), np.uint8)
    Xs = np.empty((K // 128, M), np.float32)
    _check(_load().oracle_fp8_quant_act_group(_ptr(X), M, K, K, _ptr(Xq), _ptr(Xs)),
           "fp8_quant_act_group")
    return Xq, Xs


def int8_quant_rows(A: np.ndarray):
    """A uint16 [R,K] -> (Q int8 [R,K], S float32 [R]); per-row symmetric."""
    A = _bits16(A)
    R, K = A.shape
    Q = np.empty((R, K), np.int8)
    S = np.empty((R,), np.float32)
    _check(_load().oracle_int8_quant_rows(_ptr(A), R, K, K, _ptr(Q), _ptr(S)),
           "int8_quant_rows")
    return Q, S


def fp8_quant_tensor(X: np.ndarray):
    """X uint16 [R,C] -> (Xq uint8 [R,C], scale float32): one scale for the tensor."""
    X = _bits16(X)
    R, C = X.shape
    Xq = np.empty((R, C), np.uint8)
    sc = np.empty((1,), np.float32)
    _check(_load().oracle_fp8_quant_tensor(_ptr(X), R, C, C, _ptr(Xq), _ptr(sc)), "fp8_quant_tensor")
    return Xq, sc[0]


def fp8_quant_with_scale(X: np.ndarray, scale: float):
    X = _bits16(X)
    R, C = X.shape
    Xq = np.empty((R, C), np.uint8)
    _check(_load().oracle_fp8_quant_with_scale(_ptr(X), R, C, C, float(scale), _ptr(Xq)),
           "fp8_quant_with_scale")
    return Xq


int8_quant_weight_channel = int8_quant_rows
int8_quant_act_token = int8_quant_rows


# ---------------------------------------------------------------- GEMMs

def fp8_gemm(Xq, Xs, Wq, Ws) -> np.ndarray:
    """fp64 reference of the block-scaled FP8 GEMM; returns Y float64 [M,N]."""
    Xq = np.ascontiguousarray(Xq, np.uint8)
    Wq = np.ascontiguousarray(Wq, np.uint8)
    Xs = np.ascontiguousarray(Xs, np.float32)
    Ws = np.ascontiguousarray(Ws, np.float32)
    M, K = Xq.shape
    N = Wq.shape[0]
    assert Wq.shape == (N, K) and Xs.shape == (K // 128, M) and Ws.shape == (N // 128, K // 128)
    Y = np.empty((M, N), np.float64)
    _check(_load().oracle_fp8_gemm(_ptr(Xq), _ptr(Xs), _ptr(Wq), _ptr(Ws), M, N, K, _ptr(Y)),
           "fp8_gemm")
    return Y


def fp8_gemm_grouped(Xq, Xs, Wq, Ws, offsets) -> np.ndarray:
    """Grouped (mixture-of-experts) block-scaled FP8 GEMM (FP8-RL, Abstract: the
    FP8 rollout stack serves dense and MoE models).  The T token rows of Xq are
    grouped by expert: rows offsets[e] .. offsets[e+1]-1 go through expert e's
    weights Wq[e] [N,K] with scales Ws[e] [N/128, K/128], which is the dense GEMM
    above applied to each group.  Xs is [K/128, T].  Returns Y float64 [T, N]."""
    Wq = np.ascontiguousarray(Wq, np.uint8)
    Ws = np.ascontiguousarray(Ws, np.float32)
    E, N, K = Wq.shape
    T = Xq.shape[0]
    off = np.asarray(offsets, np.int64)
    assert off.shape == (E + 1,) and off[0] == 0 and off[-1] == T and np.all(np.diff(off) >= 0)
    assert Ws.shape == (E, N // 128, K // 128)
    Y = np.zeros((T, N), np.float64)
    for e in range(E):
        a, b = int(off[e]), int(off[e + 1])
        if b > a:
            Y[a:b] = fp8_gemm(Xq[a:b], Xs[:, a:b], Wq[e], Ws[e])
    return Y


def bf16_matmul_f64(X: np.ndarray, W: np.ndarray) -> np.ndarray:
    X = _bits16(X)
    W = _bits16(W)
    M, K = X.shape
    N = W.shape[0]
    Y = np.empty((M, N), np.float64)
    _check(_load().oracle_bf16_matmul_f64(_ptr(X), K, _ptr(W), K, M, N, K, _ptr(Y)),
           "bf16_matmul_f64")
    return Y


def int8_gemm(Xq, Xs, Wq, Ws):
    """Returns (acc int32 [M,N], Y bf16 bits uint16 [M,N])."""
    Xq = np.ascontiguousarray(Xq, np.int8)
    Wq = np.ascontiguousarray(Wq, np.int8)
    Xs = np.ascontiguousarray(Xs, np.float32)
    Ws = np.ascontiguousarray(Ws, np.float32)
    M, K = Xq.shape
    N = Wq.shape[0]
    acc = np.empty((M, N), np.int32)
    Y = np.empty((M, N), np.uint16)
    _check(_load().oracle_int8_gemm(_ptr(Xq), _ptr(Xs), _ptr(Wq), _ptr(Ws), M, N, K,
                                    _ptr(acc), _ptr(Y)), "int8_gemm")
    return acc, Y


def fp8_gemm_tolerance(y_ref: np.ndarray) -> np.ndarray:
    """Per-element bound |y - y_ref| <= 2^-7 |y_ref| + 1e-3 rms(y_ref), rms over the
    whole [M,N] output (the tolerance the library's FP8 GEMM is held to)."""
    rms = float(np.sqrt(np.mean(np.square(y_ref)))) if y_ref.size else 0.0
    return np.abs(y_ref) * 2.0 ** -7 + 1e-3 * rms


# ---------------------------------------------------------------- rollout correction

def rollout_is(logp_train, logp_rollout, mask, log_clip: float, mode: int):
    """Token-level TIS (mode 0) / MIS (mode 1) weights (float64) and stats
    [valid, clipped_or_masked, sum_w, sum_logratio]."""
    lt = np.ascontiguousarray(logp_train, np.float32).ravel()
    lr = np.ascontiguousarray(logp_rollout, np.float32).ravel()
    mk = np.ascontiguousarray(mask, np.uint8).ravel()
    n = lt.size
    w = np.empty(n, np.float64)
    st = np.empty(4, np.float64)
    _check(_load().oracle_rollout_is(_ptr(lt), _ptr(lr), _ptr(mk), n, float(log_clip), int(mode),
                                     _ptr(w), _ptr(st)), "rollout_is")
    return w.reshape(np.shape(logp_train)), st


# ---------------------------------------------------------------- mismatch

def logits_kl(P, Q) -> np.ndarray:
    """Per-row KL(softmax(P) || softmax(Q)) in fp64 for bf16 logits (uint16 bits)
    [M, V]: the train-inference mismatch of a quantized rollout (FlashRL write-up,
    Fig. 2, right), P the higher-precision logits, Q the quantized ones."""
    P = _bits16(P)
    Q = _bits16(Q)
    assert P.shape == Q.shape and P.ndim == 2
    M, V = P.shape
    kl = np.empty(M, np.float64)
    _check(_load().oracle_logits_kl(_ptr(P), V, _ptr(Q), V, M, V, _ptr(kl)), "logits_kl")
    return kl
