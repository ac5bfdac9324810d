"""Python binding of libfp8rl.so (include/fp8rl.h): the same names as the C ABI,
torch CUDA tensors in and out, argument marshalling only.  Every step of the
computation runs in the library's CUDA kernels; there is no fallback path, and
``load()`` raises if the shared library has not been built.

Tensors: bf16 inputs are ``torch.bfloat16``; E4M3 codes are ``torch.uint8``
(view them as ``torch.float8_e4m3fn`` if wanted); INT8 codes ``torch.int8``;
scales ``torch.float32``.  Outputs that are not passed in are allocated with
``torch.empty`` on the input's device.  Work is enqueued on the current torch
stream of that device unless ``stream`` is given.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

STATUS = {0: "FP8RL_OK", 1: "FP8RL_ERR_NULL", 2: "FP8RL_ERR_SHAPE", 3: "FP8RL_ERR_ALIGN",
          4: "FP8RL_ERR_WORKSPACE", 5: "FP8RL_ERR_CUDA", 6: "FP8RL_ERR_UNSUPPORTED",
          7: "FP8RL_ERR_TIMEOUT", 8: "FP8RL_ERR_DEVICE"}

# Every symbol the header declares (the CPU test checks the library exports them).
EXPORTS = ("fp8rl_status_string", "fp8rl_abi_version", "fp8rl_quant_weight_block",
           "fp8rl_quant_weight_block_grouped", "fp8rl_quant_act_group",
           "fp8rl_gemm_workspace_bytes", "fp8rl_gemm_w8a8_block", "fp8rl_gemm_w8a8_block_ex",
           "fp8rl_gemm_w8a8_block_grouped",
           "fp8rl_linear_workspace_bytes", "fp8rl_linear_kernel_count", "fp8rl_linear_w8a8_block",
           "int8rl_quant_weight_channel", "int8rl_quant_act_token",
           "int8rl_gemm_workspace_bytes", "int8rl_gemm_w8a8", "fp8rl_check_device_error",
           "fp8rl_gemm_kernel_count", "int8rl_gemm_kernel_count",
           "fp8rl_kv_workspace_bytes", "fp8rl_quant_kv_tensor", "fp8rl_quant_kv_with_scale",
           "fp8rl_quant_kv_tensor_noalloc", "fp8rl_rollout_is_workspace_bytes",
           "fp8rl_rollout_is_weights", "fp8rl_logits_kl_workspace_bytes", "fp8rl_logits_kl")


class Fp8rlError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} "
                         f"({_lib.fp8rl_status_string(status).decode() if _lib else ''})")


class FP8RL_WDESC(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("Wq", ctypes.c_void_p), ("Ws", ctypes.c_void_p),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("ldw", ctypes.c_int64)]


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None):
    """Load libfp8rl.so (built by ``precision_rl_rollout_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or _build.LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libfp8rl.so not found at {p}: build it with "
                               "`python -m precision_rl_rollout_gb300.build` (needs nvcc)")
        lib = ctypes.CDLL(p)
        P, I, Z, S = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p
        lib.fp8rl_status_string.restype = ctypes.c_char_p
        lib.fp8rl_status_string.argtypes = [ctypes.c_int]
        lib.fp8rl_abi_version.restype = ctypes.c_int
        lib.fp8rl_abi_version.argtypes = []
        lib.fp8rl_quant_weight_block.argtypes = [P, I, I, I, P, P, S]
        lib.fp8rl_quant_weight_block_grouped.argtypes = [ctypes.POINTER(FP8RL_WDESC), ctypes.c_int, S]
        lib.fp8rl_quant_act_group.argtypes = [P, I, I, I, P, P, S]
        lib.fp8rl_gemm_workspace_bytes.restype = Z
        lib.fp8rl_gemm_workspace_bytes.argtypes = [I, I, I]
        lib.fp8rl_gemm_kernel_count.restype = ctypes.c_int
        lib.fp8rl_gemm_kernel_count.argtypes = [I, I, I, Z]
        lib.int8rl_gemm_kernel_count.restype = ctypes.c_int
        lib.int8rl_gemm_kernel_count.argtypes = [I, I, I, Z]
        lib.fp8rl_gemm_w8a8_block.argtypes = [P, P, P, P, I, I, I, P, I, P, Z, S]
        lib.fp8rl_gemm_w8a8_block_ex.argtypes = [P, P, P, P, I, I, I, P, I, P, Z, ctypes.c_uint, S]
        lib.fp8rl_gemm_w8a8_block_grouped.argtypes = [P, P, P, P, P, I, I, I, I, I, P, I, S]
        lib.fp8rl_linear_workspace_bytes.restype = Z
        lib.fp8rl_linear_workspace_bytes.argtypes = [I, I, I]
        lib.fp8rl_linear_w8a8_block.argtypes = [P, I, P, P, I, I, I, P, I, P, P, P, Z, S]
        lib.fp8rl_linear_kernel_count.restype = ctypes.c_int
        lib.fp8rl_linear_kernel_count.argtypes = [I, I, I, Z, ctypes.c_int]
        lib.int8rl_quant_weight_channel.argtypes = [P, I, I, I, P, P, S]
        lib.int8rl_quant_act_token.argtypes = [P, I, I, I, P, P, S]
        lib.int8rl_gemm_workspace_bytes.restype = Z
        lib.int8rl_gemm_workspace_bytes.argtypes = [I, I, I]
        lib.int8rl_gemm_w8a8.argtypes = [P, P, P, P, I, I, I, P, I, P, P, Z, S]
        lib.fp8rl_check_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
        lib.fp8rl_kv_workspace_bytes.restype = Z
        lib.fp8rl_kv_workspace_bytes.argtypes = [I, I]
        lib.fp8rl_quant_kv_tensor.argtypes = [P, I, I, I, P, P, P, Z, S]
        lib.fp8rl_quant_kv_with_scale.argtypes = [P, I, I, I, P, P, S]
        lib.fp8rl_quant_kv_tensor_noalloc.argtypes = [P, I, I, I, P, P, S]
        lib.fp8rl_logits_kl_workspace_bytes.restype = Z
        lib.fp8rl_logits_kl_workspace_bytes.argtypes = [I, I]
        lib.fp8rl_logits_kl.argtypes = [P, I, P, I, I, I, P, P, Z, S]
        lib.fp8rl_rollout_is_workspace_bytes.restype = Z
        lib.fp8rl_rollout_is_workspace_bytes.argtypes = [I]
        lib.fp8rl_rollout_is_weights.argtypes = [P, P, P, I, ctypes.c_float, ctypes.c_int, P, P, P, Z, S]
        for name in EXPORTS:
            if name not in ("fp8rl_status_string", "fp8rl_abi_version", "fp8rl_gemm_workspace_bytes",
                            "int8rl_gemm_workspace_bytes", "fp8rl_kv_workspace_bytes",
                            "fp8rl_rollout_is_workspace_bytes", "fp8rl_linear_workspace_bytes",
                            "fp8rl_logits_kl_workspace_bytes"):
                getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def _ck(rc: int, where: str):
    if rc != 0:
        raise Fp8rlError(rc, where)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(t: torch.Tensor, stream):
    if stream is None:
        stream = torch.cuda.current_stream(t.device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _rowmajor(t: torch.Tensor, name: str):
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D tensor with unit column stride")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    return t.stride(0)


def _need(t, shape, dtype, device, name):
    if t is None:
        return torch.empty(shape, dtype=dtype, device=device)
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name}: expected contiguous {dtype} {tuple(shape)}, got {t.dtype} {tuple(t.shape)}")
    return t


# ------------------------------------------------------------------ ABI mirror

def fp8rl_status_string(status: int) -> str:
    return load().fp8rl_status_string(status).decode()


def fp8rl_abi_version() -> int:
    return load().fp8rl_abi_version()


def fp8rl_quant_weight_block(W, Wq=None, Ws=None, stream=None):
    """W bf16 [N,K] -> (Wq uint8 [N,K], Ws fp32 [N/128, K/128])."""
    lib = load()
    ldw = _rowmajor(W, "W")
    N, K = W.shape
    Wq = _need(Wq, (N, K), torch.uint8, W.device, "Wq")
    Ws = _need(Ws, (N // 128, K // 128), torch.float32, W.device, "Ws")
    _ck(lib.fp8rl_quant_weight_block(_p(W), N, K, ldw, _p(Wq), _p(Ws), _stream(W, stream)),
        "fp8rl_quant_weight_block")
    return Wq, Ws


def fp8rl_quant_weight_block_grouped(items, stream=None):
    """items: sequence of (W, Wq, Ws) with preallocated outputs."""
    lib = load()
    arr = (FP8RL_WDESC * len(items))()
    for i, (W, Wq, Ws) in enumerate(items):
        ldw = _rowmajor(W, "W")
        N, K = W.shape
        _need(Wq, (N, K), torch.uint8, W.device, "Wq")
        _need(Ws, (N // 128, K // 128), torch.float32, W.device, "Ws")
        arr[i] = FP8RL_WDESC(W.data_ptr(), Wq.data_ptr(), Ws.data_ptr(), N, K, ldw)
    dev_t = items[0][0] if items else torch.empty(0, device="cuda")
    _ck(lib.fp8rl_quant_weight_block_grouped(arr, len(items), _stream(dev_t, stream)),
        "fp8rl_quant_weight_block_grouped")


class GroupedRequant:
    """A fixed set of (W, Wq, Ws) for repeated fp8rl_quant_weight_block_grouped
    calls (one per RL step): the descriptor array is marshalled once, so a call
    costs one C-ABI call on the host."""

    def __init__(self, items):
        if not items or len(items) > 256:
            raise ValueError("1 to 256 tensors per grouped requant")
        self.lib = load()
        self.items = list(items)                      # keeps the tensors alive
        self.arr = (FP8RL_WDESC * len(self.items))()
        for i, (W, Wq, Ws) in enumerate(self.items):
            ldw = _rowmajor(W, "W")
            N, K = W.shape
            _need(Wq, (N, K), torch.uint8, W.device, "Wq")
            _need(Ws, (N // 128, K // 128), torch.float32, W.device, "Ws")
            self.arr[i] = FP8RL_WDESC(W.data_ptr(), Wq.data_ptr(), Ws.data_ptr(), N, K, ldw)

    def __call__(self, stream=None):
        _ck(self.lib.fp8rl_quant_weight_block_grouped(self.arr, len(self.items),
                                                      _stream(self.items[0][0], stream)),
            "fp8rl_quant_weight_block_grouped")


def fp8rl_quant_act_group(X, Xq=None, Xs=None, stream=None):
    """X bf16 [M,K] -> (Xq uint8 [M,K], Xs fp32 [K/128, M])."""
    lib = load()
    ldx = _rowmajor(X, "X")
    M, K = X.shape
    Xq = _need(Xq, (M, K), torch.uint8, X.device, "Xq")
    Xs = _need(Xs, (K // 128, M), torch.float32, X.device, "Xs")
    _ck(lib.fp8rl_quant_act_group(_p(X), M, K, ldx, _p(Xq), _p(Xs), _stream(X, stream)),
        "fp8rl_quant_act_group")
    return Xq, Xs


def fp8rl_gemm_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load().fp8rl_gemm_workspace_bytes(M, N, K))


FP8RL_GEMM_WEIGHTS_STABLE = 1


def fp8rl_gemm_w8a8_block(Xq, Xs, Wq, Ws, Y=None, workspace=None, stream=None, weights_stable=False):
    """-> Y bf16 [M,N].  weights_stable=True passes FP8RL_GEMM_WEIGHTS_STABLE
    (the kernel issued right before this call on the stream did not write Wq)."""
    lib = load()
    M, K = Xq.shape
    N = Wq.shape[0]
    Y = Y if Y is not None else torch.empty((M, N), dtype=torch.bfloat16, device=Wq.device)
    ldy = _rowmajor(Y, "Y") if M > 0 else N
    need = lib.fp8rl_gemm_workspace_bytes(M, N, K)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=Wq.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if weights_stable:
        _ck(lib.fp8rl_gemm_w8a8_block_ex(_p(Xq), _p(Xs), _p(Wq), _p(Ws), M, N, K, _p(Y), ldy,
                                         _p(workspace), wbytes, FP8RL_GEMM_WEIGHTS_STABLE, _stream(Wq, stream)),
            "fp8rl_gemm_w8a8_block_ex")
    else:
        _ck(lib.fp8rl_gemm_w8a8_block(_p(Xq), _p(Xs), _p(Wq), _p(Ws), M, N, K, _p(Y), ldy,
                                      _p(workspace), wbytes, _stream(Wq, stream)),
            "fp8rl_gemm_w8a8_block")
    return Y


def fp8rl_gemm_w8a8_block_grouped(Xq, Xs, Wq, Ws, expert_offsets, max_tokens_per_expert=None, Y=None,
                                  stream=None):
    """Mixture-of-experts GEMM.  Xq [T,K] (rows grouped by expert), Xs [K/128,T],
    Wq [E,N,K], Ws [E,N/128,K/128], expert_offsets int32 [E+1] on the device.
    max_tokens_per_expert: host-side bound on any expert's token count (T if None).
    -> Y bf16 [T,N]."""
    lib = load()
    T, K = Xq.shape
    E, N = Wq.shape[0], Wq.shape[1]
    if expert_offsets.dtype != torch.int32 or not expert_offsets.is_cuda or expert_offsets.numel() != E + 1:
        raise ValueError("expert_offsets must be a CUDA int32 tensor of E+1 entries")
    Y = Y if Y is not None else torch.empty((T, N), dtype=torch.bfloat16, device=Wq.device)
    ldy = _rowmajor(Y, "Y") if T > 0 else N
    bound = T if max_tokens_per_expert is None else int(max_tokens_per_expert)
    _ck(lib.fp8rl_gemm_w8a8_block_grouped(_p(Xq), _p(Xs), _p(Wq), _p(Ws), _p(expert_offsets), E, T, N, K,
                                          bound, _p(Y), ldy, _stream(Wq, stream)),
        "fp8rl_gemm_w8a8_block_grouped")
    return Y


def fp8rl_linear_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load().fp8rl_linear_workspace_bytes(M, N, K))


def fp8rl_linear_w8a8_block(X, Wq, Ws, Y=None, Xq=None, Xs=None, want_codes=False, workspace=None,
                            stream=None):
    """X bf16 [M,K] -> Y bf16 [M,N] (and (Xq, Xs) when want_codes or Xq/Xs are given)."""
    lib = load()
    ldx = _rowmajor(X, "X")
    M, K = X.shape
    N = Wq.shape[0]
    Y = Y if Y is not None else torch.empty((M, N), dtype=torch.bfloat16, device=Wq.device)
    ldy = _rowmajor(Y, "Y") if M > 0 else N
    if want_codes or Xq is not None or Xs is not None:
        Xq = _need(Xq, (M, K), torch.uint8, X.device, "Xq")
        Xs = _need(Xs, (K // 128, M), torch.float32, X.device, "Xs")
    need = lib.fp8rl_linear_workspace_bytes(M, N, K)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=Wq.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _ck(lib.fp8rl_linear_w8a8_block(_p(X), ldx, _p(Wq), _p(Ws), M, N, K, _p(Y), ldy, _p(Xq), _p(Xs),
                                    _p(workspace), wbytes, _stream(Wq, stream)),
        "fp8rl_linear_w8a8_block")
    return (Y, Xq, Xs) if Xq is not None else Y


def int8rl_quant_weight_channel(W, Wq=None, Ws=None, stream=None):
    """W bf16 [N,K] -> (Wq int8 [N,K], Ws fp32 [N])."""
    lib = load()
    ldw = _rowmajor(W, "W")
    N, K = W.shape
    Wq = _need(Wq, (N, K), torch.int8, W.device, "Wq")
    Ws = _need(Ws, (N,), torch.float32, W.device, "Ws")
    _ck(lib.int8rl_quant_weight_channel(_p(W), N, K, ldw, _p(Wq), _p(Ws), _stream(W, stream)),
        "int8rl_quant_weight_channel")
    return Wq, Ws


def int8rl_quant_act_token(X, Xq=None, Xs=None, stream=None):
    """X bf16 [M,K] -> (Xq int8 [M,K], Xs fp32 [M])."""
    lib = load()
    ldx = _rowmajor(X, "X")
    M, K = X.shape
    Xq = _need(Xq, (M, K), torch.int8, X.device, "Xq")
    Xs = _need(Xs, (M,), torch.float32, X.device, "Xs")
    _ck(lib.int8rl_quant_act_token(_p(X), M, K, ldx, _p(Xq), _p(Xs), _stream(X, stream)),
        "int8rl_quant_act_token")
    return Xq, Xs


def fp8rl_gemm_kernel_count(M: int, N: int, K: int, workspace_bytes: int) -> int:
    return int(load().fp8rl_gemm_kernel_count(M, N, K, workspace_bytes))


def fp8rl_linear_kernel_count(M: int, N: int, K: int, workspace_bytes: int, want_codes: bool = False) -> int:
    return int(load().fp8rl_linear_kernel_count(M, N, K, workspace_bytes, 1 if want_codes else 0))


def int8rl_gemm_kernel_count(M: int, N: int, K: int, workspace_bytes: int) -> int:
    return int(load().int8rl_gemm_kernel_count(M, N, K, workspace_bytes))


def int8rl_gemm_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load().int8rl_gemm_workspace_bytes(M, N, K))


def int8rl_gemm_w8a8(Xq, Xs, Wq, Ws, Y=None, acc=None, want_acc=False, workspace=None, stream=None):
    """-> Y bf16 [M,N] (and the int32 accumulators when want_acc or acc is given)."""
    lib = load()
    M, K = Xq.shape
    N = Wq.shape[0]
    Y = Y if Y is not None else torch.empty((M, N), dtype=torch.bfloat16, device=Wq.device)
    ldy = _rowmajor(Y, "Y") if M > 0 else N
    if want_acc and acc is None:
        acc = torch.empty((M, N), dtype=torch.int32, device=Wq.device)
    need = lib.int8rl_gemm_workspace_bytes(M, N, K)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=Wq.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _ck(lib.int8rl_gemm_w8a8(_p(Xq), _p(Xs), _p(Wq), _p(Ws), M, N, K, _p(Y), ldy, _p(acc),
                             _p(workspace), wbytes, _stream(Wq, stream)), "int8rl_gemm_w8a8")
    return (Y, acc) if acc is not None else Y


def fp8rl_kv_workspace_bytes(R: int, C: int) -> int:
    return int(load().fp8rl_kv_workspace_bytes(R, C))


def fp8rl_quant_kv_tensor(KV, KVq=None, scale=None, workspace=None, stream=None):
    """KV bf16 [R,C] -> (KVq uint8 [R,C], scale fp32 [1]): per-tensor scale recalibrated."""
    lib = load()
    ld = _rowmajor(KV, "KV")
    R, C = KV.shape
    KVq = _need(KVq, (R, C), torch.uint8, KV.device, "KVq")
    scale = _need(scale, (1,), torch.float32, KV.device, "scale")
    need = lib.fp8rl_kv_workspace_bytes(R, C)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=KV.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _ck(lib.fp8rl_quant_kv_tensor(_p(KV), R, C, ld, _p(KVq), _p(scale), _p(workspace), wbytes,
                                  _stream(KV, stream)), "fp8rl_quant_kv_tensor")
    return KVq, scale


def fp8rl_quant_kv_with_scale(KV, scale, KVq=None, stream=None):
    """KV bf16 [R,C], scale fp32 [1] (device) -> KVq uint8 [R,C]."""
    lib = load()
    ld = _rowmajor(KV, "KV")
    R, C = KV.shape
    KVq = _need(KVq, (R, C), torch.uint8, KV.device, "KVq")
    _need(scale, (1,), torch.float32, KV.device, "scale")
    _ck(lib.fp8rl_quant_kv_with_scale(_p(KV), R, C, ld, _p(scale), _p(KVq), _stream(KV, stream)),
        "fp8rl_quant_kv_with_scale")
    return KVq


def fp8rl_quant_kv_tensor_noalloc(KV, KVq, scale, stream=None):
    """As fp8rl_quant_kv_tensor, but with the library's own scratch instead of a
    workspace, for callers that cannot allocate; KVq and scale must be given."""
    lib = load()
    ld = _rowmajor(KV, "KV")
    R, C = KV.shape
    _need(KVq, (R, C), torch.uint8, KV.device, "KVq")
    _need(scale, (1,), torch.float32, KV.device, "scale")
    _ck(lib.fp8rl_quant_kv_tensor_noalloc(_p(KV), R, C, ld, _p(KVq), _p(scale), _stream(KV, stream)),
        "fp8rl_quant_kv_tensor_noalloc")
    return KVq, scale


FP8RL_IS_TRUNCATE = 0
FP8RL_IS_MASK = 1


def fp8rl_rollout_is_workspace_bytes(n: int) -> int:
    return int(load().fp8rl_rollout_is_workspace_bytes(n))


def fp8rl_rollout_is_weights(logp_train, logp_rollout, mask=None, log_clip: float = 0.6931472,
                             mode: int = FP8RL_IS_TRUNCATE, weights=None, stats=None, workspace=None,
                             stream=None):
    """fp32 log-probs [...] (same shape, contiguous) -> (weights fp32 [...], stats fp64 [4])."""
    lib = load()
    if logp_train.shape != logp_rollout.shape or not logp_train.is_contiguous() or not logp_rollout.is_contiguous():
        raise ValueError("logp_train and logp_rollout must be contiguous tensors of the same shape")
    n = logp_train.numel()
    weights = _need(weights, tuple(logp_train.shape), torch.float32, logp_train.device, "weights")
    stats = _need(stats, (4,), torch.float64, logp_train.device, "stats")
    if mask is not None and (mask.dtype != torch.uint8 or mask.numel() != n or not mask.is_contiguous()):
        raise ValueError("mask must be a contiguous uint8 tensor with one byte per token")
    need = lib.fp8rl_rollout_is_workspace_bytes(n)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=logp_train.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _ck(lib.fp8rl_rollout_is_weights(_p(logp_train), _p(logp_rollout), _p(mask), n, float(log_clip), int(mode),
                                     _p(weights), _p(stats), _p(workspace), wbytes,
                                     _stream(logp_train, stream)), "fp8rl_rollout_is_weights")
    return weights, stats


def fp8rl_check_device_error() -> int:
    """Synchronizes the device; returns the raw device error word (0 if none)."""
    lib = load()
    w = ctypes.c_uint32(0)
    rc = lib.fp8rl_check_device_error(ctypes.byref(w))
    if rc not in (0, 7, 8):
        raise Fp8rlError(rc, "fp8rl_check_device_error")
    return int(w.value)


def fp8rl_logits_kl_workspace_bytes(M: int, V: int) -> int:
    return int(load().fp8rl_logits_kl_workspace_bytes(M, V))


def fp8rl_logits_kl(P, Q, kl=None, workspace=None, stream=None):
    """Per-row KL(softmax(P) || softmax(Q)) of bf16 logits [M, V] -> fp32 [M]."""
    lib = load()
    ldp, ldq = _rowmajor(P, "P"), _rowmajor(Q, "Q")
    if P.shape != Q.shape:
        raise ValueError("P and Q must have the same shape")
    M, V = P.shape
    kl = _need(kl, (M,), torch.float32, P.device, "kl")
    need = lib.fp8rl_logits_kl_workspace_bytes(M, V)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=P.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _ck(lib.fp8rl_logits_kl(_p(P), ldp, _p(Q), ldq, M, V, _p(kl), _p(workspace), wbytes, _stream(P, stream)),
        "fp8rl_logits_kl")
    return kl
