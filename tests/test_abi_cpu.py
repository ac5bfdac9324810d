"""CPU checks of the C ABI: the library loads, exports every function that
include/fp8rl.h declares, and rejects invalid arguments synchronously, before
any CUDA call (these paths never touch a device, so they run without a GPU).
Also checks that the product package never reaches the oracle."""
import ctypes
import os
import re

import pytest

from precision_rl_rollout_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8rl.h")
A = 0x10000  # a 16-byte-aligned fake device address: validation never dereferences it


@pytest.fixture(scope="module")
def lib():
    try:
        build.build()
    except RuntimeError as e:  # no nvcc on this machine
        pytest.skip(str(e))
    return binding.load()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_binding_exports():
    assert _declared_functions() == sorted(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
    version = int(re.search(r"#define FP8RL_ABI_VERSION (\d+)", open(HEADER).read()).group(1))
    assert lib.fp8rl_abi_version() == version
    for s in range(9):
        assert lib.fp8rl_status_string(s).decode().startswith(binding.STATUS[s])


def test_quant_weight_block_validation(lib):
    q = lib.fp8rl_quant_weight_block
    assert q(None, 128, 128, 128, A, A, None) == 1                  # NULL W
    assert q(A, 100, 128, 128, A, A, None) == 2                     # N % 128
    assert q(A, 128, 200, 200, A, A, None) == 2                     # K % 128
    assert q(A, 128, 256, 128, A, A, None) == 2                     # ldw < K
    assert q(A + 2, 128, 128, 128, A, A, None) == 3                 # misaligned W
    assert q(A, 128, 128, 132, A, A, None) == 3                     # row pitch 264 B
    assert q(A, 128, 128, 128, A + 8, A, None) == 3                 # misaligned Wq
    assert q(A, 128, 128, 128, None, A, None) == 1
    assert q(A, 0, 128, 128, A, A, None) == 0                       # empty: nothing launched


def test_grouped_requant_validates_every_descriptor_first(lib):
    D = binding.FP8RL_WDESC
    good = D(A, A, A, 128, 128, 128)
    bad = D(A, A, A, 128, 100, 128)
    arr = (D * 3)(good, good, bad)
    assert lib.fp8rl_quant_weight_block_grouped(arr, 3, None) == 2
    assert lib.fp8rl_quant_weight_block_grouped(None, 2, None) == 1
    assert lib.fp8rl_quant_weight_block_grouped(arr, -1, None) == 2
    empty = (D * 2)(D(A, A, A, 0, 128, 128), D(A, A, A, 0, 256, 256))
    assert lib.fp8rl_quant_weight_block_grouped(empty, 2, None) == 0


def test_act_quant_validation(lib):
    q = lib.fp8rl_quant_act_group
    assert q(A, 4, 100, 100, A, A, None) == 2
    assert q(A, -1, 128, 128, A, A, None) == 2
    assert q(A, 4, 128, 128, None, A, None) == 1
    assert q(A, 4, 128, 128, A, A + 2, None) == 3
    assert q(A, 0, 128, 128, A, A, None) == 0


def test_linear_validation(lib):
    f = lib.fp8rl_linear_w8a8_block
    #      X  ldx  Wq Ws  M   N    K   Y  ldy  Xq  Xs  ws   bytes
    assert f(A, 128, A, A, 8, 128, 256, A, 128, None, None, None, 0, None) == 2  # ldx < K
    assert f(A, 256, A, A, 8, 100, 256, A, 128, None, None, None, 0, None) == 2  # N % 128
    assert f(A, 256, A, A, 8, 128, 200, A, 128, None, None, None, 0, None) == 2  # K % 128
    assert f(A, 256, A, A, 8, 256, 256, A, 128, None, None, None, 0, None) == 2  # ldy < N
    assert f(None, 256, A, A, 8, 128, 256, A, 128, None, None, None, 0, None) == 1
    assert f(A, 256, None, A, 8, 128, 256, A, 128, None, None, None, 0, None) == 1
    assert f(A, 256, A, A, 8, 128, 256, None, 128, None, None, None, 0, None) == 1
    assert f(A, 256, A, A, 8, 128, 256, A, 128, A, None, None, 0, None) == 1    # Xq without Xs
    assert f(A + 2, 256, A, A, 8, 128, 256, A, 128, None, None, None, 0, None) == 3
    assert f(A, 260, A, A, 8, 128, 256, A, 128, None, None, None, 0, None) == 3  # row pitch 520 B
    assert f(A, 256, A, A, 8, 128, 256, A, 128, A + 8, A, None, 0, None) == 3
    assert f(A, 256, A, A, 2 ** 21, 128, 256, A, 128, A, A, None, 0, None) == 6  # above the M limit
    assert f(A, 256, A, A, 0, 128, 256, A, 128, None, None, None, 0, None) == 0  # empty batch
    # the workspace holds the codes and scales unless the caller passes Xq and Xs
    assert lib.fp8rl_linear_workspace_bytes(0, 128, 256) == 0
    need = lib.fp8rl_linear_workspace_bytes(65, 128, 256)
    assert need >= 65 * 256 + 65 * 2 * 4
    assert f(A, 256, A, A, 65, 128, 256, A, 128, None, None, A, need - 1, None) == 4
    assert f(A, 256, A, A, 65, 128, 256, A, 128, None, None, None, 0, None) == 4


def test_grouped_gemm_validation(lib):
    g = lib.fp8rl_gemm_w8a8_block_grouped
    #      Xq Xs Wq Ws off E  T   N    K    bound Y  ldy
    assert g(A, A, A, A, A, 0, 8, 128, 256, 8, A, 128, None) == 2      # no experts
    assert g(A, A, A, A, A, 4, -1, 128, 256, 8, A, 128, None) == 2     # negative T
    assert g(A, A, A, A, A, 4, 8, 100, 256, 8, A, 128, None) == 2      # N % 128
    assert g(A, A, A, A, A, 4, 8, 128, 256, 0, A, 128, None) == 2      # bound < 1
    assert g(A, A, A, A, A, 4, 8, 128, 256, 9, A, 128, None) == 2      # bound > T
    assert g(A, A, A, A, None, 4, 8, 128, 256, 8, A, 128, None) == 1   # offsets
    assert g(A, A, A, A, A + 2, 4, 8, 128, 256, 8, A, 128, None) == 3
    assert g(A, A, A, A, A, 4, 8, 128, 33024, 8, A, 128, None) == 6    # K above the decode limit
    assert g(A, A, A, A, A, 70000, 8, 128, 256, 8, A, 128, None) == 6  # grid z above 65535
    assert g(A, A, A, A, A, 4, 0, 128, 256, 8, A, 128, None) == 0      # no tokens: nothing launched


def test_logits_kl_validation(lib):
    f = lib.fp8rl_logits_kl
    ws = lib.fp8rl_logits_kl_workspace_bytes(4, 1000)
    assert ws == 4 * 1 * 32
    assert lib.fp8rl_logits_kl_workspace_bytes(2, 8193) == 2 * 3 * 32       # 32 bytes per 4096 logits
    #      P  ldp  Q  ldq  M  V     kl ws bytes
    assert f(A, 1000, A, 1000, 4, 0, A, A, ws, None) == 2         # V < 1
    assert f(A, 996, A, 1000, 4, 1000, A, A, ws, None) == 2       # ldp < V
    assert f(None, 1000, A, 1000, 4, 1000, A, A, ws, None) == 1
    assert f(A, 1000, A, 1000, 4, 1000, None, A, ws, None) == 1
    assert f(A, 1004, A, 1004, 4, 1000, A, A, ws, None) == 3      # row pitch 2008 B
    assert f(A, 1000, A + 2, 1000, 4, 1000, A, A, ws, None) == 3
    assert f(A, 1000, A, 1000, 4, 1000, A, A, ws - 1, None) == 4
    assert f(A, 1000, A, 1000, 70000, 1000, A, A, 1 << 40, None) == 6
    assert f(A, 1000, A, 1000, 0, 1000, A, None, 0, None) == 0    # nothing to do


def test_gemm_validation(lib):
    g = lib.fp8rl_gemm_w8a8_block
    ws = lib.fp8rl_gemm_workspace_bytes(64, 256, 256)
    assert g(A, A, A, A, 4, 100, 128, A, 100, None, ws, None) == 2   # N % 128
    assert g(A, A, A, A, 4, 128, 100, A, 128, None, ws, None) == 2   # K % 128
    assert g(A, A, A, A, 4, 128, 128, A, 64, None, ws, None) == 2    # ldy < N
    assert g(A, A, None, A, 4, 128, 128, A, 128, None, ws, None) == 1
    assert g(A + 4, A, A, A, 4, 128, 128, A, 128, None, ws, None) == 3
    assert g(A, A, A, A, 4, 128, 128, A, 132, None, ws, None) == 3   # row pitch 264 B
    assert g(A, A, A, A, 0, 128, 128, A, 128, None, ws, None) == 0   # empty batch
    e = lib.fp8rl_gemm_w8a8_block_ex
    assert e(A, A, A, A, 4, 100, 128, A, 100, None, ws, 1, None) == 2   # same validation
    assert e(A, A, A, A, 0, 128, 128, A, 128, None, ws, 1, None) == 0   # empty batch, known flag
    assert e(A, A, A, A, 0, 128, 128, A, 128, None, ws, 2, None) == 6   # unknown flag bit
    assert e(A, A, A, A, 0, 128, 128, A, 128, None, ws, 0x80000000, None) == 6
    i = lib.int8rl_gemm_w8a8
    assert i(A, A, A, A, 4, 128, 140032, A, 128, None, None, 0, None) == 6  # K * 127^2 >= 2^31
    assert i(A, A, A, A, 4, 128, 128, A, 128, A + 4, None, 0, None) == 3    # acc alignment
    assert i(A, A, A, A, 0, 128, 128, A, 128, None, None, 0, None) == 0


def test_int8_workspace_by_path(lib):
    # 4096 tokens with plenty of 128 x 256 tiles: fp16 copies of X and W and
    # nothing else (no split); a batch of 32 tokens needs none
    M, N, K = 4096, 7168, 5120
    assert lib.int8rl_gemm_workspace_bytes(M, N, K) == (M + N) * K * 2
    assert lib.int8rl_gemm_workspace_bytes(32, N, K) == 0
    assert lib.int8rl_gemm_workspace_bytes(64, N, K) == 0
    # 65 .. 256 tokens (and up to 512 on layers of 2^27 weights or more): the
    # 256-token kernel's fp16 copy of X, plus whole int32 partial tiles (256
    # tokens x 128 weight rows) of the K ranges when it splits K
    for M, N, K in [(65, 7168, 5120), (256, 7168, 5120), (256, 5120, 27648), (300, 55296, 5120),
                    (512, 5120, 27648)]:
        need = lib.int8rl_gemm_workspace_bytes(M, N, K)
        x16 = -(-(M * K * 2) // 16) * 16
        assert need >= x16 and (need - x16) % (256 * 128 * 4) == 0, (M, N, K, need)
        tiles = -(-M // 256) * (N // 128)
        assert (need - x16) // (256 * 128 * 4) in [s * tiles for s in (0, 2, 3, 4, 5, 6, 7, 8)]
    # 300 tokens on a layer below 2^27 weights: the large-batch path, with the
    # copies alone when its tiles fill the GPU, plus int32 partial tiles of
    # 128 x 256 when they are few (N = 2688: 33 tiles)
    assert lib.int8rl_gemm_workspace_bytes(300, 7168, 5120) == (300 + 7168) * 5120 * 2
    need = lib.int8rl_gemm_workspace_bytes(300, 2688, 4096)
    assert need > (300 + 2688) * 4096 * 2
    assert (need - (300 + 2688) * 4096 * 2) % (128 * 256 * 4) == 0


def test_fp8_gemm_workspace_is_whole_partial_tiles(lib):
    # whatever path a shape takes, its workspace is a whole number of fp32
    # partial tiles (decode: 128 channels x 16..128 tokens; prefill: 128 x 256)
    for M, N, K in [(1, 4608, 3584), (16, 3584, 18944), (32, 5120, 5120), (64, 3584, 18944),
                    (256, 5120, 27648), (300, 256, 4096)]:
        ws = lib.fp8rl_gemm_workspace_bytes(M, N, K)
        assert ws % (128 * 16 * 4) == 0, (M, N, K, ws)


def test_gemm_kernel_counts(lib):
    for f in (lib.fp8rl_gemm_kernel_count, lib.int8rl_gemm_kernel_count):
        assert f(0, 4608, 3584, 0) == 0
        assert f(4, 100, 3584, 0) == -2                   # N % 128
        assert f(4, 4608, 100, 0) == -2                   # K % 128
    for M, N, K in [(1, 4608, 3584), (64, 3584, 18944), (300, 256, 4096), (8192, 5120, 27648)]:
        # without a workspace every path launches one kernel; with the queried one, one or two
        assert lib.fp8rl_gemm_kernel_count(M, N, K, 0) == 1
        assert lib.fp8rl_gemm_kernel_count(M, N, K, lib.fp8rl_gemm_workspace_bytes(M, N, K)) in (1, 2)
    assert lib.int8rl_gemm_kernel_count(32, 7168, 5120, 0) == 1
    assert lib.int8rl_gemm_kernel_count(4096, 7168, 5120, lib.int8rl_gemm_workspace_bytes(4096, 7168, 5120)) == 2
    assert lib.int8rl_gemm_kernel_count(4096, 7168, 5120, 0) == 1
    # the 256-token path: X conversion and GEMM, plus the reduction of a K split
    for M, N, K in [(128, 7168, 5120), (256, 55296, 5120), (256, 5120, 27648)]:
        ws = lib.int8rl_gemm_workspace_bytes(M, N, K)
        split = (ws - M * K * 2) // (256 * 128 * 4 * (N // 128))
        assert lib.int8rl_gemm_kernel_count(M, N, K, ws) == (3 if split > 1 else 2)
        assert lib.int8rl_gemm_kernel_count(M, N, K, ws - 16) == 1     # too little: small-batch kernel


def test_linear_kernel_counts(lib):
    f = lib.fp8rl_linear_kernel_count
    assert f(0, 4608, 3584, 0, 0) == 0
    assert f(4, 100, 3584, 0, 0) == -2
    for M, N, K in [(1, 4608, 3584), (16, 3584, 18944), (32, 5120, 5120), (64, 3584, 18944), (300, 256, 4096)]:
        ws = lib.fp8rl_linear_workspace_bytes(M, N, K)
        gws = lib.fp8rl_gemm_workspace_bytes(M, N, K)
        # the quantizer plus the GEMM's kernels, with or without the codes back
        for want in (0, 1):
            assert f(M, N, K, ws, want) == 1 + lib.fp8rl_gemm_kernel_count(M, N, K, gws)
        # without the workspace the GEMM gives up its memory split
        assert f(M, N, K, 0, 0) == 1 + lib.fp8rl_gemm_kernel_count(M, N, K, 0)


def test_gemm_workspace_query_is_monotone(lib):
    for f in (lib.fp8rl_gemm_workspace_bytes, lib.int8rl_gemm_workspace_bytes):
        a = f(1, 4608, 3584)
        b = f(256, 4608, 3584)
        assert 0 <= a <= b or b == 0


def test_int8_quant_validation(lib):
    q = lib.int8rl_quant_weight_channel
    assert q(A, 4, 65536, 65536, A, A, None) == 6                   # K above the register-resident limit
    assert q(A, 4, 100, 100, A, A, None) == 2
    assert lib.int8rl_quant_act_token(A, 4, 128, 128, None, A, None) == 1


def test_product_package_never_reaches_the_oracle():
    pkg = os.path.join(ROOT, "precision_rl_rollout_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp", ".c")):
                text = open(os.path.join(dirpath, f), errors="ignore").read()
                assert not re.search(r"(import\s+oracle|from\s+oracle|\boracle\.|liboracle|oracle/)", text), \
                    f"{f} references the oracle package"


def test_kv_quant_validation(lib):
    q = lib.fp8rl_quant_kv_tensor
    ws = lib.fp8rl_kv_workspace_bytes(64, 1024)
    assert ws == 8 * ((64 * 1024 // 8 + 2047) // 2048 + 1)
    assert q(A, 64, 1020, 1024, A, A, A, ws, None) == 2                 # C % 8
    assert q(A, 64, 1024, 1000, A, A, A, ws, None) == 2                 # ld < C
    assert q(A, 64, 1024, 1024, A, None, A, ws, None) == 1               # scale
    assert q(A, 64, 1024, 1024, A, A, A, ws - 1, None) == 4              # workspace too small
    assert q(A, 64, 1024, 1024, A + 8, A, A, ws, None) == 3              # KVq alignment
    assert q(A, 64, 1024, 1024, A, A, A + 4, ws, None) == 3              # workspace: 8-byte slots
    w = lib.fp8rl_quant_kv_with_scale
    assert w(A, 64, 1024, 1024, None, A, None) == 1
    assert w(A, 0, 1024, 1024, A, A, None) == 0                          # empty: nothing launched


def test_kv_quant_noalloc_validation(lib):
    q = lib.fp8rl_quant_kv_tensor_noalloc
    assert q(A, 64, 1020, 1024, A, A, None) == 2                         # C % 8
    assert q(A, 64, 1024, 1000, A, A, None) == 2                         # ld < C
    assert q(None, 64, 1024, 1024, A, A, None) == 1                      # KV
    assert q(A, 64, 1024, 1024, None, A, None) == 1                      # KVq
    assert q(A, 64, 1024, 1024, A, None, None) == 1                      # scale
    assert q(A, 64, 1024, 1024, A + 8, A, None) == 3                     # KVq alignment
    assert q(A, 64, 1024, 1024, A, A + 2, None) == 3                     # scale alignment
    # above the library array's 16384 x 16384 values: refused before any launch
    assert q(A, 16384 * 16384 // 1024 + 1, 1024, 1024, A, A, None) == 6
    assert q(A, 16385, 16384, 16384, A, A, None) == 6


def test_rollout_is_validation(lib):
    f = lib.fp8rl_rollout_is_weights
    ws = lib.fp8rl_rollout_is_workspace_bytes(10000)
    assert ws == 8 + 3 * 32                  # header word + one 32-byte record per 4096 tokens
    assert f(A, A, None, 10000, ctypes.c_float(0.5), 2, A, A, A, ws, None) == 2      # bad mode
    assert f(A, A, None, 10000, ctypes.c_float(0.5), 0, A, None, A, ws, None) == 1   # stats NULL
    assert f(A, A, None, 10000, ctypes.c_float(0.5), 0, A, A + 4, A, ws, None) == 3  # stats alignment
    assert f(A, A, None, 10000, ctypes.c_float(0.5), 0, A, A, A, ws - 8, None) == 4  # workspace
