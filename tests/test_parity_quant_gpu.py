"""GPU parity of the quantizers against the CPU oracle: codes and scales must be
bit-exact.  Small cases are compared in full (several blocks, ragged token
counts, strided inputs, planted edge cases); the Qwen2.5-7B/32B shapes are
compared on sampled blocks/rows plus properties that hold at any size."""
import numpy as np
import pytest
import torch

import oracle
from precision_rl_rollout_gb300 import binding as fb
from precision_rl_rollout_gb300 import synth
from parity_util import (act_cpu, bits_u32, host, sample_blocks, sample_rows, weight_cpu)

pytestmark = pytest.mark.gpu


def _cmp_weight_block(W_cpu: torch.Tensor, Wq_gpu, Ws_gpu, what):
    want_q, want_s = oracle.fp8_quant_weight_block(synth.bf16_bits(W_cpu))
    got_q, got_s = host(Wq_gpu), host(Ws_gpu)
    assert np.array_equal(bits_u32(got_s), bits_u32(want_s)), f"{what}: scales differ"
    bad = np.argwhere(got_q != want_q)
    assert bad.size == 0, f"{what}: {len(bad)} codes differ, first {bad[:4].tolist()}"


def test_fp8_weight_requant_tiny(cuda_lib):
    W = weight_cpu(synth.TINY.N, synth.TINY.K, synth.seed_for(1, 0))
    Wq, Ws = fb.fp8rl_quant_weight_block(W.cuda())
    _cmp_weight_block(W, Wq, Ws, "tiny")


def test_fp8_weight_requant_edge_cases_and_strided_input(cuda_lib):
    W = synth.edge_case_weight(384, 512, seed=31)
    wide = torch.zeros(384, 640, dtype=torch.bfloat16)
    wide[:, :512] = W
    Wd = wide.cuda()[:, :512]                       # ldw = 640 > K
    Wq, Ws = fb.fp8rl_quant_weight_block(Wd)
    _cmp_weight_block(W, Wq, Ws, "edge")


@pytest.mark.parametrize("shape", synth.QWEN25_7B, ids=lambda s: s.name)
def test_fp8_weight_requant_qwen7b_sampled(cuda_lib, shape):
    W = weight_cpu(shape.N, shape.K, synth.seed_for(2, 0))
    Wq, Ws = fb.fp8rl_quant_weight_block(W.cuda())
    torch.cuda.synchronize()
    # any size: no NaN code, and every block's largest magnitude code is 448 (0x7E)
    mag = (Wq & 0x7F)
    assert not bool((mag == 0x7F).any())
    blkmax = mag.view(shape.N // 128, 128, shape.K // 128, 128).amax(dim=(1, 3))
    assert bool((blkmax == 0x7E).all())
    Wq_h, Ws_h = host(Wq), host(Ws)
    for nb, kb in sample_blocks(shape.N // 128, shape.K // 128, 40, seed=shape.K + shape.N):
        blk = W[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128].contiguous()
        q, s = oracle.fp8_quant_weight_block(synth.bf16_bits(blk))
        assert bits_u32(Ws_h[nb, kb:kb + 1])[0] == bits_u32(s)[0, 0], (nb, kb)
        assert np.array_equal(Wq_h[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128], q), (nb, kb)


def test_grouped_requant_matches_oracle_across_launches(cuda_lib):
    # more tensors than one grouped launch takes, with mixed shapes and pitches
    rng = np.random.default_rng(8)
    items, cpu = [], []
    for i in range(300):
        N = 128 * int(rng.integers(1, 3))
        K = 128 * int(rng.integers(1, 4))
        pad = 8 * int(rng.integers(0, 3))
        Wc = synth.weight(N, K, 5000 + i, std=float(10.0 ** rng.uniform(-3, 1)))
        big = torch.zeros(N, K + pad, dtype=torch.bfloat16)
        big[:, :K] = Wc
        Wd = big.cuda()[:, :K]
        items.append((Wd, torch.empty(N, K, dtype=torch.uint8, device="cuda"),
                      torch.empty(N // 128, K // 128, dtype=torch.float32, device="cuda")))
        cpu.append(Wc)
    fb.fp8rl_quant_weight_block_grouped(items)
    for i in list(range(0, 300, 7)) + [255, 256, 299]:
        _cmp_weight_block(cpu[i], items[i][1], items[i][2], f"grouped[{i}]")


def test_grouped_requant_qwen32b_full_model_sampled(cuda_lib):
    # the full-model requant as timed: 64 layers x 4 Qwen2.5-32B weights (256
    # tensors, 31.2 G values, 62.4 GB) after a policy update, in one grouped
    # launch; sampled blocks of the first, a middle and the last layer of
    # every shape -- corner blocks and seeded interior ones -- against the oracle
    items = []
    for layer in range(synth.QWEN25_32B_LAYERS):
        for i, s in enumerate(synth.QWEN25_32B):
            seed = synth.seed_for(4, 0) + 1000 * layer + i
            W = synth.weight_bf16_direct(s.N, s.K, seed, device="cuda")
            synth.policy_update_(W, seed + 500)
            items.append((W, torch.empty(s.N, s.K, dtype=torch.uint8, device="cuda"),
                          torch.empty(s.N // 128, s.K // 128, dtype=torch.float32, device="cuda")))
    fb.GroupedRequant(items)()
    torch.cuda.synchronize()
    nshapes = len(synth.QWEN25_32B)
    for layer in (0, 37, synth.QWEN25_32B_LAYERS - 1):
        for i, s in enumerate(synth.QWEN25_32B):
            W, Wq, Ws = items[layer * nshapes + i]
            Ws_h = host(Ws)
            for nb, kb in sample_blocks(s.N // 128, s.K // 128, 12, seed=layer * 10 + i):
                blk = W[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128].contiguous().cpu()
                q, sc = oracle.fp8_quant_weight_block(synth.bf16_bits(blk))
                got = host(Wq[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128])
                assert bits_u32(Ws_h[nb, kb:kb + 1])[0] == bits_u32(sc)[0, 0], (layer, s.name, nb, kb)
                assert np.array_equal(got, q), (layer, s.name, nb, kb)
    del items
    torch.cuda.empty_cache()
    assert fb.fp8rl_check_device_error() == 0


@pytest.mark.parametrize("M,K", [(1, 128), (5, 256), (16, 256), (17, 384), (33, 3584),
                                 (64, 3584), (257, 640)])
def test_fp8_act_quant_full(cuda_lib, M, K):
    X = act_cpu(M, K, synth.seed_for(1, 1) + M)
    Xq, Xs = fb.fp8rl_quant_act_group(X.cuda())
    want_q, want_s = oracle.fp8_quant_act_group(synth.bf16_bits(X))
    assert np.array_equal(bits_u32(host(Xs)), bits_u32(want_s))
    assert np.array_equal(host(Xq), want_q)


def test_fp8_act_quant_edge_rows_and_empty(cuda_lib):
    X = synth.edge_case_activation(11, 640, seed=3)
    Xq, Xs = fb.fp8rl_quant_act_group(X.cuda())
    want_q, want_s = oracle.fp8_quant_act_group(synth.bf16_bits(X))
    assert np.array_equal(bits_u32(host(Xs)), bits_u32(want_s))
    assert np.array_equal(host(Xq), want_q)
    Xq0, Xs0 = fb.fp8rl_quant_act_group(torch.empty(0, 256, dtype=torch.bfloat16, device="cuda"))
    assert Xq0.shape == (0, 256) and Xs0.shape == (2, 0)


@pytest.mark.parametrize("M", synth.DECODE_M_SWEEP)
@pytest.mark.parametrize("K", [5120, 27648])
def test_fp8_act_quant_qwen32b_decode(cuda_lib, M, K):
    X = act_cpu(M, K, synth.seed_for(3, 1))
    Xq, Xs = fb.fp8rl_quant_act_group(X.cuda())
    want_q, want_s = oracle.fp8_quant_act_group(synth.bf16_bits(X))
    assert np.array_equal(bits_u32(host(Xs)), bits_u32(want_s))
    assert np.array_equal(host(Xq), want_q)


@pytest.mark.parametrize("M,K", [(8191, 3456), (4096, 5120)])
def test_fp8_act_quant_large_full(cuda_lib, M, K):
    # large enough for several groups per thread; 8191 x 3456 leaves a ragged
    # last token tile (15 of 16) and a ragged last group range (27 = 6 x 4 + 3)
    X = act_cpu(M, K, synth.seed_for(4, 1) + K)
    Xq, Xs = fb.fp8rl_quant_act_group(X.cuda())
    want_q, want_s = oracle.fp8_quant_act_group(synth.bf16_bits(X))
    assert np.array_equal(bits_u32(host(Xs)), bits_u32(want_s))
    assert np.array_equal(host(Xq), want_q)


def test_fp8_act_quant_prefill_sampled(cuda_lib):
    M, K = synth.PREFILL_M, 27648
    X = act_cpu(M, K, synth.seed_for(4, 1))
    Xq, Xs = fb.fp8rl_quant_act_group(X.cuda())
    rows = sample_rows(M, 24, seed=4)
    want_q, want_s = oracle.fp8_quant_act_group(synth.bf16_bits(X[rows]))
    assert np.array_equal(bits_u32(host(Xs)[:, rows]), bits_u32(want_s))
    assert np.array_equal(host(Xq)[rows], want_q)


# K spans every row-kernel instance: 128-thread CTAs with 1..8 chunks of 8 per
# thread (K <= 8192), then 256-thread CTAs with 6, 8, 12 and 16
@pytest.mark.parametrize("R,K", [(1, 128), (7, 256), (3, 1152), (3, 2944), (3, 4096), (128, 5120),
                                 (3, 6016), (3, 8192), (3, 8320), (3, 16384), (3, 24576), (33, 27648)])
def test_int8_row_quant_full(cuda_lib, R, K):
    A = act_cpu(R, K, 77 + R)
    for fn in (fb.int8rl_quant_weight_channel, fb.int8rl_quant_act_token):
        Q, S = fn(A.cuda())
        want_q, want_s = oracle.int8_quant_rows(synth.bf16_bits(A))
        assert np.array_equal(bits_u32(host(S)), bits_u32(want_s))
        assert np.array_equal(host(Q), want_q)


def test_int8_row_quant_edge_and_strided(cuda_lib):
    A = synth.edge_case_activation(9, 384, seed=12)
    wide = torch.zeros(9, 512, dtype=torch.bfloat16)
    wide[:, :384] = A
    Q, S = fb.int8rl_quant_act_token(wide.cuda()[:, :384])
    want_q, want_s = oracle.int8_quant_rows(synth.bf16_bits(A))
    assert np.array_equal(bits_u32(host(S)), bits_u32(want_s))
    assert np.array_equal(host(Q), want_q)


@pytest.mark.parametrize("shape", synth.QWEN25_32B, ids=lambda s: s.name)
def test_int8_weight_quant_qwen32b_sampled(cuda_lib, shape):
    W = weight_cpu(shape.N, shape.K, synth.seed_for(5, 0))
    Q, S = fb.int8rl_quant_weight_channel(W.cuda())
    rows = sample_rows(shape.N, 32, seed=shape.N)
    want_q, want_s = oracle.int8_quant_rows(synth.bf16_bits(W[rows]))
    assert np.array_equal(bits_u32(host(S)[rows]), bits_u32(want_s))
    assert np.array_equal(host(Q)[rows], want_q)
    assert int(Q.abs().amax(dim=1).min()) == 127


def test_no_device_error_recorded(cuda_lib):
    assert fb.fp8rl_check_device_error() == 0


# ------------------------------------------------------------------ FP8 KV-cache, per-tensor scale

@pytest.mark.parametrize("R,C,ld", [(1, 8, 8), (3, 136, 144), (64, 1024, 1024), (300, 1024, 1032),
                                    (2049, 1024, 1024), (8192, 1024, 1024)])
def test_fp8_kv_tensor_quant_full(cuda_lib, R, C, ld):
    X = act_cpu(R, C, 9000 + R + C)
    wide = torch.zeros(R, ld, dtype=torch.bfloat16)
    wide[:, :C] = X
    KVq, scale = fb.fp8rl_quant_kv_tensor(wide.cuda()[:, :C])
    want_q, want_s = oracle.fp8_quant_tensor(synth.bf16_bits(X))
    assert bits_u32(host(scale))[0] == np.float32(want_s).view(np.uint32)
    assert np.array_equal(host(KVq), want_q)
    # the with-scale entry point on the same scale gives the same codes
    KVq2 = fb.fp8rl_quant_kv_with_scale(wide.cuda()[:, :C], scale)
    assert np.array_equal(host(KVq2), want_q)


def test_fp8_kv_tensor_quant_edge_rows_and_empty(cuda_lib):
    X = synth.edge_case_activation(11, 640, seed=13)
    KVq, scale = fb.fp8rl_quant_kv_tensor(X.cuda())
    want_q, want_s = oracle.fp8_quant_tensor(synth.bf16_bits(X))
    assert bits_u32(host(scale))[0] == np.float32(want_s).view(np.uint32)
    assert np.array_equal(host(KVq), want_q)
    KVq0, s0 = fb.fp8rl_quant_kv_tensor(torch.empty(0, 64, dtype=torch.bfloat16, device="cuda"))
    assert KVq0.shape == (0, 64) and float(s0[0]) == 1.0


def test_fp8_kv_tensor_quant_qwen32b_cache_sampled(cuda_lib):
    # a rollout-sized K cache: 64 sequences x 2048 tokens, 8 kv heads x 128
    R, C = 64 * 2048, 1024
    X = synth.activation(R, C, synth.seed_for(6, 0), device="cuda")
    KVq, scale = fb.fp8rl_quant_kv_tensor(X)
    want_q, want_s = oracle.fp8_quant_tensor(synth.bf16_bits(X))
    assert bits_u32(host(scale))[0] == np.float32(want_s).view(np.uint32)
    assert np.array_equal(host(KVq), want_q)


@pytest.mark.parametrize("R,where", [(9728, "last"), (9728, "first"), (9744, "last")])
def test_fp8_kv_tensor_quant_one_pass_boundary(cuda_lib, R, where):
    # 9728 x 1024 is 608 slices of 16384 values (every slice's CTA resident at
    # four per SM on 152 SMs: one pass); 9744 x 1024 is 609 (one CTA per SM
    # over ranges kept partly on chip).  The tensor amax sits in the first or
    # last slice only.
    C = 1024
    X = act_cpu(R, C, 9100 + R)
    r, c = (R - 1, C - 1) if where == "last" else (0, 0)
    X[r, c] = -1000.0
    ws = torch.empty(fb.fp8rl_kv_workspace_bytes(R, C), dtype=torch.uint8, device="cuda")
    KVq, scale = fb.fp8rl_quant_kv_tensor(X.cuda(), workspace=ws)
    want_q, want_s = oracle.fp8_quant_tensor(synth.bf16_bits(X))
    assert bits_u32(host(scale))[0] == np.float32(want_s).view(np.uint32)
    assert np.array_equal(host(KVq), want_q)
    assert fb.fp8rl_check_device_error() == 0


KV_BATCH_CHUNKS = 4 * 1024    # 16-byte chunks per batch of the resident kernel (4 rounds of 1024 threads)


@pytest.mark.parametrize("R,C,where", [(9744, 1024, "last"), (20011, 1032, "first"), (20011, 1032, "last"),
                                       (32768, 1024, "smem"), (60000, 1024, "tmem"), (60000, 1024, "reread"),
                                       (60000, 1024, "last")])
def test_fp8_kv_tensor_quant_resident_path(cuda_lib, R, C, where):
    # Contiguous tensors above the one-pass size: one CTA per SM; the tensor's
    # batches of 4096 chunks are dealt to the CTAs in turn (CTA b takes batches
    # b, b + G, ...), and each CTA's first 7 stay on chip (4 in tensor memory,
    # then 3 in shared memory) between the amax and the encode; later ones are
    # read again.  On 152 SMs: 9744 x 1024 gives 2-3 batches per CTA, 20011 x
    # 1032 4-5 (ragged last batch), 32768 x 1024 6-7 (all on chip, read once),
    # 60000 x 1024 12-13 (5-6 read again).  The tensor amax sits in the first or
    # last value, or in a batch held in tensor memory, in shared memory or read
    # again.
    X = act_cpu(R, C, 9500 + R + C)
    G = torch.cuda.get_device_properties(0).multi_processor_count
    batch = {"first": 0, "last": None,
             "tmem": 1 * G + 5,            # CTA 5's second batch
             "smem": 5 * G + 7,            # CTA 7's sixth
             "reread": 9 * G + 3}[where]   # CTA 3's tenth
    total = R * (C // 8)
    chunk = total - 1 if batch is None else min(batch * KV_BATCH_CHUNKS + 1234, total - 1)
    e = chunk * 8 + 5
    X[e // C, e % C] = -1000.0
    ws = torch.empty(fb.fp8rl_kv_workspace_bytes(R, C), dtype=torch.uint8, device="cuda")
    KVq, scale = fb.fp8rl_quant_kv_tensor(X.cuda(), workspace=ws)
    want_q, want_s = oracle.fp8_quant_tensor(synth.bf16_bits(X))
    assert bits_u32(host(scale))[0] == np.float32(want_s).view(np.uint32)
    assert np.array_equal(host(KVq), want_q)
    assert fb.fp8rl_check_device_error() == 0


@pytest.mark.parametrize("kind", ["zeros", "tiny", "ties"])
def test_fp8_kv_tensor_quant_resident_path_special_values(cuda_lib, kind):
    # The resident path (40000 x 1024: 8-9 batches per CTA on 152 SMs, so
    # batches held in tensor memory, in shared memory and read again) on
    # special tensors: all zero with half the rows -0.0 (scale 1, codes 0x00
    # and 0x80); every value below 1e-37, bf16 subnormals among them (scale
    # below 2^-90: the encode takes the IEEE division); amax exactly 448
    # (scale 1) with rows of E4M3 ties and subnormal codes spread over the
    # tensor.
    R, C = 40000, 1024
    if kind == "zeros":
        X = torch.zeros(R, C, dtype=torch.bfloat16)
        X[1::2] = -0.0
    elif kind == "tiny":
        X = (act_cpu(R, C, 9700).float() * 1e-38).to(torch.bfloat16)
    else:
        X = act_cpu(R, C, 9701).float().clamp(-400.0, 400.0)
        ties = torch.tensor([448.0, 17.0, -18.0, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10, 1.5, -0.4375,
                             -2.0 ** -7, 2.0 ** -8 * 1.0625, 240.0, 232.0])
        for r in (0, R // 7, R // 3, R // 2, R - 1):
            X[r] = ties.repeat(C // ties.numel() + 1)[:C]
        X = X.to(torch.bfloat16)
    ws = torch.empty(fb.fp8rl_kv_workspace_bytes(R, C), dtype=torch.uint8, device="cuda")
    KVq, scale = fb.fp8rl_quant_kv_tensor(X.cuda(), workspace=ws)
    want_q, want_s = oracle.fp8_quant_tensor(synth.bf16_bits(X))
    if kind != "tiny":
        assert float(want_s) == 1.0
    else:
        assert float(want_s) < 2.0 ** -90
    assert bits_u32(host(scale))[0] == np.float32(want_s).view(np.uint32)
    assert np.array_equal(host(KVq), want_q)
    assert fb.fp8rl_check_device_error() == 0


@pytest.mark.parametrize("R,C,ld", [(9744, 1024, 1032), (20011, 1032, 1040)])
def test_fp8_kv_tensor_quant_strided_above_one_pass(cuda_lib, R, C, ld):
    # rows with a pitch, above the one-pass size: the three-launch path
    X = act_cpu(R, C, 9600 + R)
    X[R - 1, C - 1] = 2000.0
    wide = torch.zeros(R, ld, dtype=torch.bfloat16)
    wide[:, :C] = X
    ws = torch.empty(fb.fp8rl_kv_workspace_bytes(R, C), dtype=torch.uint8, device="cuda")
    KVq, scale = fb.fp8rl_quant_kv_tensor(wide.cuda()[:, :C], workspace=ws)
    want_q, want_s = oracle.fp8_quant_tensor(synth.bf16_bits(X))
    assert bits_u32(host(scale))[0] == np.float32(want_s).view(np.uint32)
    assert np.array_equal(host(KVq), want_q)
    assert fb.fp8rl_check_device_error() == 0


def test_fp8_kv_tensor_quant_reused_workspace_takes_no_stale_slot(cuda_lib):
    # the same workspace for a tensor with a large amax, then one with a small
    # amax: the second call's scale must come from its own slices only
    R, C = 4096, 1024
    ws = torch.empty(fb.fp8rl_kv_workspace_bytes(R, C), dtype=torch.uint8, device="cuda")
    big = act_cpu(R, C, 9201)
    big[R // 2, 7] = 3000.0
    small = act_cpu(R, C, 9202) * 0.01
    for X in (big, small, big, small):
        KVq, scale = fb.fp8rl_quant_kv_tensor(X.cuda(), workspace=ws)
        want_q, want_s = oracle.fp8_quant_tensor(synth.bf16_bits(X))
        assert bits_u32(host(scale))[0] == np.float32(want_s).view(np.uint32)
        assert np.array_equal(host(KVq), want_q)
    assert fb.fp8rl_check_device_error() == 0


@pytest.mark.parametrize("R", [4096, 16384])
def test_fp8_kv_tensor_quant_graph_replays_recalibrate(cuda_lib, R):
    # one call captured in a CUDA graph (4096 x 1024: the one-pass kernel;
    # 16384 x 1024: one CTA per SM, partly on chip), replayed after new data is copied into its
    # input: every replay recalibrates the scale from that data (the one-pass
    # call's tag advances on the device, so a replay never accepts a slot left
    # by the one before), checked against the oracle each time
    C = 1024
    X = torch.empty(R, C, dtype=torch.bfloat16, device="cuda")
    KVq = torch.empty(R, C, dtype=torch.uint8, device="cuda")
    scale = torch.empty(1, dtype=torch.float32, device="cuda")
    ws = torch.empty(fb.fp8rl_kv_workspace_bytes(R, C), dtype=torch.uint8, device="cuda")
    inputs = []
    for i, (gain, r, c, v) in enumerate([(1.0, 7, 3, 900.0), (0.01, R - 1, C - 1, -0.5),
                                         (1.0, R // 2, 100, 2500.0), (0.001, 0, 0, 0.0)]):
        h = act_cpu(R, C, 9300 + i) * gain
        h[r, c] = v
        inputs.append(h)
    X.copy_(inputs[0])
    fb.fp8rl_quant_kv_tensor(X, KVq, scale, workspace=ws)          # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fb.fp8rl_quant_kv_tensor(X, KVq, scale, workspace=ws)
    for h in inputs + inputs[::-1]:
        X.copy_(h)
        g.replay()
        torch.cuda.synchronize()
        want_q, want_s = oracle.fp8_quant_tensor(synth.bf16_bits(h))
        assert bits_u32(host(scale))[0] == np.float32(want_s).view(np.uint32)
        assert np.array_equal(host(KVq), want_q)
    assert fb.fp8rl_check_device_error() == 0


def test_fp8_kv_tensor_quant_workspace_reused_across_paths(cuda_lib):
    # one workspace for a three-launch call (rows with a pitch; its partials
    # follow the header word), one-pass calls and calls of one CTA per SM (the
    # last two share the header word's tags): each bit-exact
    C = 1024
    ws = torch.empty(fb.fp8rl_kv_workspace_bytes(16384, C), dtype=torch.uint8, device="cuda")
    for R, seed, ld in [(16384, 9401, 1040), (4096, 9402, C), (16384, 9406, C), (2048, 9403, C),
                        (16384, 9404, 1040), (16384, 9407, C), (4096, 9405, C)]:
        X = act_cpu(R, C, seed)
        wide = torch.zeros(R, ld, dtype=torch.bfloat16)
        wide[:, :C] = X
        KVq, scale = fb.fp8rl_quant_kv_tensor(wide.cuda()[:, :C], workspace=ws)
        want_q, want_s = oracle.fp8_quant_tensor(synth.bf16_bits(X))
        assert bits_u32(host(scale))[0] == np.float32(want_s).view(np.uint32)
        assert np.array_equal(host(KVq), want_q)
    assert fb.fp8rl_check_device_error() == 0
