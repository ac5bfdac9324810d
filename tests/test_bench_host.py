"""CPU checks of bench.py's host-side bookkeeping: the algorithmic bytes its
GB/s figures divide by, the input copies that keep a timed pass above L2, the
keys that tie recorded ncu traffic to a kernel's source, the clock summary and
the oracle sample's fractions."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from precision_rl_rollout_gb300 import synth  # noqa: E402


def test_7b_decode_step_bytes():
    # per layer: requant 3 B/element + 4 B/block, act quant 3 B/element + 4 B/group,
    # GEMM e4m3 W + scales + e4m3 X + scales + bf16 Y; the 7B set at 64 tokens
    total = 0
    for s in synth.QWEN25_7B:
        blocks = (s.N // 128) * (s.K // 128)
        total += 3 * s.N * s.K + 4 * blocks
        total += 3 * 64 * s.K + 4 * 64 * (s.K // 128)
        total += s.N * s.K + 4 * blocks + 64 * s.K + 4 * 64 * (s.K // 128) + 2 * 64 * s.N
    assert bench.step_bytes(synth.QWEN25_7B, 64) == total == 946375808


def test_headline_step_bytes_and_flops():
    # 64 layers of the four 32B weights requantized (3 B/value + 4 B/block), the
    # four [8192, K] inputs quantized, the four M = 8192 GEMMs
    p = bench.model_step_parts()
    elems = sum(s.N * s.K for s in synth.QWEN25_32B)
    blocks = sum((s.N // 128) * (s.K // 128) for s in synth.QWEN25_32B)
    assert elems == 487587840 and blocks == 29760
    assert p["requant_bytes"] == 64 * (3 * elems + 4 * blocks) == 93624483840
    M = 8192
    assert p["act_quant_bytes"] == sum(3 * M * s.K + 4 * M * (s.K // 128) for s in synth.QWEN25_32B)
    assert p["gemm_flops"] == 2 * M * elems
    assert p["gemm_bytes"] == sum(s.N * s.K + 4 * (s.N // 128) * (s.K // 128) + M * s.K + 4 * M * (s.K // 128)
                                  + 2 * M * s.N for s in synth.QWEN25_32B)
    assert bench.model_step_bytes() == p["requant_bytes"] + p["act_quant_bytes"] + p["gemm_bytes"]


def test_int8_gemm_bytes():
    assert bench.int8_gemm_bytes(32, 7168, 5120) == 7168 * 5120 + 4 * 7168 + 32 * 5120 + 4 * 32 + 2 * 32 * 7168


def test_copies_exceed_three_l2():
    for n in (1, 16 << 20, 100 << 20, 500 << 20, 5 << 30):
        c = bench._copies_for(n)
        assert c >= 2 and c * n >= 3 * bench.L2_BYTES


def test_traffic_key_follows_the_requant_section_only():
    csrc = os.path.join(ROOT, "precision_rl_rollout_gb300", "csrc")
    quant = open(os.path.join(csrc, "quant.cu"), "rb").read()
    common = open(os.path.join(csrc, "common.cuh"), "rb").read()
    base = bench.requant_source_sha1(quant, common)
    assert base == bench.requant_source_sha1()
    act = quant.index(b"// ---------------------------------------------------------------- FP8 activations")
    # an edit after the weight section (another quantizer) keeps the key
    assert bench.requant_source_sha1(quant + b"\n// tail edit\n", common) == base
    after = quant.index(b"\n", act) + 1                    # the line after the activation header
    assert bench.requant_source_sha1(quant[:after] + b"// x\n" + quant[after:], common) == base
    # an edit inside the weight section, or to common.cuh, changes it
    w = quant.index(b"quant_weight_block_kernel")
    assert bench.requant_source_sha1(quant[:w] + b" " + quant[w:], common) != base
    assert bench.requant_source_sha1(quant, common + b"\n") != base
    # the recorded traffic is reported exactly when the key matches, scaled by the values processed
    t = bench.traffic_or_null(1000)
    assert (t is not None) == (bench.NCU_TRAFFIC["source_sha1"] == base)
    if t is not None:
        assert t == bench.NCU_TRAFFIC["bytes_per_value"] * 1000


def test_clock_summary():
    lines = ["0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "0, 1965, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
             "0, 2070, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "garbage"]
    s = bench.summarize_clocks(lines)
    assert s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_csv_is_not_written_into_the_repository():
    c = bench.ClockSampler(0, 0)
    assert not os.path.abspath(c.path).startswith(ROOT + os.sep)


def test_step_percentiles():
    p = bench.step_percentiles([5.0, 1.0, 3.0, 2.0, 4.0])
    assert p == {"p10": 1.4, "p50": 3.0, "p90": 4.6, "n": 5}
    assert bench.step_percentiles([]) is None
    one = bench.step_percentiles([7.0])
    assert one["p10"] == one["p50"] == one["p90"] == 7.0
