"""Host-side pieces of the benchmark, no GPU.

The roofline's numerator: the bytes one decode step must move, counted by
hand for the Llama-1B and Llama-8B shapes and compared with the benchmark's
count (weights, norm gains, the LM head, one embedding row per sequence, and
the KV read over slots 0..pos of every layer and sequence — the minimal
bytes that "9 · Quand ne pas le faire", §9.1, asks to count). And the clock
record of the timed region: the throttle reasons that void a measurement
are read from the sampled lines."""
import bench
from decode_megakernel_03_gb300 import synth


def test_llama1b_bytes_by_hand():
    # per layer: Wq 2048x2048, Wk and Wv 512x2048, Wo 2048x2048, gate/up/down
    # 8192x2048 each, two norm gains of 2048; bf16 = 2 bytes
    layer = 2 * (2048 * 2048 + 2 * 512 * 2048 + 2048 * 2048 + 3 * 8192 * 2048 + 2 * 2048)
    assert layer == 121_643_008
    # 16 layers, the final norm, the tied LM head (the embedding, 128256 rows),
    # one embedding row for the one sequence
    weights = 16 * layer + 2 * 2048 + 2 * 128256 * 2048 + 2 * 2048
    assert weights == 2_471_632_896
    # KV: 16 layers x (k, v) x 8 kv-heads x 64 dims x 2 bytes per position
    per_pos = 16 * 2 * 8 * 64 * 2
    assert per_pos == 32_768
    w, kv = bench.algorithmic_bytes(synth.LLAMA_1B, 1, [512])
    assert w == weights
    assert kv == per_pos * 513  # slots 0..512, the new one included


def test_llama8b_and_batch_bytes_by_hand():
    # 8B shape: hidden 4096, 32 heads of 128 (8 kv-heads), ffn 14336, untied
    layer = 2 * (4096 * 4096 + 2 * 1024 * 4096 + 4096 * 4096 + 3 * 14336 * 4096 + 2 * 4096)
    weights = 32 * layer + 2 * 4096 + 2 * 128256 * 4096 + 2 * 4096
    w, kv = bench.algorithmic_bytes(synth.LLAMA_8B, 1, [2048])
    assert w == weights
    assert kv == 32 * 2 * 8 * 128 * 2 * 2049
    # batch: one embedding row and one KV range per sequence; weights once
    w8, kv8 = bench.algorithmic_bytes(synth.LLAMA_1B, 8, [100 + b for b in range(8)])
    w1, _ = bench.algorithmic_bytes(synth.LLAMA_1B, 1, [0])
    assert w8 == w1 + 7 * 2 * 2048
    assert kv8 == 32_768 * sum(101 + b for b in range(8))


def test_clock_record_reads_the_throttle_reasons():
    c = bench.ClockSampler()
    # index, clocks.sm, clocks.max.sm, power.draw, reasons.active, then
    # hw_slowdown, hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap
    c.lines = ["0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
               "0, 1995, 2070, 1390.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
               "0, 2070, 2070, 1200.0, 0x0000000000000008, Active, Not Active, Not Active, Not Active",
               "garbled line"]
    s = c.summary()
    assert s["samples"] == 3
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert bench.ClockSampler().summary()["reasons"] == ["unsampled"]
