"""CPU checks of bench.py's bookkeeping: peaks, algorithmic bytes, traffic
lookup and launch counts (no GPU, no timing)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from bidirectional_masked_linear_gb300 import synth  # noqa: E402


def test_peaks_fall_back_without_measurements():
    hbm, bf16, src = bench._peaks()
    assert hbm > 0 and bf16 > 0 and src in ("measured", "fallback")


def test_algorithmic_bytes_vit_b():
    w = synth.WORKLOADS["vit_b"]
    # 3 bf16 inputs + fp32 output per (token, head, feature), plus the LION-S decays
    assert bench.algorithmic_bytes(w, "s") == w.B * w.H * w.L * (644)
    assert bench.algorithmic_bytes(w, "lit") == w.B * w.H * w.L * 640
    # bf16 output: 2 bytes instead of 4 per output value
    assert bench.algorithmic_bytes(w, "s", out_bytes=2) == w.B * w.H * w.L * 516


def test_traffic_is_null_for_unknown_kernels():
    w = synth.WORKLOADS["vit_b"]
    assert bench.traffic_bytes(w, "s", 32) == (None, None)
    t, per = bench.traffic_bytes(w, "s", 128)
    assert t is None or (t > 0 and abs(sum(per.values()) - t) < 1)


def test_traffic_covers_every_kernel_of_the_call(monkeypatch):
    """The long path's figure is the sum over its two kernels (pre-pass and
    main pass), and one kernel without a capture at its current sources makes
    the whole figure null."""
    w = synth.WORKLOADS["hires_2496"]
    kernels = bench._CALL_KERNELS[(128, True)]
    assert len(kernels) == 2
    table = {(name, bench._sources_sha(files), w.name, "s", 128): 1000.0 * (n + 1)
             for n, (name, files) in enumerate(kernels.items())}
    monkeypatch.setattr(bench, "TRAFFIC_PER_HEAD", table)
    t, per = bench.traffic_bytes(w, "s", 128)
    assert t == 3000.0 * w.B * w.H and len(per) == 2
    table.pop(next(iter(table)))
    assert bench.traffic_bytes(w, "s", 128) == (None, None)


def test_launch_counts():
    vit = synth.WORKLOADS["vit_b"]
    hires = synth.WORKLOADS["hires_2496"]
    assert bench.kernels_per_call("chunk", 128, vit) == 1
    assert bench.kernels_per_call("chunk", 64, vit) == 1
    assert bench.kernels_per_call("chunk", 64, hires) == 3
    assert bench.kernels_per_call("chunk", 128, hires) == 2   # the main pass chains the segments
    # every head one segment (B*H at least the SMs, or fewer heads than half
    # the SMs can split): pre-pass and main pass, no segment scan
    assert bench.long_segments(hires, 152) == 6
    assert bench.long_segments(synth.WORKLOADS["bert_large"], 152) == 1
    assert bench.long_segments(synth.WORKLOADS["lra_4096"], 152) == 1
    assert bench.kernels_per_call("chunk", 128, synth.WORKLOADS["bert_large"]) == 2
    assert bench.kernels_per_call("chunk", 128, synth.WORKLOADS["lra_4096"]) == 2
    assert bench.kernels_per_call("chunk", 64, synth.WORKLOADS["lra_4096"]) == 2
    assert bench.kernels_per_call("chunk", 64, hires) == 3
    assert bench.kernels_per_call("chunk", 32, hires) == 1
    # features, the column CTAs, and with few heads the combination of the
    # two sweeps run apart
    assert bench.kernels_per_call("rnn", 0, hires) == 3
    assert bench.kernels_per_call("rnn", 0, vit) == 2
    assert bench.kernels_per_call("rnn", 0, synth.WORKLOADS["lra_4096"]) == 2
    assert bench.kernels_per_call("rnn", 0, synth.WORKLOADS["tiny_d_fp32"]) == 2   # 64 tokens
    assert bench.kernels_per_call("full", 0, vit, "s") == 3   # prefix, features, the tiled pass
    assert bench.kernels_per_call("full", 0, vit, "d") == 2
    assert bench.kernels_per_call("full", 0, synth.WORKLOADS["tiny_d_fp32"], "d") == 1


def test_traffic_keys_follow_the_kernel_that_runs():
    # every sources list names files that exist, so a hash can be taken
    shas = set()
    for key, kernels in bench._CALL_KERNELS.items():
        for name, files in kernels.items():
            for rel in files:
                assert os.path.exists(os.path.join(ROOT, rel)), (key, name, rel)
            shas.add(bench._sources_sha(files))
    assert len(shas) == 3


def test_config_lines_cover_the_scope_configurations():
    """Every configuration's workload, mask, form and chunk length has a line
    (the headline ViT-B LION-S chunk 128 is measured separately)."""
    lines = set(bench.CONFIG_LINES)
    assert ("tiny_d_fp32", "d", "chunk", 16) in lines
    assert ("vit_t_s", "s", "chunk", 64) in lines
    for m in ("lit", "d", "s"):
        assert ("vit_b", m, "full", 0) in lines
        for c in (32, 64, 128):
            assert ("vit_b", m, "chunk", c) in lines
    for m in ("d", "s"):
        for c in (64, 128):
            assert ("bert_large", m, "chunk", c) in lines
        assert ("hires_2496", m, "rnn", 0) in lines and ("hires_2496", m, "chunk", 128) in lines
    for name, *_ in lines:
        assert name in synth.WORKLOADS


def test_oracle_baseline_forms():
    """The CPU baseline times the brute force on the ViT-length workloads and
    the recurrent form on the longer ones, as the measurement plan names."""
    assert "brute-force" in bench._oracle_sample("tiny_d_fp32", "d", 0.0, 1)["sample"]
    assert "recurrent" in bench._oracle_sample("bert_large", "s", 0.0, 1)["sample"]


def test_backward_flops_and_peak():
    w = synth.WORKLOADS["vit_b"]
    # six L x L x d products of 2 L^2 d flops per head
    assert bench.bwd_flops(w) == 6 * 2 * w.B * w.H * w.L ** 2 * w.d
    assert abs(bench.FP32_ALU_PEAK_TFLOPS - 80.54) < 0.01


def test_backward_launch_counts():
    # phi, rows, columns; + dl (D, S); + batch sum (D); + prefix (S, tiled d >= 64)
    assert bench.bwd_launches("lit", 64) == 3
    assert bench.bwd_launches("d", 64) == 5
    assert bench.bwd_launches("s", 64) == 5
    assert bench.bwd_launches("s", 32) == 4
    assert bench.bwd_launches("d", 16) == 5


def test_stream_bytes():
    # ViT-B heads, d = 64: S and z read and written in fp32, bf16 q, k, v in
    assert bench.stream_bytes(64, 12, 64) == 64 * 12 * (2 * (64 * 64 + 64) * 4 + 3 * 64 * 2 + 4 + 64 * 4 + 4)


def test_reordered_flops_launches_and_orders():
    w = synth.WORKLOADS["vit_b"]
    assert bench.reorder_flops(w) == 2 * 2 * w.B * w.H * w.L ** 2 * w.d
    assert bench.reorder_launches("s") == 4 and bench.reorder_launches("d") == 3
    o = bench.vit_grid_orders(197)
    assert tuple(o.shape) == (2, 197)
    for row in o:   # permutations, class token first
        assert sorted(row.tolist()) == list(range(197)) and int(row[0]) == 0
    assert o[1, 1:15].tolist() == [1 + 14 * r for r in range(14)]   # first column of the grid
    r = bench.vit_grid_orders(11)   # not 1 + a square: identity and reversal
    assert r[1].tolist() == list(range(10, -1, -1))

