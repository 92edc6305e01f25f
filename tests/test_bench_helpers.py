"""Host-side helpers of bench.py that run without a GPU."""
import numpy as np

import bench
from transformer_esm_layer_gb300 import synth


def test_cpu_oracle_train_sample_covers_whole_sequences():
    wl = synth.make_workload("tiny_fp32")
    w = synth.model_weights(wl.geometry, wl.seed, "fp32")
    toks, dt, done = bench.cpu_oracle_train_sample(wl, bench.f64_weights(w), 0.0)
    assert done == [0] and toks == wl.lengths[0] and dt > 0
    toks, dt, done = bench.cpu_oracle_train_sample(wl, bench.f64_weights(w), 1e9)
    assert done == list(range(len(wl.lengths))) and toks == int(np.sum(wl.lengths))


def test_fp4_workload_and_layer_override():
    """The NVFP4 3B workload is the FP8 one (same model, batch and seed) with every layer in
    FP4; a smaller layer count for a profiler case keeps the per-layer list in step."""
    fp8, fp4 = synth.make_workload("esm3b_fp8"), synth.make_workload("esm3b_fp4")
    assert fp4.lengths == fp8.lengths and fp4.seed == fp8.seed and fp4.precision == fp8.precision == "fp8"
    assert fp8.layer_precision is None and fp4.layer_precision == ["fp4"] * fp4.geometry.num_layers
    wl = bench.workload_for_rank(0, 8192, 1, "esm3b_fp4")
    assert wl.geometry.num_layers == 1 and wl.layer_precision == ["fp4"] and wl.total_tokens == 8192
    assert "NVFP4" in bench.workload_text(wl)
    assert bench.workload_for_rank(0, None, 3, "esm650m").layer_precision is None
