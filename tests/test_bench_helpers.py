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
