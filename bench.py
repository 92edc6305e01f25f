#!/usr/bin/env python
"""Throughput of the ESM-2 650M packed encoder forward on GB300.

One step = one full forward (embedding, 33 layers, final LayerNorm) over a packed batch
of 16384 tokens (47 sequences, log-normal lengths, seed 2) already resident in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torchrun: one global batch of N x 16384 tokens is split across the ranks
by work (the sequences of a packed batch are independent, so ranks need no data
exchange); value = all tokens / max-over-ranks time.  Rank 0 prints one JSON line.  --impl reference times
the float64 CPU oracle on the host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "ESM-2 650M packed fwd tokens/s on 1 GB300; achieved TFLOP/s vs dense BF16 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-train", action="store_true", help="skip the training-step measurement")
    ap.add_argument("--no-configs", action="store_true", help="skip the other configured workloads (tiny fp32, one "
                                                               "650M layer, padded 650M, 3B FP8)")
    ap.add_argument("--no-graph", action="store_true", help="launch the kernels eagerly instead of replaying "
                                                             "one captured CUDA graph per step")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target CPU time of the oracle sample")
    ap.add_argument("--layers", type=int, default=None, help="fewer layers: small case for profiler captures only")
    ap.add_argument("--tokens", type=int, default=None, help="other batch size: small case for captures only")
    ap.add_argument("--workload", choices=("esm650m", "esm650m_padded", "esm3b_fp8", "esm3b_fp4"), default="esm650m",
                    help="esm650m (the headline), esm650m_padded (same sequences as [B,1024] with a key padding "
                         "mask), esm3b_fp8 (3B encoder, E4M3 GEMMs, 32768 tokens), esm3b_fp4 (the same with NVFP4 "
                         "GEMMs in every layer)")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload_for_rank(rank: int, tokens=None, layers=None, name: str = "esm650m"):
    import dataclasses
    from transformer_esm_layer_gb300 import synth
    wl = synth.make_workload(name)
    default_T = wl.total_tokens
    tokens = default_T if tokens is None else tokens
    if rank > 0 or tokens != default_T:  # another batch with the same length distribution
        rng = np.random.default_rng([wl.seed, rank, tokens])
        wl.lengths = synth.lognormal_lengths(rng, total=tokens)
        wl.seed = wl.seed * 1000 + rank
    if layers is not None and layers != wl.geometry.num_layers:
        wl.geometry = dataclasses.replace(wl.geometry, num_layers=layers)
        if wl.layer_precision:
            wl.layer_precision = [wl.layer_precision[i % len(wl.layer_precision)] for i in range(layers)]
    return wl


def workload_text(wl) -> str:
    g = wl.geometry
    size = {2560: "ESM-2 3B", 1280: "ESM-2 650M"}.get(g.hidden, "tiny ESM-style")
    prec = {"fp8": "E4M3 GEMMs with per-tensor delayed scaling (history 16)", "fp32": "fp32"}.get(wl.precision, "bf16")
    if wl.layer_precision and set(wl.layer_precision) == {"fp4"}:
        prec = ("NVFP4 GEMMs (E2M1 values, E4M3 scale per 16, per-tensor current scaling) in every layer, "
                "bf16 attention and LayerNorm")
    lengths = (f"lengths {list(wl.lengths)}" if len(wl.lengths) <= 4 else
               "log-normal lengths (median 300, sigma 0.6) clipped to [32,1024]")
    txt = (f"{wl.name}: {size} encoder ({g.num_layers} layers, hidden {g.hidden}, {g.heads} heads, FFN {g.ffn}, "
           f"vocab 33), {prec}, weights N(0,0.02), {wl.total_tokens} tokens in {len(wl.lengths)} sequences, "
           f"{lengths}, seed {wl.seed}" + ("" if wl.final_ln else ", no final LayerNorm"))
    if wl.padded_len:
        txt += f"; padded layout [{len(wl.lengths)}, {wl.padded_len}] with a key padding mask"
    else:
        txt += "; packed (THD)"
    return txt


def algorithmic_flops(wl):
    """FLOPs one forward must do: per layer 2T(4d^2 + 2df) in the four linear maps plus
    4 d sum(L_i^2) in attention (QK^T and PV over each sequence only)."""
    g = wl.geometry
    T, d, f = wl.total_tokens, g.hidden, g.ffn
    L2 = float(np.sum(np.asarray(wl.lengths, np.float64) ** 2))
    per_class = {"gemm_qkv": 2.0 * T * 3 * d * d, "gemm_oproj": 2.0 * T * d * d, "gemm_fc1": 2.0 * T * f * d,
                 "gemm_fc2": 2.0 * T * d * f, "attention": 4.0 * d * L2}
    return {k: v * g.num_layers for k, v in per_class.items()}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms in the background."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "200"]
        if gpu_id:
            cmd += ["-i", gpu_id]
        try:
            self.p = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.flush()
        with open(self.f.name) as fh:
            rows = [r.strip().split(", ") for r in fh if r.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            if len(r) < 8:
                continue
            try:
                sm.append(float(r[0]))
                mx.append(float(r[1]))
            except ValueError:
                continue
            for n, v in zip(names, r[4:8]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def gemm_traffic_record():
    """DRAM bytes per GEMM launch from the committed ncu summary, if it was taken on the
    current GEMM source (null otherwise)."""
    p = os.path.join(ROOT, "profiles", "gemm_tc_dram_traffic.json")
    src = os.path.join(ROOT, "transformer_esm_layer_gb300", "csrc", "gemm_tc.cu")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    with open(src, "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()[:16]
    return rec if rec.get("gemm_tc_sha256_16") == h else None


def cpu_oracle_sample(wl, w64, seconds: float, prec: str = "bf16", enc=None):
    """Time the float64 oracle on whole sequences of the workload until `seconds` pass
    (for FP8 with the scales the GPU path holds, read back through the C ABI)."""
    from oracle import esm_oracle as O
    from transformer_esm_layer_gb300 import synth
    tok = synth.workload_tokens(wl)
    cu = O.cu_seqlens(wl.lengths)
    kw = {}
    if prec == "fp8" and enc is not None:
        sc = enc.fp8_scales()
        kw["fp8_state"] = [{k: float(sc[l, i]) for i, k in enumerate(O.FP8_TENSORS)} for l in range(sc.shape[0])]
        if wl.layer_precision and "fp4" in wl.layer_precision:
            s4 = enc.fp4_scales()  # the last forward's scales: the whole batch's amaxes
            kw["fp4_state"] = [({k: float(s4[l, i]) for i, k in enumerate(O.FP8_TENSORS)} if p == "fp4" else None)
                               for l, p in enumerate(wl.layer_precision)]
    done, toks = [], 0
    t0 = time.perf_counter()
    for i in range(len(wl.lengths)):
        O.encode_sequence(tok[cu[i]:cu[i + 1]], w64, wl.geometry.heads, final_ln=True, **kw)
        done.append(i)
        toks += wl.lengths[i]
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return toks, dt, done


def cpu_oracle_train_sample(wl, w64, seconds: float, seed: int = 0):
    """Time the float64 oracle's training step (forward recomputed, then every gradient) on
    whole sequences of the workload, with a seeded dL/d(output), until `seconds` pass."""
    from oracle import backward as B
    from oracle import esm_oracle as O
    from transformer_esm_layer_gb300 import synth
    tok = synth.workload_tokens(wl)
    cu = O.cu_seqlens(wl.lengths)
    rng = np.random.default_rng(seed)
    done, toks = [], 0
    t0 = time.perf_counter()
    for i in range(len(wl.lengths)):
        L = int(wl.lengths[i])
        B.encode_sequence_backward(tok[cu[i]:cu[i + 1]], w64, wl.geometry.heads,
                                   rng.standard_normal((L, wl.geometry.hidden)), final_ln=True)
        done.append(i)
        toks += L
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return toks, dt, done


def f64_weights(w):
    return {"emb": np.asarray(w["emb"], np.float64),
            "layers": [{k: np.asarray(v, np.float64) for k, v in l.items()} for l in w["layers"]],
            "lnf_g": np.asarray(w["lnf_g"], np.float64), "lnf_b": np.asarray(w["lnf_b"], np.float64)}


def run_reference(args):
    """The float64 oracle on the host cores: each step encodes one whole sequence of the
    workload (cycling through them in order)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from oracle import esm_oracle as O
    from transformer_esm_layer_gb300 import synth
    wl = workload_for_rank(0)
    w = f64_weights(synth.model_weights(wl.geometry, wl.seed, "bf16"))
    tok = synth.workload_tokens(wl)
    cu = O.cu_seqlens(wl.lengths)
    B = len(wl.lengths)
    for s in range(args.warmup):
        i = s % B
        O.encode_sequence(tok[cu[i]:cu[i + 1]], w, wl.geometry.heads, final_ln=True)
    toks, t = 0, 0.0
    for s in range(args.steps):
        i = (args.warmup + s) % B
        t0 = time.perf_counter()
        O.encode_sequence(tok[cu[i]:cu[i + 1]], w, wl.geometry.heads, final_ln=True)
        t += time.perf_counter() - t0
        toks += wl.lengths[i]
    value = toks / t
    cores = len(os.sched_getaffinity(0))
    sample = f"one whole sequence per step, cycling through the {B} sequences of the workload (seed 2); {toks} tokens timed"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "esm650m", "tokens_per_step": f"{toks / args.steps:.0f} (mean)"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def _timed_replays(step, steps, stream):
    """Time `steps` calls of step() with one CUDA event between consecutive calls (on the
    launching stream): returns the per-step durations in ms and their sum."""
    import torch
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record(stream)
    for i in range(steps):
        step()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    return per, ev[0].elapsed_time(ev[-1])


def attention_roofline(wl, ms_per_step, executed_flops, pk, clock_mhz, num_sms):
    """The attention kernel against its three ceilings: tensor (bf16 MMA FLOPs), the
    exponential unit (one 2^x per score; 32 results per SM per clock, the ex2.approx.f32
    rate measured on GB300 with a throughput probe) and HBM (Q, K, V read once and O
    written once)."""
    g = wl.geometry
    L2 = float(np.sum(np.asarray(wl.lengths, np.float64) ** 2))
    T = wl.total_tokens
    exps = L2 * g.heads * g.num_layers
    bytes_ = T * 4.0 * g.hidden * 2 * g.num_layers
    sec = ms_per_step / 1e3
    clock = clock_mhz if clock_mhz else float(pk.get("sm_max_mhz", 2070.0))
    exp_peak = 32.0 * num_sms * clock * 1e6
    return {"kernel": "attention_tc_kernel (tcgen05, bf16)", "ms_per_step": ms_per_step,
            "tensor": {"achieved_tflops": executed_flops / sec / 1e12, "peak": float(pk["bf16_tflops"]),
                       "frac": executed_flops / sec / 1e12 / float(pk["bf16_tflops"]),
                       "flops_per_step": executed_flops, "peak_source": "bf16_tflops (burst), measured"},
            "exp_unit": {"achieved_per_s": exps / sec, "peak_per_s": exp_peak, "frac": exps / sec / exp_peak,
                         "exps_per_step": exps,
                         "peak_source": f"32 per SM per clock (measured ex2.approx.f32 rate) x {num_sms} SMs x "
                                        f"{clock:.0f} MHz (sampled median)"},
            "hbm": {"achieved_gbs": bytes_ / sec / 1e9, "peak": float(pk["hbm_gbs"]),
                    "frac": bytes_ / sec / 1e9 / float(pk["hbm_gbs"]), "bytes_per_step": bytes_}}


def measure_forward(wl, dev, args, w_np=None, want_e2e=False, world=1, rank=0, global_tokens=None,
                    tok_np=None, clock_sampler=None):
    """One workload's forward: warm-up, CUDA-graph capture, `args.steps` timed replays with an
    event between replays (median / min / mean), then an eager pass with the library's
    per-kernel event profile.  Returns (result dict, state for the headline's extra legs)."""
    import torch
    import torch.distributed as dist

    from transformer_esm_layer_gb300 import synth
    from transformer_esm_layer_gb300.binding import DeviceWeights, EsmEncoder, packed_inputs

    g = wl.geometry
    prec = wl.precision
    padded = wl.padded_len is not None
    if w_np is None:
        w_np = synth.model_weights(g, wl.seed, prec)
    dw = DeviceWeights(w_np, prec, device=dev)
    if tok_np is None:
        tok_np = synth.workload_tokens(wl)
    global_tokens = wl.total_tokens if global_tokens is None else global_tokens
    tok, cu = packed_inputs(tok_np, wl.lengths, device=dev)
    T, B, maxL = wl.total_tokens, len(wl.lengths), max(wl.lengths)
    enc = EsmEncoder.from_geometry(g, prec, final_ln=wl.final_ln)
    fp4 = bool(wl.layer_precision) and set(wl.layer_precision) == {"fp4"}
    if wl.layer_precision:
        enc.set_layer_precision(list(wl.layer_precision))
    stream = torch.cuda.current_stream()
    torch.cuda.reset_peak_memory_stats(dev)
    if padded:
        S = wl.padded_len
        tok_pad = torch.from_numpy(synth.pad_tokens(tok_np, wl.lengths, S)).to(dev)
        lens_dev = torch.tensor(wl.lengths, dtype=torch.int32, device=dev)
        ws = enc.workspace(B * S, B, dev)
        out = torch.empty(B, S, g.hidden, dtype=enc.out_dtype, device=dev)

        def eager_step(st=stream):
            enc.forward_padded(dw, tok_pad, lens_dev, out=out, workspace=ws, stream=st)
    else:
        ws = enc.workspace(T, B, dev)
        out = torch.empty(T, g.hidden, dtype=enc.out_dtype, device=dev)

        def eager_step(st=stream):
            enc.forward(dw, tok, cu, maxL, out=out, workspace=ws, stream=st)

    # FP8 delayed scaling needs a full amax history before timing
    for _ in range(max(args.warmup, 3, 16 if prec == "fp8" else 0)):
        eager_step()
    enc.check(stream)
    step = eager_step
    launches_per_step = None
    if not args.no_graph:
        # one step = one replay of the captured forward (all of its kernels, same work)
        graph = torch.cuda.CUDAGraph()
        enc.get_profile(reset=True)
        with torch.cuda.graph(graph):
            eager_step(None)  # None: the capturing stream torch makes current
        launches_per_step = enc.get_profile(reset=True)["total_launches"]
        graph.replay()
        torch.cuda.synchronize()
        enc.check(stream)

        def step():
            graph.replay()

    # ---------------------------------------------------------------- timed region
    enc.get_profile(reset=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = clock_sampler() if clock_sampler else None
    if sampler:
        time.sleep(0.4)
    per, total_ms = _timed_replays(step, args.steps, stream)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    launches = enc.get_profile(reset=True)["total_launches"]
    if launches_per_step is not None:  # graph replays do not pass through the library
        launches = launches_per_step * args.steps
    enc.check(stream)
    ms = total_ms
    if world > 1:
        t = torch.tensor([ms], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    ms_step = ms / args.steps
    peak_mem = torch.cuda.max_memory_allocated(dev)

    # ---------------------------------------------------------------- per-kernel device times
    enc.set_profiling(True)
    prof_steps = min(args.steps, 10)
    for _ in range(prof_steps):
        eager_step()
    prof = enc.get_profile(reset=True)
    enc.set_profiling(False)
    flops = algorithmic_flops(wl)
    total_flops = sum(flops.values())
    executed = dict(flops)
    if padded:  # the GEMMs run over all B*S rows, attention over every query row of each row
        rows = B * wl.padded_len
        for c_ in ("gemm_qkv", "gemm_oproj", "gemm_fc1", "gemm_fc2"):
            executed[c_] = flops[c_] * rows / T
        executed["attention"] = 4.0 * g.hidden * wl.padded_len * float(np.sum(wl.lengths)) * g.num_layers
    pk, pk_src = peaks()
    gemm_classes = ("gemm_qkv", "gemm_oproj", "gemm_fc1", "gemm_fc2")
    per_kernel = {c_: {"ms_per_step": prof[c_]["ms"] / prof_steps,
                       "launches_per_step": prof[c_]["launches"] / prof_steps}
                  for c_ in ("gemm_qkv", "attention", "gemm_oproj", "gemm_fc1", "gemm_fc2", "layernorm", "other")}
    for c_ in list(gemm_classes) + ["attention"]:
        m_ = per_kernel[c_]["ms_per_step"]
        per_kernel[c_]["tflops"] = executed[c_] / (m_ / 1e3) / 1e12 if m_ else None
    # a contraction takes the peak of its own dtype: E4M3 = 2 x the measured bf16 (nominal 4.5 / 2.25),
    # NVFP4 = 6 x (nominal 13.5 / 2.25)
    dtype_mult = 6.0 if fp4 else (2.0 if prec == "fp8" else 1.0)
    peak_note = {6.0: " x 6 (NVFP4/bf16 nominal ratio)", 2.0: " x 2 (E4M3/bf16 nominal ratio)", 1.0: ""}[dtype_mult]
    peak_burst = float(pk["bf16_tflops"]) * dtype_mult
    peak_sust = float(pk["bf16_tflops_sustained"]) * dtype_mult
    roofline = None
    attn = None
    if prec != "fp32":
        gemm_ms = sum(prof[c_]["ms"] for c_ in gemm_classes) / prof_steps
        gemm_launches = sum(prof[c_]["launches"] for c_ in gemm_classes) / prof_steps
        gemm_flops = sum(executed[c_] for c_ in gemm_classes)
        gemm_tflops = gemm_flops / (gemm_ms / 1e3) / 1e12
        traffic = gemm_traffic_record()
        kname = ("gemm_nvfp4_kernel (tcgen05 block-scaled E2M1, all four linear maps; the operand "
                 "quantisation kernels are timed under 'other')" if fp4 else
                 f"gemm_tc_kernel (tcgen05 {'e4m3' if prec == 'fp8' else 'bf16'}, all four linear maps)")
        roofline = {"bound": "tensor", "kernel": kname,
                    "achieved": gemm_tflops, "peak": peak_burst, "unit": "TFLOP/s", "frac": gemm_tflops / peak_burst,
                    "peak_source": f"bf16_tflops (burst), {pk_src}" + peak_note,
                    "peak_sustained": peak_sust, "frac_vs_sustained": gemm_tflops / peak_sust,
                    "flops_per_launch": gemm_flops / gemm_launches if gemm_launches else None,
                    "avg_launch_ms": gemm_ms / gemm_launches if gemm_launches else None,
                    "traffic": traffic.get("dram_bytes_per_launch") if (traffic and wl.name == "esm650m"
                                                                        and args.layers is None
                                                                        and args.tokens is None) else None,
                    "traffic_source": traffic.get("source") if traffic else None}
        clock = clocks.get("sm_mhz") if clocks else None
        attn = attention_roofline(wl, per_kernel["attention"]["ms_per_step"], executed["attention"], pk, clock,
                                  torch.cuda.get_device_properties(dev).multi_processor_count)
    srt = sorted(per)
    res = {"workload": workload_text(wl), "tokens_per_s": global_tokens / (ms_step / 1e3),
           "tokens_per_s_median_step": global_tokens / (statistics.median(per) / 1e3),
           "ms_per_step": ms_step, "ms_per_step_median": statistics.median(per), "ms_per_step_min": srt[0],
           "steps": args.steps, "tflops": total_flops * (global_tokens / T) / (ms_step / 1e3) / 1e12,
           "mfu_vs_burst_peak": total_flops / (ms_step / 1e3) / 1e12 / peak_burst,
           "mfu_vs_sustained_peak": total_flops / (ms_step / 1e3) / 1e12 / peak_sust,
           "peak_dtype": ("nvfp4 (6 x measured bf16)" if fp4 else
                          "e4m3 (2 x measured bf16)" if prec == "fp8" else "bf16 (measured)"),
           "algorithmic_gflop_per_step_per_gpu": total_flops / 1e9,
           "padded_over_packed_flops": (sum(executed.values()) / total_flops) if padded else None,
           "max_memory_allocated_gb": peak_mem / 2**30, "roofline": roofline, "attention_roofline": attn,
           "per_kernel": per_kernel, "launches_per_step": launches_per_step, "gpu_launches": launches,
           "clocks": clocks, "dtype": "e2m1" if fp4 else {"fp8": "e4m3", "fp32": "f32"}.get(prec, "bf16"),
           "timing": "CUDA graph replay of the whole forward" if not args.no_graph else "eager launches"}
    state = {"enc": enc, "dw": dw, "tok": tok, "cu": cu, "ws": ws, "out": out, "w_np": w_np, "tok_np": tok_np,
             "T": T, "B": B, "maxL": maxL, "stream": stream, "flops": flops, "total_flops": total_flops,
             "gemm_classes": gemm_classes}
    return res, state


def run_ours(args):
    import torch
    import torch.distributed as dist

    from transformer_esm_layer_gb300 import build as _build
    from transformer_esm_layer_gb300 import synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    _build.build()
    dev = torch.device("cuda", torch.cuda.current_device())

    wl = workload_for_rank(0, args.tokens, args.layers, args.workload)
    g = wl.geometry
    prec = wl.precision
    padded = wl.padded_len is not None
    tok_np = synth.workload_tokens(wl)
    global_tokens = wl.total_tokens
    if world > 1:
        # one global batch of world x T tokens, split by work; each GPU encodes its share
        from transformer_esm_layer_gb300 import sharding
        rng = np.random.default_rng([wl.seed, 7, world])
        g_lengths = synth.lognormal_lengths(rng, total=world * wl.total_tokens)
        g_tokens = synth.tokens_for_lengths(np.random.default_rng([wl.seed, 8, world]), g_lengths)
        mine = sharding.shard_by_work(g_lengths, world, g.hidden, g.ffn)[rank]
        tok_np, wl.lengths = sharding.local_batch(g_tokens, g_lengths, mine)
        global_tokens = len(g_tokens)
    gpu_id = None
    try:
        gpu_id = str(torch.cuda.get_device_properties(dev).uuid)
        gpu_id = gpu_id if gpu_id.startswith("GPU-") else "GPU-" + gpu_id
    except Exception:
        gpu_id = None

    head, st = measure_forward(wl, dev, args, world=world, rank=rank, global_tokens=global_tokens, tok_np=tok_np,
                               clock_sampler=lambda: ClockSampler(gpu_id))
    enc, dw, tok, cu, ws, out = st["enc"], st["dw"], st["tok"], st["cu"], st["ws"], st["out"]
    T, B, maxL, stream, w_np = st["T"], st["B"], st["maxL"], st["stream"], st["w_np"]
    flops, total_flops, gemm_classes = st["flops"], st["total_flops"], st["gemm_classes"]
    ms_step = head["ms_per_step"]
    value = head["tokens_per_s"]

    # ---------------------------------------------------------------- end to end (host buffers)
    e2e = None
    if not padded:
        tok_h = torch.from_numpy(tok_np.astype(np.int32)).pin_memory()
        cu_h = torch.from_numpy(synth.cu_seqlens_from_lengths(wl.lengths)).pin_memory()
        out_h = torch.empty(T, g.hidden, dtype=enc.out_dtype).pin_memory()
        out_view = out_h.view(torch.int16 if enc.out_dtype == torch.bfloat16 else torch.int32).numpy()
        tok_view, cu_view = tok_h.numpy(), cu_h.numpy()
        n_e2e = args.steps
        # two untimed calls: the first runs eagerly, the second captures the call's CUDA graph
        # (pinned buffers), which later calls replay
        for _ in range(2):
            enc.forward_host(dw, tok_view, cu_view, maxL, out_view, ws, stream=stream)
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            enc.forward_host(dw, tok_view, cu_view, maxL, out_view, ws, stream=stream)
        dt = (time.perf_counter() - t0) / n_e2e
        if world > 1:
            t = torch.tensor([dt], dtype=torch.float64, device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            dt = float(t.item())
        e2e = {"value": global_tokens / dt, "unit": "tokens/s", "h2d_bytes_per_step": 4 * T + 4 * (B + 1),
               "d2h_bytes_per_step": out.element_size() * T * g.hidden, "ms_per_step": dt * 1e3,
               "call": "esm_encoder_forward_host (pinned host buffers in and out)"}

    # ---------------------------------------------------------------- masked-LM head (next step)
    mlm = None
    if not padded and prec == "bf16":
        from transformer_esm_layer_gb300.binding import DeviceLmHead
        lm = DeviceLmHead(synth.lm_head_weights(g, wl.seed, prec, w_np["emb"]), prec, device=dev)
        tg = torch.from_numpy(synth.mlm_targets(tok_np, wl.seed)).to(dev)
        hws = enc.lm_head_workspace(T, dev)
        lsum = torch.zeros(1, dtype=torch.float32, device=dev)
        cnt = torch.zeros(1, dtype=torch.int32, device=dev)
        logits = torch.empty(T, g.vocab, dtype=torch.float32, device=dev)
        for _ in range(3):
            enc.lm_head(lm, out, targets=tg, logits=logits, loss_sum=lsum, count=cnt, workspace=hws, stream=stream)
        per, tot = _timed_replays(lambda: enc.lm_head(lm, out, targets=tg, logits=logits, loss_sum=lsum, count=cnt,
                                                      workspace=hws, stream=stream), 10, stream)
        enc.check(stream)
        mms = tot / 10
        mlm = {"call": "esm_encoder_lm_head (dense+GELU, LayerNorm, logits vs tied embedding, masked CE)",
               "ms_per_call": mms, "ms_per_call_median": statistics.median(per), "tokens_per_s": T / (mms / 1e3),
               "scored_tokens": int(cnt.item()),
               "mean_loss_random_weights": float(lsum.item()) / max(1, int(cnt.item()))}
        del hws, logits
        # the head's backward from the mean masked loss: recomputed head forward, dL/d(hidden)
        # and every head parameter's gradient
        from transformer_esm_layer_gb300.binding import LM_HEAD_NAMES
        dhid = torch.empty(T, g.hidden, dtype=torch.float32, device=dev)
        hgrads = {k: torch.empty(tuple(lm.t[k].shape), dtype=torch.float32, device=dev) for k in LM_HEAD_NAMES}
        bws = enc.lm_head_backward_workspace(T, dev)
        bwd_call = lambda: enc.lm_head_backward(lm, out, tg, d_hidden=dhid, grads=hgrads, loss_sum=lsum, count=cnt,
                                                workspace=bws, stream=stream)
        for _ in range(3):
            bwd_call()
        per_b, tot_b = _timed_replays(bwd_call, 10, stream)
        enc.check(stream)
        mlm["backward_call"] = "esm_encoder_lm_head_backward (head forward recomputed, dL/d(hidden), head gradients)"
        mlm["backward_ms_per_call"] = tot_b / 10
        mlm["backward_ms_per_call_median"] = statistics.median(per_b)
        del dhid, hgrads, bws

    # ---------------------------------------------------------------- training step (forward that keeps
    # its activations + backward: every parameter's gradient), same batch
    train = None
    if not padded and prec == "bf16" and not args.no_train:
        from transformer_esm_layer_gb300.binding import DeviceGrads
        tb = enc.train_buffer(T, dev)
        grads = DeviceGrads(g, g.num_layers, device=dev)
        d_out = torch.randn(T, g.hidden, dtype=torch.float32, device=dev,
                            generator=torch.Generator(device=dev).manual_seed(wl.seed))

        def train_fwd():
            enc.forward_train(dw, tok, cu, maxL, tb, ws, out=out, stream=stream)

        allreduce_bytes = 0

        def train_bwd():
            nonlocal allreduce_bytes
            enc.backward(dw, d_out, grads, tb, ws, stream=stream)
            if world > 1:  # data parallel: every rank holds the gradient of the whole global batch
                from transformer_esm_layer_gb300 import sharding as _sh
                allreduce_bytes = _sh.allreduce_gradients(grads.tensors())

        for _ in range(2):
            train_fwd()
            train_bwd()
        enc.check(stream)
        n_tr = 5
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n_tr + 1)]
        ev[0].record(stream)
        for i in range(n_tr):
            train_fwd()
            ev[2 * i + 1].record(stream)
            train_bwd()
            ev[2 * i + 2].record(stream)
        torch.cuda.synchronize()
        enc.check(stream)
        f_all = [ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(n_tr)]
        b_all = [ev[2 * i + 1].elapsed_time(ev[2 * i + 2]) for i in range(n_tr)]
        f_ms, b_ms = sum(f_all) / n_tr, sum(b_all) / n_tr
        enc.set_profiling(True)
        enc.get_profile(reset=True)
        train_fwd()
        fprof = enc.get_profile(reset=True)
        train_bwd()
        bprof = enc.get_profile(reset=True)
        enc.set_profiling(False)
        # backward work: two products per linear map (input and weight gradient) and five
        # per attention tile pair (S, dP, dV, dK, dQ) against the forward's two
        bwd_flops = 2.0 * sum(flops[c] for c in gemm_classes) + 2.5 * flops["attention"]
        bg_ms = bprof["gemm_backward"]["ms"]
        train = {"calls": "esm_encoder_forward_train + esm_encoder_backward (all parameter gradients, fp32)"
                          + (" + NCCL all-reduce (sum) of the gradients" if world > 1 else ""),
                 "gradient_allreduce_bytes_per_rank": allreduce_bytes if world > 1 else 0,
                 "ms_per_step": f_ms + b_ms, "ms_per_step_min": min(f + b for f, b in zip(f_all, b_all)),
                 "ms_forward_train": f_ms, "ms_backward": b_ms,
                 "tokens_per_s": global_tokens / ((f_ms + b_ms) / 1e3),
                 "backward_tflops": bwd_flops / (b_ms / 1e3) / 1e12,
                 "step_tflops": (total_flops + bwd_flops) / ((f_ms + b_ms) / 1e3) / 1e12,
                 "backward_gemm": {"ms": bg_ms, "launches": bprof["gemm_backward"]["launches"],
                                   "tflops": 2.0 * sum(flops[c] for c in gemm_classes) / (bg_ms / 1e3) / 1e12
                                   if bg_ms else None},
                 "backward_per_class_ms": {c: bprof[c]["ms"] for c in ("attention", "layernorm", "gemm_backward",
                                                                       "other")},
                 "forward_train_per_class_ms": {c: fprof[c]["ms"] for c in ("gemm_qkv", "attention", "gemm_oproj",
                                                                            "gemm_fc1", "gemm_fc2", "layernorm",
                                                                            "other")},
                 "train_buffer_gb": tb.numel() / 2**30}
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            try:  # an auxiliary figure: a failure here must not cost the benchmark line
                toks_c, dt_c, done_c = cpu_oracle_train_sample(wl, f64_weights(w_np), args.cpu_seconds, wl.seed)
                train["cpu_baseline"] = {
                    "value": toks_c / dt_c, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
                    "sample": f"{len(done_c)} whole sequence(s) of the workload ({toks_c} tokens): forward and every "
                              f"gradient through all {g.num_layers} layers in float64 numpy, {dt_c:.1f} s"}
            except Exception as e:  # noqa: BLE001
                train["cpu_baseline"] = {"error": f"{type(e).__name__}: {e}"}
        del tb, grads

    # ---------------------------------------------------------------- CPU baseline (oracle)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        toks, dt, done = cpu_oracle_sample(wl, f64_weights(w_np), args.cpu_seconds, prec, enc)
        cpu = {"value": toks / dt, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
               "sample": f"{len(done)} whole sequence(s) of the workload (indices {done}, {toks} tokens) through all "
                         f"{g.num_layers} layers in float64 numpy, {dt:.1f} s"}

    # ---------------------------------------------------------------- the other configured workloads
    configs = None
    if world == 1 and not args.no_configs and args.workload == "esm650m" and args.layers is None \
            and args.tokens is None:
        del st
        configs = {}
        for name in ("tiny_fp32", "layer650m", "esm650m_padded", "esm3b_fp8", "esm3b_fp4"):
            try:  # a side measurement: a failure here must not cost the benchmark line
                wl2 = synth.make_workload(name)
                reuse = w_np if name == "esm650m_padded" else None  # same model and seed as the headline
                r2, st2 = measure_forward(wl2, dev, args, w_np=reuse)
                del st2
                torch.cuda.empty_cache()
                configs[name] = r2
            except Exception as e:  # noqa: BLE001
                configs[name] = {"error": f"{type(e).__name__}: {e}"}

    if world > 1:
        dist.barrier()
    if rank == 0:
        metric = {"esm650m": METRIC,
                  "esm650m_padded": "ESM-2 650M padded [B,1024] fwd tokens/s (real tokens) on 1 GB300; achieved "
                                    "TFLOP/s vs dense BF16 peak",
                  "esm3b_fp8": "ESM-2 3B packed FP8 fwd tokens/s on 1 GB300; achieved TFLOP/s vs dense FP8 peak",
                  "esm3b_fp4": "ESM-2 3B packed NVFP4 fwd tokens/s on 1 GB300; achieved TFLOP/s vs dense FP4 peak"
                  }[args.workload]
        line = {"metric": metric, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_step, "ms_per_step_median": head["ms_per_step_median"],
                "ms_per_step_min": head["ms_per_step_min"], "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": head["dtype"], "data": "synthetic",
                "config": {"workload": head["workload"], "tokens_per_step_per_gpu": T, "sequences": B,
                           "max_seqlen": maxL,
                           "l2": "no flush: inputs larger than L2 ("
                                 f"{sum(t.numel() * t.element_size() for l in dw.layers for t in l.values()) / 2**30:.2f} GB "
                                 f"of weights read per step plus {ws.numel() / 2**30:.2f} GB of activations vs the "
                                 "129 MB L2)",
                           "parallelism": "single GPU" if world == 1 else
                           f"{world} replicas, one global batch of {global_tokens} tokens split by work "
                           "(longest-first greedy), no collective on the data path"},
                "tflops": head["tflops"], "mfu_vs_burst_peak": head["mfu_vs_burst_peak"],
                "mfu_vs_sustained_peak": head["mfu_vs_sustained_peak"], "peak_dtype": head["peak_dtype"],
                "algorithmic_gflop_per_step_per_gpu": head["algorithmic_gflop_per_step_per_gpu"],
                "max_memory_allocated_gb": head["max_memory_allocated_gb"],
                "roofline": head["roofline"], "attention_roofline": head["attention_roofline"],
                "per_kernel": head["per_kernel"], "padded_over_packed_flops": head["padded_over_packed_flops"],
                "cpu_baseline": cpu, "e2e": e2e, "mlm_head": mlm, "train_step": train, "configs": configs,
                "clocks": head["clocks"], "gpu_launches": head["gpu_launches"], "timing": head["timing"],
                "context": "pages' own figure: 59.2% model-FLOP utilisation, ESM-2 650M training, batch 46, A100"}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
