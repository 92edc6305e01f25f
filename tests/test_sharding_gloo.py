"""Multi-GPU host logic on CPU: sequence sharding for independent replicas, checked with a
world-size-2 gloo process group (no GPU needed)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from transformer_esm_layer_gb300 import sharding, synth


def test_shard_by_work_is_a_balanced_partition():
    wl = synth.make_workload("esm650m")
    g = wl.geometry
    for world in (1, 2, 4, 8):
        parts = sharding.shard_by_work(wl.lengths, world, g.hidden, g.ffn)
        flat = sorted(i for p in parts for i in p)
        assert flat == list(range(len(wl.lengths)))            # every sequence exactly once
        costs = [sum(sharding.sequence_cost(wl.lengths[i], g.hidden, g.ffn) for i in p) for p in parts]
        biggest = max(sharding.sequence_cost(L, g.hidden, g.ffn) for L in wl.lengths)
        assert max(costs) - min(costs) <= biggest + 1e-6      # greedy bound: within one sequence


def test_local_batch_keeps_sequences_intact():
    lengths = [3, 5, 2, 7]
    tok = np.arange(sum(lengths), dtype=np.int32)
    t, l = sharding.local_batch(tok, lengths, [1, 3])
    assert l == [5, 7]
    assert t.tolist() == list(range(3, 8)) + list(range(10, 17))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # every rank builds the same global batch and takes its own share, as bench.py does
        rng = np.random.default_rng([2, 99])
        lengths = synth.lognormal_lengths(rng, total=world * 4096)
        tokens = synth.tokens_for_lengths(np.random.default_rng([2, 98]), lengths)
        parts = sharding.shard_by_work(lengths, world, 1280, 5120)
        mine = parts[rank]
        toks, lens = sharding.local_batch(tokens, lengths, mine)
        # what each rank would hand to esm_encoder_forward: valid packed inputs
        cu = synth.cu_seqlens_from_lengths(lens)
        assert cu[0] == 0 and cu[-1] == len(toks) and np.all(np.diff(cu) >= 1)
        # the ranks agree on the partition and together cover the batch exactly once
        got = [None] * world
        dist.all_gather_object(got, mine)
        flat = sorted(i for p in got for i in p)
        ok = flat == list(range(len(lengths))) and got == parts
        # token counts add up to the global batch
        n = torch.tensor([len(toks)], dtype=torch.int64)
        dist.all_reduce(n)
        ok = ok and int(n.item()) == len(tokens)
        q.put((rank, ok))
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_sharding():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    results = dict(q.get(timeout=10) for _ in range(world))
    assert all(p.exitcode == 0 for p in procs)
    assert results == {0: True, 1: True}


SMALL = synth.Geometry(num_layers=2, hidden=16, heads=2, ffn=32, vocab=33)


def _grad_worker(rank, world, port, q):
    """Each rank backpropagates its share of one packed batch (float64 oracle), the gradients
    are summed with allreduce_gradients, and every rank compares with the gradient of the
    whole batch."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from oracle import backward as B
        from oracle import esm_oracle as O
        rng = np.random.default_rng(5)
        lengths = [9, 4, 7, 1, 12]
        tokens = synth.tokens_for_lengths(rng, lengths).astype(np.int64)
        w = synth.model_weights(SMALL, 5, "fp32", ln_random=True)
        T = len(tokens)
        d_out = np.random.default_rng(6).standard_normal((T, SMALL.hidden))
        cu = O.cu_seqlens(lengths)
        mine = sharding.shard_by_work(lengths, world, SMALL.hidden, SMALL.ffn)[rank]
        toks, lens = sharding.local_batch(tokens, lengths, mine)
        d_mine = np.concatenate([d_out[cu[i]:cu[i + 1]] for i in mine]) if mine else np.zeros((0, SMALL.hidden))

        def flat(g):
            return [g["emb"]] + [l[n] for l in g["layers"] for n in B.PARAM_NAMES] + [g["lnf_g"], g["lnf_b"]]

        if lens:
            part = flat(B.encode_packed_backward(toks.astype(np.int64), O.cu_seqlens(lens), w, SMALL.heads, d_mine))
        else:
            part = [np.zeros_like(a) for a in flat(B.encode_packed_backward(tokens, cu, w, SMALL.heads, d_out))]
        tens = [torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64)) for a in part]
        nbytes = sharding.allreduce_gradients(tens, bucket_bytes=4096)  # several buckets
        full = flat(B.encode_packed_backward(tokens, cu, w, SMALL.heads, d_out))
        err = max(float(np.abs(t.numpy() - f).max() / (np.abs(f).max() + 1e-300)) for t, f in zip(tens, full))
        q.put((rank, err < 1e-12 and nbytes == sum(a.size * 8 for a in full)))
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_gradient_allreduce_equals_whole_batch_gradient():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_grad_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    results = dict(q.get(timeout=10) for _ in range(world))
    assert results == {0: True, 1: True}


def _loss_grad_worker(rank, world, port, q):
    """A data-parallel step from the masked-LM loss: each rank encodes its share, takes the
    loss backward with the global scored count (all-reduced first), backpropagates through
    the encoder, and the gradients are summed.  Every rank compares with the gradient of the
    whole batch's mean loss (float64 oracle); the shares have different scored counts."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from oracle import backward as B
        from oracle import esm_oracle as O
        lengths = [9, 4, 7, 1, 12]
        tokens = synth.tokens_for_lengths(np.random.default_rng(7), lengths).astype(np.int64)
        w = synth.model_weights(SMALL, 7, "fp32", ln_random=True)
        head = synth.lm_head_weights(SMALL, 7, "fp32", w["emb"])
        targets = synth.mlm_targets(tokens, 7, rate=0.4).astype(np.int64)
        cu = O.cu_seqlens(lengths)
        mine = sharding.shard_by_work(lengths, world, SMALL.hidden, SMALL.ffn)[rank]
        toks, lens = sharding.local_batch(tokens, lengths, mine)
        t_mine = np.concatenate([targets[cu[i]:cu[i + 1]] for i in mine])
        n_global = int(sharding.global_scored_count(torch.from_numpy(t_mine)).item())
        counts = [None] * world
        dist.all_gather_object(counts, int((t_mine != -100).sum()))

        def step(tk, cuv, tg, count):
            hid = O.encode_packed(tk, cuv, w, SMALL.heads)
            hid = np.concatenate([hid[i] for i in range(len(cuv) - 1)])
            rh = B.lm_head_backward(hid, head, tg, count=count)
            ge = B.encode_packed_backward(tk, cuv, w, SMALL.heads, rh["hidden"])
            flat = [ge["emb"] + rh["emb"]] + [rh[k] for k in ("dense_w", "dense_b", "ln_g", "ln_b", "bias")]
            return flat + [l[n] for l in ge["layers"] for n in B.PARAM_NAMES] + [ge["lnf_g"], ge["lnf_b"]]

        part = step(toks.astype(np.int64), O.cu_seqlens(lens), t_mine, n_global)
        tens = [torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64)) for a in part]
        sharding.allreduce_gradients(tens, bucket_bytes=4096)
        full = step(tokens, cu, targets, None)
        err = max(float(np.abs(t.numpy() - f).max() / (np.abs(f).max() + 1e-300)) for t, f in zip(tens, full))
        ok = err < 1e-12 and n_global == int((targets != -100).sum()) and counts[0] != counts[1]
        q.put((rank, ok))
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_training_step_from_the_loss_equals_whole_batch_gradient():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_loss_grad_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    results = dict(q.get(timeout=10) for _ in range(world))
    assert results == {0: True, 1: True}
