"""Float64 CPU oracle of the backward pass of the packed ESM-2 encoder (training).

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the benchmark's
CPU-baseline / reference arm may import this module.  The CUDA library never calls it and
shares no code with it.

Sources (page title, section):

* "生物大模型训练加速实战：基于PyTorch与NVIDIA BioNeMo的Transformer优化指南" (hotelren.com),
  §3.2 (the packed model trains over ``cu_seqlens``: the training loop calls ``backward``
  on the packed forward) and §6 (the FP8 training loop with ``loss.backward()``).
* "深入源码NVIDIA ESM-2 TransformerEngine优化的实现原理与技术细节" (mlqm.cn), the training
  sections (the same layer stack under autograd).

The pages name the backward pass but never write it out; what it computes is fixed by the
forward: the exact gradients of the forward in ``esm_oracle`` (chain rule, written here
step by step in the reverse order of the forward).  Every function is pinned in
tests/test_oracle_backward_pins.py by central finite differences of the float64 forward,
adjoint identities and invariants of the forward (a constant added to all keys of a
sequence, a constant added to a LayerNorm input row).

Readings: gradients are taken of a scalar loss whose gradient with respect to the encoder
output is given (``d_out``); parameters shared by the sequences of a packed batch receive
the sum of the per-sequence gradients; the embedding table's gradient is the scatter-add of
``emb_scale`` times the gradient of the embedded rows.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import numpy as np
from scipy.special import erf

from .esm_oracle import LN_EPS, ROPE_BASE, attention, encoder_layer, gelu, layer_norm, rope

PARAM_NAMES = ("ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o", "ln2_g", "ln2_b", "w_1", "b_1", "w_2", "b_2")


def layer_norm_backward(x: np.ndarray, gamma: np.ndarray, dy: np.ndarray, eps: float = LN_EPS):
    """Gradients of y = (x - mean) / sqrt(var + eps) * gamma + beta (rows of x) given dL/dy.

    With xhat the normalised row, r = 1 / sqrt(var + eps) and g = dy * gamma:
    dx = r * (g - mean(g) - xhat * mean(g * xhat)); dgamma = sum_rows dy * xhat;
    dbeta = sum_rows dy."""
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    r = 1.0 / np.sqrt(var + eps)
    xhat = (x - mu) * r
    g = dy * gamma
    dx = r * (g - g.mean(axis=-1, keepdims=True) - xhat * (g * xhat).mean(axis=-1, keepdims=True))
    return dx, (dy * xhat).sum(axis=0), dy.sum(axis=0)


def gelu_grad(a: np.ndarray) -> np.ndarray:
    """Derivative of the exact GELU a * Phi(a): Phi(a) + a * phi(a), phi the normal density."""
    return 0.5 * (1.0 + erf(a / np.sqrt(2.0))) + a * np.exp(-0.5 * a * a) / np.sqrt(2.0 * np.pi)


def rope_backward(g: np.ndarray, pos: np.ndarray, base: float = ROPE_BASE) -> np.ndarray:
    """Gradient through the rotary embedding: each pair (j, j + dh/2) was turned by the angle
    p * base^(-2j/dh), so its gradient turns back by the same angle (the transpose of a
    rotation).  g is [L, H, dh]."""
    dh = g.shape[-1]
    half = dh // 2
    j = np.arange(half, dtype=np.float64)
    theta = base ** (-2.0 * j / dh)
    phi = pos.astype(np.float64)[:, None] * theta[None, :]
    c = np.cos(phi)[:, None, :]
    s = np.sin(phi)[:, None, :]
    ga, gb = g[..., :half], g[..., half:]
    return np.concatenate([ga * c + gb * s, gb * c - ga * s], axis=-1)


def attention_backward(q: np.ndarray, k: np.ndarray, v: np.ndarray, do: np.ndarray):
    """Gradients of o = softmax(q k^T / sqrt(dh)) v (one sequence, all keys visible) with
    respect to q, k, v; all [L, H, dh].

    Per head: P = softmax(S), dV = P^T dO, dP = dO V^T, dS = P * (dP - rowsum(P * dP)),
    dq = dS k / sqrt(dh), dk = dS^T q / sqrt(dh)."""
    dh = q.shape[-1]
    sc = 1.0 / np.sqrt(dh)
    qh, kh, vh, doh = (t.transpose(1, 0, 2) for t in (q, k, v, do))  # [H, L, dh]
    s = np.matmul(qh, kh.transpose(0, 2, 1)) * sc
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p = p / p.sum(axis=-1, keepdims=True)
    dv = np.matmul(p.transpose(0, 2, 1), doh)
    dp = np.matmul(doh, vh.transpose(0, 2, 1))
    ds = p * (dp - (p * dp).sum(axis=-1, keepdims=True))
    dq = np.matmul(ds, kh) * sc
    dk = np.matmul(ds.transpose(0, 2, 1), qh) * sc
    return tuple(t.transpose(1, 0, 2) for t in (dq, dk, dv))


def attention_lse(q: np.ndarray, k: np.ndarray) -> np.ndarray:
    """log sum_j exp(q_i . k_j / sqrt(dh)) per query and head ([L, H], natural log): the
    softmax normaliser a training forward keeps for its backward."""
    dh = q.shape[-1]
    s = np.einsum("ihd,jhd->hij", q, k) / np.sqrt(dh)
    m = s.max(axis=-1, keepdims=True)
    return (m[..., 0] + np.log(np.exp(s - m).sum(axis=-1))).T


def encoder_layer_backward(x: np.ndarray, pos: np.ndarray, w: Dict[str, np.ndarray], heads: int,
                           d_out: np.ndarray, eps: float = LN_EPS, rope_base: float = ROPE_BASE):
    """Backward of one pre-LN layer (the forward of ``esm_oracle.encoder_layer``) on one
    sequence: returns (dL/dx, {parameter name: gradient}).  The forward intermediates are
    recomputed from x."""
    L, d = x.shape
    dh = d // heads
    # forward, keeping what the backward needs
    y = layer_norm(x, w["ln1_g"], w["ln1_b"], eps)
    qkv = y @ w["w_qkv"].T + w["b_qkv"]
    q = rope(qkv[:, :d].reshape(L, heads, dh), pos, rope_base)
    k = rope(qkv[:, d:2 * d].reshape(L, heads, dh), pos, rope_base)
    v = qkv[:, 2 * d:].reshape(L, heads, dh)
    o = attention(q, k, v).reshape(L, d)
    x1 = x + o @ w["w_o"].T + w["b_o"]
    z = layer_norm(x1, w["ln2_g"], w["ln2_b"], eps)
    a = z @ w["w_1"].T + w["b_1"]
    u = gelu(a)
    g = {}
    # MLP block: x2 = x1 + u W2^T + b2
    g["w_2"] = d_out.T @ u
    g["b_2"] = d_out.sum(axis=0)
    da = (d_out @ w["w_2"]) * gelu_grad(a)
    g["w_1"] = da.T @ z
    g["b_1"] = da.sum(axis=0)
    dx1, g["ln2_g"], g["ln2_b"] = layer_norm_backward(x1, w["ln2_g"], da @ w["w_1"], eps)
    dx1 = dx1 + d_out
    # attention block: x1 = x + o Wo^T + bo
    g["w_o"] = dx1.T @ o
    g["b_o"] = dx1.sum(axis=0)
    do = (dx1 @ w["w_o"]).reshape(L, heads, dh)
    dq, dk, dv = attention_backward(q, k, v, do)
    dq = rope_backward(dq, pos, rope_base)
    dk = rope_backward(dk, pos, rope_base)
    dqkv = np.concatenate([dq.reshape(L, d), dk.reshape(L, d), dv.reshape(L, d)], axis=1)
    g["w_qkv"] = dqkv.T @ y
    g["b_qkv"] = dqkv.sum(axis=0)
    dx, g["ln1_g"], g["ln1_b"] = layer_norm_backward(x, w["ln1_g"], dqkv @ w["w_qkv"], eps)
    return dx + dx1, g


def encode_sequence_backward(tokens: np.ndarray, weights: Dict, heads: int, d_out: np.ndarray,
                             final_ln: bool = True, emb_scale: float = 1.0, eps: float = LN_EPS,
                             rope_base: float = ROPE_BASE, num_layers: Optional[int] = None) -> Dict:
    """Gradients of one sequence's encoder (``esm_oracle.encode_sequence``) given dL/d(out).

    Returns {"emb": [vocab, d], "layers": [{name: grad}], "lnf_g", "lnf_b", "x0": dL/d(embedded
    rows)}."""
    tokens = np.asarray(tokens, dtype=np.int64)
    emb = np.asarray(weights["emb"], dtype=np.float64)
    layers = weights["layers"] if num_layers is None else weights["layers"][:num_layers]
    lw = [{k: np.asarray(v, np.float64) for k, v in wl.items()} for wl in layers]
    pos = np.arange(len(tokens))
    xs = [emb_scale * emb[tokens]]
    for wl in lw:
        xs.append(encoder_layer(xs[-1], pos, wl, heads, eps, rope_base))
    out = {}
    dx = np.asarray(d_out, np.float64)
    if final_ln:
        gf = np.asarray(weights["lnf_g"], np.float64)
        dx, out["lnf_g"], out["lnf_b"] = layer_norm_backward(xs[-1], gf, dx, eps)
    grads: List[Dict[str, np.ndarray]] = [None] * len(lw)
    for li in range(len(lw) - 1, -1, -1):
        dx, grads[li] = encoder_layer_backward(xs[li], pos, lw[li], heads, dx, eps, rope_base)
    out["layers"] = grads
    out["x0"] = dx
    de = np.zeros_like(emb)
    for t, tok in enumerate(tokens):
        de[tok] += emb_scale * dx[t]
    out["emb"] = de
    return out


def encode_packed_backward(token_ids: np.ndarray, cu: Sequence[int], weights: Dict, heads: int,
                           d_out: np.ndarray, final_ln: bool = True, **kw) -> Dict:
    """Backward of the packed forward: sequences are independent, so each is differentiated
    on its own and the parameter gradients add up over the sequences.  d_out is [T, d];
    the result's "x0" is [T, d]."""
    total = None
    x0 = np.zeros((int(cu[-1]), np.asarray(weights["emb"]).shape[1]))
    for i in range(len(cu) - 1):
        a, b = int(cu[i]), int(cu[i + 1])
        gi = encode_sequence_backward(token_ids[a:b], weights, heads, d_out[a:b], final_ln, **kw)
        x0[a:b] = gi["x0"]
        if total is None:
            total = gi
        else:
            total["emb"] = total["emb"] + gi["emb"]
            for n in ("lnf_g", "lnf_b"):
                if n in gi:
                    total[n] = total[n] + gi[n]
            for lt, lg in zip(total["layers"], gi["layers"]):
                for n in PARAM_NAMES:
                    lt[n] = lt[n] + lg[n]
    total["x0"] = x0
    return total


# --------------------------------------------------------------------------- masked-LM head
def lm_head_backward(h: np.ndarray, w: Dict[str, np.ndarray], targets: Sequence[int],
                     count: Optional[int] = None):
    """Gradients of the mean masked-LM loss L = sum_scored CE / count (the forward of
    ``esm_oracle.lm_head`` and ``masked_lm_loss``) with respect to the hidden states h [T, d]
    and the head's parameters.  The embedding E is tied: the gradient returned for it is the
    head's part only (the encoder's embedding gradient adds to it).

    ``count`` is the number of scored tokens the mean is taken over: by default those of
    ``targets``.  When a batch is split over data-parallel ranks, each rank passes the
    scored count of the whole batch, so that every rank differentiates its own share of the
    same loss and the ranks' gradients add up to the batch gradient.

    With logits l = z E^T + b, z = LN(u), u = GELU(a), a = h Wd^T + bd:
    dl = (softmax(l) - onehot(target)) / count on scored rows (0 elsewhere),
    dE = dl^T z, db = sum dl, dz = dl E, then LayerNorm, GELU' and the dense map backward."""
    from .esm_oracle import IGNORE_INDEX
    h = np.asarray(h, np.float64)
    wd = np.asarray(w["dense_w"], np.float64)
    E = np.asarray(w["emb"], np.float64)
    a = h @ wd.T + np.asarray(w["dense_b"], np.float64)
    u = gelu(a)
    lg, lb = np.asarray(w["ln_g"], np.float64), np.asarray(w["ln_b"], np.float64)
    z = layer_norm(u, lg, lb)
    logits = z @ E.T + np.asarray(w["bias"], np.float64)
    t = np.asarray(targets, np.int64)
    scored = t != IGNORE_INDEX
    if count is None:
        count = int(scored.sum())
    dl = np.zeros_like(logits)
    if count > 0 and scored.any():
        m = logits.max(axis=1, keepdims=True)
        p = np.exp(logits - m)
        p /= p.sum(axis=1, keepdims=True)
        rows = np.nonzero(scored)[0]
        dl[rows] = p[rows]
        dl[rows, t[scored]] -= 1.0
        dl /= count
    g = {"emb": dl.T @ z, "bias": dl.sum(axis=0)}
    du, g["ln_g"], g["ln_b"] = layer_norm_backward(u, lg, dl @ E)
    da = du * gelu_grad(a)
    g["dense_w"] = da.T @ h
    g["dense_b"] = da.sum(axis=0)
    g["hidden"] = da @ wd
    return g
