"""Float64 CPU oracle of the ESM-2 encoder forward on packed variable-length sequences.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the benchmark's
CPU-baseline / reference arm may import this module.  The CUDA library never calls it and
shares no code with it.  It is deliberately plain: one sequence at a time, one layer at a
time, with numpy's float64 matmul as the only library step.

Sources (page title, section):

* "生物大模型训练加速实战：基于PyTorch与NVIDIA BioNeMo的Transformer优化指南" (hotelren.com),
  §3.1 (the layer holds self-attention, LayerNorm, fc1, fc2; ``te.TransformerLayer`` as an
  encoder layer), §3.2 (THD packing: ``flat_tokens = cat(seqs)``,
  ``cu_seqlens = cumsum([0] + lengths)``, ``max_seqlen``; ``PackedEsm.forward`` runs the
  embedding then every layer over ``cu_seqlens``), §4.1 (FP8 ``DelayedScaling`` with
  ``amax_compute_algo="max"``).
* "深入源码NVIDIA ESM-2 TransformerEngine优化的实现原理与技术细节" (mlqm.cn): sections
  旋转位置编码集成 (rotary embedding of size hidden // heads), 注意力掩码优化 (padding mask,
  bshd), 权重融合技术 (fused QKV parameters), 序列长度优化 (1026 positions, vocab 33).
* BioNeMo ESM-2 model card (docs.nvda.net.cn), 模型概述 / 描述 (bidirectional BERT-style
  encoder), 输出 (one embedding vector per residue).
* "Accelerating transformer training with NVIDIA Transformer Engine" (aikraft.ru), section
  "Рецепт FP8: Delayed Scaling" (E4M3 forward format, amax history 16, max).
* Masked-LM head: the mlqm.cn walkthrough loads the model as ``AutoModelForMaskedLM``
  (section on usage) and the BioNeMo model card's accuracy benchmark (竞争性基准测试 / 准确率)
  reports masked-LM perplexity; neither lists the head's layers.

Readings where the pages are silent (each also applied by the CUDA path):
pre-LayerNorm blocks; LayerNorm eps 1e-5 with the biased variance; exact erf GELU; RoPE
base 10000 with rotate-half pairs (j, j + head_dim/2), applied to q and k after the bias,
positions restarting at 0 at each sequence start; scores scaled by 1/sqrt(head_dim);
no dropout; an optional final LayerNorm; embedding scale 1.  The FP8 workload states that
attention stays in bf16: its oracle rounds the attention operands q, k, v to bfloat16.
Masked-LM head (silent on the pages): the ESM-2 head of that model family, dense d -> d with
bias, exact GELU, LayerNorm, then logits against the (tied) token embedding plus a vocabulary
bias; the loss is the mean cross-entropy over the masked positions (target -100 = not
scored), and perplexity is exp of that mean.

Parity pins: every function here is checked in tests/test_oracle_pins.py against closed
forms, invariants, brute force or an independent library formulation.  The only part with
no pin is trained-model behaviour (perplexity), which needs weights and data that are
not available: parity unpinned for that part.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import numpy as np
from scipy.special import erf

LN_EPS = 1e-5
ROPE_BASE = 10000.0
E4M3_MAX = 448.0


# --------------------------------------------------------------------------- packing
def cu_seqlens(lengths: Sequence[int]) -> np.ndarray:
    """Offsets of the packed batch: cumsum([0] + lengths) (THD packing, §3.2 step 1)."""
    out = [0]
    for L in lengths:
        out.append(out[-1] + int(L))
    return np.asarray(out, dtype=np.int64)


def pack_index(cu: Sequence[int]):
    """For every packed token t: its sequence index seg_id[t] and its position inside that
    sequence pos_id[t] = t - cu[seg_id[t]].  Plain enumeration, sequence by sequence."""
    T = int(cu[-1])
    pos = np.zeros(T, dtype=np.int64)
    seg = np.zeros(T, dtype=np.int64)
    for i in range(len(cu) - 1):
        for p, t in enumerate(range(int(cu[i]), int(cu[i + 1]))):
            pos[t] = p
            seg[t] = i
    return pos, seg


# --------------------------------------------------------------------------- pieces
def layer_norm(x: np.ndarray, gamma: np.ndarray, beta: np.ndarray, eps: float = LN_EPS) -> np.ndarray:
    """LayerNorm over the last axis: (x - mean) / sqrt(var + eps) * gamma + beta, var biased."""
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * gamma + beta


def gelu(a: np.ndarray) -> np.ndarray:
    """Exact GELU: a * Phi(a) with Phi the standard normal CDF, written through erf."""
    return a * 0.5 * (1.0 + erf(a / np.sqrt(2.0)))


def rope(u: np.ndarray, pos: np.ndarray, base: float = ROPE_BASE) -> np.ndarray:
    """Rotary position embedding (rotary section of the mlqm.cn walkthrough) on u[L, H, dh].

    For j < dh/2 the pair (u_j, u_{j+dh/2}) at position p turns by the angle
    p * base^(-2j/dh)."""
    dh = u.shape[-1]
    half = dh // 2
    j = np.arange(half, dtype=np.float64)
    theta = base ** (-2.0 * j / dh)
    phi = pos.astype(np.float64)[:, None] * theta[None, :]
    c = np.cos(phi)[:, None, :]
    s = np.sin(phi)[:, None, :]
    a, b = u[..., :half], u[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, n_keys: Optional[int] = None) -> np.ndarray:
    """Bidirectional softmax attention inside one sequence; q, k, v are [L, H, dh].

    Every query sees every key of its own sequence (the model card's bidirectional
    encoder).  With ``n_keys`` only the first n_keys keys are visible (padding mask)."""
    dh = q.shape[-1]
    if n_keys is not None:
        k, v = k[:n_keys], v[:n_keys]
    qh = q.transpose(1, 0, 2)             # [H, L, dh]
    kh = k.transpose(1, 2, 0)             # [H, dh, Lk]
    s = np.matmul(qh, kh) / np.sqrt(dh)   # [H, L, Lk]
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p = p / p.sum(axis=-1, keepdims=True)
    o = np.matmul(p, v.transpose(1, 0, 2))  # [H, L, dh]
    return o.transpose(1, 0, 2)


# --------------------------------------------------------------------------- bf16
def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bfloat16 value (ties to even): keep the top 8 significand bits
    of the float32 nearest to x.  (Used where a workload fixes bf16 operands.)"""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = ((u + 0x7FFF + lsb) >> 16) << 16
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------- FP8 (E4M3)
def e4m3_round(x: np.ndarray) -> np.ndarray:
    """Round to the nearest OCP FP8 E4M3 value (ties to even), saturating at +-448.

    E4M3: 4 exponent bits with bias 7, 3 mantissa bits, subnormal spacing 2^-9, largest
    finite value 1.75 * 2^8 = 448.  Inside the binade [2^e, 2^(e+1)) (e >= -6) the
    values are spaced 2^(e-3); below 2^-6 the spacing stays 2^-9."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, ex = np.frexp(a)                      # a = m * 2^ex, m in [0.5, 1)
    e = np.maximum(ex - 1, -6).astype(np.float64)
    q = np.ldexp(1.0, (e - 3).astype(np.int64))
    r = np.round(a / q) * q                  # numpy rounds half to even
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, x)


def fp8_fake_quant(a: np.ndarray, scale: float) -> np.ndarray:
    """A GEMM operand as the FP8 path sees it: deq(q(a * scale)) / scale."""
    return e4m3_round(a * scale) / scale


def fp8_scale_update(history: np.ndarray, scale: float, amax: float):
    """Delayed scaling with the max algorithm (§4.1 of the hotelren.com guide; the
    aikraft.ru FP8 recipe): push this call's amax into the history (dropping the oldest),
    then scale = 448 / max(history).  A zero or non-finite max keeps the old scale."""
    h = np.concatenate([[amax], np.asarray(history, dtype=np.float64)[:-1]])
    m = h.max()
    new_scale = E4M3_MAX / m if (np.isfinite(m) and m > 0) else scale
    return h, float(new_scale)


FP8_TENSORS = ("x_qkv", "w_qkv", "x_o", "w_o", "x_1", "w_1", "x_2", "w_2")


# --------------------------------------------------------------------------- layer / encoder
FP8_WEIGHTS = ("w_qkv", "w_o", "w_1", "w_2")


def fp8_quantised_weights(w: Dict[str, np.ndarray], fp8_scales: Dict[str, float]) -> Dict[str, np.ndarray]:
    """The four linear weights of one layer as the FP8 path sees them, deq(q(w * s_w)) / s_w
    with each weight's own per-tensor scale.  A weight has one scale per call, so this is
    the same for every sequence of the call; the other entries are returned unchanged."""
    out = dict(w)
    for k in FP8_WEIGHTS:
        out[k] = fp8_fake_quant(np.asarray(w[k], np.float64), fp8_scales[k])
    return out


def encoder_layer(x: np.ndarray, pos: np.ndarray, w: Dict[str, np.ndarray], heads: int,
                  eps: float = LN_EPS, rope_base: float = ROPE_BASE, n_keys: Optional[int] = None,
                  fp8_scales: Optional[Dict[str, float]] = None, amax_out: Optional[Dict[str, float]] = None,
                  bf16_attention: bool = False, weights_quantised: bool = False,
                  fp4_scales: Optional[Dict[str, float]] = None):
    """One pre-LN encoder layer on one sequence x[L, d] (float64).

    y = LN1(x); [q|k|v] = y Wqkv^T + bqkv; RoPE on q, k; o = attention(q, k, v);
    x += o Wo^T + bo; z = LN2(x); u = GELU(z W1^T + b1); x += u W2^T + b2.

    With ``fp8_scales`` every GEMM operand (the four activations and four weights) is
    replaced by its E4M3 fake-quantised value; ``amax_out`` then receives max|.| of each
    operand before quantisation.  ``weights_quantised`` says the four weights in ``w`` are
    already fake-quantised with these scales (``fp8_quantised_weights``), so only the
    activations are quantised here.  ``bf16_attention`` rounds the attention operands q, k, v
    to bfloat16 (the FP8 workload keeps attention in bf16).

    With ``fp4_scales`` (tensor scales S of the eight operands, named as for FP8) every GEMM
    operand is replaced by its NVFP4 value (``fp4.nvfp4_fake_quant`` along the reduction axis
    with that S); the activations are the bf16 tensors the layer holds (LayerNorm outputs,
    attention output, GELU output), so they are rounded to bfloat16 before quantisation."""
    L, d = x.shape
    dh = d // heads

    def mm(a, wname, aname):
        wt = w[wname]
        if fp4_scales is not None:
            from . import fp4
            a = fp4.nvfp4_fake_quant(bf16_round(a), S=fp4_scales[aname])[0]
            wt = fp4.nvfp4_fake_quant(wt, S=fp4_scales[wname])[0]
        elif fp8_scales is not None:
            if amax_out is not None:
                amax_out[aname] = max(amax_out.get(aname, 0.0), float(np.abs(a).max(initial=0.0)))
                if not weights_quantised:
                    amax_out[wname] = float(np.abs(wt).max())
            a = fp8_fake_quant(a, fp8_scales[aname])
            if not weights_quantised:
                wt = fp8_fake_quant(wt, fp8_scales[wname])
        return a @ wt.T

    y = layer_norm(x, w["ln1_g"], w["ln1_b"], eps)
    qkv = mm(y, "w_qkv", "x_qkv") + w["b_qkv"]
    q = qkv[:, :d].reshape(L, heads, dh)
    k = qkv[:, d:2 * d].reshape(L, heads, dh)
    v = qkv[:, 2 * d:].reshape(L, heads, dh)
    q = rope(q, pos, rope_base)
    k = rope(k, pos, rope_base)
    if bf16_attention:
        q, k, v = bf16_round(q), bf16_round(k), bf16_round(v)
    o = attention(q, k, v, n_keys).reshape(L, d)
    x = x + mm(o, "w_o", "x_o") + w["b_o"]
    z = layer_norm(x, w["ln2_g"], w["ln2_b"], eps)
    u = gelu(mm(z, "w_1", "x_1") + w["b_1"])
    x = x + mm(u, "w_2", "x_2") + w["b_2"]
    return x


def _f64_layer(wl: Dict[str, np.ndarray]) -> Dict[str, np.ndarray]:
    return {k: np.asarray(v, dtype=np.float64) for k, v in wl.items()}


def encode_sequence(tokens: np.ndarray, weights: Dict, heads: int, final_ln: bool = True,
                    emb_scale: float = 1.0, eps: float = LN_EPS, rope_base: float = ROPE_BASE,
                    num_layers: Optional[int] = None, n_keys: Optional[int] = None,
                    fp8_state: Optional[List[Dict[str, float]]] = None,
                    amax_out: Optional[List[Dict[str, float]]] = None, bf16_attention: bool = False,
                    fp4_state: Optional[List[Optional[Dict[str, float]]]] = None) -> np.ndarray:
    """Encode ONE sequence (token ids [L]) through the embedding, the layers and the
    optional final LayerNorm.  Positions are 0..L-1.  ``fp4_state[l]`` (tensor scales, or
    None) makes layer l an NVFP4 layer."""
    tokens = np.asarray(tokens, dtype=np.int64)
    emb = np.asarray(weights["emb"], dtype=np.float64)
    x = emb_scale * emb[tokens]
    pos = np.arange(len(tokens))
    layers = weights["layers"] if num_layers is None else weights["layers"][:num_layers]
    for li, wl in enumerate(layers):
        f4 = None if fp4_state is None else fp4_state[li]
        x = encoder_layer(x, pos, _f64_layer(wl), heads, eps, rope_base, n_keys,
                          None if (fp8_state is None or f4 is not None) else fp8_state[li],
                          None if amax_out is None else amax_out[li], bf16_attention, fp4_scales=f4)
    if final_ln:
        x = layer_norm(x, np.asarray(weights["lnf_g"], np.float64), np.asarray(weights["lnf_b"], np.float64), eps)
    return x


def encode_packed(token_ids: np.ndarray, cu: Sequence[int], weights: Dict, heads: int,
                  final_ln: bool = True, seq_subset: Optional[Sequence[int]] = None,
                  emb_scale: float = 1.0, eps: float = LN_EPS, rope_base: float = ROPE_BASE,
                  num_layers: Optional[int] = None, n_keys: Optional[int] = None,
                  fp8_state: Optional[List[Dict[str, float]]] = None,
                  amax_out: Optional[List[Dict[str, float]]] = None,
                  bf16_attention: bool = False,
                  fp4_state: Optional[List[Optional[Dict[str, float]]]] = None) -> Dict[int, np.ndarray]:
    """The packed forward: every sequence [cu[i], cu[i+1]) is encoded on its own, with the
    same steps as ``encode_sequence``; the loop runs layer by layer over the sequences so
    that a layer's weights are converted (and, with an FP8 state, fake-quantised with their
    per-tensor scales) once for the whole call, as the weights are the same for every
    sequence.  Returns {sequence index: [L_i, d] float64}.  ``seq_subset`` limits the work to
    some sequences (packed sequences never interact, so each output is exact on its own)."""
    idx = list(range(len(cu) - 1)) if seq_subset is None else list(seq_subset)
    emb = np.asarray(weights["emb"], dtype=np.float64)
    xs = {i: emb_scale * emb[np.asarray(token_ids[int(cu[i]):int(cu[i + 1])], dtype=np.int64)] for i in idx}
    layers = weights["layers"] if num_layers is None else weights["layers"][:num_layers]
    for li, wl in enumerate(layers):
        f4 = None if fp4_state is None else fp4_state[li]
        scales = None if (fp8_state is None or f4 is not None) else fp8_state[li]
        wl64 = _f64_layer(wl)
        pre = scales is not None and amax_out is None
        if pre:
            wl64 = fp8_quantised_weights(wl64, scales)
        for i in idx:
            xs[i] = encoder_layer(xs[i], np.arange(len(xs[i])), wl64, heads, eps, rope_base, n_keys, scales,
                                  None if amax_out is None else amax_out[li], bf16_attention, weights_quantised=pre,
                                  fp4_scales=f4)
        del wl64
    if final_ln:
        g, b = np.asarray(weights["lnf_g"], np.float64), np.asarray(weights["lnf_b"], np.float64)
        xs = {i: layer_norm(x, g, b, eps) for i, x in xs.items()}
    return xs


def encode_padded(token_ids: np.ndarray, seq_lens: Sequence[int], weights: Dict, heads: int,
                  final_ln: bool = True, seq_subset: Optional[Sequence[int]] = None, **kw) -> Dict[int, np.ndarray]:
    """The padded [B, S] forward with a key padding mask.  Row b's queries see keys
    0..len_b-1 only, so its valid rows equal the sequence encoded alone; rows >= len_b
    of the output are defined as zero."""
    B, S = token_ids.shape
    idx = range(B) if seq_subset is None else seq_subset
    out = {}
    for b in idx:
        L = int(seq_lens[b])
        full = np.zeros((S, np.asarray(weights["emb"]).shape[1]))
        full[:L] = encode_sequence(token_ids[b, :L], weights, heads, final_ln, **kw)
        out[b] = full
    return out


# --------------------------------------------------------------------------- masked-LM head
IGNORE_INDEX = -100


def lm_head(h: np.ndarray, w: Dict[str, np.ndarray]) -> np.ndarray:
    """Logits [T, vocab] of final hidden states h [T, d]: dense + GELU, LayerNorm, then the
    tied embedding as the output projection plus the vocabulary bias."""
    h = np.asarray(h, np.float64)
    z = gelu(h @ np.asarray(w["dense_w"], np.float64).T + np.asarray(w["dense_b"], np.float64))
    z = layer_norm(z, np.asarray(w["ln_g"], np.float64), np.asarray(w["ln_b"], np.float64))
    return z @ np.asarray(w["emb"], np.float64).T + np.asarray(w["bias"], np.float64)


def masked_lm_loss(logits: np.ndarray, targets: Sequence[int]):
    """Per-token cross-entropy log(sum_v exp(l_v)) - l_target (0 where target == -100), the
    sum over scored tokens and their count."""
    logits = np.asarray(logits, np.float64)
    t = np.asarray(targets, np.int64)
    m = logits.max(axis=1)
    lse = m + np.log(np.exp(logits - m[:, None]).sum(axis=1))
    scored = t != IGNORE_INDEX
    per = np.zeros(len(t))
    per[scored] = lse[scored] - logits[np.nonzero(scored)[0], t[scored]]
    return per, float(per.sum()), int(scored.sum())
