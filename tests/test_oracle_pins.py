"""Pins of the float64 oracle against facts that do not come from the oracle itself:
closed forms, invariants, brute force on tiny inputs, the values printed in
tests/golden/, and independent library formulations (torch float64 CPU ops).

Each test is chosen so that a plausible mistake in the oracle (a dropped term, a wrong
sign or index, a transposed operand, a wrong rounding rule) fails at least one of them."""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import esm_oracle as O
from transformer_esm_layer_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------- packing
def test_packing_golden():
    g = _gold("packing.json")
    assert O.cu_seqlens(g["lengths"]).tolist() == g["cu_seqlens"]
    assert max(g["lengths"]) == g["max_seqlen"]
    pos, seg = O.pack_index(g["cu_seqlens"])
    for t, p in g["pos_id_at"].items():
        assert pos[int(t)] == p
    for t, s in g["seg_id_at"].items():
        assert seg[int(t)] == s


def test_pack_index_vs_repeat_formulation():
    lengths = [1, 2, 127, 128, 129, 1024, 3, 1]
    cu = O.cu_seqlens(lengths)
    pos, seg = O.pack_index(cu)
    seg2 = np.repeat(np.arange(len(lengths)), lengths)
    pos2 = np.arange(cu[-1]) - cu[seg2]
    assert np.array_equal(pos, pos2) and np.array_equal(seg, seg2)
    assert np.array_equal(synth.cu_seqlens_from_lengths(lengths), cu.astype(np.int32))


def test_pack_index_empty_sequences():
    cu = [0, 0, 3, 3, 5]
    pos, seg = O.pack_index(cu)
    assert pos.tolist() == [0, 1, 2, 0, 1]
    assert seg.tolist() == [1, 1, 1, 3, 3]


# --------------------------------------------------------------------------- LayerNorm
def test_layernorm_closed_forms():
    rng = np.random.default_rng(0)
    gamma = rng.standard_normal(48)
    beta = rng.standard_normal(48)
    # a constant row normalises to beta
    x = np.full((3, 48), 2.5)
    assert np.allclose(O.layer_norm(x, gamma, beta), beta, atol=1e-12)
    # gamma=1, beta=0: mean 0 and variance var/(var+eps)
    x = rng.standard_normal((5, 48)) * 3 + 1
    y = O.layer_norm(x, np.ones(48), np.zeros(48), eps=1e-5)
    var = x.var(axis=-1)
    assert np.allclose(y.mean(axis=-1), 0, atol=1e-12)
    assert np.allclose(y.var(axis=-1), var / (var + 1e-5), rtol=1e-12)


def test_layernorm_vs_torch():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((7, 96)) * 2 - 0.5
    g = rng.standard_normal(96)
    b = rng.standard_normal(96)
    ref = F.layer_norm(torch.from_numpy(x), (96,), torch.from_numpy(g), torch.from_numpy(b), eps=1e-5).numpy()
    assert np.allclose(O.layer_norm(x, g, b), ref, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------- GELU
def test_gelu_closed_forms():
    assert O.gelu(np.array([0.0]))[0] == 0.0
    x = np.linspace(-6, 6, 101)
    # gelu(x) - gelu(-x) = x  (Phi(x) + Phi(-x) = 1)
    assert np.allclose(O.gelu(x) - O.gelu(-x), x, atol=1e-14)
    # gelu(1) = Phi(1) = 0.841344746068542948...
    assert abs(O.gelu(np.array([1.0]))[0] - 0.8413447460685429) < 1e-15
    for v in (-3.0, -0.7, 0.3, 2.2):
        assert abs(O.gelu(np.array([v]))[0] - v * 0.5 * (1 + math.erf(v / math.sqrt(2)))) < 1e-15


def test_gelu_vs_torch_exact():
    x = np.linspace(-8, 8, 1001)
    ref = F.gelu(torch.from_numpy(x), approximate="none").numpy()
    assert np.allclose(O.gelu(x), ref, rtol=1e-13, atol=1e-15)
    # and it is NOT the tanh approximation
    tanh_ref = F.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    assert np.abs(O.gelu(x) - tanh_ref).max() > 1e-5


# --------------------------------------------------------------------------- RoPE
def _rope_complex(u, pos, base=10000.0):
    """Independent formulation: the pair (u_j, u_{j+half}) is the complex number
    u_j + i u_{j+half}, multiplied by exp(i p theta_j)."""
    half = u.shape[-1] // 2
    z = torch.complex(torch.from_numpy(u[..., :half]), torch.from_numpy(u[..., half:]))
    theta = torch.tensor([base ** (-2.0 * j / u.shape[-1]) for j in range(half)], dtype=torch.float64)
    ang = torch.from_numpy(pos.astype(np.float64))[:, None] * theta[None, :]
    rot = torch.polar(torch.ones_like(ang), ang)[:, None, :]
    w = z * rot
    return np.concatenate([w.real.numpy(), w.imag.numpy()], axis=-1)


def test_rope_vs_complex_and_invariants():
    rng = np.random.default_rng(2)
    for dh in (16, 64):
        u = rng.standard_normal((37, 3, dh))
        pos = np.arange(37) * 13 % 1026
        r = O.rope(u, pos)
        assert np.allclose(r, _rope_complex(u, pos), rtol=1e-12, atol=1e-12)
        # position 0 is the identity
        assert np.allclose(O.rope(u[:1], np.array([0])), u[:1], atol=0)
        # norms are preserved
        assert np.allclose(np.linalg.norm(r, axis=-1), np.linalg.norm(u, axis=-1), rtol=1e-12)


def test_rope_relative_position_invariant():
    """q.k after RoPE depends only on the offset p_q - p_k."""
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 1, 64))
    k = rng.standard_normal((1, 1, 64))
    for off in (0, 1, 7, 300):
        vals = []
        for shift in (0, 5, 111, 700):
            rq = O.rope(q, np.array([shift + off]))
            rk = O.rope(k, np.array([shift]))
            vals.append(float((rq * rk).sum()))
        assert np.allclose(vals, vals[0], rtol=1e-10, atol=1e-12)
    # and it does change with the offset
    a = float((O.rope(q, np.array([3])) * O.rope(k, np.array([0]))).sum())
    b = float((O.rope(q, np.array([4])) * O.rope(k, np.array([0]))).sum())
    assert abs(a - b) > 1e-6


# --------------------------------------------------------------------------- attention
def _attention_bruteforce(q, k, v):
    L, H, dh = q.shape
    out = np.zeros_like(q)
    for h in range(H):
        for t in range(L):
            s = [sum(q[t, h, c] * k[j, h, c] for c in range(dh)) / math.sqrt(dh) for j in range(L)]
            m = max(s)
            e = [math.exp(x - m) for x in s]
            z = sum(e)
            for c in range(dh):
                out[t, h, c] = sum(e[j] / z * v[j, h, c] for j in range(L))
    return out


def test_attention_bruteforce_tiny():
    rng = np.random.default_rng(4)
    q, k, v = (rng.standard_normal((5, 2, 4)) for _ in range(3))
    assert np.allclose(O.attention(q, k, v), _attention_bruteforce(q, k, v), rtol=1e-12, atol=1e-13)


def test_attention_vs_torch_sdpa():
    rng = np.random.default_rng(5)
    q, k, v = (rng.standard_normal((33, 4, 16)) * 2 for _ in range(3))
    tq, tk, tv = (torch.from_numpy(a).permute(1, 0, 2) for a in (q, k, v))
    ref = F.scaled_dot_product_attention(tq, tk, tv).permute(1, 0, 2).numpy()
    assert np.allclose(O.attention(q, k, v), ref, rtol=1e-11, atol=1e-12)
    # padding mask: only the first 20 keys are visible
    mask = torch.zeros(33, 33, dtype=torch.bool)
    mask[:, :20] = True
    ref_m = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask).permute(1, 0, 2).numpy()
    assert np.allclose(O.attention(q, k, v, n_keys=20), ref_m, rtol=1e-11, atol=1e-12)


def test_attention_special_cases():
    rng = np.random.default_rng(6)
    # one token: the output is v
    q, k, v = (rng.standard_normal((1, 3, 8)) for _ in range(3))
    assert np.allclose(O.attention(q, k, v), v)
    # all keys equal: the output is the mean of V
    q = rng.standard_normal((6, 2, 8))
    k = np.repeat(rng.standard_normal((1, 2, 8)), 6, axis=0)
    v = rng.standard_normal((6, 2, 8))
    assert np.allclose(O.attention(q, k, v), np.broadcast_to(v.mean(axis=0), v.shape))
    # softmax rows sum to one: V = ones gives ones
    k = rng.standard_normal((6, 2, 8))
    assert np.allclose(O.attention(q, k, np.ones_like(v)), 1.0)
    # permuting keys and values together changes nothing (bidirectional, no positions)
    perm = rng.permutation(6)
    assert np.allclose(O.attention(q, k, v), O.attention(q, k[perm], v[perm]))


# --------------------------------------------------------------------------- layer / model
def _torch_layer(x, pos, w, heads, eps=1e-5):
    """Independent formulation of the pre-LN layer with torch float64 modules."""
    t = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    X = t(x)
    L, d = X.shape
    dh = d // heads
    y = F.layer_norm(X, (d,), t(w["ln1_g"]), t(w["ln1_b"]), eps)
    q, k, v = F.linear(y, t(w["w_qkv"]), t(w["b_qkv"])).split(d, dim=-1)
    q = torch.from_numpy(_rope_complex(q.reshape(L, heads, dh).numpy(), pos))
    k = torch.from_numpy(_rope_complex(k.reshape(L, heads, dh).numpy(), pos))
    v = v.reshape(L, heads, dh)
    o = F.scaled_dot_product_attention(q.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1))
    X = X + F.linear(o.transpose(0, 1).reshape(L, d), t(w["w_o"]), t(w["b_o"]))
    z = F.layer_norm(X, (d,), t(w["ln2_g"]), t(w["ln2_b"]), eps)
    X = X + F.linear(F.gelu(F.linear(z, t(w["w_1"]), t(w["b_1"]))), t(w["w_2"]), t(w["b_2"]))
    return X.numpy()


def _scaled_weights(g, seed, ln_random=True, scale=10.0):
    w = synth.model_weights(g, seed, "fp32", ln_random=ln_random)
    # enlarge the linear weights so attention is far from uniform and every term matters
    for wl in w["layers"]:
        for k in ("w_qkv", "w_o", "w_1", "w_2", "b_qkv", "b_o", "b_1", "b_2"):
            wl[k] = wl[k] * scale
    return w


def test_layer_vs_torch_formulation():
    g = synth.TINY
    w = _scaled_weights(g, 11)
    rng = np.random.default_rng(7)
    x = rng.standard_normal((23, g.hidden))
    pos = np.arange(23)
    wl = {k: np.asarray(v, np.float64) for k, v in w["layers"][0].items()}
    assert np.allclose(O.encoder_layer(x, pos, wl, g.heads), _torch_layer(x, pos, wl, g.heads),
                       rtol=1e-10, atol=1e-10)


def test_zero_weights_layer_is_identity_and_model_is_final_ln_of_embedding():
    g = synth.TINY
    w = synth.model_weights(g, 0, "fp32", ln_random=True)
    for wl in w["layers"]:
        for k in ("w_qkv", "b_qkv", "w_o", "b_o", "w_1", "b_1", "w_2", "b_2"):
            wl[k] = np.zeros_like(wl[k])
    tok = np.array([0, 5, 9, 23, 2])
    x = np.asarray(w["emb"], np.float64)[tok]
    wl = {k: np.asarray(v, np.float64) for k, v in w["layers"][0].items()}
    assert np.array_equal(O.encoder_layer(x, np.arange(5), wl, g.heads), x)
    out = O.encode_sequence(tok, w, g.heads, final_ln=True)
    assert np.allclose(out, O.layer_norm(x, w["lnf_g"], w["lnf_b"]), atol=1e-12)


def test_packed_equals_joint_block_diagonal_formulation():
    """The oracle encodes each packed sequence alone.  An independent joint formulation
    (one [T, d] tensor, positions from the repeat formula, a block-diagonal attention
    mask from cu_seqlens) must give the same hidden states."""
    g = synth.TINY
    w = _scaled_weights(g, 12)
    lengths = [5, 1, 9, 3]
    cu = O.cu_seqlens(lengths)
    tok = synth.tokens_for_lengths(np.random.default_rng(8), lengths)
    ref = O.encode_packed(tok, cu, w, g.heads, final_ln=True)
    T = int(cu[-1])
    seg = np.repeat(np.arange(len(lengths)), lengths)
    pos = np.arange(T) - cu[seg]
    t = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    X = t(w["emb"])[torch.from_numpy(tok.astype(np.int64))]
    d, H = g.hidden, g.heads
    dh = d // H
    mask = torch.from_numpy(seg[:, None] == seg[None, :])
    for wl in w["layers"]:
        y = F.layer_norm(X, (d,), t(wl["ln1_g"]), t(wl["ln1_b"]), 1e-5)
        q, k, v = F.linear(y, t(wl["w_qkv"]), t(wl["b_qkv"])).split(d, dim=-1)
        q = torch.from_numpy(_rope_complex(q.reshape(T, H, dh).numpy(), pos))
        k = torch.from_numpy(_rope_complex(k.reshape(T, H, dh).numpy(), pos))
        o = F.scaled_dot_product_attention(q.transpose(0, 1), k.transpose(0, 1),
                                           v.reshape(T, H, dh).transpose(0, 1), attn_mask=mask)
        X = X + F.linear(o.transpose(0, 1).reshape(T, d), t(wl["w_o"]), t(wl["b_o"]))
        z = F.layer_norm(X, (d,), t(wl["ln2_g"]), t(wl["ln2_b"]), 1e-5)
        X = X + F.linear(F.gelu(F.linear(z, t(wl["w_1"]), t(wl["b_1"]))), t(wl["w_2"]), t(wl["b_2"]))
    X = F.layer_norm(X, (d,), t(w["lnf_g"]), t(w["lnf_b"]), 1e-5).numpy()
    for i in range(len(lengths)):
        assert np.allclose(ref[i], X[cu[i]:cu[i + 1]], rtol=1e-9, atol=1e-10)


def test_padded_equals_packed_and_masked_formulation():
    g = synth.TINY
    w = _scaled_weights(g, 13)
    lengths = [6, 2, 9]
    S = 12
    tok = synth.tokens_for_lengths(np.random.default_rng(9), lengths)
    cu = O.cu_seqlens(lengths)
    padded = synth.pad_tokens(tok, lengths, S)
    pk = O.encode_packed(tok, cu, w, g.heads)
    pd = O.encode_padded(padded, lengths, w, g.heads)
    for b, L in enumerate(lengths):
        assert np.allclose(pd[b][:L], pk[b], atol=1e-12)
        assert np.all(pd[b][L:] == 0)
    # joint masked formulation for one padded row: pad tokens are present as queries and
    # as (masked) keys; valid rows must be unaffected by them
    b, L = 0, lengths[0]
    X = np.asarray(w["emb"], np.float64)[padded[b]]
    t = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    d, H = g.hidden, g.heads
    dh = d // H
    mask = torch.zeros(S, S, dtype=torch.bool)
    mask[:, :L] = True
    Xt = t(X)
    for wl in w["layers"]:
        y = F.layer_norm(Xt, (d,), t(wl["ln1_g"]), t(wl["ln1_b"]), 1e-5)
        q, k, v = F.linear(y, t(wl["w_qkv"]), t(wl["b_qkv"])).split(d, dim=-1)
        q = torch.from_numpy(_rope_complex(q.reshape(S, H, dh).numpy(), np.arange(S)))
        k = torch.from_numpy(_rope_complex(k.reshape(S, H, dh).numpy(), np.arange(S)))
        o = F.scaled_dot_product_attention(q.transpose(0, 1), k.transpose(0, 1),
                                           v.reshape(S, H, dh).transpose(0, 1), attn_mask=mask)
        Xt = Xt + F.linear(o.transpose(0, 1).reshape(S, d), t(wl["w_o"]), t(wl["b_o"]))
        z = F.layer_norm(Xt, (d,), t(wl["ln2_g"]), t(wl["ln2_b"]), 1e-5)
        Xt = Xt + F.linear(F.gelu(F.linear(z, t(wl["w_1"]), t(wl["b_1"]))), t(wl["w_2"]), t(wl["b_2"]))
    Xt = F.layer_norm(Xt, (d,), t(w["lnf_g"]), t(w["lnf_b"]), 1e-5).numpy()
    assert np.allclose(pd[b][:L], Xt[:L], rtol=1e-9, atol=1e-10)


def test_segment_permutation_permutes_outputs():
    g = synth.TINY
    w = _scaled_weights(g, 14)
    lengths = [4, 7, 2]
    tok = synth.tokens_for_lengths(np.random.default_rng(10), lengths)
    cu = O.cu_seqlens(lengths)
    out = O.encode_packed(tok, cu, w, g.heads)
    order = [2, 0, 1]
    seqs = [tok[cu[i]:cu[i + 1]] for i in order]
    tok2 = np.concatenate(seqs)
    cu2 = O.cu_seqlens([lengths[i] for i in order])
    out2 = O.encode_packed(tok2, cu2, w, g.heads)
    for j, i in enumerate(order):
        assert np.array_equal(out2[j], out[i])


# --------------------------------------------------------------------------- bf16
def test_bf16_round_vs_torch_cast():
    rng = np.random.default_rng(18)
    x = np.concatenate([rng.standard_normal(50000) * s for s in (1e-3, 1.0, 300.0)])
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.bf16_round(x.astype(np.float32)), ref)
    # exact halfway cases go to the even significand
    assert O.bf16_round(np.array([1.0 + 2.0 ** -8]))[0] == 1.0
    assert O.bf16_round(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 1.0 + 2.0 ** -6


def test_bf16_attention_operands_are_rounded():
    g = synth.TINY
    w = _scaled_weights(g, 19)
    wl = {k: np.asarray(v, np.float64) for k, v in w["layers"][0].items()}
    rng = np.random.default_rng(20)
    x = rng.standard_normal((9, g.hidden))
    a = O.encoder_layer(x, np.arange(9), wl, g.heads)
    b = O.encoder_layer(x, np.arange(9), wl, g.heads, bf16_attention=True)
    rel = np.linalg.norm(a - b) / np.linalg.norm(a)
    assert 0 < rel < 2e-2
    # rounding already-bf16 operands is the identity: attention on bf16 values is unchanged
    q = O.bf16_round(rng.standard_normal((5, 2, 8)))
    assert np.array_equal(O.bf16_round(q), q)


# --------------------------------------------------------------------------- FP8
def _e4m3_decode(code: int) -> float:
    """Decode one E4M3 byte from its bit fields (OCP definition)."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * m * 2.0 ** -9
    return s * (1 + m / 8.0) * 2.0 ** (e - 7)


def test_e4m3_exhaustive_codes():
    gold = _gold("fp8_recipe.json")
    vals = np.array([_e4m3_decode(c) for c in range(256)])
    finite = vals[np.isfinite(vals)]
    pos = np.unique(finite[finite > 0])
    assert len(pos) == gold["e4m3_finite_positive_count"]
    assert pos.max() == gold["e4m3_max"] and pos.min() == gold["e4m3_min_subnormal"]
    # every representable value is a fixed point of the rounding
    assert np.array_equal(O.e4m3_round(finite), finite)
    # midpoints round to the neighbour with the even mantissa (code with low bit 0)
    codes = [c for c in range(1, 0x7E)]
    for c in codes:
        lo, hi = _e4m3_decode(c), _e4m3_decode(c + 1)
        mid = 0.5 * (lo + hi)
        want = lo if (c & 1) == 0 else hi
        assert O.e4m3_round(np.array([mid]))[0] == want, (c, lo, hi)
        assert O.e4m3_round(np.array([-mid]))[0] == -want
        # just off the midpoint goes to the nearer value
        assert O.e4m3_round(np.array([mid - (hi - lo) * 1e-3]))[0] == lo
        assert O.e4m3_round(np.array([mid + (hi - lo) * 1e-3]))[0] == hi
    # saturation
    assert np.array_equal(O.e4m3_round(np.array([448.0, 460.0, 1e6, -1e6])), [448.0, 448.0, 448.0, -448.0])


def test_e4m3_vs_torch_cast():
    rng = np.random.default_rng(15)
    x = np.concatenate([rng.standard_normal(20000) * s for s in (0.003, 0.05, 1.0, 60.0)])
    x = x[np.abs(x) < 440]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(O.e4m3_round(x), ref)


def test_fp8_scale_update():
    gold = _gold("fp8_recipe.json")
    n = gold["amax_history_len"]
    h = np.zeros(n)
    h, s = O.fp8_scale_update(h, 1.0, 0.0)
    assert s == 1.0                                   # zero max keeps the old scale
    h, s = O.fp8_scale_update(h, 1.0, gold["scale_example"]["history_max"])
    assert s == gold["scale_example"]["scale"]        # 448 / 3.5 = 128
    h, s = O.fp8_scale_update(h, s, 1.0)              # a smaller amax does not lower the max
    assert s == 128.0
    for _ in range(n - 1):
        h, s = O.fp8_scale_update(h, s, 1.0)
    assert s == 448.0                                 # 3.5 rolled out after n calls
    assert len(h) == n


def test_fp8_fake_quant_layer_close_to_exact():
    """With scales from the operands' own amax, the FP8 layer stays within a few percent
    of the exact layer (E4M3 has a 3-bit mantissa: relative rounding error <= 2^-4)."""
    g = synth.TINY
    w = synth.model_weights(g, 16, "fp32")
    wl = {k: np.asarray(v, np.float64) for k, v in w["layers"][0].items()}
    rng = np.random.default_rng(17)
    x = rng.standard_normal((31, g.hidden))
    amax = {}
    ones = {k: 1.0 for k in O.FP8_TENSORS}
    O.encoder_layer(x, np.arange(31), wl, g.heads, fp8_scales=ones, amax_out=amax)
    scales = {k: 448.0 / amax[k] for k in O.FP8_TENSORS}
    exact = O.encoder_layer(x, np.arange(31), wl, g.heads)
    q8 = O.encoder_layer(x, np.arange(31), wl, g.heads, fp8_scales=scales)
    rel = np.linalg.norm(q8 - exact) / np.linalg.norm(exact)
    assert 0 < rel < 5e-2
    # and the amax of a weight is its max |value|
    assert amax["w_o"] == np.abs(wl["w_o"]).max()


# --------------------------------------------------------------------------- geometry
def _param_count(g):
    d, f, V = g.hidden, g.ffn, g.vocab
    per_layer = 4 * d + (3 * d * d + 3 * d) + (d * d + d) + (f * d + f) + (d * f + d)
    return V * d + g.num_layers * per_layer + 2 * d


def test_geometry_golden():
    gold = _gold("esm2_geometry.json")
    for key, g in (("esm2_650m", synth.ESM2_650M), ("esm2_3b", synth.ESM2_3B)):
        G = gold[key]
        assert (g.num_layers, g.hidden, g.heads, g.ffn, g.vocab, g.max_positions, g.head_dim) == \
            (G["num_layers"], G["hidden"], G["heads"], G["ffn"], G["vocab"], G["max_positions"], G["head_dim"])
        n = _param_count(g)
        # the encoder layout reproduces the nominal size within 10%
        assert abs(n / G["nominal_params"] - 1) < 0.1, n
    assert gold["max_residues"] + 2 <= synth.ESM2_650M.max_positions


# --------------------------------------------------------------------------- masked-LM head
def _lm_weights(d=48, V=33, seed=5):
    r = np.random.default_rng(seed)
    return {"dense_w": r.standard_normal((d, d)) * 0.2, "dense_b": r.standard_normal(d) * 0.1,
            "ln_g": 1 + 0.1 * r.standard_normal(d), "ln_b": 0.1 * r.standard_normal(d),
            "emb": r.standard_normal((V, d)) * 0.3, "bias": r.standard_normal(V) * 0.1}


def test_lm_head_zero_dense_gives_embedding_of_ln_bias():
    """dense = 0: GELU(0) = 0, LayerNorm of a constant row is beta, so every token's logits
    are emb . beta + bias."""
    w = _lm_weights()
    w["dense_w"][:] = 0
    w["dense_b"][:] = 0
    h = np.random.default_rng(1).standard_normal((7, 48))
    got = O.lm_head(h, w)
    want = w["emb"] @ w["ln_b"] + w["bias"]
    assert np.allclose(got, np.broadcast_to(want, got.shape), atol=1e-12)


def test_lm_head_vs_torch_formulation():
    w = _lm_weights()
    h = np.random.default_rng(2).standard_normal((9, 48))
    th = torch.from_numpy(h)
    z = F.gelu(F.linear(th, torch.from_numpy(w["dense_w"]), torch.from_numpy(w["dense_b"])))
    z = F.layer_norm(z, (48,), torch.from_numpy(w["ln_g"]), torch.from_numpy(w["ln_b"]), eps=1e-5)
    ref = F.linear(z, torch.from_numpy(w["emb"]), torch.from_numpy(w["bias"])).numpy()
    assert np.allclose(O.lm_head(h, w), ref, atol=1e-12, rtol=1e-12)


def test_masked_lm_loss_bruteforce_and_invariants():
    r = np.random.default_rng(3)
    logits = r.standard_normal((6, 33)) * 4
    targets = [0, 5, O.IGNORE_INDEX, 32, 7, O.IGNORE_INDEX]
    per, total, n = O.masked_lm_loss(logits, targets)
    for i, t in enumerate(targets):  # plain loops with math.exp / math.log
        if t == O.IGNORE_INDEX:
            assert per[i] == 0.0
            continue
        z = sum(math.exp(v) for v in logits[i])
        assert abs(per[i] - (math.log(z) - logits[i, t])) < 1e-12
    assert n == 4 and abs(total - per.sum()) < 1e-12
    # shift invariance, uniform logits -> log(V), a dominant target logit -> ~0
    per2, _, _ = O.masked_lm_loss(logits + 123.0, targets)
    assert np.allclose(per2, per, atol=1e-9)
    perU, totU, _ = O.masked_lm_loss(np.zeros((3, 33)), [1, 2, 3])
    assert np.allclose(perU, math.log(33)) and abs(totU - 3 * math.log(33)) < 1e-12
    big = np.zeros((1, 33))
    big[0, 4] = 60.0
    assert O.masked_lm_loss(big, [4])[1] < 1e-20
    # torch cross_entropy with ignore_index, summed
    ref = F.cross_entropy(torch.from_numpy(logits), torch.tensor(targets), ignore_index=-100, reduction="sum")
    assert abs(total - float(ref)) < 1e-10
