"""Pins of the float64 backward oracle against facts that do not come from it: central
finite differences of the float64 forward (``oracle.esm_oracle``, itself pinned in
test_oracle_pins.py), adjoint identities, invariances of the forward, and an independent
torch float64 formulation differentiated by autograd.

A dropped term, a wrong sign, a transposed operand or a missing scale anywhere in the
chain rule moves at least one finite-difference check by far more than its tolerance."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import logsumexp

from oracle import backward as B
from oracle import esm_oracle as O
from transformer_esm_layer_gb300 import synth

SMALL = synth.Geometry(num_layers=2, hidden=16, heads=2, ffn=32, vocab=33)


def _fd(f, x, idx, h=1e-6):
    """Central difference of scalar f at x along coordinate idx."""
    xp = x.copy()
    xm = x.copy()
    xp[idx] += h
    xm[idx] -= h
    return (f(xp) - f(xm)) / (2 * h)


def _sample_idx(rng, shape, n):
    return [tuple(int(rng.integers(0, s)) for s in shape) for _ in range(n)]


def _small_weights(seed, scale=4.0, layers=2):
    w = synth.model_weights(SMALL, seed, "fp32", ln_random=True, num_layers=layers)
    w = {"emb": np.asarray(w["emb"], np.float64) * 20, "lnf_g": np.asarray(w["lnf_g"], np.float64),
         "lnf_b": np.asarray(w["lnf_b"], np.float64),
         "layers": [{k: np.asarray(v, np.float64) for k, v in wl.items()} for wl in w["layers"]]}
    for wl in w["layers"]:  # larger weights: every term of the chain rule matters
        for k in ("w_qkv", "w_o", "w_1", "w_2", "b_qkv", "b_o", "b_1", "b_2"):
            wl[k] = wl[k] * scale * 10
    return w


# --------------------------------------------------------------------------- pieces
def test_gelu_grad_closed_form_and_finite_differences():
    assert B.gelu_grad(np.array([0.0]))[0] == pytest.approx(0.5, abs=1e-15)
    # far tails: the derivative tends to 0 (left) and 1 (right)
    assert abs(B.gelu_grad(np.array([-12.0]))[0]) < 1e-20
    assert B.gelu_grad(np.array([12.0]))[0] == pytest.approx(1.0, abs=1e-15)
    a = np.linspace(-6, 6, 97)
    fd = (O.gelu(a + 1e-6) - O.gelu(a - 1e-6)) / 2e-6
    assert np.allclose(B.gelu_grad(a), fd, rtol=1e-7, atol=1e-8)


def test_layer_norm_backward_finite_differences_and_invariants():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4, 12)) * 2 + 0.3
    g = rng.standard_normal(12) + 1
    b = rng.standard_normal(12)
    dy = rng.standard_normal((4, 12))
    dx, dg, db = B.layer_norm_backward(x, g, dy)
    J = lambda xx: float((O.layer_norm(xx, g, b) * dy).sum())
    for idx in _sample_idx(rng, x.shape, 12):
        assert dx[idx] == pytest.approx(_fd(J, x, idx), rel=1e-6, abs=1e-8)
    Jg = lambda gg: float((O.layer_norm(x, gg, b) * dy).sum())
    Jb = lambda bb: float((O.layer_norm(x, g, bb) * dy).sum())
    for i in range(12):
        assert dg[i] == pytest.approx(_fd(Jg, g, (i,)), rel=1e-6, abs=1e-8)
        assert db[i] == pytest.approx(_fd(Jb, b, (i,)), rel=1e-6, abs=1e-8)
    # adding a constant to a row leaves LN unchanged, so each row of dx sums to zero
    assert np.allclose(dx.sum(axis=1), 0, atol=1e-12)
    # with eps = 0, scaling a row leaves LN unchanged: dx is orthogonal to x - mean
    dx0, _, _ = B.layer_norm_backward(x, g, dy, eps=0.0)
    assert np.allclose((dx0 * (x - x.mean(axis=1, keepdims=True))).sum(axis=1), 0, atol=1e-11)


def test_rope_backward_is_the_adjoint_of_rope():
    rng = np.random.default_rng(4)
    u = rng.standard_normal((9, 3, 8))
    gr = rng.standard_normal((9, 3, 8))
    pos = rng.integers(0, 1000, 9)
    lhs = float((O.rope(u, pos) * gr).sum())
    rhs = float((u * B.rope_backward(gr, pos)).sum())
    assert lhs == pytest.approx(rhs, rel=1e-12)
    # and, a rotation, it undoes RoPE
    assert np.allclose(B.rope_backward(O.rope(u, pos), pos), u, atol=1e-12)


def test_attention_lse_normalises_the_softmax():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((7, 2, 8)) * 3
    k = rng.standard_normal((7, 2, 8)) * 3
    lse = B.attention_lse(q, k)
    s = np.einsum("ihd,jhd->ihj", q, k) / np.sqrt(8)
    assert np.allclose(lse, logsumexp(s, axis=-1), rtol=1e-13, atol=1e-13)


def test_attention_backward_finite_differences_and_invariants():
    rng = np.random.default_rng(6)
    L, H, dh = 6, 2, 8
    q, k, v, do = (rng.standard_normal((L, H, dh)) * 2 for _ in range(4))
    dq, dk, dv = B.attention_backward(q, k, v, do)
    for name, t, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        def J(tt, name=name):
            a = {"q": q, "k": k, "v": v}
            a[name] = tt
            return float((O.attention(a["q"], a["k"], a["v"]) * do).sum())
        for idx in _sample_idx(rng, t.shape, 10):
            assert g[idx] == pytest.approx(_fd(J, t, idx), rel=1e-6, abs=1e-8), name
    # adding one vector to every key shifts each query's scores by a constant: sum_j dk_j = 0
    assert np.allclose(dk.sum(axis=0), 0, atol=1e-12)
    # the softmax rows sum to one: sum_j dv_j = sum_i do_i
    assert np.allclose(dv.sum(axis=0), do.sum(axis=0), atol=1e-12)


# --------------------------------------------------------------------------- layer / encoder
def test_layer_backward_finite_differences():
    rng = np.random.default_rng(7)
    w = _small_weights(8)["layers"][0]
    L = 7
    x = rng.standard_normal((L, SMALL.hidden)) * 2
    pos = np.arange(L)
    d_out = rng.standard_normal((L, SMALL.hidden))
    dx, grads = B.encoder_layer_backward(x, pos, w, SMALL.heads, d_out)
    J = lambda xx: float((O.encoder_layer(xx, pos, w, SMALL.heads) * d_out).sum())
    for idx in _sample_idx(rng, x.shape, 10):
        assert dx[idx] == pytest.approx(_fd(J, x, idx), rel=1e-5, abs=1e-7)
    for name in B.PARAM_NAMES:
        def Jp(pp, name=name):
            ww = dict(w)
            ww[name] = pp
            return float((O.encoder_layer(x, pos, ww, SMALL.heads) * d_out).sum())
        assert grads[name].shape == w[name].shape
        for idx in _sample_idx(rng, w[name].shape, 6):
            assert grads[name][idx] == pytest.approx(_fd(Jp, w[name], idx), rel=1e-5, abs=1e-7), name


def test_packed_encoder_backward_finite_differences():
    """Two sequences packed, two layers, final LayerNorm, embedding table."""
    rng = np.random.default_rng(9)
    w = _small_weights(10)
    lengths = [5, 3]
    cu = O.cu_seqlens(lengths)
    tok = synth.tokens_for_lengths(rng, lengths).astype(np.int64)
    T = int(cu[-1])
    d_out = rng.standard_normal((T, SMALL.hidden))
    g = B.encode_packed_backward(tok, cu, w, SMALL.heads, d_out, emb_scale=0.7)

    def J(ww):
        outs = O.encode_packed(tok, cu, ww, SMALL.heads, emb_scale=0.7)
        return float(sum((outs[i] * d_out[cu[i]:cu[i + 1]]).sum() for i in range(len(lengths))))

    def perturbed(path, pp):
        ww = {"emb": w["emb"], "lnf_g": w["lnf_g"], "lnf_b": w["lnf_b"], "layers": [dict(x) for x in w["layers"]]}
        if len(path) == 1:
            ww[path[0]] = pp
        else:
            ww["layers"][path[0]][path[1]] = pp
        return ww

    for name in ("emb", "lnf_g", "lnf_b"):
        used = np.unique(tok) if name == "emb" else None
        for idx in _sample_idx(rng, w[name].shape, 6):
            if name == "emb" and rng.random() < 0.7:
                idx = (int(rng.choice(used)), idx[1])
            assert g[name][idx] == pytest.approx(_fd(lambda pp: J(perturbed((name,), pp)), w[name], idx),
                                                 rel=1e-5, abs=1e-7), name
    for li in range(2):
        for name in B.PARAM_NAMES:
            base = w["layers"][li][name]
            for idx in _sample_idx(rng, base.shape, 3):
                fd = _fd(lambda pp: J(perturbed((li, name), pp)), base, idx)
                assert g["layers"][li][name][idx] == pytest.approx(fd, rel=1e-5, abs=1e-7), (li, name)
    # tokens that never occur get no embedding gradient
    unused = np.setdiff1d(np.arange(SMALL.vocab), tok)
    assert np.all(g["emb"][unused] == 0)


def _torch_encoder(tok, w, heads, emb_scale, params):
    """Independent torch float64 formulation of one sequence's encoder, differentiable in
    the tensors of ``params`` (same keys as the weights)."""
    L = len(tok)
    d = w["emb"].shape[1]
    dh = d // heads
    half = dh // 2
    pos = torch.arange(L, dtype=torch.float64)
    theta = 10000.0 ** (-torch.arange(half, dtype=torch.float64) * 2 / dh)
    rot = torch.polar(torch.ones(L, half, dtype=torch.float64), pos[:, None] * theta[None, :])[:, None, :]

    def rope_t(u):  # pairs (j, j + half) as complex numbers times e^{i phi}
        z = torch.complex(u[..., :half], u[..., half:]) * rot
        return torch.cat([z.real, z.imag], dim=-1)

    X = params["emb"][torch.as_tensor(tok)] * emb_scale
    for lp in params["layers"]:
        y = F.layer_norm(X, (d,), lp["ln1_g"], lp["ln1_b"], 1e-5)
        q, k, v = F.linear(y, lp["w_qkv"], lp["b_qkv"]).split(d, dim=-1)
        q, k, v = (t.reshape(L, heads, dh) for t in (q, k, v))
        q, k = rope_t(q), rope_t(k)
        o = F.scaled_dot_product_attention(q.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1))
        X = X + F.linear(o.transpose(0, 1).reshape(L, d), lp["w_o"], lp["b_o"])
        z = F.layer_norm(X, (d,), lp["ln2_g"], lp["ln2_b"], 1e-5)
        X = X + F.linear(F.gelu(F.linear(z, lp["w_1"], lp["b_1"])), lp["w_2"], lp["b_2"])
    return F.layer_norm(X, (d,), params["lnf_g"], params["lnf_b"], 1e-5)


def test_encoder_backward_vs_torch_autograd():
    rng = np.random.default_rng(11)
    w = _small_weights(12, scale=2.0)
    tok = synth.tokens_for_lengths(rng, [9]).astype(np.int64)
    d_out = rng.standard_normal((9, SMALL.hidden))
    g = B.encode_sequence_backward(tok, w, SMALL.heads, d_out, emb_scale=1.3)
    t = lambda a: torch.tensor(np.asarray(a, np.float64), requires_grad=True)
    params = {"emb": t(w["emb"]), "lnf_g": t(w["lnf_g"]), "lnf_b": t(w["lnf_b"]),
              "layers": [{k: t(v) for k, v in wl.items()} for wl in w["layers"]]}
    out = _torch_encoder(tok, w, SMALL.heads, 1.3, params)
    (out * torch.from_numpy(d_out)).sum().backward()
    for name in ("emb", "lnf_g", "lnf_b"):
        assert np.allclose(g[name], params[name].grad.numpy(), rtol=1e-9, atol=1e-10), name
    for li, lp in enumerate(params["layers"]):
        for name in B.PARAM_NAMES:
            assert np.allclose(g["layers"][li][name], lp[name].grad.numpy(), rtol=1e-9, atol=1e-10), (li, name)


# --------------------------------------------------------------------------- masked-LM head
def _lm_weights(d=16, V=33, seed=21):
    rng = np.random.default_rng(seed)
    return {"dense_w": rng.standard_normal((d, d)) * 0.4, "dense_b": rng.standard_normal(d) * 0.2,
            "ln_g": 1 + 0.1 * rng.standard_normal(d), "ln_b": 0.1 * rng.standard_normal(d),
            "emb": rng.standard_normal((V, d)), "bias": 0.1 * rng.standard_normal(V)}


def _mean_loss(h, w, t):
    _, s, n = O.masked_lm_loss(O.lm_head(h, w), t)
    return s / n


def test_lm_head_backward_finite_differences():
    rng = np.random.default_rng(22)
    w = _lm_weights()
    h = rng.standard_normal((9, 16)) * 1.5
    t = rng.integers(0, 33, 9)
    t[[1, 4, 7]] = -100
    g = B.lm_head_backward(h, w, t)
    for idx in _sample_idx(rng, h.shape, 10):
        assert g["hidden"][idx] == pytest.approx(_fd(lambda hh: _mean_loss(hh, w, t), h, idx), rel=1e-6, abs=1e-8)
    for name in ("dense_w", "dense_b", "ln_g", "ln_b", "emb", "bias"):
        def J(pp, name=name):
            ww = dict(w)
            ww[name] = pp
            return _mean_loss(h, ww, t)
        for idx in _sample_idx(rng, w[name].shape, 6):
            assert g[name][idx] == pytest.approx(_fd(J, w[name], idx), rel=1e-6, abs=1e-8), name
    # the loss gradient of each scored row of logits sums to zero, so the bias gradient does too
    assert abs(g["bias"].sum()) < 1e-12


def test_lm_head_backward_vs_torch_autograd_and_unscored_rows():
    rng = np.random.default_rng(23)
    w = _lm_weights(seed=24)
    h = rng.standard_normal((7, 16))
    t = np.array([3, -100, 5, 32, -100, 0, 7])
    g = B.lm_head_backward(h, w, t)
    T_ = lambda a: torch.tensor(np.asarray(a, np.float64), requires_grad=True)
    P = {k: T_(v) for k, v in w.items()}
    H = T_(h)
    a = F.linear(H, P["dense_w"], P["dense_b"])
    z = F.layer_norm(F.gelu(a), (16,), P["ln_g"], P["ln_b"], 1e-5)
    logits = F.linear(z, P["emb"], P["bias"])
    loss = F.cross_entropy(logits, torch.from_numpy(t), ignore_index=-100, reduction="mean")
    loss.backward()
    assert np.allclose(g["hidden"], H.grad.numpy(), rtol=1e-10, atol=1e-12)
    for k in P:
        assert np.allclose(g[k], P[k].grad.numpy(), rtol=1e-10, atol=1e-12), k
    # unscored rows get no gradient; nothing scored gives zero everywhere
    assert np.all(g["hidden"][[1, 4]] == 0)
    g0 = B.lm_head_backward(h, w, np.full(7, -100))
    assert all(np.all(v == 0) for v in g0.values())


def test_lm_head_backward_with_a_global_count():
    """With the mean taken over a given count N (the scored tokens of a whole data-parallel
    batch), the gradient is that of sum_scored CE / N: checked by finite differences of that
    loss, and torch autograd of cross-entropy with reduction "sum" divided by N.  Two shares
    of a batch with uneven scored counts, each differentiated with the batch's count, add up
    to the whole batch's gradient."""
    rng = np.random.default_rng(25)
    w = _lm_weights(seed=26)
    h = rng.standard_normal((11, 16))
    t = rng.integers(0, 33, 11)
    t[[0, 2, 3, 9]] = -100
    N = 17
    g = B.lm_head_backward(h, w, t, count=N)

    def loss_over_n(hh, ww):
        _, s, _ = O.masked_lm_loss(O.lm_head(hh, ww), t)
        return s / N

    for idx in _sample_idx(rng, h.shape, 8):
        assert g["hidden"][idx] == pytest.approx(_fd(lambda hh: loss_over_n(hh, w), h, idx), rel=1e-6, abs=1e-8)
    for idx in _sample_idx(rng, w["emb"].shape, 4):
        def J(pp):
            ww = dict(w)
            ww["emb"] = pp
            return loss_over_n(h, ww)
        assert g["emb"][idx] == pytest.approx(_fd(J, w["emb"], idx), rel=1e-6, abs=1e-8)
    T_ = lambda a: torch.tensor(np.asarray(a, np.float64), requires_grad=True)
    P = {k: T_(v) for k, v in w.items()}
    H = T_(h)
    z = F.layer_norm(F.gelu(F.linear(H, P["dense_w"], P["dense_b"])), (16,), P["ln_g"], P["ln_b"], 1e-5)
    loss = F.cross_entropy(F.linear(z, P["emb"], P["bias"]), torch.from_numpy(t), ignore_index=-100,
                           reduction="sum") / N
    loss.backward()
    assert np.allclose(g["hidden"], H.grad.numpy(), rtol=1e-10, atol=1e-12)
    for k in P:
        assert np.allclose(g[k], P[k].grad.numpy(), rtol=1e-10, atol=1e-12), k
    # split into two shares with 4 and 3 scored tokens: each uses the batch count
    whole = B.lm_head_backward(h, w, t)
    n_all = int((t != -100).sum())
    a, b = slice(0, 6), slice(6, 11)
    ga = B.lm_head_backward(h[a], w, t[a], count=n_all)
    gb = B.lm_head_backward(h[b], w, t[b], count=n_all)
    assert int((t[a] != -100).sum()) != int((t[b] != -100).sum())
    assert np.allclose(np.concatenate([ga["hidden"], gb["hidden"]]), whole["hidden"], rtol=0, atol=1e-14)
    for k in ("dense_w", "dense_b", "ln_g", "ln_b", "emb", "bias"):
        assert np.allclose(ga[k] + gb[k], whole[k], rtol=1e-12, atol=1e-14), k
