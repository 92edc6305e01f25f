"""Parity of the training path (forward that keeps activations, backward) with the float64
oracle in oracle/backward.py, called through the C ABI.

Tolerances (relative L2 over all compared elements):
* fp32 arithmetic on exact inputs (LayerNorm backward, the GEMMs with float32 output on
  bf16-representable operands): 1e-4, the fp32 bound of the forward.
* one bf16 rounding of the result (bf16-output GEMM): 1e-2, the bf16 bound of the forward.
* attention backward (bf16 P and dS operands, bf16 outputs): 1e-2.
* encoder gradients: 2e-2.  The forward's bf16 bound is 1e-2 for outputs that pass through
  about four bf16-rounded operands per layer; a parameter gradient of the backward is a
  product of one rounded forward activation and one rounded backward gradient per GEMM,
  and the backward chain rounds twice as many tensors per layer (activations kept by the
  forward and the gradients of the backward), so its bound is twice the forward's."""
import numpy as np
import pytest

from oracle import backward as B
from oracle import esm_oracle as O
from tests._util import ensure_built, rel_l2, to_np
from transformer_esm_layer_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SMALL = synth.Geometry(num_layers=2, hidden=256, heads=4, ffn=512)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def _enc(g, precision="bf16", final_ln=True, **kw):
    from transformer_esm_layer_gb300.binding import EsmEncoder
    return EsmEncoder.from_geometry(g, precision, final_ln, **kw)


def _bf16(a):
    return synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(np.asarray(a, np.float32)))


def _dev(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda", dtype)


# --------------------------------------------------------------------------- GEMMs
@pytest.mark.parametrize("M,N,K", [(300, 320, 512), (1000, 1280, 5120), (129, 3840, 1280)])
def test_gemm_dgrad_fp32_and_bf16(M, N, K):
    """out = dY W with W [N, K] read MN-major (an input gradient through a linear map)."""
    rng = np.random.default_rng(M + N)
    dY = _bf16(rng.standard_normal((M, N)))
    W = _bf16(rng.standard_normal((N, K)) * 0.05)
    ref = dY.astype(np.float64) @ W.astype(np.float64)
    enc = _enc(SMALL)
    out = torch.empty(M, K, dtype=torch.float32, device="cuda")
    enc.op_gemm_dgrad(_dev(dY, torch.bfloat16), _dev(W, torch.bfloat16), out)
    assert enc.check_status() == 0
    assert rel_l2(to_np(out), ref) < 1e-4
    outb = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    enc.op_gemm_dgrad(_dev(dY, torch.bfloat16), _dev(W, torch.bfloat16), outb)
    assert rel_l2(to_np(outb), ref) < 1e-2


@pytest.mark.parametrize("M,N,K", [(700, 512, 256), (16384, 1280, 1280), (2000, 5120, 1280), (1, 256, 256),
                                   (0, 256, 512)])
def test_gemm_wgrad_split_k(M, N, K):
    """dW = dY^T X summed over M tokens (both operands MN-major; the token loop split)."""
    rng = np.random.default_rng(M + 7)
    dY = _bf16(rng.standard_normal((M, N)))
    X = _bf16(rng.standard_normal((M, K)))
    enc = _enc(SMALL)
    dW = torch.full((N, K), float("nan"), dtype=torch.float32, device="cuda")
    enc.op_gemm_wgrad(_dev(dY, torch.bfloat16), _dev(X, torch.bfloat16), dW)
    assert enc.check_status() == 0
    ref = dY.astype(np.float64).T @ X.astype(np.float64)
    if M == 0:
        assert torch.count_nonzero(dW).item() == 0
    else:
        assert rel_l2(to_np(dW), ref) < 1e-4
    # without a workspace the reduction is not split: same values up to summation order
    dW2 = torch.empty_like(dW)
    tdy, tx = _dev(dY, torch.bfloat16), _dev(X, torch.bfloat16)
    assert enc.lib.esm_op_gemm_wgrad(enc.handle, tdy.data_ptr(), tx.data_ptr(), dW2.data_ptr(), M, N, K, None, 0,
                                     None) == 0
    torch.cuda.synchronize()
    if M > 0:
        assert rel_l2(to_np(dW2), ref) < 1e-4


# --------------------------------------------------------------------------- LayerNorm
@pytest.mark.parametrize("rows,cols", [(257, 1280), (3, 256), (1000, 2560)])
def test_layernorm_backward(rows, cols):
    rng = np.random.default_rng(rows)
    x = (rng.standard_normal((rows, cols)) * 2 + 0.5).astype(np.float32)
    g = _bf16(1 + 0.1 * rng.standard_normal(cols))
    dy = rng.standard_normal((rows, cols)).astype(np.float32)
    dres = rng.standard_normal((rows, cols)).astype(np.float32)
    enc = _enc(SMALL)
    tx, tdy = _dev(x, torch.float32), _dev(dy, torch.float32)
    dx = _dev(dres, torch.float32)  # accumulated in place
    dg = torch.empty(cols, dtype=torch.float32, device="cuda")
    db = torch.empty_like(dg)
    enc.op_layernorm_backward(tx, _dev(g, torch.bfloat16), tdy, dx, dx, dg, db)
    assert enc.check_status() == 0
    rdx, rdg, rdb = B.layer_norm_backward(x.astype(np.float64), g.astype(np.float64), dy.astype(np.float64))
    assert rel_l2(to_np(dx), rdx + dres) < 1e-4
    assert rel_l2(to_np(dg), rdg) < 1e-4
    assert rel_l2(to_np(db), rdb) < 1e-4


# --------------------------------------------------------------------------- attention
@pytest.mark.parametrize("lengths", [[1, 7, 130, 300, 64, 129], [1024, 3, 1], [128, 256]])
def test_attention_lse_and_backward(lengths):
    g = SMALL
    H, d = g.heads, g.hidden
    T = int(sum(lengths))
    rng = np.random.default_rng(T)
    qkv = _bf16(rng.standard_normal((T, 3 * d)) * 2.0)
    dO = _bf16(rng.standard_normal((T, d)))
    enc = _enc(g)
    cu = torch.from_numpy(synth.cu_seqlens_from_lengths(lengths)).cuda()
    tq = _dev(qkv, torch.bfloat16)
    o = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(H, T, dtype=torch.float32, device="cuda")  # head-major
    enc.op_attention_train(tq, cu, max(lengths), o, lse)
    dqkv = torch.full((T, 3 * d), float("nan"), dtype=torch.bfloat16, device="cuda")
    enc.op_attention_backward(tq, o, lse, _dev(dO, torch.bfloat16), cu, max(lengths), dqkv)
    assert enc.check_status() == 0
    cu_np = O.cu_seqlens(lengths)
    ref_lse = np.zeros((T, H))
    ref = np.zeros((T, 3 * d))
    for i in range(len(lengths)):
        a, b = int(cu_np[i]), int(cu_np[i + 1])
        L = b - a
        q = qkv[a:b, :d].reshape(L, H, 64).astype(np.float64)
        k = qkv[a:b, d:2 * d].reshape(L, H, 64).astype(np.float64)
        v = qkv[a:b, 2 * d:].reshape(L, H, 64).astype(np.float64)
        ref_lse[a:b] = B.attention_lse(q, k)
        dq, dk, dv = B.attention_backward(q, k, v, dO[a:b].reshape(L, H, 64).astype(np.float64))
        ref[a:b] = np.concatenate([dq.reshape(L, d), dk.reshape(L, d), dv.reshape(L, d)], axis=1)
    assert np.abs(to_np(lse).T - ref_lse).max() < 1e-4 * np.abs(ref_lse).max() + 1e-5
    got = to_np(dqkv)
    for name, sl in (("dq", slice(0, d)), ("dk", slice(d, 2 * d)), ("dv", slice(2 * d, 3 * d))):
        assert rel_l2(got[:, sl], ref[:, sl]) < 1e-2, name


# --------------------------------------------------------------------------- encoder
def _train_case(g, lengths, seed, emb_scale=1.0, final_ln=True):
    rng = np.random.default_rng(seed)
    w = synth.model_weights(g, seed, "bf16", ln_random=True)
    tok = synth.tokens_for_lengths(rng, lengths)
    T = int(sum(lengths))
    d_out = rng.standard_normal((T, g.hidden)).astype(np.float32)
    from transformer_esm_layer_gb300.binding import DeviceGrads, DeviceWeights, packed_inputs
    enc = _enc(g, final_ln=final_ln, emb_scale=emb_scale)
    dw = DeviceWeights(w, "bf16")
    t_tok, t_cu = packed_inputs(tok, lengths)
    ws = enc.workspace(T, len(lengths))
    tb = enc.train_buffer(T)
    out = enc.forward_train(dw, t_tok, t_cu, max(lengths), tb, ws)
    grads = DeviceGrads(g, g.num_layers)
    enc.backward(dw, _dev(d_out, torch.float32), grads, tb, ws)
    assert enc.check_status() == 0
    ref = B.encode_packed_backward(tok, O.cu_seqlens(lengths), w, g.heads, d_out.astype(np.float64),
                                   final_ln=final_ln, emb_scale=emb_scale)
    return enc, w, tok, out, grads, ref


def _check_grads(grads, ref, g, tol, final_ln=True):
    worst = {}
    worst["emb"] = rel_l2(to_np(grads.emb), ref["emb"])
    if final_ln:
        worst["lnf_g"] = rel_l2(to_np(grads.lnf_g), ref["lnf_g"])
        worst["lnf_b"] = rel_l2(to_np(grads.lnf_b), ref["lnf_b"])
    for li in range(g.num_layers):
        for n in B.PARAM_NAMES:
            worst[f"{li}.{n}"] = rel_l2(to_np(grads.layers[li][n]), ref["layers"][li][n])
    bad = {k: v for k, v in worst.items() if not v < tol}
    assert not bad, (bad, max(worst.values()))
    return worst


@pytest.mark.parametrize("lengths", [[5, 130, 77, 1, 260], [300]])
def test_encoder_backward_small(lengths):
    g = SMALL
    enc, w, tok, out, grads, ref = _train_case(g, lengths, 21, emb_scale=0.88)
    # the training forward gives the forward's output
    cu = O.cu_seqlens(lengths)
    fwd = O.encode_packed(tok, cu, w, g.heads, emb_scale=0.88)
    got = to_np(out)
    assert rel_l2(got, np.concatenate([fwd[i] for i in range(len(lengths))])) < 1e-2
    _check_grads(grads, ref, g, 2e-2)


def test_encoder_backward_without_final_ln():
    g = SMALL
    enc, w, tok, out, grads, ref = _train_case(g, [40, 200, 3], 5, final_ln=False)
    _check_grads(grads, ref, g, 2e-2, final_ln=False)


def test_encoder_backward_650m_width_one_layer():
    """One ESM-2 650M layer (hidden 1280, 20 heads, ffn 5120) on ~1.5K tokens."""
    g = synth.Geometry(num_layers=1, hidden=1280, heads=20, ffn=5120)
    enc, w, tok, out, grads, ref = _train_case(g, [700, 513, 129, 1, 200], 33)
    _check_grads(grads, ref, g, 2e-2)


def test_backward_rejects_mismatched_buffers_and_other_precisions():
    from transformer_esm_layer_gb300.binding import DeviceGrads, DeviceWeights, EsmError, packed_inputs
    g = SMALL
    lengths = [30, 20]
    w = synth.model_weights(g, 1, "bf16")
    tok = synth.tokens_for_lengths(np.random.default_rng(1), lengths)
    enc = _enc(g)
    dw = DeviceWeights(w, "bf16")
    grads = DeviceGrads(g, g.num_layers)
    t_tok, t_cu = packed_inputs(tok, lengths)
    ws = enc.workspace(50, 2)
    tb = enc.train_buffer(50)
    d_out = torch.zeros(50, g.hidden, dtype=torch.float32, device="cuda")
    with pytest.raises(EsmError):  # no training forward yet
        enc.backward(dw, d_out, grads, tb, ws)
    enc.forward_train(dw, t_tok, t_cu, 30, tb, ws)
    with pytest.raises(EsmError):  # another buffer than the forward's
        enc.backward(dw, d_out, grads, enc.train_buffer(50), ws)
    with pytest.raises(EsmError):  # a buffer too small
        enc.forward_train(dw, t_tok, t_cu, 30, tb[:1024], ws)
    enc.backward(dw, d_out, grads, tb, ws)
    assert enc.check_status() == 0
    # zero upstream gradient: every parameter gradient is zero
    for l in grads.layers:
        for t in l.values():
            assert torch.count_nonzero(t).item() == 0
    assert torch.count_nonzero(grads.emb).item() == 0
    # an inference forward on the same workspace withdraws the pending backward
    enc.forward(dw, t_tok, t_cu, 30, workspace=ws)
    with pytest.raises(EsmError):
        enc.backward(dw, d_out, grads, tb, ws)
    enc8 = _enc(g, "fp8")
    with pytest.raises(EsmError):
        enc8.train_buffer(50)


def test_encoder_backward_3b_width_one_layer():
    """One ESM-2 3B layer (hidden 2560, 40 heads, ffn 10240): the wider LayerNorm backward
    and GEMM shapes."""
    g = synth.Geometry(num_layers=1, hidden=2560, heads=40, ffn=10240)
    enc, w, tok, out, grads, ref = _train_case(g, [300, 129, 1, 64], 44)
    _check_grads(grads, ref, g, 2e-2)


def test_backward_is_repeatable():
    """Every reduction over tokens runs in a fixed order: gradients computed before the first
    attention backward (the last layer's fc2 and final LayerNorm) are bitwise identical across
    calls; the rest differ only by the arrival order of the fp32 dQ additions."""
    from transformer_esm_layer_gb300.binding import DeviceGrads, DeviceWeights, packed_inputs
    g = SMALL
    lengths = [200, 57, 3]
    rng = np.random.default_rng(3)
    w = synth.model_weights(g, 3, "bf16", ln_random=True)
    tok = synth.tokens_for_lengths(rng, lengths)
    T = int(sum(lengths))
    d_out = _dev(rng.standard_normal((T, g.hidden)), torch.float32)
    enc = _enc(g)
    dw = DeviceWeights(w, "bf16")
    t_tok, t_cu = packed_inputs(tok, lengths)
    ws = enc.workspace(T, len(lengths))
    tb = enc.train_buffer(T)
    runs = []
    for _ in range(2):
        enc.forward_train(dw, t_tok, t_cu, max(lengths), tb, ws)
        gr = DeviceGrads(g, g.num_layers)
        enc.backward(dw, d_out, gr, tb, ws)
        runs.append(gr)
    assert enc.check_status() == 0
    a, b = runs
    last = g.num_layers - 1
    for n in ("w_2", "b_2"):
        assert torch.equal(a.layers[last][n], b.layers[last][n]), n
    assert torch.equal(a.lnf_g, b.lnf_g) and torch.equal(a.lnf_b, b.lnf_b)
    for li in range(g.num_layers):
        for n in B.PARAM_NAMES:
            assert rel_l2(to_np(a.layers[li][n]), to_np(b.layers[li][n])) < 1e-5, (li, n)
    assert rel_l2(to_np(a.emb), to_np(b.emb)) < 1e-5


# --------------------------------------------------------------------------- masked-LM head
def _head_case(g, T, seed, rate=0.3):
    from transformer_esm_layer_gb300.binding import DeviceLmHead
    rng = np.random.default_rng(seed)
    w = synth.model_weights(g, seed, "bf16")
    head = synth.lm_head_weights(g, seed, "bf16", w["emb"])
    tok = rng.integers(4, 24, T).astype(np.int32)
    targets = synth.mlm_targets(tok, seed, rate=rate)
    h = _bf16(rng.standard_normal((T, g.hidden)))
    return head, DeviceLmHead(head, "bf16"), targets, h


@pytest.mark.parametrize("T,rate", [(300, 0.3), (37, 1.0), (64, 0.0)])
def test_lm_head_backward(T, rate):
    g = SMALL
    head, dh, targets, h = _head_case(g, T, 31, rate)
    enc = _enc(g)
    lsum = torch.zeros(1, dtype=torch.float32, device="cuda")
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    d_hidden, grads = enc.lm_head_backward(dh, _dev(h, torch.bfloat16), torch.from_numpy(targets).cuda(),
                                           loss_sum=lsum, count=cnt)
    assert enc.check_status() == 0
    ref = B.lm_head_backward(h.astype(np.float64), head, targets)
    n = int((targets != -100).sum())
    assert int(cnt.item()) == n
    if n == 0:
        assert torch.count_nonzero(d_hidden).item() == 0
        assert all(torch.count_nonzero(v).item() == 0 for v in grads.values())
        return
    assert rel_l2(to_np(d_hidden), ref["hidden"]) < 2e-2
    for k in ("dense_w", "dense_b", "ln_g", "ln_b", "emb", "bias"):
        assert rel_l2(to_np(grads[k]), ref[k]) < 2e-2, k


def test_lm_head_backward_with_a_global_count():
    """loss_count: the mean is taken over a count given by the caller (the scored tokens of a
    whole data-parallel batch) instead of this call's own."""
    g = SMALL
    head, dh, targets, h = _head_case(g, 200, 32, 0.3)
    enc = _enc(g)
    n_local = int((targets != -100).sum())
    n_global = 3 * n_local + 5
    d_hidden, grads = enc.lm_head_backward(dh, _dev(h, torch.bfloat16), torch.from_numpy(targets).cuda(),
                                           loss_count=torch.tensor([n_global], dtype=torch.int32, device="cuda"))
    assert enc.check_status() == 0
    ref = B.lm_head_backward(h.astype(np.float64), head, targets, count=n_global)
    assert rel_l2(to_np(d_hidden), ref["hidden"]) < 2e-2
    for k in ("dense_w", "dense_b", "ln_g", "ln_b", "emb", "bias"):
        assert rel_l2(to_np(grads[k]), ref[k]) < 2e-2, k


def test_training_step_from_masked_lm_loss():
    """forward_train -> masked-LM head backward -> encoder backward, against the oracle chain
    (the tied embedding's gradient is the head's part plus the encoder's part)."""
    from transformer_esm_layer_gb300.binding import DeviceGrads, DeviceLmHead, DeviceWeights, packed_inputs
    g = SMALL
    lengths = [90, 33, 140]
    rng = np.random.default_rng(41)
    w = synth.model_weights(g, 41, "bf16", ln_random=True)
    head = synth.lm_head_weights(g, 41, "bf16", w["emb"])
    tok = synth.tokens_for_lengths(rng, lengths)
    targets = synth.mlm_targets(tok, 41, rate=0.25)
    T = int(sum(lengths))
    enc = _enc(g)
    dw = DeviceWeights(w, "bf16")
    t_tok, t_cu = packed_inputs(tok, lengths)
    ws = enc.workspace(T, len(lengths))
    tb = enc.train_buffer(T)
    out = enc.forward_train(dw, t_tok, t_cu, max(lengths), tb, ws)
    d_hidden, hg = enc.lm_head_backward(DeviceLmHead(head, "bf16"), out, torch.from_numpy(targets).cuda())
    grads = DeviceGrads(g, g.num_layers)
    enc.backward(dw, d_hidden, grads, tb, ws)
    assert enc.check_status() == 0
    cu = O.cu_seqlens(lengths)
    hid = O.encode_packed(tok, cu, w, g.heads)
    hid = np.concatenate([hid[i] for i in range(len(lengths))])
    rh = B.lm_head_backward(hid, head, targets)
    ref = B.encode_packed_backward(tok, cu, w, g.heads, rh["hidden"])
    assert rel_l2(to_np(d_hidden), rh["hidden"]) < 2e-2
    for k in ("dense_w", "dense_b", "ln_g", "ln_b", "bias"):
        assert rel_l2(to_np(hg[k]), rh[k]) < 2e-2, k
    assert rel_l2(to_np(hg["emb"]) + to_np(grads.emb), rh["emb"] + ref["emb"]) < 2e-2
    _check_grads(grads, ref, g, 2e-2)
