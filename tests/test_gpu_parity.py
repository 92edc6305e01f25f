"""Parity of the CUDA path (called through the C ABI) with the float64 oracle.

Tolerances (relative L2 over all compared elements): fp32 1e-4, bf16 1e-2, FP8 5e-2 for
final hidden states; packing indices bit-exact.  Kernel-level checks use tighter bounds
derived from the arithmetic (stated at each test)."""
import dataclasses

import numpy as np
import pytest

from oracle import esm_oracle as O
from tests._util import ensure_built, rel_l2, to_np
from transformer_esm_layer_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def _enc(g, precision, final_ln=True, **kw):
    from transformer_esm_layer_gb300.binding import EsmEncoder
    return EsmEncoder.from_geometry(g, precision, final_ln, **kw)


SMALL = synth.Geometry(num_layers=2, hidden=256, heads=4, ffn=512)


def _bf16(a):
    return synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(np.asarray(a, np.float32)))


def _dev(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda", dtype)


# --------------------------------------------------------------------------- packing
@pytest.mark.parametrize("lengths", [[17, 40, 7], [1, 2, 127, 128, 129, 1024, 3], [5, 0, 0, 9, 0], [1026, 1]])
def test_pack_index_bit_exact(lengths):
    enc = _enc(SMALL, "bf16")
    cu = torch.from_numpy(synth.cu_seqlens_from_lengths(lengths)).cuda()
    T = int(sum(lengths))
    pos, seg = enc.debug_pack_index(cu, T, max(lengths))
    assert enc.check_status() == 0
    opos, oseg = O.pack_index(O.cu_seqlens(lengths))
    assert np.array_equal(pos.cpu().numpy(), opos) and np.array_equal(seg.cpu().numpy(), oseg)


@pytest.mark.parametrize("cu", [[1, 5, 9], [0, 6, 4, 9], [0, 4, 8], [0, 3, 9]])
def test_bad_cu_seqlens_is_reported(cu):
    enc = _enc(SMALL, "bf16")
    T = 9
    pos, seg = enc.debug_pack_index(torch.tensor(cu, dtype=torch.int32, device="cuda"), T, 5)
    assert enc.check_status() == 3  # ESM_ERR_BAD_CU_SEQLENS
    assert enc.check_status() == 0  # the check clears the latch
    assert pos.min().item() >= 0 and seg.min().item() >= 0


# --------------------------------------------------------------------------- LayerNorm
@pytest.mark.parametrize("precision,cols,tol", [("bf16", 1280, 8e-3), ("bf16", 256, 8e-3), ("fp32", 64, 1e-6)])
def test_layernorm(precision, cols, tol):
    g = synth.Geometry(1, cols, cols // 64 if precision != "fp32" else 4, 4 * cols)
    enc = _enc(g, precision)
    rng = np.random.default_rng(0)
    x = (rng.standard_normal((333, cols)) * 3 + rng.standard_normal((333, 1)) * 2).astype(np.float32)
    gm = rng.standard_normal(cols).astype(np.float32)
    bt = rng.standard_normal(cols).astype(np.float32)
    pdt = torch.float32 if precision == "fp32" else torch.bfloat16
    if precision != "fp32":
        gm, bt = _bf16(gm), _bf16(bt)
    y = torch.empty(333, cols, dtype=pdt, device="cuda")
    enc.op_layernorm(_dev(x, torch.float32), _dev(gm, pdt), _dev(bt, pdt), y)
    torch.cuda.synchronize()
    ref = O.layer_norm(x.astype(np.float64), gm.astype(np.float64), bt.astype(np.float64))
    assert rel_l2(to_np(y), ref) < tol  # bf16 output rounding: ~2^-9 / sqrt(3) rms


# --------------------------------------------------------------------------- GEMMs
@pytest.mark.parametrize("M", [1, 128, 300, 1000])
def test_gemm_bias_f32_tcgen05(M):
    """bf16 x bf16 products are exact in fp32; only the fp32 summation order differs
    from the float64 reference: rel L2 ~ 1e-7."""
    enc = _enc(SMALL, "bf16")
    rng = np.random.default_rng(M)
    K, N = 320, 512
    A = _bf16(rng.standard_normal((M, K)))
    B = _bf16(rng.standard_normal((N, K)))
    b = _bf16(rng.standard_normal(N))
    out = torch.empty(M, N, dtype=torch.float32, device="cuda")
    enc.op_gemm("bias_f32", _dev(A, torch.bfloat16), _dev(B, torch.bfloat16), _dev(b, torch.bfloat16), out)
    assert enc.check_status() == 0
    ref = A.astype(np.float64) @ B.astype(np.float64).T + b
    assert rel_l2(to_np(out), ref) < 1e-5


def test_gemm_large_k_and_many_tiles():
    enc = _enc(SMALL, "bf16")
    rng = np.random.default_rng(5)
    M, K, N = 1500, 5120, 1280
    A = _bf16(rng.standard_normal((M, K)))
    B = _bf16(rng.standard_normal((N, K)) * 0.02)
    out = torch.empty(M, N, dtype=torch.float32, device="cuda")
    enc.op_gemm("bias_f32", _dev(A, torch.bfloat16), _dev(B, torch.bfloat16), None, out)
    assert enc.check_status() == 0
    ref = A.astype(np.float64) @ B.astype(np.float64).T
    assert rel_l2(to_np(out), ref) < 1e-5


def test_gemm_epilogues():
    g = SMALL
    enc = _enc(g, "bf16")
    rng = np.random.default_rng(9)
    M, d, f = 333, g.hidden, g.ffn
    A = _bf16(rng.standard_normal((M, d)))
    Wqkv = _bf16(rng.standard_normal((3 * d, d)) * 0.05)
    bqkv = _bf16(rng.standard_normal(3 * d) * 0.1)
    pos = rng.integers(0, 1026, size=M).astype(np.int32)
    qkv = torch.empty(M, 3 * d, dtype=torch.bfloat16, device="cuda")
    enc.op_gemm("qkv_rope", _dev(A, torch.bfloat16), _dev(Wqkv, torch.bfloat16), _dev(bqkv, torch.bfloat16), qkv,
                pos_id=torch.from_numpy(pos).cuda())
    lin = A.astype(np.float64) @ Wqkv.astype(np.float64).T + bqkv
    H = g.heads
    ref = lin.copy()
    ref[:, :d] = O.rope(lin[:, :d].reshape(M, H, 64), pos).reshape(M, d)
    ref[:, d:2 * d] = O.rope(lin[:, d:2 * d].reshape(M, H, 64), pos).reshape(M, d)
    assert rel_l2(to_np(qkv), ref) < 5e-3
    # GELU
    W1 = _bf16(rng.standard_normal((f, d)) * 0.05)
    b1 = _bf16(rng.standard_normal(f) * 0.1)
    u = torch.empty(M, f, dtype=torch.bfloat16, device="cuda")
    enc.op_gemm("gelu", _dev(A, torch.bfloat16), _dev(W1, torch.bfloat16), _dev(b1, torch.bfloat16), u)
    ref = O.gelu(A.astype(np.float64) @ W1.astype(np.float64).T + b1)
    assert rel_l2(to_np(u), ref) < 5e-3
    # residual: x += A W^T + b
    W2 = _bf16(rng.standard_normal((d, f)) * 0.05)
    b2 = _bf16(rng.standard_normal(d) * 0.1)
    U = _bf16(rng.standard_normal((M, f)))
    x0 = rng.standard_normal((M, d)).astype(np.float32)
    x = _dev(x0, torch.float32)
    enc.op_gemm("residual", _dev(U, torch.bfloat16), _dev(W2, torch.bfloat16), _dev(b2, torch.bfloat16), x)
    assert enc.check_status() == 0
    ref = x0 + U.astype(np.float64) @ W2.astype(np.float64).T + b2
    assert rel_l2(to_np(x), ref) < 1e-5


def test_gemm_residual_with_half_width_tail_tiles():
    """M=5000, N=1280: 100 tiles of 256 x 256 on the persistent grid, so the last ones run as
    256 x 128 halves (and the last row band is ragged); x += A W^T + b against float64."""
    enc = _enc(SMALL, "bf16")
    rng = np.random.default_rng(13)
    M, K, N = 5000, 1280, 1280
    A = _bf16(rng.standard_normal((M, K)))
    W = _bf16(rng.standard_normal((N, K)) * 0.05)
    b = _bf16(rng.standard_normal(N) * 0.1)
    x0 = rng.standard_normal((M, N)).astype(np.float32)
    x = _dev(x0, torch.float32)
    enc.op_gemm("residual", _dev(A, torch.bfloat16), _dev(W, torch.bfloat16), _dev(b, torch.bfloat16), x)
    assert enc.check_status() == 0
    ref = x0 + A.astype(np.float64) @ W.astype(np.float64).T + b
    got = to_np(x)
    assert rel_l2(got, ref) < 1e-5
    assert np.max(np.abs(got - ref)) < 1e-3  # every column block, including the half tiles


def test_gelu_epilogue_within_bf16_rounding():
    """The GELU epilogue on a sweep of 16384 bf16 inputs x (a GEMM whose only nonzero
    product per output is 1 * x, so the accumulator holds x exactly).  The epilogue's fp32
    GELU has an absolute error below 3e-7 max(1, |x|) (erf approximation 1.5e-7 of
    Abramowitz & Stegun 7.1.26 plus single-instruction rcp/exp2), so each bf16 output lies
    within half a bf16 ulp of GELU(x) plus that bound; for x >= -1 all but the near-tie
    cases equal the round-to-nearest-even bf16 of the float64 GELU."""
    enc = _enc(SMALL, "bf16")
    M, K, N = 256, 64, 256
    rng = np.random.default_rng(11)
    xs = np.concatenate([np.linspace(-12.0, 12.0, K * N - 512), rng.standard_normal(256) * 1e-3,
                         rng.standard_normal(256) * 3.0])
    B = _bf16(rng.permutation(xs)).reshape(N, K)
    A = np.zeros((M, K), np.float32)
    A[np.arange(M), np.arange(M) % K] = 1.0
    u = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    enc.op_gemm("gelu", _dev(A, torch.bfloat16), _dev(B, torch.bfloat16), _dev(np.zeros(N), torch.bfloat16), u)
    assert enc.check_status() == 0
    x = B.T[np.arange(M) % K].astype(np.float64)  # x[m, n] = B[n, m % K]
    exact = O.gelu(x)
    got = to_np(u)
    mag = np.maximum(np.abs(exact), 1e-38)
    half_ulp = 2.0 ** (np.floor(np.log2(mag)) - 8)
    bound = half_ulp + 3e-7 * np.maximum(1.0, np.abs(x))
    assert np.all(np.abs(got - exact) <= bound)
    # Where Phi(x) is not small (x >= -1) the fp32 error is ~1e-6 relative: rounding ties only.
    # (Below, GELU is x * Phi(x) with Phi(x) tiny and the 3e-7 absolute error dominates.)
    keep = x >= -1.0
    assert np.mean(got[keep] == O.bf16_round(exact[keep])) > 0.99


def test_gemm_fp32_simt():
    enc = _enc(synth.TINY, "fp32")
    rng = np.random.default_rng(3)
    M, K, N = 77, 64, 192
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = rng.standard_normal((N, K)).astype(np.float32)
    b = rng.standard_normal(N).astype(np.float32)
    out = torch.empty(M, N, dtype=torch.float32, device="cuda")
    enc.op_gemm("bias_f32", _dev(A, torch.float32), _dev(B, torch.float32), _dev(b, torch.float32), out)
    torch.cuda.synchronize()
    assert rel_l2(to_np(out), A.astype(np.float64) @ B.T.astype(np.float64) + b) < 1e-6


# --------------------------------------------------------------------------- attention
@pytest.mark.parametrize("lengths", [[1, 2, 63, 64, 65, 127, 128, 129, 200], [1024, 7, 333], [1],
                                     [256, 257, 383, 384, 385, 3, 512, 640]])
def test_attention_bf16(lengths):
    g = SMALL
    enc = _enc(g, "bf16")
    rng = np.random.default_rng(len(lengths))
    T, d, H = sum(lengths), g.hidden, g.heads
    qkv = _bf16(rng.standard_normal((T, 3 * d)) * 1.5)
    o = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    cu = torch.from_numpy(synth.cu_seqlens_from_lengths(lengths)).cuda()
    enc.op_attention(_dev(qkv, torch.bfloat16), cu, max(lengths), o)
    assert enc.check_status() == 0
    got = to_np(o)
    c = O.cu_seqlens(lengths)
    q64 = qkv.astype(np.float64)
    for i, L in enumerate(lengths):
        s = slice(c[i], c[i + 1])
        ref = O.attention(q64[s, :d].reshape(L, H, 64), q64[s, d:2 * d].reshape(L, H, 64),
                          q64[s, 2 * d:].reshape(L, H, 64)).reshape(L, d)
        # P and O rounded to bf16: ~2^-9 relative each
        assert rel_l2(got[s], ref) < 1e-2, (i, L)


def test_attention_fp32():
    g = synth.TINY
    enc = _enc(g, "fp32")
    lengths = [17, 40, 7]
    rng = np.random.default_rng(1)
    T, d, H = sum(lengths), g.hidden, g.heads
    qkv = rng.standard_normal((T, 3 * d)).astype(np.float32)
    o = torch.empty(T, d, dtype=torch.float32, device="cuda")
    cu = torch.from_numpy(synth.cu_seqlens_from_lengths(lengths)).cuda()
    enc.op_attention(_dev(qkv, torch.float32), cu, 40, o)
    torch.cuda.synchronize()
    got = to_np(o)
    c = O.cu_seqlens(lengths)
    dh = d // H
    q64 = qkv.astype(np.float64)
    for i, L in enumerate(lengths):
        s = slice(c[i], c[i + 1])
        ref = O.attention(q64[s, :d].reshape(L, H, dh), q64[s, d:2 * d].reshape(L, H, dh),
                          q64[s, 2 * d:].reshape(L, H, dh)).reshape(L, d)
        assert rel_l2(got[s], ref) < 1e-6


# --------------------------------------------------------------------------- forward
def _run_packed(g, precision, w, tokens, lengths, final_ln=True):
    from transformer_esm_layer_gb300.binding import DeviceWeights, packed_inputs
    enc = _enc(g, precision, final_ln)
    dw = DeviceWeights(w, precision)
    tok, cu = packed_inputs(tokens, lengths)
    out = enc.forward(dw, tok, cu, max(lengths))
    enc.check()
    return enc, dw, to_np(out)


def test_forward_tiny_fp32_config(margin):
    """The tiny fp32 workload: 2 layers, hidden 64, 4 heads, lengths 17/40/7."""
    wl = synth.make_workload("tiny_fp32")
    g = wl.geometry
    w = synth.model_weights(g, wl.seed, "fp32")
    tok = synth.workload_tokens(wl)
    _, _, got = _run_packed(g, "fp32", w, tok, wl.lengths)
    ref = O.encode_packed(tok, O.cu_seqlens(wl.lengths), w, g.heads, final_ln=True)
    ref = np.concatenate([ref[i] for i in range(len(wl.lengths))])
    assert margin("tiny fp32 encoder", rel_l2(got, ref), 1e-4) < 1e-4


def test_forward_bf16_two_layers_ragged(margin):
    g = synth.Geometry(num_layers=2, hidden=1280, heads=20, ffn=5120)
    lengths = [1, 2, 130, 64, 257, 1024, 33]
    w = synth.model_weights(g, 21, "bf16", ln_random=True)
    tok = synth.tokens_for_lengths(np.random.default_rng(21), lengths)
    _, _, got = _run_packed(g, "bf16", w, tok, lengths)
    ref = O.encode_packed(tok, O.cu_seqlens(lengths), w, g.heads, final_ln=True)
    ref = np.concatenate([ref[i] for i in range(len(lengths))])
    assert margin("650M width x2, ragged lengths", rel_l2(got, ref), 1e-2) < 1e-2


def test_forward_single_layer_workload(margin):
    """One ESM-2 650M layer, 16 log-normal sequences, no final LN."""
    wl = synth.make_workload("layer650m")
    g = wl.geometry
    w = synth.model_weights(g, wl.seed, "bf16")
    tok = synth.workload_tokens(wl)
    _, _, got = _run_packed(g, "bf16", w, tok, wl.lengths, final_ln=False)
    c = O.cu_seqlens(wl.lengths)
    ref = O.encode_packed(tok, c, w, g.heads, final_ln=False)
    worst = max(rel_l2(got[c[i]:c[i + 1]], ref[i]) for i in range(len(wl.lengths)))
    assert margin("one 650M layer workload, worst of 16 sequences", worst, 1e-2) < 1e-2


def test_packed_equals_each_sequence_alone_bitwise():
    g = synth.Geometry(num_layers=2, hidden=1280, heads=20, ffn=5120)
    lengths = [70, 1, 200, 129]
    w = synth.model_weights(g, 22, "bf16")
    tok = synth.tokens_for_lengths(np.random.default_rng(22), lengths)
    enc, dw, got = _run_packed(g, "bf16", w, tok, lengths)
    from transformer_esm_layer_gb300.binding import packed_inputs
    c = O.cu_seqlens(lengths)
    for i, L in enumerate(lengths):
        t1, cu1 = packed_inputs(tok[c[i]:c[i + 1]], [L])
        alone = to_np(enc.forward(dw, t1, cu1, L))
        assert np.array_equal(alone, got[c[i]:c[i + 1]]), i


def test_padded_equals_packed():
    g = synth.Geometry(num_layers=2, hidden=1280, heads=20, ffn=5120)
    lengths = [70, 1, 200, 129]
    S = 256
    w = synth.model_weights(g, 23, "bf16")
    tok = synth.tokens_for_lengths(np.random.default_rng(23), lengths)
    enc, dw, packed = _run_packed(g, "bf16", w, tok, lengths)
    padded = torch.from_numpy(synth.pad_tokens(tok, lengths, S)).cuda()
    lens = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    out = to_np(enc.forward_padded(dw, padded, lens, check=True))
    c = O.cu_seqlens(lengths)
    for b, L in enumerate(lengths):
        assert rel_l2(out[b, :L], packed[c[b]:c[b + 1]]) < 1e-3, b
        assert np.all(out[b, L:] == 0)
    ref = O.encode_padded(padded.cpu().numpy(), lengths, w, g.heads)
    for b, L in enumerate(lengths):
        assert rel_l2(out[b, :L], ref[b][:L]) < 1e-2


# --------------------------------------------------------------------------- errors
def test_forward_host_matches_device_forward():
    """esm_encoder_forward_host (host token ids / cu_seqlens in, host bf16 hidden states out,
    copies inside the call) gives exactly the device-buffer forward."""
    from transformer_esm_layer_gb300.binding import DeviceWeights, packed_inputs
    g = SMALL
    enc = _enc(g, "bf16")
    w = synth.model_weights(g, 6, "bf16", ln_random=True)
    lengths = [33, 1, 200, 7]
    tok = synth.tokens_for_lengths(np.random.default_rng(6), lengths)
    dw = DeviceWeights(w, "bf16")
    t, cu = packed_inputs(tok, lengths)
    dev_out = enc.forward(dw, t, cu, max(lengths)).view(torch.int16).cpu().numpy()
    T = len(tok)
    host_out = np.zeros((T, g.hidden), np.int16)
    ws = enc.workspace(T, len(lengths), torch.device("cuda"))
    enc.forward_host(dw, np.ascontiguousarray(tok, np.int32), synth.cu_seqlens_from_lengths(lengths), max(lengths),
                     host_out, ws)
    assert enc.check_status() == 0
    assert np.array_equal(host_out, dev_out)


def test_forward_host_pinned_graph_replays():
    """With pinned host buffers esm_encoder_forward_host replays a CUDA graph of the whole call
    from its second call on (the first runs eagerly).  Every call gives exactly the
    device-buffer forward, including after a change of host buffers and inputs."""
    from transformer_esm_layer_gb300.binding import DeviceWeights, packed_inputs
    g = SMALL
    enc = _enc(g, "bf16")
    w = synth.model_weights(g, 7, "bf16", ln_random=True)
    dw = DeviceWeights(w, "bf16")
    ws = enc.workspace(400, 8, torch.device("cuda"))
    for lengths, seed in (([33, 1, 200, 7], 7), ([90, 2, 5], 8)):
        tok = synth.tokens_for_lengths(np.random.default_rng(seed), lengths)
        t, cu = packed_inputs(tok, lengths)
        dev_out = enc.forward(dw, t, cu, max(lengths)).view(torch.int16).cpu().numpy()
        T = len(tok)
        tok_h = torch.from_numpy(np.ascontiguousarray(tok, np.int32)).pin_memory()
        cu_h = torch.from_numpy(synth.cu_seqlens_from_lengths(lengths)).pin_memory()
        out_h = torch.zeros(T, g.hidden, dtype=torch.int16).pin_memory()
        for call in range(4):  # eager, capture, replay, replay
            out_h.zero_()
            enc.forward_host(dw, tok_h.numpy(), cu_h.numpy(), max(lengths), out_h.numpy(), ws)
            assert enc.check_status() == 0
            assert np.array_equal(out_h.numpy(), dev_out), (lengths, call)


def test_fp8_forward_one_layer_3b_width(margin):
    """One layer of the 3B geometry (hidden 2560, 40 heads, ffn 10240) with E4M3 GEMMs against
    the oracle with the same scales (5e-2; attention in bf16)."""
    g = synth.Geometry(num_layers=1, hidden=2560, heads=40, ffn=10240)
    lengths = [300, 77, 1, 650]
    enc, w, tok, st, out = _fp8_run(g, lengths, 34)
    scales = enc.fp8_scales(st)
    fp8_state = [{k: float(scales[0, i]) for i, k in enumerate(O.FP8_TENSORS)}]
    c = O.cu_seqlens(lengths)
    ref = O.encode_packed(tok, c, w, g.heads, final_ln=True, fp8_state=fp8_state, bf16_attention=True)
    ref = np.concatenate([ref[i] for i in range(len(lengths))])
    assert margin("one 3B-width FP8 layer", rel_l2(out, ref), 5e-2) < 5e-2


def test_token_out_of_range_reported():
    g = SMALL
    enc = _enc(g, "bf16")
    from transformer_esm_layer_gb300.binding import DeviceWeights, packed_inputs
    dw = DeviceWeights(synth.model_weights(g, 1, "bf16"), "bf16")
    tok, cu = packed_inputs(np.array([0, 5, 40, 2], np.int32), [4])
    enc.forward(dw, tok, cu, 4)
    assert enc.check_status() == 4  # ESM_ERR_TOKEN_RANGE


def test_host_side_argument_errors():
    from transformer_esm_layer_gb300.binding import DeviceWeights, EsmError, packed_inputs
    g = SMALL
    enc = _enc(g, "bf16")
    dw = DeviceWeights(synth.model_weights(g, 1, "bf16"), "bf16")
    tok, cu = packed_inputs(np.array([0, 5, 6, 2], np.int32), [4])
    small_ws = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(EsmError) as e:
        enc.forward(dw, tok, cu, 4, workspace=small_ws)
    assert e.value.status == 5
    with pytest.raises(EsmError) as e:
        enc.forward(dw, tok, cu, 2000)  # max_seqlen above max_positions
    assert e.value.status == 1
    with pytest.raises(EsmError) as e:
        _enc(synth.Geometry(1, 96, 3, 256), "bf16")  # head_dim 32 is not a bf16 geometry
    assert e.value.status == 2


# --------------------------------------------------------------------------- FP8 (E4M3)
# E4M3 keeps 3 mantissa bits: quantising ONE operand of the forward already moves the final
# hidden states by ~3% rel L2, and a 1e-6 perturbation anywhere upstream flips enough
# roundings to move a multi-layer FP8 result by ~1%.  So the FP8 path is pinned exactly at
# the operation level (E4M3 GEMM on E4M3 inputs; LayerNorm -> E4M3 codes), end to end at
# the stated 5e-2 on one layer, and at depth by its accuracy against the exact forward.
_FP8_G = synth.Geometry(num_layers=1, hidden=1280, heads=20, ffn=5120)


def _fp8_codes(rng, shape, table):
    codes = rng.integers(0, 256, size=shape).astype(np.uint8)
    codes[np.isnan(table[codes])] = 0
    return codes


def test_fp8_gemm_exact_on_e4m3_inputs():
    """tcgen05 kind::f8f6f4 GEMM: products of E4M3 values are exact in fp32, so the only
    difference from the float64 reference is fp32 accumulation: about K/32 rounded adds of
    partial sums whose cancellation factor sum|ab| / |sum ab| is ~sqrt(K) for random signs,
    i.e. ~ sqrt(K/32) * 2^-24 * sqrt(K) = 5e-5 at K = 5120 in the worst case; rms well
    below.  Bound: 2e-5."""
    from tests._util import e4m3_table
    table = e4m3_table()
    enc = _enc(_FP8_G, "fp8")
    rng = np.random.default_rng(40)
    for M, N, K in ((300, 512, 1280), (1, 256, 5120), (1000, 1280, 1280)):
        A = _fp8_codes(rng, (M, K), table)
        B = _fp8_codes(rng, (N, K), table)
        b = _bf16(rng.standard_normal(N))
        sa, sb = 3.0, 0.25
        out = torch.empty(M, N, dtype=torch.float32, device="cuda")
        enc.op_gemm_fp8("bias_f32", torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(),
                        torch.tensor([sa], device="cuda"), torch.tensor([sb], device="cuda"),
                        _dev(b, torch.bfloat16), out)
        assert enc.check_status() == 0
        ref = table[A] @ table[B].T / (sa * sb) + b
        assert rel_l2(to_np(out), ref) < 2e-5, (M, N, K)
    # GELU epilogue (bf16 output)
    M, N, K = 200, 5120, 1280
    A = _fp8_codes(rng, (M, K), table)
    B = _fp8_codes(rng, (N, K), table)
    b = _bf16(rng.standard_normal(N))
    u = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    enc.op_gemm_fp8("gelu", torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(),
                    torch.tensor([1e3], device="cuda"), torch.tensor([2e2], device="cuda"),
                    _dev(b, torch.bfloat16), u)
    ref = O.gelu(table[A] @ table[B].T / 2e5 + b)
    assert rel_l2(to_np(u), ref) < 5e-3


def test_fp8_layernorm_codes_match_oracle_rounding():
    """LayerNorm -> E4M3: the codes equal the oracle's round-to-nearest-even of LN(x)*scale
    except where fp32 and float64 LN(x) straddle a rounding midpoint (then the two codes are
    neighbours); the amax is max |LN(x)|."""
    from tests._util import e4m3_table
    table = e4m3_table()
    enc = _enc(_FP8_G, "fp8")
    rng = np.random.default_rng(41)
    rows, cols = 333, 1280
    x = (rng.standard_normal((rows, cols)) * 2 + 0.5).astype(np.float32)
    g = _bf16(1 + 0.3 * rng.standard_normal(cols))
    bt = _bf16(0.3 * rng.standard_normal(cols))
    scale = 61.0
    y = torch.empty(rows, cols, dtype=torch.uint8, device="cuda")
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    enc.op_layernorm_e4m3(_dev(x, torch.float32), _dev(g, torch.bfloat16), _dev(bt, torch.bfloat16), y,
                          torch.tensor([scale], device="cuda"), amax)
    torch.cuda.synchronize()
    ln = O.layer_norm(x.astype(np.float64), g.astype(np.float64), bt.astype(np.float64))
    ref = O.e4m3_round(ln * scale)
    got = table[y.cpu().numpy()]
    diff = got != ref
    assert diff.mean() < 1e-3
    if diff.any():
        r, gv = ref[diff], got[diff]
        assert np.all(np.abs(gv - r) <= np.abs(r) / 8 + 2.0 ** -9)  # one E4M3 step apart
    assert abs(amax.item() / np.abs(ln).max() - 1) < 1e-5


def _fp8_run(g, lengths, seed, calls=3, layer_precision=None):
    from transformer_esm_layer_gb300.binding import DeviceWeights, EsmEncoder, packed_inputs
    w = synth.model_weights(g, seed, "fp8")
    tok = synth.tokens_for_lengths(np.random.default_rng(seed), lengths)
    enc = EsmEncoder.from_geometry(g, "fp8", final_ln=True, amax_history_len=16)
    if layer_precision is not None:
        enc.set_layer_precision(layer_precision)
    dw = DeviceWeights(w, "fp8")
    t, cu = packed_inputs(tok, lengths)
    st0 = enc.get_fp8_state()
    assert np.all(enc.fp8_scales(st0) == 1.0) and np.all(enc.fp8_history(st0) == 0.0)
    for _ in range(calls):
        enc.forward(dw, t, cu, max(lengths))
    enc.check()
    st = enc.get_fp8_state()
    out = to_np(enc.forward(dw, t, cu, max(lengths)))
    enc.check()
    return enc, w, tok, st, out


def test_fp8_forward_one_layer_and_delayed_scaling(margin):
    """One 650M-width layer with E4M3 GEMMs (history 16, max), attention in bf16.  After
    three warm-up calls the scales are read back; the next call matches the oracle using
    those scales within 5e-2, and that call's state update is exact: the history rolls by
    one, weight amaxes equal max |w|, activation amaxes match, scale = 448 / max(history)."""
    g = _FP8_G
    lengths = [300, 1, 129, 64, 700]
    enc, w, tok, st, out = _fp8_run(g, lengths, 31)
    scales, hist = enc.fp8_scales(st), enc.fp8_history(st)
    assert np.all(scales > 1.0)
    fp8_state = [{k: float(scales[l, i]) for i, k in enumerate(O.FP8_TENSORS)} for l in range(g.num_layers)]
    amax = [dict() for _ in range(g.num_layers)]
    c = O.cu_seqlens(lengths)
    ref = O.encode_packed(tok, c, w, g.heads, final_ln=True, fp8_state=fp8_state, amax_out=amax,
                          bf16_attention=True)
    ref = np.concatenate([ref[i] for i in range(len(lengths))])
    assert margin("one 650M-width FP8 layer", rel_l2(out, ref), 5e-2) < 5e-2
    st2 = enc.get_fp8_state()
    hist2, scales2 = enc.fp8_history(st2), enc.fp8_scales(st2)
    for l in range(g.num_layers):
        for i, k in enumerate(O.FP8_TENSORS):
            assert np.array_equal(hist2[l, i, 1:], hist[l, i, :-1])    # rolled by one
            if k.startswith("w_"):
                assert hist2[l, i, 0] == np.float32(amax[l][k])          # weights: exact
            else:
                assert abs(hist2[l, i, 0] / amax[l][k] - 1) < 0.05, (l, k)
            assert scales2[l, i] == np.float32(448.0) / hist2[l, i].max()


@pytest.mark.parametrize("layers", [("bf16", "fp8"), ("fp8", "bf16")])
def test_per_layer_precision_mixed_bf16_and_fp8(layers):
    """layer_precision: one layer with E4M3 GEMMs and one with bf16 GEMMs (650M width).  The
    forward matches the oracle with E4M3 fake-quantisation on the FP8 layer only (5e-2, one
    FP8 layer); the bf16 layer's scales stay 1 and its amax history stays empty."""
    g = synth.Geometry(num_layers=2, hidden=1280, heads=20, ffn=5120)
    lengths = [300, 1, 129, 64, 700]
    enc, w, tok, st, out = _fp8_run(g, lengths, 33, layer_precision=list(layers))
    scales, hist = enc.fp8_scales(st), enc.fp8_history(st)
    fp8_state = [({k: float(scales[l, i]) for i, k in enumerate(O.FP8_TENSORS)} if layers[l] == "fp8" else None)
                 for l in range(2)]
    c = O.cu_seqlens(lengths)
    ref = O.encode_packed(tok, c, w, g.heads, final_ln=True, fp8_state=fp8_state, bf16_attention=True)
    ref = np.concatenate([ref[i] for i in range(len(lengths))])
    assert rel_l2(out, ref) < 5e-2
    for l in range(2):
        if layers[l] == "bf16":
            assert np.all(scales[l] == 1.0) and np.all(hist[l] == 0.0)
        else:
            assert np.all(scales[l] > 1.0)


def test_layer_precision_rejections():
    from transformer_esm_layer_gb300.binding import EsmEncoder, EsmError
    g = synth.Geometry(num_layers=2, hidden=256, heads=4, ffn=512)
    enc8 = EsmEncoder.from_geometry(g, "fp8")
    enc8.set_layer_precision(["fp8", "fp4"])             # NVFP4 layers on an FP8 handle
    with pytest.raises(EsmError, match="UNSUPPORTED"):
        enc8.set_layer_precision(["fp8", "fp32"])
    with pytest.raises(EsmError, match="INVALID_ARG"):
        enc8.set_layer_precision(["fp8"])                # wrong layer count
    enc16 = EsmEncoder.from_geometry(g, "bf16")
    with pytest.raises(EsmError, match="UNSUPPORTED"):
        enc16.set_layer_precision(["bf16", "fp8"])       # FP8 layers need an FP8 handle
    with pytest.raises(EsmError, match="UNSUPPORTED"):
        enc16.set_layer_precision(["bf16", "fp4"])       # so do NVFP4 layers
    enc16.set_layer_precision(["bf16", "bf16"])
    with pytest.raises(EsmError, match="UNSUPPORTED"):
        EsmEncoder.from_geometry(g, "fp4")


def test_fp8_forward_depth_accuracy(margin):
    """Two 650M-width layers: the GPU's FP8 forward is as close to the exact (unquantised)
    forward as the oracle's own FP8 forward with the same scales, and the two FP8 results
    differ by less than two independent FP8 evaluations would (sqrt(2) x the FP8 error)."""
    g = synth.Geometry(num_layers=2, hidden=1280, heads=20, ffn=5120)
    lengths = [300, 1, 129, 64, 700]
    enc, w, tok, st, out = _fp8_run(g, lengths, 32)
    scales = enc.fp8_scales(st)
    fp8_state = [{k: float(scales[l, i]) for i, k in enumerate(O.FP8_TENSORS)} for l in range(g.num_layers)]
    c = O.cu_seqlens(lengths)
    cat = lambda d: np.concatenate([d[i] for i in range(len(lengths))])
    ref8 = cat(O.encode_packed(tok, c, w, g.heads, final_ln=True, fp8_state=fp8_state, bf16_attention=True))
    exact = cat(O.encode_packed(tok, c, w, g.heads, final_ln=True))
    e_oracle = rel_l2(ref8, exact)
    e_gpu = rel_l2(out, exact)
    margin("two 650M-width FP8 layers vs the oracle's FP8 forward", rel_l2(out, ref8), 5e-2)
    assert e_oracle > 1e-2                      # quantisation really happened on both sides
    assert e_gpu < 1.25 * e_oracle, (e_gpu, e_oracle)
    assert rel_l2(out, ref8) < np.sqrt(2) * e_oracle


# --------------------------------------------------------------------------- CUDA graph
def test_forward_captured_in_cuda_graph_replays_bitwise():
    """The whole forward (about 7 launches per layer) captured into one CUDA graph and
    replayed gives exactly the eager result."""
    from transformer_esm_layer_gb300.binding import DeviceWeights, EsmEncoder, packed_inputs
    g = synth.Geometry(num_layers=2, hidden=1280, heads=20, ffn=5120)
    lengths = [130, 7, 300]
    w = synth.model_weights(g, 24, "bf16")
    tok = synth.tokens_for_lengths(np.random.default_rng(24), lengths)
    enc = EsmEncoder.from_geometry(g, "bf16")
    dw = DeviceWeights(w, "bf16")
    t, cu = packed_inputs(tok, lengths)
    ws = enc.workspace(sum(lengths), len(lengths))
    eager = enc.forward(dw, t, cu, max(lengths), workspace=ws).clone()
    out = torch.zeros_like(eager)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        enc.forward(dw, t, cu, max(lengths), out=out, workspace=ws)  # uncaptured call on this stream
    torch.cuda.current_stream().wait_stream(side)
    with torch.cuda.graph(graph):
        enc.forward(dw, t, cu, max(lengths), out=out, workspace=ws)
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    enc.check()


# --------------------------------------------------------------------------- failure detection
def test_bounded_wait_times_out_and_context_stays_usable():
    """A device wait on a barrier nothing arrives at gives up after its limit (50 ms here),
    the host reads ESM_ERR_TIMEOUT, and the next forward runs normally."""
    import time
    from transformer_esm_layer_gb300.binding import DeviceWeights, packed_inputs
    g = SMALL
    enc = _enc(g, "bf16")
    t0 = time.perf_counter()
    enc.debug_wait_timeout(50_000)
    assert enc.check_status() == 7  # ESM_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    assert enc.check_status() == 0
    dw = DeviceWeights(synth.model_weights(g, 3, "bf16"), "bf16")
    tok, cu = packed_inputs(np.array([0, 5, 6, 9, 2], np.int32), [5])
    out = enc.forward(dw, tok, cu, 5)
    enc.check()
    assert torch.isfinite(out.float()).all()


# --------------------------------------------------------------------------- masked-LM head
def _lm_case(g, precision, seed, T):
    w = synth.model_weights(g, seed, precision, num_layers=1)
    head = synth.lm_head_weights(g, seed, precision, w["emb"])
    rng = np.random.default_rng(seed)
    h = rng.standard_normal((T, g.hidden)).astype(np.float32)
    if precision != "fp32":
        h = _bf16(h)
    tokens = rng.integers(0, g.vocab, size=T).astype(np.int32)
    targets = synth.mlm_targets(tokens, seed)
    return head, h, targets


@pytest.mark.parametrize("precision,g,T,tol", [("bf16", synth.ESM2_650M, 1000, 1e-2), ("bf16", SMALL, 333, 1e-2),
                                               ("bf16", dataclasses.replace(SMALL, vocab=8), 257, 1e-2),
                                               ("bf16", dataclasses.replace(SMALL, vocab=20), 100, 1e-2),
                                               ("bf16", dataclasses.replace(SMALL, vocab=64), 333, 1e-2),
                                               ("fp32", synth.TINY, 77, 1e-5)])
def test_lm_head_logits_and_loss(precision, g, T, tol):
    """Logits (relative L2) and masked cross-entropy against the float64 oracle; the scored
    count is exact.  bf16: the dense output and the LayerNorm output are rounded to bf16
    (~2^-9 relative each), so logits agree to ~1e-2.  The bf16 logits run in blocks of 8
    vocabulary rows: vocabularies of 8, 20 (a partly padded block) and 64 (eight blocks)
    besides the model's 33."""
    from transformer_esm_layer_gb300.binding import DeviceLmHead
    enc = _enc(g, precision)
    head, h, targets = _lm_case(g, precision, 21, T)
    dh = DeviceLmHead(head, precision)
    dt = torch.float32 if precision == "fp32" else torch.bfloat16
    hid = _dev(h, dt)
    tg = torch.from_numpy(targets).cuda()
    logits = torch.empty(T, g.vocab, dtype=torch.float32, device="cuda")
    tl = torch.empty(T, dtype=torch.float32, device="cuda")
    ls = torch.zeros(1, dtype=torch.float32, device="cuda")
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    enc.lm_head(dh, hid, targets=tg, logits=logits, token_loss=tl, loss_sum=ls, count=cnt)
    assert enc.check_status() == 0
    ref = O.lm_head(h.astype(np.float64), head)
    per, total, n = O.masked_lm_loss(ref, targets)
    assert rel_l2(to_np(logits), ref) < tol
    assert int(cnt.item()) == n
    got_per = to_np(tl)
    assert np.all(got_per[targets == -100] == 0.0)
    assert abs(float(ls.item()) - total) <= tol * total + 1e-6
    assert abs(float(ls.item()) - float(np.sum(got_per, dtype=np.float64))) <= 1e-3 * max(1.0, total)


def test_lm_head_after_encoder_forward_and_bad_target():
    """The head on the encoder's own output (2 layers, ragged sequences) against the oracle
    encode + head; a target outside the vocabulary is not scored and latches
    ESM_ERR_TOKEN_RANGE; the loss sum is bitwise reproducible."""
    from transformer_esm_layer_gb300.binding import DeviceLmHead, DeviceWeights, packed_inputs
    g = SMALL
    enc = _enc(g, "bf16")
    w = synth.model_weights(g, 4, "bf16", ln_random=True)
    head = synth.lm_head_weights(g, 4, "bf16", w["emb"])
    lengths = [5, 130, 1, 77]
    tokens = synth.tokens_for_lengths(np.random.default_rng(4), lengths)
    tok, cu = packed_inputs(tokens, lengths)
    T = len(tokens)
    dw = DeviceWeights(w, "bf16")
    out = torch.empty(T, g.hidden, dtype=torch.bfloat16, device="cuda")
    enc.forward(dw, tok, cu, max(lengths), out)
    targets = synth.mlm_targets(tokens, 9, rate=0.5)
    tg = torch.from_numpy(targets).cuda()
    dh = DeviceLmHead(head, "bf16")
    logits = torch.empty(T, g.vocab, dtype=torch.float32, device="cuda")
    ls = torch.zeros(1, dtype=torch.float32, device="cuda")
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    enc.lm_head(dh, out, targets=tg, logits=logits, loss_sum=ls, count=cnt)
    assert enc.check_status() == 0
    hid = O.encode_packed(tokens, O.cu_seqlens(lengths), w, g.heads)
    hid = np.concatenate([hid[i] for i in range(len(lengths))])
    ref = O.lm_head(hid, head)
    assert rel_l2(to_np(logits), ref) < 2e-2
    _, total, n = O.masked_lm_loss(ref, targets)
    assert int(cnt.item()) == n and abs(float(ls.item()) - total) < 2e-2 * total
    first = float(ls.item())
    enc.lm_head(dh, out, targets=tg, loss_sum=ls, count=cnt)
    assert float(ls.item()) == first
    bad = targets.copy()
    bad[0] = 40
    enc.lm_head(dh, out, targets=torch.from_numpy(bad).cuda(), loss_sum=ls, count=cnt)
    assert enc.check_status() == 4  # ESM_ERR_TOKEN_RANGE
