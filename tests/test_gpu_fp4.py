"""NVFP4 (block-scaled E2M1) operands and GEMM on the tensor cores against the FP4 oracle.

* Quantisation: the tensor scale S, the E4M3 block scales and the E2M1 codes equal the
  oracle's (float64) except where fp32 and float64 straddle a rounding midpoint, then the
  two results are neighbouring codes.
* GEMM exactness: the product of the GPU's own quantised operands, decoded in numpy from their
  bytes (codes, the atom-ordered scales) and multiplied in float64, agrees with the tensor-core
  result up to fp32 accumulation: this pins the block-scaled MMA, the scale-factor layout in
  tensor memory and the epilogue's 1 / (S_A S_B).
* Epilogues: residual add, GELU and RoPE on the same decoded product, element by element.
* End to end: the GEMM of bf16 inputs quantised on the GPU against the oracle's fake-quantised
  product (nvfp4_fake_quant of both operands), and FP4 layers in an encoder against the
  oracle's FP4 forward (criteria relative to the recipe's own quantisation error)."""
import numpy as np
import pytest

from oracle import fp4 as F4
from tests._util import e4m3_table, ensure_built, rel_l2
from transformer_esm_layer_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


@pytest.fixture(scope="module")
def enc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()
    from transformer_esm_layer_gb300.binding import EsmEncoder
    return EsmEncoder(1, 256, 4, 512, precision="bf16")


def _bf16(a):
    return synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(np.asarray(a, np.float32))).astype(np.float64)


def _codes(codes, scales, rows, K):
    """E2M1 values q [rows, K] and E4M3 block scales sb [rows, K/16] of a GPU NVFP4 operand,
    from its bytes (value k in the low nibble of byte k/2 for even k; scales in atom order)."""
    c = codes.astype(np.int64)
    nib = np.stack([c & 0xF, c >> 4], axis=-1).reshape(rows, K)
    q = np.where(nib & 8, -1.0, 1.0) * E2M1[nib & 7]
    r = np.arange(rows)[:, None]
    k16 = np.arange(K // 16)[None, :]
    off = ((r // 128) * (K // 64) + k16 // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (k16 % 4)
    return q, e4m3_table()[scales[off]]


def _decode(codes, scales, S, rows, K):
    """float64 values of a GPU NVFP4 operand from its bytes: E2M1 values times the block
    scales, divided by the tensor scale."""
    q, sb = _codes(codes, scales, rows, K)
    return (q.reshape(rows, K // 16, 16) * sb[..., None]).reshape(rows, K) / S, sb


def _case(rng, rows, K):
    x = rng.standard_normal((rows, K)) * np.exp(rng.standard_normal((rows, 1)))  # rows of varied magnitude
    x[0, :16] = 0.0                                                               # one all-zero block
    x[1, 16:32] *= 1e-3                                                           # one tiny block
    return _bf16(x)


def _quant(enc, x):
    return enc.op_quantize_nvfp4(torch.from_numpy(x.astype(np.float32)).cuda().to(torch.bfloat16))


def test_nvfp4_quantize_matches_oracle(enc):
    """S to fp32 rounding; block scales and E2M1 codes equal to the oracle's (S in float64)
    except where a rounding midpoint decides (then neighbouring codes)."""
    rng = np.random.default_rng(50)
    rows, K = 256, 768
    x = _case(rng, rows, K)
    codes, scales, amax, scale = _quant(enc, x)
    torch.cuda.synchronize()
    _, sb_o, S_o = F4.nvfp4_fake_quant(x)
    S = float(scale.item())
    assert float(amax.item()) == np.abs(x).max()
    assert abs(S / S_o - 1) < 1e-6
    q, sb = _codes(codes.cpu().numpy(), scales.cpu().numpy(), rows, K)
    diff = sb != sb_o
    assert diff.mean() < 2e-3
    assert np.all(np.abs(sb[diff] - sb_o[diff]) <= sb_o[diff] / 8 + 2.0 ** -9)
    xb = x.reshape(rows, K // 16, 16)
    q_o = np.where(sb_o[..., None] > 0, F4.e2m1_round(xb * S_o / np.where(sb_o > 0, sb_o, 1.0)[..., None]), 0.0)
    q_o = q_o.reshape(rows, K)
    qd = (q != q_o) & np.repeat(~diff, 16, axis=1)
    assert qd.mean() < 2e-3
    idx_step = np.abs(np.searchsorted(E2M1, np.abs(q[qd])) - np.searchsorted(E2M1, np.abs(q_o[qd])))
    assert np.all(idx_step <= 1) and np.all(np.sign(q[qd]) * np.sign(q_o[qd]) >= 0)
    assert np.all(q[0, :16] == 0.0) and np.all(sb[0, 0] == 0.0)


def _fp32_codes(x, K):
    """E2M1 code nibbles (sign bit 3) and E4M3 block scales of a bf16 operand with every
    decision taken in fp32 as the kernel takes it: S = RN(2688 / amax), sb = E4M3(RN(RN(bmax /
    6) S)), q = E2M1(RN(RN(x S) / sb)) with ties to even; 0 for a block whose scale is 0."""
    f = np.float32
    x32 = x.astype(f)
    S = f(2688.0) / np.abs(x32).max()
    xb = x32.reshape(x.shape[0], K // 16, 16)
    u = (np.abs(xb).max(axis=-1) / f(6.0)) * S
    sb = F4.e4m3_round(u.astype(np.float64))
    safe = np.where(sb > 0, sb, 1.0).astype(f)
    q = (xb * S) / safe[..., None]                 # two fp32 steps, each correctly rounded
    mag = F4.e2m1_round(np.abs(q).astype(np.float64))
    idx = np.searchsorted(E2M1, mag)
    nib = np.where(np.signbit(q), 8, 0) | idx
    nib = np.where(sb[..., None] > 0, nib, 0)
    return nib.reshape(x.shape[0], K), sb, S


def test_nvfp4_quantize_fp32_decisions_exact(enc):
    """Every code nibble and block scale equals the fp32 decision, on inputs built to hit
    E2M1 rounding midpoints exactly: the amax is 21, so S = 2688 / 21 = 128 exactly; each
    block's largest value is 3 sb / 64 for a chosen E4M3 scale sb (all 126 finite positive
    ones), so the block scale is exactly sb; the other values are +-t sb / 128 for E2M1 values
    and midpoints t (quotient exactly t, so ties to even decide) and their bf16 neighbours
    one step up or down (quotients just off the midpoints), and a few -0 and bf16 subnormals.
    A random operand follows.  This pins the kernel's quotient (a reciprocal corrected by an
    FMA, no per-value division) to IEEE division."""
    from tests._util import e4m3_table
    rng = np.random.default_rng(56)
    table = e4m3_table()
    sbs = table[1:0x7F]
    points = np.array([0.25, 0.5, 0.75, 1.0, 1.25, 1.5, 1.75, 2.0, 2.5, 3.0, 3.5, 4.0, 5.0, 6.0])
    rows, K = 256, 768
    nblk = rows * K // 16
    blocks = np.zeros((nblk, 16))
    sb_pick = sbs[np.arange(nblk) % len(sbs)]
    blocks[:, 0] = 3 * sb_pick / 64
    t = rng.choice(points, size=(nblk, 15)) * rng.choice([-1.0, 1.0], size=(nblk, 15))
    bits = synth.f32_to_bf16_bits((t * sb_pick[:, None] / 128).astype(np.float32)).astype(np.int64)
    step = rng.integers(-1, 2, size=bits.shape)                   # -1, 0, +1 bf16 steps
    bits = np.where((bits & 0x7FFF) != 0, bits + step, bits)
    vals = synth.bf16_bits_to_f32(bits.astype(np.uint16)).astype(np.float64)
    blocks[:, 1:] = np.minimum(np.abs(vals), 3 * sb_pick[:, None] / 64) * np.sign(vals)
    x = blocks.reshape(rows, K)
    x[5, 17] = -0.0
    x[6, 33] = synth.bf16_bits_to_f32(np.array([0x0003], np.uint16))[0]
    x[0, 0] = 21.0                                                # the tensor's amax
    x = _bf16(x)
    for i, case in enumerate((x, _case(rng, rows, K))):
        codes, scales, amax, scale = _quant(enc, case)
        torch.cuda.synchronize()
        c = codes.cpu().numpy().astype(np.int64)
        nib = np.stack([c & 0xF, c >> 4], axis=-1).reshape(rows, K)
        want, sb_want, S = _fp32_codes(case, K)
        _, sb = _codes(codes.cpu().numpy(), scales.cpu().numpy(), rows, K)
        assert float(scale.item()) == float(S) and (i > 0 or float(S) == 128.0)
        assert np.array_equal(sb, sb_want)
        # magnitudes exactly; the sign bit wherever the magnitude is not zero (a signed zero
        # code has the value of an unsigned one)
        bad = np.argwhere(((nib & 7) != (want & 7)) | (((want & 7) != 0) & ((nib & 8) != (want & 8))))
        assert len(bad) == 0, (i, len(bad), bad[:5], nib[tuple(bad[0])], want[tuple(bad[0])])
        if i == 0:   # the construction reached the ties it was built for
            q_exact = case.reshape(rows, K // 16, 16) * 128.0 / np.where(sb_want > 0, sb_want, 1.0)[..., None]
            ties = np.isin(np.abs(q_exact), [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
            assert ties.sum() > 1000


@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (256, 384, 1280), (384, 256, 512)])
def test_nvfp4_gemm_exact_on_its_operands(enc, M, N, K):
    """fp32 accumulation of E2M1 x E2M1 products scaled by E4M3 x E4M3 block scales: exact
    products, about K/64 rounded partial sums; bound 2e-5 relative L2 (as for the E4M3 GEMM)."""
    rng = np.random.default_rng(M + N + K)
    A, B = _case(rng, M, K), _bf16(_case(rng, N, K) * 0.05)
    bias = _bf16(rng.standard_normal(N))
    qa, qb = _quant(enc, A), _quant(enc, B)
    out = enc.op_gemm_nvfp4(qa, qb, bias=torch.from_numpy(bias.astype(np.float32)).cuda().to(torch.bfloat16))
    assert enc.check_status() == 0
    da, _ = _decode(qa[0].cpu().numpy(), qa[1].cpu().numpy(), float(qa[3].item()), M, K)
    db, _ = _decode(qb[0].cpu().numpy(), qb[1].cpu().numpy(), float(qb[3].item()), N, K)
    ref = da @ db.T + bias
    got = out.to(torch.float64).cpu().numpy()
    assert rel_l2(got, ref) < 2e-5, rel_l2(got, ref)


def test_nvfp4_gemm_matches_oracle_fake_quant(enc, margin):
    rng = np.random.default_rng(51)
    M, N, K = 256, 512, 1280
    A, B = _case(rng, M, K), _bf16(_case(rng, N, K) * 0.02)
    out = enc.op_gemm_nvfp4(_quant(enc, A), _quant(enc, B))
    assert enc.check_status() == 0
    ref = F4.nvfp4_fake_quant(A)[0] @ F4.nvfp4_fake_quant(B)[0].T
    e = rel_l2(out.to(torch.float64).cpu().numpy(), ref)
    margin("NVFP4 GEMM vs the oracle's fake-quantised product", e, 5e-3)
    assert e < 5e-3
    # and the quantisation error itself, against the unquantised product (for the record)
    margin("NVFP4 GEMM vs the exact product (record)", rel_l2(out.to(torch.float64).cpu().numpy(), A @ B.T), 2e-1)


@pytest.mark.parametrize("epi", ["residual", "gelu", "qkv_rope"])
def test_nvfp4_gemm_epilogues(enc, epi):
    """The epilogues an FP4 layer uses, on the GPU's own quantised operands (decoded from their
    bytes and multiplied in float64): the residual add in fp32, GELU (exact erf) and RoPE at
    random positions (hidden 256, 4 heads of 64) each followed by one bf16 rounding, so every
    element is within 2^-8 of its value (plus a small absolute term for fp32 accumulation)."""
    from oracle import esm_oracle as O
    rng = np.random.default_rng({"residual": 53, "gelu": 54, "qkv_rope": 55}[epi])
    M, K, d = 256, 512, 256
    N = {"residual": d, "gelu": 1024, "qkv_rope": 3 * d}[epi]
    A, B = _case(rng, M, K), _bf16(_case(rng, N, K) * 0.05)
    bias = _bf16(rng.standard_normal(N) * 0.1)
    qa, qb = _quant(enc, A), _quant(enc, B)
    da, _ = _decode(qa[0].cpu().numpy(), qa[1].cpu().numpy(), float(qa[3].item()), M, K)
    db, _ = _decode(qb[0].cpu().numpy(), qb[1].cpu().numpy(), float(qb[3].item()), N, K)
    v = da @ db.T + bias
    bias_t = torch.from_numpy(bias.astype(np.float32)).cuda().to(torch.bfloat16)
    if epi == "residual":
        x0 = rng.standard_normal((M, N)).astype(np.float32)
        out = torch.from_numpy(x0).cuda()
        enc.op_gemm_nvfp4(qa, qb, bias=bias_t, out=out, epi="residual")
        ref, rel = x0 + v, 0.0
    elif epi == "gelu":
        out = enc.op_gemm_nvfp4(qa, qb, bias=bias_t, epi="gelu")
        ref, rel = O.gelu(v), 2.0 ** -8
    else:
        pos = rng.integers(0, 1026, size=M).astype(np.int32)
        out = enc.op_gemm_nvfp4(qa, qb, bias=bias_t, epi="qkv_rope", pos_id=torch.from_numpy(pos).cuda())
        ref = v.copy()
        ref[:, :d] = O.rope(v[:, :d].reshape(M, 4, 64), pos).reshape(M, d)
        ref[:, d:2 * d] = O.rope(v[:, d:2 * d].reshape(M, 4, 64), pos).reshape(M, d)
        rel = 2.0 ** -8
    assert enc.check_status() == 0
    got = out.to(torch.float64).cpu().numpy()
    rms = np.sqrt(np.mean(ref ** 2))
    err = np.abs(got - ref) - (rel * np.abs(ref) + 2e-5 * rms)
    assert err.max() <= 0, (epi, np.unravel_index(err.argmax(), err.shape), err.max())


def test_nvfp4_argument_errors(enc):
    from transformer_esm_layer_gb300.binding import EsmError
    x = torch.zeros(100, 256, dtype=torch.bfloat16, device="cuda")   # rows not a multiple of 128
    with pytest.raises(EsmError, match="INVALID_ARG"):
        enc.op_quantize_nvfp4(x)
    y = torch.zeros(128, 200, dtype=torch.bfloat16, device="cuda")   # cols not a multiple of 256
    with pytest.raises(EsmError, match="INVALID_ARG"):
        enc.op_quantize_nvfp4(y)
    q = enc.op_quantize_nvfp4(torch.zeros(128, 256, dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(EsmError, match="INVALID_ARG"):   # RoPE without positions
        enc.op_gemm_nvfp4(q, q, epi="qkv_rope")
    pos = torch.zeros(128, dtype=torch.int32, device="cuda")
    with pytest.raises(EsmError, match="INVALID_ARG"):   # N = 128 is not 3 * hidden
        enc.op_gemm_nvfp4(q, q, epi="qkv_rope", pos_id=pos)


@pytest.mark.parametrize("layers", [("fp4",), ("fp4", "fp8"), ("bf16", "fp4")])
def test_fp4_layers_in_an_encoder(layers, margin):
    """layer_precision with NVFP4 layers (650M width, ragged lengths, final LayerNorm) against
    the oracle with the GPU's tensor scales: the FP8 layer's delayed scales (state read before
    the compared call) and each FP4 layer's current scales (read after it).

    No tolerance is stated for FP4.  The operations are pinned exactly above (codes and
    scales, the GEMM on its operands, the GEMM against the oracle's fake quantisation on the
    same bf16 inputs).  At layer level two evaluations of one FP4 recipe differ by E2M1
    rounding flips seeded by any upstream rounding difference (here the attention's bf16
    probabilities), each flip a whole E2M1 step (25-50% of the value), so the bound is set by
    the recipe's own quantisation noise e_q (the oracle's FP4 forward against the exact one):
    (i) the GPU is as accurate as the recipe, |e_gpu - e_q| <= 2% of e_q, and (ii) the GPU is
    closer to the oracle's FP4 forward than that noise, rel L2 <= 0.75 e_q."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()
    from oracle import esm_oracle as O
    from transformer_esm_layer_gb300.binding import DeviceWeights, EsmEncoder, packed_inputs
    g = synth.Geometry(num_layers=len(layers), hidden=1280, heads=20, ffn=5120)
    lengths = [300, 1, 129, 64, 700]
    w = synth.model_weights(g, 61, "fp8")
    tok = synth.tokens_for_lengths(np.random.default_rng(61), lengths)
    enc = EsmEncoder.from_geometry(g, "fp8", final_ln=True, amax_history_len=16)
    enc.set_layer_precision(list(layers))
    dw = DeviceWeights(w, "fp8")
    t, cu = packed_inputs(tok, lengths)
    for _ in range(3):
        enc.forward(dw, t, cu, max(lengths))
    enc.check()
    s8 = enc.fp8_scales(enc.get_fp8_state())
    out = enc.forward(dw, t, cu, max(lengths))
    enc.check()
    s4 = enc.fp4_scales()
    got = out.to(torch.float64).cpu().numpy()
    assert np.isfinite(got).all()
    fp8_state = [({k: float(s8[l, i]) for i, k in enumerate(O.FP8_TENSORS)} if p == "fp8" else None)
                 for l, p in enumerate(layers)]
    fp4_state = [({k: float(s4[l, i]) for i, k in enumerate(O.FP8_TENSORS)} if p == "fp4" else None)
                 for l, p in enumerate(layers)]
    for l, p in enumerate(layers):
        assert (np.all(s4[l] > 0) if p == "fp4" else np.all(s4[l] == 0)), (l, s4[l])
    c = O.cu_seqlens(lengths)
    ref = O.encode_packed(tok, c, w, g.heads, final_ln=True, fp8_state=fp8_state, fp4_state=fp4_state,
                          bf16_attention=True)
    ref = np.concatenate([ref[i] for i in range(len(lengths))])
    exact = O.encode_packed(tok, c, w, g.heads, final_ln=True)
    exact = np.concatenate([exact[i] for i in range(len(lengths))])
    e, e_q, e_gpu = rel_l2(got, ref), rel_l2(ref, exact), rel_l2(got, exact)
    margin(f"layers {layers}: GPU vs exact against the recipe's own error, |e_gpu - e_q| / e_q",
           abs(e_gpu - e_q) / e_q, 2e-2)
    margin(f"layers {layers}: GPU vs the oracle's quantised forward, in units of e_q = {e_q:.3f}", e / e_q, 0.75)
    assert abs(e_gpu - e_q) <= 2e-2 * e_q
    assert e <= 0.75 * e_q
