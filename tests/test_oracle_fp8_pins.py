"""Pins of the oracle's FP8 (E4M3, per-tensor delayed scaling) branch.

Sources: the aikraft.ru Transformer Engine summary, section on the FP8 recipe (delayed
scaling, E4M3 forward format, one scale per tensor) and §4.1 of the hotelren.com guide.

* ``fp8_fake_quant`` on values the E4M3 code table fixes (round to nearest, ties to the
  even mantissa, saturation at 448, the subnormal binade), with the scale multiplied in
  before rounding and divided out after.
* The tensor -> scale mapping of ``encoder_layer``: every one of the eight scales is given a
  distinct value, each call of the fake-quantiser is recorded, and an independent torch
  float64 formulation of the layer (torch's ``float8_e4m3fn`` cast, ``layer_norm``, ``gelu``,
  ``scaled_dot_product_attention``, RoPE as a complex rotation) checks that each scale meets
  exactly the operand of the GEMM it belongs to and that the layer output follows.
"""
import numpy as np
import pytest

from oracle import esm_oracle as O
from tests._util import e4m3_table

torch = pytest.importorskip("torch")


def _table_values():
    t = e4m3_table()
    return np.unique(t[np.isfinite(t)])


@pytest.mark.parametrize("a,expected_code_value", [
    (1.0, 128.0),                   # 128 = 2^7 is a code
    (136.0 / 128, 128.0),           # midpoint of 128 (mantissa 000) and 144 (001): even -> 128
    (152.0 / 128, 160.0),           # midpoint of 144 (001) and 160 (010): even -> 160
    (150.0 / 128, 144.0),           # below that midpoint
    (0.3, 40.0),                    # 38.4 in [32, 64) (spacing 4) -> 40
    (3.5, 448.0),                   # the largest finite code
    (3.5 + 1e-9, 448.0),            # saturates
    (4.0, 448.0),
    (-1000.0, -448.0),
    (1.5 * 2.0 ** -9 / 128, 2.0 ** -8),  # subnormal midpoint of 2^-9 (odd) and 2^-8 (even)
    (2.0 ** -11 / 128, 0.0),        # below half of the smallest subnormal
])
def test_fake_quant_on_table_values(a, expected_code_value):
    """deq(q(a * 128)) / 128 with the rounded value taken from the E4M3 code table."""
    assert abs(expected_code_value) in set(np.abs(_table_values())) or expected_code_value == 0.0
    got = O.fp8_fake_quant(np.array([a]), 128.0)[0]
    assert got == expected_code_value / 128.0


def test_fake_quant_result_is_a_scaled_table_value():
    """Every output times the scale is an E4M3 code value, and it is the nearest one."""
    rng = np.random.default_rng(3)
    vals = _table_values()
    for scale in (0.75, 61.0, 4096.0):
        a = rng.standard_normal(2000) * rng.choice([1e-4, 1e-2, 1.0, 10.0], size=2000)
        q = O.fp8_fake_quant(a, scale) * scale
        assert np.all(np.isin(q, vals))
        clipped = np.clip(a * scale, -448.0, 448.0)
        nearest = np.min(np.abs(vals[None, :] - clipped[:, None]), axis=1)
        assert np.allclose(np.abs(q - clipped), nearest, rtol=0, atol=1e-15)


def _torch_fq(a, s):
    """E4M3 fake quantisation through torch's own float8_e4m3fn cast (saturated first: the
    cast itself maps values above 448 to NaN)."""
    t = torch.as_tensor(a, dtype=torch.float64) * s
    t = t.clamp(-448.0, 448.0)
    return t.to(torch.float8_e4m3fn).to(torch.float64) / s


def _torch_layer_fp8(x, w, heads, scales):
    """Independent float64 formulation of one FP8 pre-LN layer (bf16 attention operands):
    returns the eight GEMM operands before quantisation and the layer output."""
    import torch.nn.functional as F
    t = lambda a: torch.as_tensor(np.asarray(a, np.float64))
    X = t(x)
    L, d = X.shape
    dh = d // heads
    ops = {}
    y = F.layer_norm(X, (d,), t(w["ln1_g"]), t(w["ln1_b"]), eps=1e-5)
    ops["x_qkv"], ops["w_qkv"] = y, t(w["w_qkv"])
    qkv = _torch_fq(y, scales["x_qkv"]) @ _torch_fq(t(w["w_qkv"]), scales["w_qkv"]).T + t(w["b_qkv"])
    q, k, v = (qkv[:, i * d:(i + 1) * d].reshape(L, heads, dh) for i in range(3))
    half = dh // 2
    theta = 10000.0 ** (-2.0 * torch.arange(half, dtype=torch.float64) / dh)
    rot = torch.polar(torch.ones(L, half, dtype=torch.float64), torch.arange(L, dtype=torch.float64)[:, None] * theta)

    def rope(u):
        zc = torch.complex(u[..., :half], u[..., half:]) * rot[:, None, :]
        return torch.cat([zc.real, zc.imag], dim=-1)

    bf = lambda u: u.to(torch.float32).to(torch.bfloat16).to(torch.float64)
    q, k, v = bf(rope(q)), bf(rope(k)), bf(v)
    o = F.scaled_dot_product_attention(q.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1))
    o = o.transpose(0, 1).reshape(L, d)
    ops["x_o"], ops["w_o"] = o, t(w["w_o"])
    X = X + _torch_fq(o, scales["x_o"]) @ _torch_fq(t(w["w_o"]), scales["w_o"]).T + t(w["b_o"])
    z = F.layer_norm(X, (d,), t(w["ln2_g"]), t(w["ln2_b"]), eps=1e-5)
    ops["x_1"], ops["w_1"] = z, t(w["w_1"])
    u = F.gelu(_torch_fq(z, scales["x_1"]) @ _torch_fq(t(w["w_1"]), scales["w_1"]).T + t(w["b_1"]))
    ops["x_2"], ops["w_2"] = u, t(w["w_2"])
    X = X + _torch_fq(u, scales["x_2"]) @ _torch_fq(t(w["w_2"]), scales["w_2"]).T + t(w["b_2"])
    return ops, X


def _layer_case(seed=11, L=7, d=32, heads=2, f=64):
    rng = np.random.default_rng(seed)
    w = {"ln1_g": 1 + 0.2 * rng.standard_normal(d), "ln1_b": 0.2 * rng.standard_normal(d),
         "w_qkv": 0.2 * rng.standard_normal((3 * d, d)), "b_qkv": 0.1 * rng.standard_normal(3 * d),
         "w_o": 0.2 * rng.standard_normal((d, d)), "b_o": 0.1 * rng.standard_normal(d),
         "ln2_g": 1 + 0.2 * rng.standard_normal(d), "ln2_b": 0.2 * rng.standard_normal(d),
         "w_1": 0.2 * rng.standard_normal((f, d)), "b_1": 0.1 * rng.standard_normal(f),
         "w_2": 0.2 * rng.standard_normal((d, f)), "b_2": 0.1 * rng.standard_normal(d)}
    x = rng.standard_normal((L, d))
    # eight distinct scales, none of which saturates these operands
    scales = dict(zip(O.FP8_TENSORS, (3.0, 5.0, 7.0, 11.0, 13.0, 17.0, 19.0, 23.0)))
    return x, w, heads, scales


def test_fp8_layer_tensor_to_scale_mapping(monkeypatch):
    x, w, heads, scales = _layer_case()
    calls = []
    real = O.fp8_fake_quant

    def recording(a, s):
        out = real(a, s)
        calls.append((float(s), np.array(a, copy=True), out))
        return out

    monkeypatch.setattr(O, "fp8_fake_quant", recording)
    got = O.encoder_layer(x, np.arange(x.shape[0]), w, heads, fp8_scales=scales, bf16_attention=True)
    monkeypatch.setattr(O, "fp8_fake_quant", real)
    assert len(calls) == 8
    by_scale = {s: (a, q) for s, a, q in calls}
    assert sorted(by_scale) == sorted(scales.values())          # every scale used exactly once
    ops, ref = _torch_layer_fp8(x, w, heads, scales)
    for name, s in scales.items():
        a, q = by_scale[s]
        want = ops[name].numpy()
        assert a.shape == want.shape, name
        if name.startswith("w_"):
            assert np.array_equal(a, want), name                # the weight itself
        else:
            assert np.allclose(a, want, rtol=0, atol=1e-12), name
        assert np.allclose(q, _torch_fq(a, s).numpy(), rtol=0, atol=0), name
    assert np.allclose(got, ref.numpy(), rtol=0, atol=1e-12)


def test_fp8_saturating_scale_changes_only_its_own_gemm():
    """A scale so large that every element of its operand saturates to +-448/s: the layer
    output then follows the torch formulation with that one operand replaced, and moves away
    from the unchanged layer."""
    x, w, heads, scales = _layer_case(seed=12)
    base = O.encoder_layer(x, np.arange(x.shape[0]), w, heads, fp8_scales=scales, bf16_attention=True)
    for name in O.FP8_TENSORS:
        sc = dict(scales)
        sc[name] = 1e7
        got = O.encoder_layer(x, np.arange(x.shape[0]), w, heads, fp8_scales=sc, bf16_attention=True)
        _, ref = _torch_layer_fp8(x, w, heads, sc)
        assert np.allclose(got, ref.numpy(), rtol=0, atol=1e-12), name
        assert np.abs(got - base).max() > 1e-3, name


def test_weights_quantised_once_per_call_equal_quantising_per_sequence():
    """encode_packed runs layer by layer and fake-quantises each FP8 layer's weights once per
    call; encode_sequence quantises them inside every layer call of one sequence: the outputs
    are identical (bf16 and FP8 layers mixed)."""
    from transformer_esm_layer_gb300 import synth
    g = synth.Geometry(num_layers=3, hidden=64, heads=1, ffn=128)
    w = synth.model_weights(g, 3, "fp8", ln_random=True)
    lengths = [5, 9, 1]
    tok = synth.tokens_for_lengths(np.random.default_rng(0), lengths)
    sc = dict(zip(O.FP8_TENSORS, (3.0, 400.0, 5.0, 300.0, 7.0, 200.0, 9.0, 100.0)))
    st = [sc, None, sc]
    c = O.cu_seqlens(lengths)
    once = O.encode_packed(tok, c, w, g.heads, fp8_state=st, bf16_attention=True)
    for i in range(len(lengths)):
        alone = O.encode_sequence(tok[c[i]:c[i + 1]], w, g.heads, fp8_state=st, bf16_attention=True)
        assert np.array_equal(once[i], alone)
