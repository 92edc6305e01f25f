"""Pins of the FP4 (E2M1, block-scaled) oracle: the code table from its bit fields, ties,
saturation, and the block-scaling invariants and error bound."""
import numpy as np
import pytest

from oracle import fp4 as F4
from oracle import esm_oracle as O


def _e2m1_decode(code: int) -> float:
    """Value of a 4-bit E2M1 code from its fields: sign, 2 exponent bits (bias 1), 1 mantissa
    bit; exponent 0 is subnormal (0 or 0.5)."""
    s = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    return s * (m * 0.5 if e == 0 else (1 + m / 2.0) * 2.0 ** (e - 1))


def test_e2m1_table_and_exact_round_trip():
    vals = np.array([_e2m1_decode(c) for c in range(16)])
    assert np.array_equal(np.abs(vals[:8]), F4.E2M1_VALUES)
    assert np.array_equal(F4.e2m1_round(vals), vals)  # every code is its own rounding


def test_e2m1_ties_to_even_and_saturation():
    # midpoints between neighbours go to the code with mantissa bit 0
    mids = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for x, want in mids.items():
        assert F4.e2m1_round(np.array([x]))[0] == want, x
        assert F4.e2m1_round(np.array([-x]))[0] == -want, x
    assert F4.e2m1_round(np.array([6.9, 1e9, -7.0])).tolist() == [6.0, 6.0, -6.0]
    # off-midpoint values go to the nearest code
    rng = np.random.default_rng(0)
    x = rng.uniform(-6, 6, 2000)
    r = F4.e2m1_round(x)
    d = np.abs(np.abs(x)[:, None] - F4.E2M1_VALUES[None, :]).min(axis=1)
    assert np.allclose(np.abs(np.abs(x) - np.abs(r)), d)


def test_block_scaling_invariants_and_error_bound():
    rng = np.random.default_rng(1)
    a = rng.standard_normal((8, 64)) * np.exp(rng.uniform(-3, 3, (8, 1)))  # rows of very different size
    deq, sb, S = F4.nvfp4_fake_quant(a, axis=1)
    # the largest block scale equals 448 exactly (so it is representable in E4M3)
    assert sb.max() == pytest.approx(O.E4M3_MAX, rel=1e-12)
    assert np.array_equal(O.e4m3_round(sb), sb)
    # every dequantised value is a representable E2M1 value times its block's scale
    q = deq.reshape(8, 4, 16) * S / sb[..., None]
    assert np.allclose(F4.e2m1_round(q), q, atol=1e-9)
    # error bound: half the largest E2M1 spacing of the block (2 at the top) in real units,
    # plus the block scale's own E4M3 rounding
    blk = np.abs(a.reshape(8, 4, 16)).max(axis=-1)
    err = np.abs(deq - a).reshape(8, 4, 16).max(axis=-1)
    assert np.all(err <= blk * (1.0 / 6.0 + 2 ** -3) + 1e-12)
    # scaling the whole tensor by a power of two scales the result exactly
    deq2, _, _ = F4.nvfp4_fake_quant(a * 8.0, axis=1)
    assert np.array_equal(deq2, deq * 8.0)


def test_zero_blocks_and_axis():
    a = np.zeros((3, 32))
    a[1, 16:] = np.linspace(-1, 1, 16)
    deq, sb, S = F4.nvfp4_fake_quant(a)
    assert np.all(deq[0] == 0) and np.all(deq[1, :16] == 0) and sb[0, 0] == 0
    z, _, S0 = F4.nvfp4_fake_quant(np.zeros((2, 16)))
    assert np.all(z == 0) and S0 == 1.0
    # blocks along axis 0 equal blocks along the last axis of the transpose
    b = np.random.default_rng(2).standard_normal((32, 5))
    d0, _, _ = F4.nvfp4_fake_quant(b, axis=0)
    d1, _, _ = F4.nvfp4_fake_quant(b.T, axis=-1)
    assert np.array_equal(d0, d1.T)
    with pytest.raises(ValueError):
        F4.nvfp4_fake_quant(np.ones((2, 10)))


def test_fp4_layer_tensor_to_scale_mapping(monkeypatch):
    """The NVFP4 layer of the oracle: each of the eight tensor scales meets exactly the operand
    of its GEMM (activations as the bf16 tensors the layer holds, weights as given), and the
    layer output follows an independent torch float64 composition of the recorded quantised
    operands (LayerNorm, RoPE as a complex rotation, SDPA, exact GELU, residuals)."""
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(13)
    L, d, heads, f = 5, 32, 2, 64
    w = {"ln1_g": 1 + 0.2 * rng.standard_normal(d), "ln1_b": 0.2 * rng.standard_normal(d),
         "w_qkv": 0.2 * rng.standard_normal((3 * d, d)), "b_qkv": 0.1 * rng.standard_normal(3 * d),
         "w_o": 0.2 * rng.standard_normal((d, d)), "b_o": 0.1 * rng.standard_normal(d),
         "ln2_g": 1 + 0.2 * rng.standard_normal(d), "ln2_b": 0.2 * rng.standard_normal(d),
         "w_1": 0.2 * rng.standard_normal((f, d)), "b_1": 0.1 * rng.standard_normal(f),
         "w_2": 0.2 * rng.standard_normal((d, f)), "b_2": 0.1 * rng.standard_normal(d)}
    x = rng.standard_normal((L, d))
    scales = dict(zip(O.FP8_TENSORS, (3.0, 5.0, 7.0, 11.0, 13.0, 17.0, 19.0, 23.0)))
    calls = []
    real = F4.nvfp4_fake_quant

    def recording(a, axis=-1, S=None):
        out = real(a, axis, S)
        calls.append((float(S), np.array(a, copy=True), out[0]))
        return out

    monkeypatch.setattr(F4, "nvfp4_fake_quant", recording)
    got = O.encoder_layer(x, np.arange(L), w, heads, bf16_attention=True, fp4_scales=scales)
    monkeypatch.setattr(F4, "nvfp4_fake_quant", real)
    assert len(calls) == 8
    by = {s: (a, q) for s, a, q in calls}
    assert sorted(by) == sorted(scales.values())
    t = lambda a: torch.as_tensor(np.asarray(a, np.float64))
    bf = lambda u: u.to(torch.float32).to(torch.bfloat16).to(torch.float64)
    q = lambda name: t(by[scales[name]][1])
    for name in ("w_qkv", "w_o", "w_1", "w_2"):
        assert np.array_equal(by[scales[name]][0], w[name]), name
    X = t(x)
    y = F.layer_norm(X, (d,), t(w["ln1_g"]), t(w["ln1_b"]), eps=1e-5)
    assert np.allclose(by[scales["x_qkv"]][0], bf(y).numpy(), rtol=0, atol=0)
    qkv = q("x_qkv") @ q("w_qkv").T + t(w["b_qkv"])
    dh = d // heads
    qh, kh, vh = (qkv[:, i * d:(i + 1) * d].reshape(L, heads, dh) for i in range(3))
    half = dh // 2
    theta = 10000.0 ** (-2.0 * torch.arange(half, dtype=torch.float64) / dh)
    rot = torch.polar(torch.ones(L, half, dtype=torch.float64), torch.arange(L, dtype=torch.float64)[:, None] * theta)

    def rope(u):
        zc = torch.complex(u[..., :half], u[..., half:]) * rot[:, None, :]
        return torch.cat([zc.real, zc.imag], dim=-1)

    o = F.scaled_dot_product_attention(bf(rope(qh)).transpose(0, 1), bf(rope(kh)).transpose(0, 1),
                                       bf(vh).transpose(0, 1)).transpose(0, 1).reshape(L, d)
    assert np.allclose(by[scales["x_o"]][0], bf(o).numpy(), rtol=0, atol=1e-12)
    X = X + q("x_o") @ q("w_o").T + t(w["b_o"])
    z = F.layer_norm(X, (d,), t(w["ln2_g"]), t(w["ln2_b"]), eps=1e-5)
    assert np.allclose(by[scales["x_1"]][0], bf(z).numpy(), rtol=0, atol=1e-12)
    u = F.gelu(q("x_1") @ q("w_1").T + t(w["b_1"]))
    assert np.allclose(by[scales["x_2"]][0], bf(u).numpy(), rtol=0, atol=1e-12)
    X = X + q("x_2") @ q("w_2").T + t(w["b_2"])
    assert np.allclose(got, X.numpy(), rtol=0, atol=1e-12)


def test_fp4_given_scale_equals_own_scale():
    """nvfp4_fake_quant with S given as the tensor's own 448 * 6 / amax is the default."""
    rng = np.random.default_rng(14)
    a = rng.standard_normal((3, 64))
    S = 448.0 * 6.0 / np.abs(a).max()
    d0, s0, S0 = F4.nvfp4_fake_quant(a)
    d1, s1, S1 = F4.nvfp4_fake_quant(a, S=S)
    assert S0 == S1 and np.array_equal(d0, d1) and np.array_equal(s0, s1)
