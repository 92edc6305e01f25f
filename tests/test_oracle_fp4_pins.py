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
