"""Float64 CPU oracle of FP4 (E2M1) block-scaled quantisation of GEMM operands.

TEST INFRASTRUCTURE ONLY (same rules as ``esm_oracle``).  This module fixes what an FP4
operand and an FP4 layer compute, so that the CUDA library's NVFP4 kernels can be checked
against it.

Source: the mlqm.cn walkthrough ("深入源码NVIDIA ESM-2 TransformerEngine优化的实现原理与技术细节"),
section FP8与FP4混合精度支持: ``NVEsmEncoder`` takes an ``fp4_recipe`` beside the FP8 one and
``layer_precision`` picks FP8 or FP4 per layer.  The pages give no FP4 format.  Reading (the
block-scaled FP4 of the GPUs the pages name): values in E2M1 (1 sign, 2 exponent bits with
bias 1, 1 mantissa bit: 0, 0.5, 1, 1.5, 2, 3, 4, 6), one E4M3 scale per block of 16
consecutive values along the reduction axis, and one fp32 scale per tensor chosen so that
the largest block scale is exactly representable: S = 448 * 6 / amax(tensor).

Parity pins: tests/test_oracle_fp4_pins.py (exhaustive E2M1 codes from their bit fields,
ties to even, saturation, block-scale invariants, error bound against the exact values).
"""
from __future__ import annotations

import numpy as np

from .esm_oracle import E4M3_MAX, e4m3_round

E2M1_MAX = 6.0
E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])  # codes 0..7 (sign separate)
BLOCK = 16


def e2m1_round(x: np.ndarray) -> np.ndarray:
    """Round to the nearest E2M1 value, ties to the even code (mantissa bit 0), saturating
    at +-6.  The representable magnitudes are spaced 0.5 below 2, 1 in [2, 4), 2 in [4, 6]."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E2M1_MAX)
    # distance to every code; on a tie the lower code wins only if it is even
    d = np.abs(a[..., None] - E2M1_VALUES)
    best = np.argmin(d, axis=-1)
    dmin = np.take_along_axis(d, best[..., None], axis=-1)[..., 0]
    nxt = np.minimum(best + 1, len(E2M1_VALUES) - 1)
    dn = np.take_along_axis(d, nxt[..., None], axis=-1)[..., 0]
    tie = (nxt != best) & (dn == dmin) & (best % 2 == 1)
    code = np.where(tie, nxt, best)
    return np.copysign(E2M1_VALUES[code], x)


def nvfp4_fake_quant(a: np.ndarray, axis: int = -1, S: float = None):
    """An operand as a block-scaled FP4 GEMM sees it: blocks of 16 along `axis` (its length a
    multiple of 16).  Returns (dequantised values, per-block E4M3 scales, tensor scale S).

    S = 448 * 6 / amax(a) (1 when a is all zero), or the given S (a tensor whose amax spans
    more than the values passed here, e.g. a whole packed batch of which `a` is one sequence);
    block scale sb = E4M3(amax_block / 6 * S); q = E2M1(a * S / sb) (0 for an all-zero block);
    dequantised a ~ q * sb / S."""
    a = np.asarray(a, dtype=np.float64)
    x = np.moveaxis(a, axis, -1)
    K = x.shape[-1]
    if K % BLOCK:
        raise ValueError("the blocked axis must be a multiple of 16")
    xb = x.reshape(x.shape[:-1] + (K // BLOCK, BLOCK))
    if S is None:
        amax = float(np.abs(a).max(initial=0.0))
        S = E4M3_MAX * E2M1_MAX / amax if amax > 0 else 1.0
    bmax = np.abs(xb).max(axis=-1)
    sb = e4m3_round(bmax / E2M1_MAX * S)
    safe = np.where(sb > 0, sb, 1.0)
    q = np.where(sb[..., None] > 0, e2m1_round(xb * S / safe[..., None]), 0.0)
    deq = (q * sb[..., None] / S).reshape(x.shape)
    return np.moveaxis(deq, -1, axis), sb, S
