"""Helpers shared by the test files (no arithmetic of the encoder lives here)."""
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def header_functions():
    """Names of the functions include/esm_encoder.h declares."""
    with open(os.path.join(ROOT, "include", "esm_encoder.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^ESM_API\s+[\w\s\*]+?\b(esm_\w+)\s*\(", text, flags=re.M)))


def ensure_built():
    from transformer_esm_layer_gb300 import build
    return build.build()


def to_np(t):
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def e4m3_table():
    """Value of every E4M3 byte from its bit fields (OCP layout: sign, 4 exponent bits with
    bias 7, 3 mantissa bits; 0x7F / 0xFF are NaN)."""
    vals = np.zeros(256)
    for code in range(256):
        s = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            vals[code] = np.nan
        elif e == 0:
            vals[code] = s * m * 2.0 ** -9
        else:
            vals[code] = s * (1 + m / 8.0) * 2.0 ** (e - 7)
    return vals
