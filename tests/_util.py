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
