"""Seeded synthetic inputs for the ESM-2 packed encoder: protein-length-distributed
token batches and random-init weights.

This module holds no arithmetic of the encoder itself. It only draws numbers and lays
them out, so that the float64 oracle and the CUDA library receive exactly the same
inputs. Every tensor is a plain numpy array.

Workloads (the sequence lengths include BOS and EOS):

* ``tiny_fp32``   -- 2 layers, hidden 64, 4 heads (head_dim 16), FFN 256, vocab 33,
  three sequences of lengths 17, 40, 7 (cu_seqlens = [0, 17, 57, 64]), seed 0.
* ``layer650m``   -- one ESM-2 650M layer (hidden 1280, 20 heads, FFN 5120), 16
  sequences with log-normal lengths (median 300, sigma 0.6) clipped to [32, 1024],
  seed 1.
* ``esm650m``     -- the full 33-layer 650M encoder, lengths drawn as above until the
  running total reaches 16384 tokens (the last one truncated to fill), seed 2.
* ``esm650m_padded`` -- the ``esm650m`` sequences laid out as [B, 1024] with pad id 1.
* ``esm3b_fp8``   -- the 36-layer 3B encoder (hidden 2560, 40 heads, FFN 10240), 32768
  packed tokens, seed 3.
* ``esm3b_fp4``   -- the same model and batch with every layer's linear maps in NVFP4
  (per-layer precision "fp4" on an FP8 encoder).

The geometry follows the ESM-2 model card ("BioNeMo ESM-2", model overview: 650M has 33
layers, 20 heads, hidden 1280; 3B has 36 layers, 40 heads, hidden 2560) and the NVIDIA
ESM-2 TransformerEngine walkthrough (config.json: vocab 33, 1026 positions, head size
hidden // heads).  Token ids: BOS = 0, pad = 1, EOS = 2, amino acids 4..23.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np

BOS_ID = 0
PAD_ID = 1
EOS_ID = 2
AA_LO, AA_HI = 4, 23  # inclusive range of the 20 canonical amino-acid ids

# Order in which per-layer tensors are drawn; the index is part of each tensor's seed.
LAYER_TENSORS = ("ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o",
                 "ln2_g", "ln2_b", "w_1", "b_1", "w_2", "b_2")


@dataclasses.dataclass(frozen=True)
class Geometry:
    num_layers: int
    hidden: int
    heads: int
    ffn: int
    vocab: int = 33
    max_positions: int = 1026

    @property
    def head_dim(self) -> int:
        return self.hidden // self.heads


TINY = Geometry(num_layers=2, hidden=64, heads=4, ffn=256)
ESM2_650M = Geometry(num_layers=33, hidden=1280, heads=20, ffn=5120)
ESM2_3B = Geometry(num_layers=36, hidden=2560, heads=40, ffn=10240)


@dataclasses.dataclass
class Workload:
    name: str
    geometry: Geometry
    precision: str          # "fp32" | "bf16" | "fp8"
    final_ln: bool
    seed: int
    lengths: List[int]
    padded_len: Optional[int] = None  # S for the padded [B, S] layout
    layer_precision: Optional[List[str]] = None  # per-layer GEMM precision on an fp8 encoder

    @property
    def total_tokens(self) -> int:
        return int(sum(self.lengths))


# --------------------------------------------------------------------------- lengths
def _lognormal_length(rng: np.random.Generator) -> int:
    z = rng.standard_normal()
    return int(np.clip(np.rint(np.exp(np.log(300.0) + 0.6 * z)), 32, 1024))


def lognormal_lengths(rng: np.random.Generator, count: Optional[int] = None,
                      total: Optional[int] = None) -> List[int]:
    """Draw lengths L = clip(rint(exp(ln 300 + 0.6 z)), 32, 1024) (rint = half to even).

    With ``count``: exactly that many draws. With ``total``: draw until the running sum
    reaches ``total``; the last length is cut so the sum is exactly ``total``.
    """
    out: List[int] = []
    if count is not None:
        return [_lognormal_length(rng) for _ in range(count)]
    assert total is not None and total > 0
    s = 0
    while s < total:
        L = _lognormal_length(rng)
        if s + L > total:
            L = total - s
        out.append(L)
        s += L
    return out


def cu_seqlens_from_lengths(lengths) -> np.ndarray:
    """Packed-batch offsets [0, L0, L0+L1, ...] as int32."""
    return np.concatenate([[0], np.cumsum(np.asarray(lengths, dtype=np.int64))]).astype(np.int32)


def tokens_for_lengths(rng: np.random.Generator, lengths) -> np.ndarray:
    """Flat int32 token ids: BOS, uniform amino acids 4..23, EOS per sequence."""
    T = int(sum(lengths))
    tok = rng.integers(AA_LO, AA_HI + 1, size=T, dtype=np.int64).astype(np.int32)
    cu = cu_seqlens_from_lengths(lengths)
    for i, L in enumerate(lengths):
        if L >= 1:
            tok[cu[i]] = BOS_ID
        if L >= 2:
            tok[cu[i] + L - 1] = EOS_ID
    return tok


def pad_tokens(tokens: np.ndarray, lengths, S: int) -> np.ndarray:
    """Lay packed sequences out as [B, S] with PAD_ID after each sequence."""
    cu = cu_seqlens_from_lengths(lengths)
    out = np.full((len(lengths), S), PAD_ID, dtype=np.int32)
    for i, L in enumerate(lengths):
        out[i, :L] = tokens[cu[i]:cu[i] + L]
    return out


# --------------------------------------------------------------------------- workloads
def make_workload(name: str) -> Workload:
    if name == "tiny_fp32":
        return Workload(name, TINY, "fp32", True, 0, [17, 40, 7])
    if name == "layer650m":
        g = dataclasses.replace(ESM2_650M, num_layers=1)
        rng = np.random.default_rng(1)
        return Workload(name, g, "bf16", False, 1, lognormal_lengths(rng, count=16))
    if name == "esm650m":
        rng = np.random.default_rng(2)
        return Workload(name, ESM2_650M, "bf16", True, 2, lognormal_lengths(rng, total=16384))
    if name == "esm650m_padded":
        rng = np.random.default_rng(2)
        return Workload(name, ESM2_650M, "bf16", True, 2, lognormal_lengths(rng, total=16384),
                        padded_len=1024)
    if name in ("esm3b_fp8", "esm3b_fp4"):
        rng = np.random.default_rng(3)
        lp = ["fp4"] * ESM2_3B.num_layers if name == "esm3b_fp4" else None
        return Workload(name, ESM2_3B, "fp8", True, 3, lognormal_lengths(rng, total=32768), layer_precision=lp)
    raise KeyError(name)


def workload_tokens(w: Workload) -> np.ndarray:
    """Token ids for a workload; drawn after the lengths from a stream of their own."""
    rng = np.random.default_rng([w.seed, 1000])
    return tokens_for_lengths(rng, w.lengths)


# --------------------------------------------------------------------------- weights
def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even) and return the uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + r) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal(seed_key, shape, std=0.02) -> np.ndarray:
    rng = np.random.default_rng(seed_key)
    return (rng.standard_normal(size=shape, dtype=np.float32) * np.float32(std))


def layer_weights(g: Geometry, seed: int, layer: int, ln_random: bool = False) -> Dict[str, np.ndarray]:
    """float32 weights of one layer. Linear weights and biases ~ N(0, 0.02); LayerNorm
    gamma = 1, beta = 0 (or gamma ~ 1 + N(0, 0.1), beta ~ N(0, 0.1) with ``ln_random``).
    Linear weights are [out_features, in_features]; w_qkv rows are q | k | v, each
    head-major (row h*head_dim + c)."""
    d, f = g.hidden, g.ffn
    shapes = {"ln1_g": (d,), "ln1_b": (d,), "w_qkv": (3 * d, d), "b_qkv": (3 * d,),
              "w_o": (d, d), "b_o": (d,), "ln2_g": (d,), "ln2_b": (d,),
              "w_1": (f, d), "b_1": (f,), "w_2": (d, f), "b_2": (d,)}
    out = {}
    for ti, name in enumerate(LAYER_TENSORS):
        key = [seed, 1 + layer, ti]
        if name.endswith("_g"):
            out[name] = (1.0 + _normal(key, shapes[name], 0.1)) if ln_random else np.ones(shapes[name], np.float32)
        elif name.startswith("ln"):
            out[name] = _normal(key, shapes[name], 0.1) if ln_random else np.zeros(shapes[name], np.float32)
        else:
            out[name] = _normal(key, shapes[name])
    return out


def model_weights(g: Geometry, seed: int, precision: str, ln_random: bool = False,
                  num_layers: Optional[int] = None) -> Dict:
    """All weights of an encoder as float32 arrays holding exactly the values the GPU sees
    (rounded through bfloat16 for the bf16 and fp8 precisions).

    Returns {"emb": [V,d], "layers": [dict per layer], "lnf_g": [d], "lnf_b": [d]}.
    """
    n = g.num_layers if num_layers is None else num_layers
    rnd = (lambda a: bf16_bits_to_f32(f32_to_bf16_bits(a))) if precision in ("bf16", "fp8") else (lambda a: a)
    emb = rnd(_normal([seed, 0, 0], (g.vocab, g.hidden)))
    layers = [{k: rnd(v) for k, v in layer_weights(g, seed, l, ln_random).items()} for l in range(n)]
    key = [seed, 10_000, 0]
    lnf_g = (1.0 + _normal(key, (g.hidden,), 0.1)) if ln_random else np.ones(g.hidden, np.float32)
    lnf_b = _normal([seed, 10_000, 1], (g.hidden,), 0.1) if ln_random else np.zeros(g.hidden, np.float32)
    return {"emb": emb, "layers": layers, "lnf_g": rnd(lnf_g), "lnf_b": rnd(lnf_b)}


def lm_head_weights(g: Geometry, seed: int, precision: str, emb: np.ndarray, ln_random: bool = True) -> Dict:
    """Masked-LM head weights: dense [d, d] and bias [d] ~ N(0, 0.02), LayerNorm gamma / beta
    (random around 1 / 0 with ``ln_random``), the vocabulary bias [V] ~ N(0, 0.02), and the
    output projection tied to the given token embedding [V, d]."""
    d = g.hidden
    rnd = (lambda a: bf16_bits_to_f32(f32_to_bf16_bits(a))) if precision in ("bf16", "fp8") else (lambda a: a)
    ln_g = (1.0 + _normal([seed, 20_000, 2], (d,), 0.1)) if ln_random else np.ones(d, np.float32)
    ln_b = _normal([seed, 20_000, 3], (d,), 0.1) if ln_random else np.zeros(d, np.float32)
    return {"dense_w": rnd(_normal([seed, 20_000, 0], (d, d))), "dense_b": rnd(_normal([seed, 20_000, 1], (d,))),
            "ln_g": rnd(ln_g), "ln_b": rnd(ln_b), "emb": emb,
            "bias": rnd(_normal([seed, 20_000, 4], (g.vocab,)))}


def mlm_targets(tokens: np.ndarray, seed: int, rate: float = 0.15) -> np.ndarray:
    """Masked-LM targets for a token batch: each position is scored with probability
    ``rate`` (target = its token id), otherwise -100 (not scored)."""
    rng = np.random.default_rng([seed, 30_000])
    pick = rng.random(len(tokens)) < rate
    return np.where(pick, np.asarray(tokens, np.int64), -100).astype(np.int32)


def random_lengths_case(seed: int, count: int, lo: int, hi: int) -> List[int]:
    """Uniform integer lengths in [lo, hi] for parity cases with ragged tiles."""
    rng = np.random.default_rng([seed, 77])
    return [int(x) for x in rng.integers(lo, hi + 1, size=count)]
