"""Thin ctypes binding of the C ABI in include/esm_encoder.h.

Argument marshalling only: every step of the forward runs in the CUDA library.  torch is
used for device memory and streams.  Loading fails loudly when the library has not been
built; there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional, Sequence

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libesm_encoder.so")

ESM_OK = 0
STATUS_NAMES = {0: "ESM_OK", 1: "ESM_ERR_INVALID_ARG", 2: "ESM_ERR_UNSUPPORTED", 3: "ESM_ERR_BAD_CU_SEQLENS",
                4: "ESM_ERR_TOKEN_RANGE", 5: "ESM_ERR_WORKSPACE", 6: "ESM_ERR_CUDA", 7: "ESM_ERR_TIMEOUT"}
PRECISIONS = {"fp32": 0, "bf16": 1, "fp8": 2, "fp4": 3}
EPILOGUES = {"bias_f32": 0, "qkv_rope": 1, "residual": 2, "gelu": 3}

# Every symbol the header declares (checked by the tests).
EXPORTS = ("esm_encoder_create", "esm_encoder_destroy", "esm_encoder_workspace_size", "esm_encoder_forward",
           "esm_encoder_forward_host", "esm_encoder_forward_padded", "esm_encoder_check",
           "esm_encoder_debug_pack_index", "esm_op_layernorm", "esm_op_gemm", "esm_op_attention",
           "esm_encoder_get_fp8_state", "esm_encoder_set_fp8_state", "esm_encoder_set_profiling",
           "esm_encoder_get_profile", "esm_op_attention_noalloc", "esm_op_layernorm_e4m3", "esm_op_gemm_fp8",
           "esm_encoder_debug_wait_timeout", "esm_encoder_lm_head_workspace_size", "esm_encoder_lm_head",
           "esm_encoder_set_layer_precision",
           "esm_encoder_train_buffer_size", "esm_encoder_forward_train", "esm_encoder_backward",
           "esm_op_gemm_dgrad", "esm_op_gemm_wgrad_workspace_size", "esm_op_gemm_wgrad",
           "esm_op_layernorm_backward_workspace_size", "esm_op_layernorm_backward", "esm_op_attention_train",
           "esm_op_attention_backward_workspace_size", "esm_op_attention_backward",
           "esm_encoder_lm_head_backward_workspace_size", "esm_encoder_lm_head_backward",
           "esm_op_quantize_nvfp4", "esm_op_gemm_nvfp4", "esm_encoder_get_fp4_scales", "esm_status_string")
PROFILE_CLASSES = ("gemm_qkv", "attention", "gemm_oproj", "gemm_fc1", "gemm_fc2", "layernorm", "other",
                   "gemm_backward")


class EsmError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")
        self.status = status


class EsmConfig(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int), ("hidden", ctypes.c_int), ("heads", ctypes.c_int),
                ("ffn", ctypes.c_int), ("vocab", ctypes.c_int), ("max_positions", ctypes.c_int),
                ("ln_eps", ctypes.c_float), ("rope_base", ctypes.c_float), ("emb_scale", ctypes.c_float),
                ("final_ln", ctypes.c_int), ("precision", ctypes.c_int), ("amax_history_len", ctypes.c_int)]


_PP = ctypes.POINTER(ctypes.c_void_p)


class EsmProfile(ctypes.Structure):
    _fields_ = [("ms", ctypes.c_double * 8), ("launches", ctypes.c_longlong * 8), ("total_launches", ctypes.c_longlong)]


class EsmWeights(ctypes.Structure):
    _fields_ = [("emb", ctypes.c_void_p)] + \
        [(n, _PP) for n in ("ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o", "ln2_g", "ln2_b",
                            "w_1", "b_1", "w_2", "b_2")] + \
        [("lnf_g", ctypes.c_void_p), ("lnf_b", ctypes.c_void_p)]


_PF = ctypes.POINTER(ctypes.c_void_p)
GRAD_NAMES = ("ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o", "ln2_g", "ln2_b", "w_1", "b_1", "w_2", "b_2")


class EsmGrads(ctypes.Structure):
    _fields_ = [("emb", ctypes.c_void_p)] + [(n, _PF) for n in GRAD_NAMES] + \
        [("lnf_g", ctypes.c_void_p), ("lnf_b", ctypes.c_void_p)]


LM_HEAD_NAMES = ("dense_w", "dense_b", "ln_g", "ln_b", "emb", "bias")


class EsmLmHead(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in LM_HEAD_NAMES]


class EsmLmHeadGrads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in LM_HEAD_NAMES]


_lib = None


def load_library() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                           "(run python -m transformer_esm_layer_gb300.build)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    sig = {
        "esm_encoder_create": (i32, [ctypes.POINTER(EsmConfig), ctypes.POINTER(vp)]),
        "esm_encoder_destroy": (None, [vp]),
        "esm_encoder_workspace_size": (i32, [vp, i32, i32, ctypes.POINTER(sz)]),
        "esm_encoder_forward": (i32, [vp, ctypes.POINTER(EsmWeights), vp, vp, i32, i32, i32, vp, vp, sz, vp]),
        "esm_encoder_forward_host": (i32, [vp, ctypes.POINTER(EsmWeights), vp, vp, i32, i32, i32, vp, vp, sz, vp]),
        "esm_encoder_forward_padded": (i32, [vp, ctypes.POINTER(EsmWeights), vp, vp, i32, i32, vp, vp, sz, vp]),
        "esm_encoder_check": (i32, [vp, vp]),
        "esm_encoder_set_layer_precision": (i32, [vp, ctypes.POINTER(ctypes.c_int), i32]),
        "esm_encoder_lm_head_workspace_size": (i32, [vp, i32, ctypes.POINTER(sz)]),
        "esm_encoder_lm_head": (i32, [vp, ctypes.POINTER(EsmLmHead), vp, i32, vp, vp, vp, vp, vp, vp, sz, vp]),
        "esm_encoder_debug_pack_index": (i32, [vp, vp, i32, i32, i32, vp, vp, vp, sz, vp]),
        "esm_op_layernorm": (i32, [vp, vp, vp, vp, vp, i32, i32, vp]),
        "esm_op_gemm": (i32, [vp, i32, vp, vp, vp, vp, vp, i32, i32, i32, vp]),
        "esm_op_attention": (i32, [vp, vp, vp, i32, i32, i32, vp, vp, sz, vp]),
        "esm_encoder_get_fp8_state": (i32, [vp, ctypes.POINTER(ctypes.c_float), sz]),
        "esm_encoder_set_fp8_state": (i32, [vp, ctypes.POINTER(ctypes.c_float), sz]),
        "esm_encoder_set_profiling": (i32, [vp, i32]),
        "esm_encoder_get_profile": (i32, [vp, ctypes.POINTER(EsmProfile), i32]),
        "esm_op_attention_noalloc": (i32, [vp, vp, i32, i32, i32, i32, i32, vp, vp, vp]),
        "esm_op_quantize_nvfp4": (i32, [vp, vp, i32, i32, vp, vp, vp, vp, vp]),
        "esm_encoder_get_fp4_scales": (i32, [vp, ctypes.POINTER(ctypes.c_float), sz]),
        "esm_op_gemm_nvfp4": (i32, [vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, vp]),
        "esm_op_layernorm_e4m3": (i32, [vp, vp, vp, vp, vp, i32, i32, vp, vp, vp]),
        "esm_encoder_debug_wait_timeout": (i32, [vp, i32, vp]),
        "esm_op_gemm_fp8": (i32, [vp, i32, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, vp]),
        "esm_status_string": (ctypes.c_char_p, [i32]),
        "esm_encoder_train_buffer_size": (i32, [vp, i32, ctypes.POINTER(sz)]),
        "esm_encoder_forward_train": (i32, [vp, ctypes.POINTER(EsmWeights), vp, vp, i32, i32, i32, vp, vp, sz, vp, sz,
                                            vp]),
        "esm_encoder_backward": (i32, [vp, ctypes.POINTER(EsmWeights), vp, ctypes.POINTER(EsmGrads), vp, sz, vp, sz,
                                       vp]),
        "esm_op_gemm_dgrad": (i32, [vp, vp, vp, vp, i32, i32, i32, i32, vp]),
        "esm_op_gemm_wgrad_workspace_size": (i32, [vp, i32, i32, ctypes.POINTER(sz)]),
        "esm_op_gemm_wgrad": (i32, [vp, vp, vp, vp, i32, i32, i32, vp, sz, vp]),
        "esm_op_layernorm_backward_workspace_size": (i32, [vp, i32, i32, ctypes.POINTER(sz)]),
        "esm_op_layernorm_backward": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, vp, sz, vp]),
        "esm_op_attention_train": (i32, [vp, vp, vp, i32, i32, i32, vp, vp, vp, sz, vp]),
        "esm_op_attention_backward_workspace_size": (i32, [vp, i32, i32, ctypes.POINTER(sz)]),
        "esm_op_attention_backward": (i32, [vp, vp, vp, vp, vp, vp, i32, i32, i32, vp, vp, sz, vp]),
        "esm_encoder_lm_head_backward_workspace_size": (i32, [vp, i32, ctypes.POINTER(sz)]),
        "esm_encoder_lm_head_backward": (i32, [vp, ctypes.POINTER(EsmLmHead), vp, i32, vp, vp,
                                               ctypes.POINTER(EsmLmHeadGrads), vp, vp, vp, vp, sz, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return stream.cuda_stream or None


class DeviceWeights:
    """Weights on the device in the handle's parameter dtype, plus the esm_weights struct.

    ``w`` is the dict returned by synth.model_weights (float32 arrays)."""

    def __init__(self, w: Dict, precision: str, device="cuda"):
        import torch
        dt = torch.float32 if precision == "fp32" else torch.bfloat16
        to = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device=device, dtype=dt)
        self.emb = to(w["emb"])
        self.layers = [{k: to(v) for k, v in wl.items()} for wl in w["layers"]]
        self.lnf_g = to(w["lnf_g"])
        self.lnf_b = to(w["lnf_b"])
        self._keep = []
        n = len(self.layers)
        st = EsmWeights()
        st.emb = self.emb.data_ptr()
        for name in ("ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o", "ln2_g", "ln2_b", "w_1", "b_1", "w_2", "b_2"):
            arr = (ctypes.c_void_p * max(n, 1))(*[l[name].data_ptr() for l in self.layers])
            self._keep.append(arr)
            setattr(st, name, ctypes.cast(arr, _PP))
        st.lnf_g = self.lnf_g.data_ptr()
        st.lnf_b = self.lnf_b.data_ptr()
        self.struct = st


class DeviceGrads:
    """float32 gradient buffers on the device, shaped like the weights, plus the esm_grads
    struct (esm_encoder_backward overwrites them)."""

    def __init__(self, g, num_layers: int, device="cuda"):
        import torch
        z = lambda *shape: torch.empty(*shape, dtype=torch.float32, device=device)
        d, f = g.hidden, g.ffn
        shapes = {"ln1_g": (d,), "ln1_b": (d,), "w_qkv": (3 * d, d), "b_qkv": (3 * d,), "w_o": (d, d), "b_o": (d,),
                  "ln2_g": (d,), "ln2_b": (d,), "w_1": (f, d), "b_1": (f,), "w_2": (d, f), "b_2": (d,)}
        self.emb = z(g.vocab, d)
        self.layers = [{k: z(*s) for k, s in shapes.items()} for _ in range(num_layers)]
        self.lnf_g = z(d)
        self.lnf_b = z(d)
        self._keep = []
        st = EsmGrads()
        st.emb = self.emb.data_ptr()
        for name in GRAD_NAMES:
            arr = (ctypes.c_void_p * max(num_layers, 1))(*[l[name].data_ptr() for l in self.layers])
            self._keep.append(arr)
            setattr(st, name, ctypes.cast(arr, _PF))
        st.lnf_g = self.lnf_g.data_ptr()
        st.lnf_b = self.lnf_b.data_ptr()
        self.struct = st

    def tensors(self):
        """Every gradient tensor in a fixed order (embedding, layers, final LayerNorm)."""
        return [self.emb] + [l[n] for l in self.layers for n in GRAD_NAMES] + [self.lnf_g, self.lnf_b]


class DeviceLmHead:
    """Masked-LM head weights on the device (handle's parameter dtype) plus the esm_lm_head
    struct; ``w`` is the dict of synth.lm_head_weights (its "emb" is the tied embedding)."""

    def __init__(self, w: Dict, precision: str, device="cuda"):
        import torch
        dt = torch.float32 if precision == "fp32" else torch.bfloat16
        to = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device=device, dtype=dt)
        self.t = {k: to(w[k]) for k in ("dense_w", "dense_b", "ln_g", "ln_b", "emb", "bias")}
        self.struct = EsmLmHead(*[self.t[k].data_ptr() for k in ("dense_w", "dense_b", "ln_g", "ln_b", "emb", "bias")])


class EsmEncoder:
    """One esm_encoder handle (the esm_encoder_* calls with their own names)."""

    def __init__(self, num_layers: int, hidden: int, heads: int, ffn: int, vocab: int = 33,
                 max_positions: int = 1026, precision: str = "bf16", final_ln: bool = True,
                 ln_eps: float = 1e-5, rope_base: float = 10000.0, emb_scale: float = 1.0,
                 amax_history_len: int = 16):
        self.lib = load_library()
        self.cfg = EsmConfig(num_layers, hidden, heads, ffn, vocab, max_positions, ln_eps, rope_base, emb_scale,
                             int(final_ln), PRECISIONS[precision], amax_history_len)
        self.precision = precision
        self.hidden = hidden
        self.num_layers = num_layers
        self.amax_history_len = amax_history_len
        h = ctypes.c_void_p()
        self._raise(self.lib.esm_encoder_create(ctypes.byref(self.cfg), ctypes.byref(h)), "esm_encoder_create")
        self.handle = h

    @classmethod
    def from_geometry(cls, g, precision: str, final_ln: bool = True, **kw):
        return cls(g.num_layers, g.hidden, g.heads, g.ffn, g.vocab, g.max_positions, precision, final_ln, **kw)

    @staticmethod
    def _raise(st: int, where: str):
        if st != ESM_OK:
            raise EsmError(st, where)

    def close(self):
        if getattr(self, "handle", None):
            self.lib.esm_encoder_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------------ buffers
    @property
    def out_dtype(self):
        import torch
        return torch.float32 if self.precision == "fp32" else torch.bfloat16

    def workspace_size(self, max_tokens: int, max_seqs: int) -> int:
        n = ctypes.c_size_t()
        self._raise(self.lib.esm_encoder_workspace_size(self.handle, max_tokens, max_seqs, ctypes.byref(n)),
                    "esm_encoder_workspace_size")
        return n.value

    def workspace(self, max_tokens: int, max_seqs: int, device="cuda"):
        import torch
        return torch.empty(self.workspace_size(max_tokens, max_seqs), dtype=torch.uint8, device=device)

    # ------------------------------------------------------------------ calls
    def forward(self, weights: DeviceWeights, token_ids, cu_seqlens, max_seqlen: int, out=None, workspace=None,
                stream=None, check: bool = False):
        import torch
        T = token_ids.numel()
        B = cu_seqlens.numel() - 1
        if out is None:
            out = torch.empty(T, self.hidden, dtype=self.out_dtype, device=token_ids.device)
        if workspace is None:
            workspace = self.workspace(T, B, token_ids.device)
        st = self.lib.esm_encoder_forward(self.handle, ctypes.byref(weights.struct), _ptr(token_ids),
                                          _ptr(cu_seqlens), B, T, int(max_seqlen), _ptr(out), _ptr(workspace),
                                          workspace.numel(), _stream_ptr(stream))
        self._raise(st, "esm_encoder_forward")
        if check:
            self.check(stream)
        return out

    def forward_host(self, weights: DeviceWeights, token_ids: np.ndarray, cu_seqlens: np.ndarray, max_seqlen: int,
                     out: np.ndarray, workspace, stream=None):
        """Host buffers in and out (numpy arrays, or pinned torch CPU tensors via .numpy())."""
        T = int(token_ids.size)
        B = int(cu_seqlens.size) - 1
        st = self.lib.esm_encoder_forward_host(self.handle, ctypes.byref(weights.struct),
                                               token_ids.ctypes.data, cu_seqlens.ctypes.data, B, T, int(max_seqlen),
                                               out.ctypes.data, _ptr(workspace), workspace.numel(),
                                               _stream_ptr(stream))
        self._raise(st, "esm_encoder_forward_host")
        return out

    def forward_padded(self, weights: DeviceWeights, token_ids, seq_lens, out=None, workspace=None, stream=None,
                       check: bool = False):
        import torch
        B, S = token_ids.shape
        if out is None:
            out = torch.empty(B, S, self.hidden, dtype=self.out_dtype, device=token_ids.device)
        if workspace is None:
            workspace = self.workspace(B * S, B, token_ids.device)
        st = self.lib.esm_encoder_forward_padded(self.handle, ctypes.byref(weights.struct), _ptr(token_ids),
                                                 _ptr(seq_lens), B, S, _ptr(out), _ptr(workspace), workspace.numel(),
                                                 _stream_ptr(stream))
        self._raise(st, "esm_encoder_forward_padded")
        if check:
            self.check(stream)
        return out

    def check(self, stream=None) -> int:
        st = self.lib.esm_encoder_check(self.handle, _stream_ptr(stream))
        self._raise(st, "esm_encoder_check")
        return st

    def check_status(self, stream=None) -> int:
        """Like check() but returns the status instead of raising."""
        return self.lib.esm_encoder_check(self.handle, _stream_ptr(stream))

    def debug_pack_index(self, cu_seqlens, total_tokens: int, max_seqlen: int, workspace=None, stream=None):
        import torch
        B = cu_seqlens.numel() - 1
        pos = torch.empty(max(total_tokens, 1), dtype=torch.int32, device=cu_seqlens.device)
        seg = torch.empty_like(pos)
        if workspace is None:
            workspace = self.workspace(total_tokens, B, cu_seqlens.device)
        st = self.lib.esm_encoder_debug_pack_index(self.handle, _ptr(cu_seqlens), B, total_tokens, int(max_seqlen),
                                                   _ptr(pos), _ptr(seg), _ptr(workspace), workspace.numel(),
                                                   _stream_ptr(stream))
        self._raise(st, "esm_encoder_debug_pack_index")
        return pos[:total_tokens], seg[:total_tokens]

    def debug_wait_timeout(self, timeout_us: int, stream=None):
        self._raise(self.lib.esm_encoder_debug_wait_timeout(self.handle, int(timeout_us), _stream_ptr(stream)),
                    "esm_encoder_debug_wait_timeout")

    def op_layernorm(self, x, gamma, beta, y, stream=None):
        rows, cols = x.shape
        self._raise(self.lib.esm_op_layernorm(self.handle, _ptr(x), _ptr(gamma), _ptr(beta), _ptr(y), rows, cols,
                                              _stream_ptr(stream)), "esm_op_layernorm")
        return y

    def op_gemm(self, epi: str, A, B, bias, out, pos_id=None, stream=None):
        M, K = A.shape
        N = B.shape[0]
        self._raise(self.lib.esm_op_gemm(self.handle, EPILOGUES[epi], _ptr(A), _ptr(B), _ptr(bias), _ptr(out),
                                         _ptr(pos_id), M, N, K, _stream_ptr(stream)), "esm_op_gemm")
        return out

    def op_layernorm_e4m3(self, x, gamma, beta, y, scale, amax, stream=None):
        rows, cols = x.shape
        self._raise(self.lib.esm_op_layernorm_e4m3(self.handle, _ptr(x), _ptr(gamma), _ptr(beta), _ptr(y), rows, cols,
                                                   _ptr(scale), _ptr(amax), _stream_ptr(stream)),
                    "esm_op_layernorm_e4m3")
        return y

    def op_gemm_fp8(self, epi: str, A, B, a_scale, b_scale, bias, out, pos_id=None, stream=None):
        M, K = A.shape
        N = B.shape[0]
        self._raise(self.lib.esm_op_gemm_fp8(self.handle, EPILOGUES[epi], _ptr(A), _ptr(B), _ptr(a_scale),
                                             _ptr(b_scale), _ptr(bias), _ptr(out), _ptr(pos_id), M, N, K,
                                             _stream_ptr(stream)), "esm_op_gemm_fp8")
        return out

    def op_attention(self, qkv, cu_seqlens, max_seqlen: int, o, workspace=None, stream=None):
        T = qkv.shape[0]
        B = cu_seqlens.numel() - 1
        if workspace is None:
            workspace = self.workspace(T, B, qkv.device)
        self._raise(self.lib.esm_op_attention(self.handle, _ptr(qkv), _ptr(cu_seqlens), B, T, int(max_seqlen),
                                              _ptr(o), _ptr(workspace), workspace.numel(), _stream_ptr(stream)),
                    "esm_op_attention")
        return o

    def set_layer_precision(self, per_layer):
        """esm_encoder_set_layer_precision: one of "fp32", "bf16", "fp8", "fp4" per layer."""
        arr = (ctypes.c_int * max(1, len(per_layer)))(*[PRECISIONS[p] for p in per_layer])
        self._raise(self.lib.esm_encoder_set_layer_precision(self.handle, arr, len(per_layer)),
                    "esm_encoder_set_layer_precision")

    def lm_head_workspace(self, T: int, device="cuda"):
        import torch
        n = ctypes.c_size_t()
        self._raise(self.lib.esm_encoder_lm_head_workspace_size(self.handle, T, ctypes.byref(n)),
                    "esm_encoder_lm_head_workspace_size")
        return torch.empty(max(int(n.value), 256), dtype=torch.uint8, device=device)

    def lm_head(self, head: "DeviceLmHead", hidden, targets=None, logits=None, token_loss=None, loss_sum=None,
                count=None, workspace=None, stream=None):
        """esm_encoder_lm_head: logits [T, vocab] / per-token masked cross-entropy / its sum and
        the number of scored tokens, into the given device tensors (any may be None)."""
        T = hidden.shape[0]
        if workspace is None:
            workspace = self.lm_head_workspace(T, hidden.device)
        self._raise(self.lib.esm_encoder_lm_head(self.handle, ctypes.byref(head.struct), _ptr(hidden), T, _ptr(targets),
                                                 _ptr(logits), _ptr(token_loss), _ptr(loss_sum), _ptr(count),
                                                 _ptr(workspace), workspace.numel(), _stream_ptr(stream)),
                    "esm_encoder_lm_head")

    # ------------------------------------------------------------------ training
    def train_buffer(self, max_tokens: int, device="cuda"):
        import torch
        n = ctypes.c_size_t()
        self._raise(self.lib.esm_encoder_train_buffer_size(self.handle, max_tokens, ctypes.byref(n)),
                    "esm_encoder_train_buffer_size")
        return torch.empty(int(n.value), dtype=torch.uint8, device=device)

    def forward_train(self, weights: DeviceWeights, token_ids, cu_seqlens, max_seqlen: int, train_buf, workspace,
                      out=None, stream=None):
        """esm_encoder_forward_train: the forward, keeping its activations in train_buf."""
        import torch
        T = token_ids.numel()
        B = cu_seqlens.numel() - 1
        if out is None:
            out = torch.empty(T, self.hidden, dtype=self.out_dtype, device=token_ids.device)
        self._raise(self.lib.esm_encoder_forward_train(self.handle, ctypes.byref(weights.struct), _ptr(token_ids),
                                                       _ptr(cu_seqlens), B, T, int(max_seqlen), _ptr(out),
                                                       _ptr(train_buf), train_buf.numel(), _ptr(workspace),
                                                       workspace.numel(), _stream_ptr(stream)),
                    "esm_encoder_forward_train")
        return out

    def backward(self, weights: DeviceWeights, d_out, grads: "DeviceGrads", train_buf, workspace, stream=None):
        """esm_encoder_backward: parameter gradients of the last forward_train, given dL/d(out)."""
        self._raise(self.lib.esm_encoder_backward(self.handle, ctypes.byref(weights.struct), _ptr(d_out),
                                                  ctypes.byref(grads.struct), _ptr(train_buf), train_buf.numel(),
                                                  _ptr(workspace), workspace.numel(), _stream_ptr(stream)),
                    "esm_encoder_backward")
        return grads

    def op_gemm_dgrad(self, dY, W, out, stream=None):
        import torch
        M, N = dY.shape
        K = W.shape[1]
        self._raise(self.lib.esm_op_gemm_dgrad(self.handle, _ptr(dY), _ptr(W), _ptr(out),
                                               int(out.dtype == torch.bfloat16), M, N, K, _stream_ptr(stream)),
                    "esm_op_gemm_dgrad")
        return out

    def op_gemm_wgrad(self, dY, X, dW, workspace=None, stream=None):
        import torch
        M, N = dY.shape
        K = X.shape[1]
        if workspace is None:
            n = ctypes.c_size_t()
            self._raise(self.lib.esm_op_gemm_wgrad_workspace_size(self.handle, N, K, ctypes.byref(n)),
                        "esm_op_gemm_wgrad_workspace_size")
            workspace = torch.empty(int(n.value), dtype=torch.uint8, device=dY.device)
        self._raise(self.lib.esm_op_gemm_wgrad(self.handle, _ptr(dY), _ptr(X), _ptr(dW), M, N, K, _ptr(workspace),
                                               0 if workspace is None else workspace.numel(), _stream_ptr(stream)),
                    "esm_op_gemm_wgrad")
        return dW

    def op_layernorm_backward(self, x, gamma, dy, dres, dx, dgamma, dbeta, stream=None):
        import torch
        rows, cols = x.shape
        n = ctypes.c_size_t()
        self._raise(self.lib.esm_op_layernorm_backward_workspace_size(self.handle, rows, cols, ctypes.byref(n)),
                    "esm_op_layernorm_backward_workspace_size")
        ws = torch.empty(int(n.value), dtype=torch.uint8, device=x.device)
        self._raise(self.lib.esm_op_layernorm_backward(self.handle, _ptr(x), _ptr(gamma), _ptr(dy), _ptr(dres),
                                                       _ptr(dx), _ptr(dgamma), _ptr(dbeta), rows, cols, _ptr(ws),
                                                       ws.numel(), _stream_ptr(stream)), "esm_op_layernorm_backward")
        return dx, dgamma, dbeta

    def op_attention_train(self, qkv, cu_seqlens, max_seqlen: int, o, lse, workspace=None, stream=None):
        T = qkv.shape[0]
        B = cu_seqlens.numel() - 1
        if workspace is None:
            workspace = self.workspace(T, B, qkv.device)
        self._raise(self.lib.esm_op_attention_train(self.handle, _ptr(qkv), _ptr(cu_seqlens), B, T, int(max_seqlen),
                                                    _ptr(o), _ptr(lse), _ptr(workspace), workspace.numel(),
                                                    _stream_ptr(stream)), "esm_op_attention_train")
        return o, lse

    def op_attention_backward(self, qkv, o, lse, d_o, cu_seqlens, max_seqlen: int, dqkv, workspace=None,
                              stream=None):
        import torch
        T = qkv.shape[0]
        B = cu_seqlens.numel() - 1
        if workspace is None:
            n = ctypes.c_size_t()
            self._raise(self.lib.esm_op_attention_backward_workspace_size(self.handle, T, B, ctypes.byref(n)),
                        "esm_op_attention_backward_workspace_size")
            workspace = torch.empty(int(n.value), dtype=torch.uint8, device=qkv.device)
        self._raise(self.lib.esm_op_attention_backward(self.handle, _ptr(qkv), _ptr(o), _ptr(lse), _ptr(d_o),
                                                       _ptr(cu_seqlens), B, T, int(max_seqlen), _ptr(dqkv),
                                                       _ptr(workspace), workspace.numel(), _stream_ptr(stream)),
                    "esm_op_attention_backward")
        return dqkv

    def lm_head_backward_workspace(self, T: int, device="cuda"):
        import torch
        n = ctypes.c_size_t()
        self._raise(self.lib.esm_encoder_lm_head_backward_workspace_size(self.handle, T, ctypes.byref(n)),
                    "esm_encoder_lm_head_backward_workspace_size")
        return torch.empty(int(n.value), dtype=torch.uint8, device=device)

    def lm_head_backward(self, head: "DeviceLmHead", hidden, targets, d_hidden=None, grads=None, loss_sum=None,
                         count=None, workspace=None, stream=None, loss_count=None):
        """esm_encoder_lm_head_backward: dL/d(hidden) (float32 [T, hidden]) and the head's
        gradients (dict of float32 device tensors shaped like the head's parameters) of the
        mean masked-LM loss.  ``loss_count`` (device int32 scalar): the scored-token count the
        mean divides by, e.g. the global batch's in data-parallel training (None: this call's)."""
        import torch
        T = hidden.shape[0]
        dev = hidden.device
        if d_hidden is None:
            d_hidden = torch.empty(T, self.hidden, dtype=torch.float32, device=dev)
        if grads is None:
            grads = {k: torch.empty(tuple(head.t[k].shape), dtype=torch.float32, device=dev) for k in LM_HEAD_NAMES}
        if workspace is None:
            workspace = self.lm_head_backward_workspace(T, dev)
        gs = EsmLmHeadGrads(*[grads[k].data_ptr() for k in LM_HEAD_NAMES])
        self._raise(self.lib.esm_encoder_lm_head_backward(self.handle, ctypes.byref(head.struct), _ptr(hidden), T,
                                                          _ptr(targets), _ptr(d_hidden), ctypes.byref(gs),
                                                          _ptr(loss_sum), _ptr(count), _ptr(loss_count),
                                                          _ptr(workspace), workspace.numel(), _stream_ptr(stream)),
                    "esm_encoder_lm_head_backward")
        return d_hidden, grads

    def op_quantize_nvfp4(self, x, stream=None):
        """esm_op_quantize_nvfp4 of a contiguous bf16 [rows, cols] CUDA tensor: returns (codes uint8
        [rows, cols/2], scales uint8 [rows * cols / 16] in the tensor-core atom order, amax and
        scale as float32 one-element tensors)."""
        import torch
        rows, cols = x.shape
        codes = torch.empty(rows, cols // 2, dtype=torch.uint8, device=x.device)
        scales = torch.empty(rows * cols // 16, dtype=torch.uint8, device=x.device)
        amax = torch.empty(1, dtype=torch.float32, device=x.device)
        scale = torch.empty(1, dtype=torch.float32, device=x.device)
        self._raise(self.lib.esm_op_quantize_nvfp4(self.handle, _ptr(x), rows, cols, _ptr(codes), _ptr(scales),
                                                   _ptr(amax), _ptr(scale), _stream_ptr(stream)), "esm_op_quantize_nvfp4")
        return codes, scales, amax, scale

    def op_gemm_nvfp4(self, a, b, bias=None, out=None, epi="bias_f32", pos_id=None, stream=None):
        """esm_op_gemm_nvfp4 of two operands returned by op_quantize_nvfp4 (A [M, K], B [N, K]):
        v = (A B^T) / (S_A S_B) + bias, then the epilogue `epi` ("bias_f32": float32 out = v;
        "residual": float32 out += v; "gelu": bf16 out = GELU(v); "qkv_rope": bf16 out = v with
        RoPE at the rows' positions pos_id)."""
        import torch
        (ac, asf, _, asc), (bc, bsf, _, bsc) = a, b
        M, N, K = ac.shape[0], bc.shape[0], 2 * ac.shape[1]
        if out is None:
            dt = torch.float32 if epi in ("bias_f32", "residual") else torch.bfloat16
            out = torch.zeros(M, N, dtype=dt, device=ac.device)
        self._raise(self.lib.esm_op_gemm_nvfp4(self.handle, EPILOGUES[epi], _ptr(ac), _ptr(asf), _ptr(asc), _ptr(bc),
                                               _ptr(bsf), _ptr(bsc), _ptr(bias), _ptr(pos_id), _ptr(out), M, N, K,
                                               _stream_ptr(stream)), "esm_op_gemm_nvfp4")
        return out

    def set_profiling(self, enable: bool):
        self._raise(self.lib.esm_encoder_set_profiling(self.handle, int(enable)), "esm_encoder_set_profiling")

    def get_profile(self, reset: bool = True) -> Dict:
        """{class: {"ms": summed device ms, "launches": n}} plus "total_launches"."""
        p = EsmProfile()
        self._raise(self.lib.esm_encoder_get_profile(self.handle, ctypes.byref(p), int(reset)),
                    "esm_encoder_get_profile")
        out = {name: {"ms": p.ms[i], "launches": int(p.launches[i])} for i, name in enumerate(PROFILE_CLASSES)}
        out["total_launches"] = int(p.total_launches)
        return out

    def fp8_state_size(self) -> int:
        return self.num_layers * 8 * (1 + self.amax_history_len)

    def get_fp8_state(self) -> np.ndarray:
        buf = np.zeros(self.fp8_state_size(), dtype=np.float32)
        self._raise(self.lib.esm_encoder_get_fp8_state(self.handle, buf.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                                       buf.size), "esm_encoder_get_fp8_state")
        return buf

    def set_fp8_state(self, buf: np.ndarray):
        buf = np.ascontiguousarray(buf, dtype=np.float32)
        self._raise(self.lib.esm_encoder_set_fp8_state(self.handle, buf.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                                       buf.size), "esm_encoder_set_fp8_state")

    def fp4_scales(self) -> np.ndarray:
        """[num_layers, 8] NVFP4 tensor scales of the last forward's FP4 layers (tensor order
        x_qkv, w_qkv, x_o, w_o, x_1, w_1, x_2, w_2; zero for other layers)."""
        buf = np.zeros(self.num_layers * 8, dtype=np.float32)
        self._raise(self.lib.esm_encoder_get_fp4_scales(self.handle, buf.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                                        buf.size), "esm_encoder_get_fp4_scales")
        return buf.reshape(self.num_layers, 8)

    def fp8_scales(self, buf: Optional[np.ndarray] = None) -> np.ndarray:
        """[num_layers, 8] scales from a state buffer (tensor order x_qkv, w_qkv, x_o, w_o, x_1, w_1, x_2, w_2)."""
        buf = self.get_fp8_state() if buf is None else buf
        return buf[:self.num_layers * 8].reshape(self.num_layers, 8)

    def fp8_history(self, buf: Optional[np.ndarray] = None) -> np.ndarray:
        buf = self.get_fp8_state() if buf is None else buf
        return buf[self.num_layers * 8:].reshape(self.num_layers, 8, self.amax_history_len)


def op_attention_noalloc(qkv, cu_seqlens, max_seqlen: int, hidden: int, heads: int, o, status=None,
                         stream=None) -> int:
    """esm_op_attention_noalloc: attention with no handle, no workspace and no allocation.

    qkv: contiguous CUDA bf16 [T, 3*hidden]; o: contiguous CUDA bf16 [T, hidden];
    cu_seqlens: contiguous int32 [B + 1] on the same device; status: optional int32 device
    tensor of one element that receives the call's device-side outcome (ESM_OK,
    ESM_ERR_BAD_CU_SEQLENS or ESM_ERR_TIMEOUT).  Raises ValueError on tensors the C side
    cannot check (wrong dtype, device, layout or shape); returns the call's status code."""
    import torch

    def need(ok, what):
        if not ok:
            raise ValueError(f"op_attention_noalloc: {what}")

    for name, t in (("qkv", qkv), ("o", o), ("cu_seqlens", cu_seqlens)):
        need(isinstance(t, torch.Tensor) and t.is_cuda, f"{name} must be a CUDA tensor")
        need(t.is_contiguous(), f"{name} must be contiguous")
        need(t.device == qkv.device, f"{name} must be on {qkv.device}")
    need(qkv.dtype == torch.bfloat16 and o.dtype == torch.bfloat16, "qkv and o must be bfloat16")
    need(cu_seqlens.dtype == torch.int32 and cu_seqlens.dim() == 1 and cu_seqlens.numel() >= 2,
         "cu_seqlens must be a 1-D int32 tensor of at least two offsets")
    need(qkv.dim() == 2 and qkv.shape[1] == 3 * hidden, f"qkv must be [T, {3 * hidden}]")
    need(o.dim() == 2 and tuple(o.shape) == (qkv.shape[0], hidden), f"o must be [{qkv.shape[0]}, {hidden}]")
    if status is not None:
        need(isinstance(status, torch.Tensor) and status.device == qkv.device and status.dtype == torch.int32
             and status.numel() >= 1, "status must be an int32 tensor on the device of qkv")
    lib = load_library()
    return lib.esm_op_attention_noalloc(_ptr(qkv), _ptr(cu_seqlens), cu_seqlens.numel() - 1, qkv.shape[0],
                                        int(max_seqlen), hidden, heads, _ptr(o), _ptr(status), _stream_ptr(stream))


def packed_inputs(tokens: np.ndarray, lengths: Sequence[int], device="cuda"):
    """Device token ids and cu_seqlens (int32) for a packed batch."""
    import torch
    from .synth import cu_seqlens_from_lengths
    tok = torch.from_numpy(np.ascontiguousarray(tokens, dtype=np.int32)).to(device)
    cu = torch.from_numpy(cu_seqlens_from_lengths(lengths)).to(device)
    return tok, cu
