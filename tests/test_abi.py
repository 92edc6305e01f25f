"""The C-ABI library builds, loads and exports every function the header declares.
No compute call is made (no GPU needed)."""
import ctypes

import pytest

from tests._util import ensure_built, header_functions
from transformer_esm_layer_gb300 import binding


@pytest.fixture(scope="module")
def lib():
    ensure_built()
    return binding.load_library()


def test_header_declares_the_boundary():
    names = header_functions()
    assert set(names) == set(binding.EXPORTS), names
    for n in ("esm_encoder_create", "esm_encoder_forward", "esm_encoder_forward_padded", "esm_encoder_destroy"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    for code in range(8):
        s = lib.esm_status_string(code)
        assert isinstance(s, bytes) and len(s) > 0
    assert lib.esm_status_string(99) == b"unknown status"


def test_null_arguments_are_rejected_without_a_device(lib):
    n = ctypes.c_size_t()
    assert lib.esm_encoder_workspace_size(None, 10, 1, ctypes.byref(n)) == 1  # ESM_ERR_INVALID_ARG
    assert lib.esm_encoder_create(None, None) == 1
    assert lib.esm_encoder_forward(None, None, None, None, 0, 0, 0, None, None, 0, None) == 1
    assert lib.esm_encoder_check(None, None) == 1
    assert lib.esm_encoder_lm_head_workspace_size(None, 10, ctypes.byref(n)) == 1
    assert lib.esm_encoder_set_layer_precision(None, None, 0) == 1
    assert lib.esm_encoder_lm_head(None, None, None, 0, None, None, None, None, None, None, 0, None) == 1
    assert lib.esm_encoder_train_buffer_size(None, 10, ctypes.byref(n)) == 1
    assert lib.esm_encoder_forward_train(None, None, None, None, 1, 1, 1, None, None, 0, None, 0, None) == 1
    assert lib.esm_encoder_backward(None, None, None, None, None, 0, None, 0, None) == 1
    assert lib.esm_op_gemm_dgrad(None, None, None, None, 0, 1, 64, 256, None) == 1
    assert lib.esm_op_gemm_wgrad_workspace_size(None, 256, 256, ctypes.byref(n)) == 1
    assert lib.esm_op_gemm_wgrad(None, None, None, None, 1, 256, 256, None, 0, None) == 1
    assert lib.esm_op_layernorm_backward_workspace_size(None, 4, 256, ctypes.byref(n)) == 1
    assert lib.esm_op_layernorm_backward(None, None, None, None, None, None, None, None, 4, 256, None, 0, None) == 1
    assert lib.esm_op_attention_train(None, None, None, 1, 1, 1, None, None, None, 0, None) == 1
    assert lib.esm_op_attention_backward_workspace_size(None, 4, 1, ctypes.byref(n)) == 1
    assert lib.esm_op_attention_backward(None, None, None, None, None, None, 1, 1, 1, None, None, 0, None) == 1
    assert lib.esm_encoder_lm_head_backward_workspace_size(None, 4, ctypes.byref(n)) == 1
    assert lib.esm_encoder_lm_head_backward(None, None, None, 1, None, None, None, None, None, None, None, 0, None) == 1
    lib.esm_encoder_destroy(None)


def test_create_without_sm103_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available() and torch.cuda.get_device_capability() == (10, 3):
        pytest.skip("a GB300 is present")
    cfg = binding.EsmConfig(2, 64, 4, 256, 33, 1026, 1e-5, 10000.0, 1.0, 1, 0, 16)
    h = ctypes.c_void_p()
    st = lib.esm_encoder_create(ctypes.byref(cfg), ctypes.byref(h))
    assert st in (2, 6)  # unsupported device, or no CUDA device at all
    assert not h.value
