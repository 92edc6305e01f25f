"""The attention entry point that allocates nothing (for callers that cannot call
cudaMalloc: allocators that own the whole device, plugin hosts that only hand out their
input and output buffers, runtimes that forbid allocation after start-up).

Its output must match the regular workspace-based entry point, on two calls in a row
with different batches (the shared scratch array keeps the previous call's contents).
This file is collected last so that a run stopping at the first failure has already run
every other test; it also passes alone in a fresh process."""
import numpy as np
import pytest

from tests._util import ensure_built, rel_l2
from transformer_esm_layer_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _bf16_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda", torch.bfloat16)


def test_noalloc_attention_matches_workspace_entry_point_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()
    from transformer_esm_layer_gb300.binding import EsmEncoder, op_attention_noalloc
    hidden, heads = 1280, 20
    enc = EsmEncoder(1, hidden, heads, 4 * hidden, precision="bf16")
    cases = [[300, 1, 64, 129, 1024, 77], [5, 900, 33]]
    for call, lengths in enumerate(cases):
        rng = np.random.default_rng(100 + call)
        T = sum(lengths)
        qkv = _bf16_dev(rng.standard_normal((T, 3 * hidden)) * 1.5)
        cu = torch.from_numpy(synth.cu_seqlens_from_lengths(lengths)).cuda()
        ref = torch.empty(T, hidden, dtype=torch.bfloat16, device="cuda")
        enc.op_attention(qkv, cu, max(lengths), ref)
        got = torch.full((T, hidden), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = op_attention_noalloc(qkv, cu, max(lengths), hidden, heads, got)
        assert st == 0
        torch.cuda.synchronize()
        g = got.to(torch.float64).cpu().numpy()
        r = ref.to(torch.float64).cpu().numpy()
        assert np.isfinite(g).all()
        assert rel_l2(g, r) < 1e-2, call


def test_noalloc_rejects_sizes_beyond_its_maximum():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()
    from transformer_esm_layer_gb300.binding import load_library
    lib = load_library()
    dummy = torch.empty(16, dtype=torch.int32, device="cuda")
    p = dummy.data_ptr()
    assert lib.esm_op_attention_noalloc(p, p, 4097, 100, 10, 1280, 20, p, None) == 1   # too many sequences
    assert lib.esm_op_attention_noalloc(p, p, 2, 65537, 10, 1280, 20, p, None) == 1    # too many tokens
    assert lib.esm_op_attention_noalloc(p, p, 2, 100, 10, 1280, 19, p, None) == 2      # head_dim != 64
