"""The attention entry point that allocates nothing (for callers that cannot call
cudaMalloc: allocators that own the whole device, plugin hosts that only hand out their
input and output buffers, runtimes that forbid allocation after start-up).

It runs the same tcgen05 attention kernel as the workspace-based entry point, so on two
calls in a row with different batches (the shared scratch array keeps the previous call's
contents) its output equals that entry point's bit for bit, and it matches the float64
oracle's attention within the bf16 tolerance.  Malformed cu_seqlens are reported through
the optional status output.  This file is collected last so that a run stopping at the
first failure has already run every other test; it also passes alone in a fresh process."""
import numpy as np
import pytest

from oracle import esm_oracle as O
from tests._util import ensure_built, rel_l2
from transformer_esm_layer_gb300 import synth

torch = pytest.importorskip("torch")


def _bf16_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda", torch.bfloat16)


def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


@pytest.mark.gpu
def test_noalloc_attention_matches_workspace_entry_point_and_oracle_twice(margin):
    _needs_gpu()
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
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        assert op_attention_noalloc(qkv, cu, max(lengths), hidden, heads, got, status=status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(got, ref), call                 # the same kernel on the same inputs
        g = got.to(torch.float64).cpu().numpy()
        q = qkv.to(torch.float64).cpu().numpy()
        c = O.cu_seqlens(lengths)
        worst = 0.0
        for i in range(len(lengths)):
            s = slice(int(c[i]), int(c[i + 1]))
            L = int(c[i + 1] - c[i])
            o = O.attention(q[s, :hidden].reshape(L, heads, 64), q[s, hidden:2 * hidden].reshape(L, heads, 64),
                            q[s, 2 * hidden:].reshape(L, heads, 64))
            worst = max(worst, rel_l2(g[s], o.reshape(L, hidden)))
        margin(f"no-allocation attention vs the oracle, call {call}", worst, 1e-2)
        assert worst < 1e-2, call


@pytest.mark.gpu
def test_noalloc_reports_malformed_cu_seqlens_and_rejects_sizes_beyond_its_maximum():
    _needs_gpu()
    from transformer_esm_layer_gb300.binding import load_library, op_attention_noalloc
    hidden, heads = 128, 2
    T = 40
    qkv = _bf16_dev(np.random.default_rng(5).standard_normal((T, 3 * hidden)))
    out = torch.empty(T, hidden, dtype=torch.bfloat16, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    bad = torch.tensor([0, 30, 20, 40], dtype=torch.int32, device="cuda")   # decreasing offsets
    assert op_attention_noalloc(qkv, bad, 30, hidden, heads, out, status=status) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 3                                         # ESM_ERR_BAD_CU_SEQLENS
    good = torch.tensor([0, 30, 40], dtype=torch.int32, device="cuda")
    assert op_attention_noalloc(qkv, good, 30, hidden, heads, out, status=status) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0                                         # the next call starts clear
    lib = load_library()
    dummy = torch.empty(16, dtype=torch.int32, device="cuda")
    p = dummy.data_ptr()
    assert lib.esm_op_attention_noalloc(p, p, 4097, 100, 10, 1280, 20, p, None, None) == 1   # too many sequences
    assert lib.esm_op_attention_noalloc(p, p, 2, 65537, 10, 1280, 20, p, None, None) == 1    # too many tokens
    assert lib.esm_op_attention_noalloc(p, p, 2, 100, 10, 1280, 19, p, None, None) == 2      # head_dim != 64
    with pytest.raises(ValueError):
        op_attention_noalloc(qkv.float(), good, 30, hidden, heads, out)                       # not bf16
    with pytest.raises(ValueError):
        op_attention_noalloc(qkv[:, :hidden], good, 30, hidden, heads, out)                   # wrong shape
    with pytest.raises(ValueError):
        op_attention_noalloc(qkv, good.long(), 30, hidden, heads, out)                        # not int32


def test_noalloc_binding_rejects_host_tensors_before_any_call():
    """The wrapper checks device, dtype, layout and shapes before it reaches the library (the
    C side cannot check what a raw pointer points to)."""
    from transformer_esm_layer_gb300.binding import op_attention_noalloc
    qkv = torch.zeros(8, 3 * 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        op_attention_noalloc(qkv, torch.tensor([0, 8], dtype=torch.int32), 8, 128, 2,
                             torch.zeros(8, 128, dtype=torch.bfloat16))
