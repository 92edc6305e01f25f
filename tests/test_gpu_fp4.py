"""NVFP4 (block-scaled E2M1) operands and GEMM on the tensor cores against the FP4 oracle.

* Quantisation: the tensor scale S, the E4M3 block scales and the E2M1 codes equal the
  oracle's (float64) except where fp32 and float64 straddle a rounding midpoint, then the
  two results are neighbouring codes.
* GEMM exactness: the product of the GPU's own quantised operands, decoded in numpy from their
  bytes (codes, the atom-ordered scales) and multiplied in float64, agrees with the tensor-core
  result up to fp32 accumulation: this pins the block-scaled MMA, the scale-factor layout in
  tensor memory and the epilogue's 1 / (S_A S_B).
* End to end: the GEMM of bf16 inputs quantised on the GPU against the oracle's fake-quantised
  product (nvfp4_fake_quant of both operands)."""
import numpy as np
import pytest

from oracle import fp4 as F4
from tests._util import e4m3_table, ensure_built, rel_l2
from transformer_esm_layer_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


@pytest.fixture(scope="module")
def enc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()
    from transformer_esm_layer_gb300.binding import EsmEncoder
    return EsmEncoder(1, 256, 4, 512, precision="bf16")


def _bf16(a):
    return synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(np.asarray(a, np.float32))).astype(np.float64)


def _decode(codes, scales, S, rows, K):
    """float64 values of a GPU NVFP4 operand from its bytes: E2M1 nibbles times the atom-ordered
    E4M3 block scales, divided by the tensor scale."""
    c = codes.astype(np.int64)
    nib = np.stack([c & 0xF, c >> 4], axis=-1).reshape(rows, K)       # value k: low nibble if k even
    q = np.where(nib & 8, -1.0, 1.0) * E2M1[nib & 7]
    r = np.arange(rows)[:, None]
    k16 = np.arange(K // 16)[None, :]
    off = ((r // 128) * (K // 64) + k16 // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (k16 % 4)
    sb = e4m3_table()[scales[off]]
    return (q.reshape(rows, K // 16, 16) * sb[..., None]).reshape(rows, K) / S, sb


def _case(rng, rows, K):
    x = rng.standard_normal((rows, K)) * np.exp(rng.standard_normal((rows, 1)))  # rows of varied magnitude
    x[0, :16] = 0.0                                                               # one all-zero block
    x[1, 16:32] *= 1e-3                                                           # one tiny block
    return _bf16(x)


def _quant(enc, x):
    return enc.op_quantize_nvfp4(torch.from_numpy(x.astype(np.float32)).cuda().to(torch.bfloat16))


def test_nvfp4_quantize_matches_oracle(enc):
    rng = np.random.default_rng(50)
    rows, K = 256, 768
    x = _case(rng, rows, K)
    codes, scales, amax, scale = _quant(enc, x)
    torch.cuda.synchronize()
    deq_o, sb_o, S_o = F4.nvfp4_fake_quant(x)
    S = float(scale.item())
    assert float(amax.item()) == np.abs(x).max()
    assert abs(S / S_o - 1) < 1e-6
    deq, sb = _decode(codes.cpu().numpy(), scales.cpu().numpy(), S, rows, K)
    # block scales: equal except at an E4M3 rounding midpoint (then neighbours)
    diff = sb != sb_o
    assert diff.mean() < 2e-3
    assert np.all(np.abs(sb[diff] - sb_o[diff]) <= sb_o[diff] / 8 + 2.0 ** -9)
    # values: equal except where a midpoint decides (then one E2M1 step apart, relative to
    # the block scale)
    same_scale = np.repeat(~diff, 16, axis=1)
    vd = (deq != deq_o) & same_scale
    assert vd.mean() < 2e-3
    step = np.repeat(sb_o, 16, axis=1) / S_o * 2.0
    assert np.all(np.abs(deq[vd] - deq_o[vd]) <= step[vd] + 1e-12)
    assert np.all(deq[0, :16] == 0.0)


@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (256, 384, 1280), (384, 256, 512)])
def test_nvfp4_gemm_exact_on_its_operands(enc, M, N, K):
    """fp32 accumulation of E2M1 x E2M1 products scaled by E4M3 x E4M3 block scales: exact
    products, about K/64 rounded partial sums; bound 2e-5 relative L2 (as for the E4M3 GEMM)."""
    rng = np.random.default_rng(M + N + K)
    A, B = _case(rng, M, K), _case(rng, N, K) * 0.05
    bias = _bf16(rng.standard_normal(N))
    qa, qb = _quant(enc, A), _quant(enc, B)
    out = enc.op_gemm_nvfp4(qa, qb, bias=torch.from_numpy(bias.astype(np.float32)).cuda().to(torch.bfloat16))
    assert enc.check_status() == 0
    da, _ = _decode(qa[0].cpu().numpy(), qa[1].cpu().numpy(), float(qa[3].item()), M, K)
    db, _ = _decode(qb[0].cpu().numpy(), qb[1].cpu().numpy(), float(qb[3].item()), N, K)
    ref = da @ db.T + bias
    got = out.to(torch.float64).cpu().numpy()
    assert rel_l2(got, ref) < 2e-5, rel_l2(got, ref)


def test_nvfp4_gemm_matches_oracle_fake_quant(enc, margin):
    rng = np.random.default_rng(51)
    M, N, K = 256, 512, 1280
    A, B = _case(rng, M, K), _case(rng, N, K) * 0.02
    out = enc.op_gemm_nvfp4(_quant(enc, A), _quant(enc, B))
    assert enc.check_status() == 0
    ref = F4.nvfp4_fake_quant(A)[0] @ F4.nvfp4_fake_quant(B)[0].T
    e = rel_l2(out.to(torch.float64).cpu().numpy(), ref)
    margin("NVFP4 GEMM vs the oracle's fake-quantised product", e, 5e-3)
    assert e < 5e-3
    # and the quantisation error itself, against the unquantised product (for the record)
    margin("NVFP4 GEMM vs the exact product (record)", rel_l2(out.to(torch.float64).cpu().numpy(), A @ B.T), 2e-1)


def test_nvfp4_argument_errors(enc):
    from transformer_esm_layer_gb300.binding import EsmError
    x = torch.zeros(100, 256, dtype=torch.bfloat16, device="cuda")   # rows not a multiple of 128
    with pytest.raises(EsmError, match="INVALID_ARG"):
        enc.op_quantize_nvfp4(x)
    y = torch.zeros(128, 200, dtype=torch.bfloat16, device="cuda")   # cols not a multiple of 256
    with pytest.raises(EsmError, match="INVALID_ARG"):
        enc.op_quantize_nvfp4(y)
