"""GPU parity of the on-device FP8 / NVFP4 encoders (tkg_quantize_*) with the
oracle's encoders (oracle/quantize.c): codes, block scales and tensor scales
must be bit-identical, since every decision is the same fp32 operation on both
sides.  Shapes cover a single block, ragged row counts, more than one grid
stride, and the full sizes of the FP8 (8192 x 8192) and NVFP4 (16384 x 16384)
workloads; inputs are the seeded fp32 draws that also feed those workloads'
encoders, plus all-zero, constant and extreme-range tensors.  The encoded
operands then go through the GEMM and must match the oracle GEMM of the
oracle-encoded operands.
"""
import numpy as np
import pytest

from tiled_tensor_core_gb300 import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def tkg():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from tiled_tensor_core_gb300 import tkg as mod
    return mod


def gpu_fp8(tkg, x):
    xd = torch.from_numpy(x).cuda()
    q = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
    s = torch.empty(1, dtype=torch.float32, device="cuda")
    tkg.tkg_quantize_fp8(x.shape[0], x.shape[1], xd, q, s)
    assert tkg.tkg_check_status() == tkg.TKG_OK
    return q.cpu().numpy(), np.float32(s.item())


def gpu_nvfp4(tkg, x):
    rows, cols = x.shape
    xd = torch.from_numpy(x).cuda()
    q = torch.empty((rows, cols // 2), dtype=torch.uint8, device="cuda")
    sf = torch.empty((rows, cols // 16), dtype=torch.uint8, device="cuda")
    g = torch.empty(1, dtype=torch.float32, device="cuda")
    tkg.tkg_quantize_nvfp4(rows, cols, xd, q, sf, g)
    assert tkg.tkg_check_status() == tkg.TKG_OK
    return q.cpu().numpy(), sf.cpu().numpy(), np.float32(g.item())


SHAPES = [(1, 16), (3, 48), (64, 256), (1000, 1024), (4097, 528)]


def special_inputs():
    yield "zeros", np.zeros((5, 64), np.float32)
    yield "constant", np.full((7, 32), -3.25, np.float32)
    x = synth.draw_fp32(77, 33, 96, "normal")
    x[0, :16] = 0.0
    x[1, 16:32] *= np.float32(1e-8)       # block scale underflows to 0
    x[2, :] *= np.float32(1e30)           # tensor amax far above the rest
    yield "mixed_range", x
    yield "tiny", (synth.draw_fp32(78, 9, 48, "normal") * np.float32(1e-30)).astype(np.float32)


@pytest.mark.parametrize("shape", SHAPES)
def test_fp8_encoder_bit_exact(tkg, oracle_mod, shape):
    x = synth.draw_fp32(100 + shape[0], *shape, "normal")
    q, s = gpu_fp8(tkg, x)
    q_ref, s_ref = oracle_mod.quantize_fp8(x)
    assert s == s_ref
    assert np.array_equal(q, q_ref)


@pytest.mark.parametrize("shape", SHAPES)
def test_nvfp4_encoder_bit_exact(tkg, oracle_mod, shape):
    x = synth.draw_fp32(200 + shape[0], *shape, "normal")
    q, sf, g = gpu_nvfp4(tkg, x)
    q_ref, sf_ref, g_ref = oracle_mod.quantize_nvfp4(x)
    assert g == g_ref
    assert np.array_equal(sf, sf_ref)
    assert np.array_equal(q, q_ref)


@pytest.mark.parametrize("name,x", list(special_inputs()))
def test_encoders_on_degenerate_inputs(tkg, oracle_mod, name, x):
    q, s = gpu_fp8(tkg, x)
    q_ref, s_ref = oracle_mod.quantize_fp8(x)
    assert s == s_ref and np.array_equal(q, q_ref)
    q, sf, g = gpu_nvfp4(tkg, x)
    q_ref, sf_ref, g_ref = oracle_mod.quantize_nvfp4(x)
    assert g == g_ref and np.array_equal(sf, sf_ref) and np.array_equal(q, q_ref)


def test_fp8_encoder_full_workload_size(tkg, oracle_mod):
    x = synth.draw_fp32(1004, 8192, 8192, "normal")
    q, s = gpu_fp8(tkg, x)
    q_ref, s_ref = oracle_mod.quantize_fp8(x)
    assert s == s_ref
    assert np.array_equal(q, q_ref)


def test_nvfp4_encoder_full_workload_size(tkg, oracle_mod):
    x = synth.draw_fp32(1005, 16384, 16384, "normal")
    q, sf, g = gpu_nvfp4(tkg, x)
    q_ref, sf_ref, g_ref = oracle_mod.quantize_nvfp4(x)
    assert g == g_ref
    assert np.array_equal(sf, sf_ref)
    assert np.array_equal(q, q_ref)


@pytest.mark.parametrize("kind", ["fp8", "nvfp4"])
def test_encoded_operands_through_the_gemm(tkg, oracle_mod, kind):
    M, N, K = 384, 520, 512
    xa = synth.draw_fp32(31, M, K, "normal")
    xb = synth.draw_fp32(32, N, K, "normal")
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    if kind == "fp8":
        (qa, sa), (qb, sb) = gpu_fp8(tkg, xa), gpu_fp8(tkg, xb)
        ops = synth.Operands("fp8", M, N, K, qa, qb, None, None, sa, sb)
    else:
        (qa, fa, ga), (qb, fb, gb) = gpu_nvfp4(tkg, xa), gpu_nvfp4(tkg, xb)
        ops = synth.Operands("nvfp4", M, N, K, qa, qb, fa, fb, ga, gb)
    from tiled_tensor_core_gb300.device import DeviceGemm
    g = DeviceGemm(ops, "cuda")
    g.run()
    assert tkg.tkg_check_status() == tkg.TKG_OK
    acc, c_ref = oracle_mod.gemm(ops)
    from gpu_util import check_against_oracle
    check_against_oracle(kind, g.c_bits(), acc, c_ref, ops.scale_a, ops.scale_b)
