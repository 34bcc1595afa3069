"""GPU checks of the GEMM's building blocks in isolation:
 * the TMA copy engine's 32/64/128-byte swizzles equal the pages' XOR formula
   (the layout the epilogue writes by hand and the MMA descriptors assume);
 * one tensor-core MMA on one tile, through the same shared-memory and
   instruction descriptors the GEMM kernels use, equals the oracle exactly on
   small-integer operands (bf16 and e4m3)."""
import numpy as np
import pytest

from oracle import swizzle as sw
from tiled_tensor_core_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def tkg():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from tiled_tensor_core_gb300 import tkg as mod
    return mod


@pytest.mark.parametrize("s", [32, 64, 128])
def test_tma_swizzle_matches_formula(tkg, oracle_mod, s):
    rng = np.random.default_rng(s)
    src = rng.integers(0, 256, size=(64, s), dtype=np.uint8)
    d_src = torch.from_numpy(src).cuda()
    d_dst = torch.zeros(64 * s, dtype=torch.uint8, device="cuda")
    assert tkg.tkg_debug_tma_swizzle_probe(s, d_src, d_dst) == tkg.TKG_OK
    img = d_dst.cpu().numpy()
    expect = np.zeros(64 * s, dtype=np.uint8)
    for r in range(64):
        for c in range(s):
            expect[sw.swizzle(r * s + c, s)] = src[r, c]
    assert np.array_equal(img, expect)


def _probe(tkg, kind, n, ksteps, a_bytes, b_bytes):
    d_a = torch.from_numpy(np.ascontiguousarray(a_bytes)).cuda()
    d_b = torch.from_numpy(np.ascontiguousarray(b_bytes)).cuda()
    d_out = torch.full((128, n), float("nan"), dtype=torch.float32, device="cuda")
    assert tkg.tkg_debug_mma_probe(kind, n, ksteps, d_a, d_b, d_out=d_out) == tkg.TKG_OK
    return d_out.cpu().numpy()


@pytest.mark.parametrize("n", [64, 128, 256])
@pytest.mark.parametrize("ksteps", [1, 4])
def test_single_tile_bf16_mma(tkg, oracle_mod, n, ksteps):
    ops = synth.small_int_operands("bf16", 128, n, 64, seed=n + ksteps)
    out = _probe(tkg, 0, n, ksteps, ops.a.view(np.uint8).reshape(128, 128), ops.b.view(np.uint8).reshape(n, 128))
    kk = 16 * ksteps
    acc, _ = oracle_mod.gemm_bf16(ops.a[:, :kk], ops.b[:, :kk])
    assert np.array_equal(out, acc)


@pytest.mark.parametrize("n", [128, 256])
@pytest.mark.parametrize("ksteps", [1, 4])
def test_single_tile_fp8_mma(tkg, oracle_mod, n, ksteps):
    ops = synth.small_int_operands("fp8", 128, n, 128, seed=7 * n + ksteps)
    out = _probe(tkg, 1, n, ksteps, ops.a, ops.b)
    kk = 32 * ksteps
    acc, _ = oracle_mod.gemm_fp8(ops.a[:, :kk], ops.b[:, :kk], 1.0, 1.0)
    assert np.array_equal(out, acc)
