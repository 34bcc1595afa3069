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


def _sf_words(sf_rows, quarter_lanes):
    """TMEM contents [128 lanes][8 columns] holding the 4 scales of each of up
    to 256 rows: row i at column i // 32, lane (i % 32) + 32 q for every
    quarter q (B's rule, and a superset of A's: lane i itself)."""
    words = np.zeros((128, 8), dtype=np.uint32)
    for i in range(sf_rows.shape[0]):
        w = int(sf_rows[i, 0]) | (int(sf_rows[i, 1]) << 8) | (int(sf_rows[i, 2]) << 16) | (int(sf_rows[i, 3]) << 24)
        for q in quarter_lanes:
            words[(i % 32) + 32 * q, i // 32] = w
    return words


@pytest.mark.parametrize("n", [128, 192, 256])
def test_single_tile_nvfp4_mma_scale_layout(tkg, oracle_mod, n):
    # one block-scaled MMA (K = 64): 4 scales per row, slice j in byte j;
    # A's row m read at lane m, column m // 32; B's row n at lane n % 32, column n // 32
    ops = synth.small_int_operands("nvfp4", 128, n, 64, seed=n)
    a_tile = np.zeros((128, 128), np.uint8)
    b_tile = np.zeros((n, 128), np.uint8)
    a_tile[:, :32] = ops.a
    b_tile[:, :32] = ops.b
    sfa = _sf_words(ops.sfa, [0, 1, 2, 3])
    sfb = _sf_words(ops.sfb, [0, 1, 2, 3])
    d_a = torch.from_numpy(a_tile).cuda()
    d_b = torch.from_numpy(b_tile).cuda()
    d_sfa = torch.from_numpy(sfa.view(np.int32)).cuda()
    d_sfb = torch.from_numpy(sfb.view(np.int32)).cuda()
    d_out = torch.full((128, n), float("nan"), dtype=torch.float32, device="cuda")
    assert tkg.tkg_debug_mma_probe(2, n, 1, d_a, d_b, d_sfa, d_sfb, [0, 0], d_out) == tkg.TKG_OK
    acc, _ = oracle_mod.gemm_nvfp4(ops.a, ops.b, ops.sfa, ops.sfb, 1.0, 1.0)
    assert np.array_equal(d_out.cpu().numpy(), acc)


def test_single_tile_nvfp4_n192_b_scales_at_an_offset(tkg, oracle_mod):
    # N = 192 reads B's scales from six columns starting at the address the MMA is given: placed
    # two columns in, the result shows the scale address, not column 0, decides where they are read
    n = 192
    ops = synth.small_int_operands("nvfp4", 128, n, 64, seed=1920)
    a_tile = np.zeros((128, 128), np.uint8)
    b_tile = np.zeros((n, 128), np.uint8)
    a_tile[:, :32] = ops.a
    b_tile[:, :32] = ops.b
    sfa = _sf_words(ops.sfa, [0, 1, 2, 3])
    sfb = np.zeros((128, 8), dtype=np.uint32)
    sfb[:, 2:] = _sf_words(ops.sfb, [0, 1, 2, 3])[:, :6]
    d_a = torch.from_numpy(a_tile).cuda()
    d_b = torch.from_numpy(b_tile).cuda()
    d_sfa = torch.from_numpy(sfa.view(np.int32)).cuda()
    d_sfb = torch.from_numpy(sfb.view(np.int32)).cuda()
    d_out = torch.full((128, n), float("nan"), dtype=torch.float32, device="cuda")
    assert tkg.tkg_debug_mma_probe(2, n, 1, d_a, d_b, d_sfa, d_sfb, [0, 2], d_out) == tkg.TKG_OK
    acc, _ = oracle_mod.gemm_nvfp4(ops.a, ops.b, ops.sfa, ops.sfb, 1.0, 1.0)
    assert np.array_equal(d_out.cpu().numpy(), acc)
