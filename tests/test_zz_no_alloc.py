"""tkg_gemm_nvfp4_noalloc: the NVFP4 GEMM for callers that cannot allocate
device memory during a call (its scale re-layout scratch is a fixed array in
the library instead of a pool allocation).  Its output must match the regular
tkg_gemm_nvfp4 within the NVFP4 tolerance, on consecutive calls that reuse the
shared array; problems whose scratch would not fit are rejected up front.

Kept in the last-collected file so that a stop-at-first-failure run has
already run every other test."""
import numpy as np
import pytest

from tiled_tensor_core_gb300 import synth

from gpu_util import SCALED_REL_FRO, bf16_bits_to_f64, rel_fro

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def tkg():
    from tiled_tensor_core_gb300 import build
    build.build()
    from tiled_tensor_core_gb300 import tkg as mod
    return mod


def test_rejects_problems_beyond_the_fixed_scratch(tkg):
    A = B = C = 1 << 20  # fake aligned addresses: the size check fails first, nothing is dereferenced
    s = tkg.tkg_scales(1 << 12, 1 << 12, 1 << 14, 1 << 14)
    # 32768^2 x 32768 needs (256 + 256) * 128 * 2 KiB = 128 MiB of scratch
    assert tkg.lib.tkg_gemm_nvfp4_noalloc(32768, 32768, 32768, A, B, C, s, None) == tkg.TKG_ERR_INVALID_ARG
    assert tkg.lib.tkg_gemm_nvfp4_noalloc(8, 8, 48, A, B, C, s, None) == tkg.TKG_ERR_INVALID_ARG


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(1000, 1000, 1024), (520, 300, 288), (4096, 4096, 4096)])
def test_noalloc_matches_regular_entry_point_twice(tkg, shape):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from tiled_tensor_core_gb300.device import DeviceGemm
    M, N, K = shape
    ops = synth.make_operands("nvfp4", M, N, K, "normal", 91 + M, 92 + N)
    g = DeviceGemm(ops, "cuda")
    g.run()
    assert tkg.tkg_check_status() == tkg.TKG_OK
    ref = bf16_bits_to_f64(g.c_bits())
    for call in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        tkg.tkg_gemm_nvfp4_noalloc(M, N, K, g.a, g.b, out, g.scales())
        assert tkg.tkg_check_status() == tkg.TKG_OK
        got = bf16_bits_to_f64(out.view(torch.int16).cpu().numpy().view(np.uint16))
        assert np.isfinite(got).all(), f"call {call}"
        assert rel_fro(got, ref) <= SCALED_REL_FRO, f"call {call}"
