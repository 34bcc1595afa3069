"""tkg_gemm_nvfp4_noalloc: the NVFP4 GEMM for callers that cannot allocate
device memory during a call — a caller whose device memory belongs to another
framework's allocator, one held to a fixed memory budget, or one that must not
let a call allocate (and so synchronise) in the middle of its own work.  The
scratch for its re-layout of the block scales is a fixed array inside the
library instead of a pool allocation.

Checked here: its output against the CPU oracle within the NVFP4 tolerance, on
two consecutive calls that reuse the shared array (including the one size that
fills the array exactly, M = N = K = 16384, on sampled rows); that warmed-up
calls leave the device's free memory unchanged; and that a problem whose
scratch would not fit is rejected before any GPU work, right at the boundary.

Kept in the last-collected file so that a stop-at-first-failure run has
already run every other test."""
import numpy as np
import pytest

import oracle
from tiled_tensor_core_gb300 import synth

from gpu_util import check_against_oracle, sample_rows

torch = pytest.importorskip("torch")

SCRATCH_BYTES = 32 << 20  # TKG_NVFP4_NOALLOC_SCRATCH_BYTES


@pytest.fixture(scope="module")
def tkg():
    from tiled_tensor_core_gb300 import build
    build.build()
    from tiled_tensor_core_gb300 import tkg as mod
    return mod


def staged_scale_bytes(M, N, K):
    """Scratch the NVFP4 kernel stages its block scales in: 2 KB per (256-deep K stage,
    128-row block) of A (rows padded to 256-row pair tiles) and of B (256-column tiles)."""
    blocks_a = -(-M // 256) * 2
    blocks_b = -(-N // 256) * 2
    return (blocks_a + blocks_b) * -(-K // 256) * 2048


def test_scratch_limit_fits_the_largest_workload_exactly():
    assert staged_scale_bytes(16384, 16384, 16384) == SCRATCH_BYTES
    assert staged_scale_bytes(16385, 16384, 16384) > SCRATCH_BYTES
    assert staged_scale_bytes(16384, 16384, 16416) > SCRATCH_BYTES


def test_rejects_problems_beyond_the_fixed_scratch(tkg):
    A = B = C = 1 << 20  # fake aligned addresses: the size check fails first, nothing is dereferenced
    s = tkg.tkg_scales(1 << 12, 1 << 12, 1 << 14, 1 << 14)
    f = tkg.lib.tkg_gemm_nvfp4_noalloc
    # just past the limit in M (one more 256-row tile) and in K (one more 256-deep stage)
    assert f(16385, 16384, 16384, A, B, C, s, None) == tkg.TKG_ERR_INVALID_ARG
    assert f(16384, 16385, 16384, A, B, C, s, None) == tkg.TKG_ERR_INVALID_ARG
    assert f(16384, 16384, 16416, A, B, C, s, None) == tkg.TKG_ERR_INVALID_ARG
    assert f(32768, 32768, 32768, A, B, C, s, None) == tkg.TKG_ERR_INVALID_ARG
    # the ordinary argument checks come first: K % 32, missing block scales
    assert f(8, 8, 48, A, B, C, s, None) == tkg.TKG_ERR_INVALID_ARG
    assert f(8, 8, 64, A, B, C, tkg.tkg_scales(1 << 12, 1 << 12, None, 1 << 14), None) == tkg.TKG_ERR_INVALID_ARG


def _run_noalloc(tkg, g, out):
    tkg.tkg_gemm_nvfp4_noalloc(g.M, g.N, g.K, g.a, g.b, out, g.scales())
    st = tkg.tkg_check_status()
    assert st == tkg.TKG_OK, tkg.status_string(st)


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(1000, 1000, 1024), (520, 300, 288), (77, 100, 96), (4096, 4096, 4096)])
def test_noalloc_matches_oracle_on_two_calls(tkg, shape):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from tiled_tensor_core_gb300.device import DeviceGemm
    M, N, K = shape
    ops = synth.make_operands("nvfp4", M, N, K, "normal", 91 + M, 92 + N)
    g = DeviceGemm(ops, "cuda")
    acc, c_ref = oracle.gemm(ops)
    for call in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        _run_noalloc(tkg, g, out)
        got = out.view(torch.int16).cpu().numpy().view(np.uint16)
        check_against_oracle("nvfp4", got, acc, c_ref, ops.scale_a, ops.scale_b)


@pytest.mark.gpu
def test_noalloc_exact_fit_workload_sampled_rows(tkg):
    """M = N = K = 16384 stages exactly TKG_NVFP4_NOALLOC_SCRATCH_BYTES of scales."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from tiled_tensor_core_gb300.device import DeviceGemm
    ops = synth.workload_operands("nvfp4_16384")
    g = DeviceGemm(ops, "cuda")
    rows = sample_rows(ops.M, 12, seed=7)
    acc, c_ref = oracle.gemm(ops, rows=rows)
    idx = torch.from_numpy(rows).cuda()
    for call in range(2):
        g.c.fill_(float("nan"))
        _run_noalloc(tkg, g, g.c)
        got = g.c[idx].view(torch.int16).cpu().numpy().view(np.uint16)
        check_against_oracle("nvfp4", got, acc, c_ref, ops.scale_a, ops.scale_b)


@pytest.mark.gpu
def test_noalloc_calls_leave_device_memory_unchanged(tkg):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from tiled_tensor_core_gb300.device import DeviceGemm
    ops = synth.make_operands("nvfp4", 2048, 1536, 2048, "normal", 5, 6)
    g = DeviceGemm(ops, "cuda")
    out = torch.empty((ops.M, ops.N), dtype=torch.bfloat16, device="cuda")
    _run_noalloc(tkg, g, out)  # first call: per-device set-up and the kernels' first load
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    torch_bytes0 = torch.cuda.memory_allocated()
    for _ in range(3):
        _run_noalloc(tkg, g, out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_allocated() == torch_bytes0
