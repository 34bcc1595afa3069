"""Parity of the CUDA GEMMs with the CPU oracle, element by element, on seeded
inputs: small multi-tile shapes with ragged edges through every compiled
variant, exact small-integer and permutation cases (bit-identical output), and
the full-size workloads in the launch configuration the benchmark times
(sampled rows the oracle computes one by one)."""
import numpy as np
import pytest

import oracle
from tiled_tensor_core_gb300 import synth

from gpu_util import check_against_oracle, run_gpu, sample_rows

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def tkg():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from tiled_tensor_core_gb300 import tkg as mod
    yield mod
    mod.tkg_set_option(mod.TKG_OPT_VARIANT, 0)


@pytest.fixture
def variant(tkg, request):
    tkg.tkg_set_option(tkg.TKG_OPT_VARIANT, request.param)
    yield request.param
    tkg.tkg_set_option(tkg.TKG_OPT_VARIANT, 0)


# the compiled variants of each kind: 256x256 and 256x512 pair tiles (bf16 / FP8; the latter with
# its K step's two MMAs sharing A through the collector buffer, and eight epilogue warps given
# their registers by a warpgroup register split), the block-scaled 256x256 pair tile (NVFP4)
KIND_VARIANTS = {"bf16": [2, 15], "fp8": [2, 15], "nvfp4": [14]}
KIND_VARIANT_PAIRS = [(k, v) for k, vs in KIND_VARIANTS.items() for v in vs]

SMALL_SHAPES = {
    "bf16": [(128, 256, 64), (256, 256, 256), (300, 520, 200), (77, 100, 40), (1, 8, 8), (513, 136, 1032),
             (1000, 1000, 512)],
    "fp8": [(128, 256, 128), (256, 256, 256), (300, 520, 208), (77, 100, 48), (1, 16, 16), (1000, 1000, 512)],
    "nvfp4": [(128, 256, 256), (256, 256, 512), (300, 520, 416), (77, 100, 96), (1, 16, 32), (1000, 1000, 1024),
              (520, 300, 288)],
}


@pytest.mark.parametrize("kind,variant", KIND_VARIANT_PAIRS, indirect=["variant"])
def test_small_shapes_match_oracle(tkg, variant, kind):
    for i, (M, N, K) in enumerate(SMALL_SHAPES[kind]):
        ops = synth.make_operands(kind, M, N, K, "normal_sqrtk" if kind == "bf16" else "normal", 31 + i, 47 + i)
        g = run_gpu(ops)
        acc, c_ref = oracle.gemm(ops)
        check_against_oracle(kind, g.c_bits(), acc, c_ref, ops.scale_a, ops.scale_b)


@pytest.mark.parametrize("kind,variant", KIND_VARIANT_PAIRS, indirect=["variant"])
@pytest.mark.parametrize("shape", [(256, 256, 256), (300, 392, 128), (129, 64, 256), (200, 264, 544)])
def test_small_integers_bit_exact(tkg, variant, kind, shape):
    M, N, K = shape
    ops = synth.small_int_operands(kind, M, N, K, seed=sum(shape))
    g = run_gpu(ops)
    _, c_ref = oracle.gemm(ops)
    assert np.array_equal(g.c_bits(), c_ref)


@pytest.mark.parametrize("kind,variant", KIND_VARIANT_PAIRS, indirect=["variant"])
@pytest.mark.parametrize("identity", [True, False])
def test_permutation_exact(tkg, variant, kind, identity):
    ops, perm = synth.permutation_operands(kind, 384, 256, seed=3, identity=identity)
    g = run_gpu(ops)
    _, c_ref = oracle.gemm(ops)
    assert np.array_equal(g.c_bits(), c_ref)


def test_output_fully_overwritten_and_repeatable(tkg):
    ops = synth.make_operands("bf16", 640, 768, 320, "normal_sqrtk", 5, 6)
    g1 = run_gpu(ops)
    first = g1.c_bits()
    g1.c.fill_(123.0)
    g1.run()
    assert tkg.tkg_check_status() == tkg.TKG_OK
    assert np.array_equal(g1.c_bits(), first)


@pytest.mark.parametrize("group_m", [1, 3, 8, 64])
def test_tile_order_does_not_change_result(tkg, group_m):
    ops = synth.make_operands("bf16", 1536, 1280, 256, "normal_sqrtk", 8, 9)
    tkg.tkg_set_option(tkg.TKG_OPT_GROUP_M, group_m)
    try:
        g = run_gpu(ops)
    finally:
        tkg.tkg_set_option(tkg.TKG_OPT_GROUP_M, 0)
    acc, c_ref = oracle.gemm(ops)
    check_against_oracle("bf16", g.c_bits(), acc, c_ref)


def test_small_grid_many_tiles_per_cta(tkg):
    ops = synth.make_operands("bf16", 2048, 2048, 128, "normal_sqrtk", 10, 11)
    tkg.tkg_set_option(tkg.TKG_OPT_MAX_CTAS, 4)
    try:
        g = run_gpu(ops)
    finally:
        tkg.tkg_set_option(tkg.TKG_OPT_MAX_CTAS, 0)
    acc, c_ref = oracle.gemm(ops)
    check_against_oracle("bf16", g.c_bits(), acc, c_ref)


# ---- full-size workloads, default (benchmarked) launch configuration -------

@pytest.mark.parametrize("name", ["bf16_256", "bf16_4096"])
def test_workload_full_compare(tkg, name):
    ops = synth.workload_operands(name)
    g = run_gpu(ops)
    acc, c_ref = oracle.gemm(ops)
    check_against_oracle(ops.kind, g.c_bits(), acc, c_ref, ops.scale_a, ops.scale_b)


@pytest.mark.parametrize("name", ["bf16_8192", "bf16_skinny", "fp8_8192", "nvfp4_16384"])
def test_workload_sampled_rows(tkg, name):
    ops = synth.workload_operands(name)
    g = run_gpu(ops)
    rows = sample_rows(ops.M, 24, seed=ops.M)
    acc, c_ref = oracle.gemm(ops, rows=rows)
    c = g.c[torch.from_numpy(rows).cuda()].view(torch.int16).cpu().numpy().view(np.uint16)
    check_against_oracle(ops.kind, c, acc, c_ref, ops.scale_a, ops.scale_b)


def test_nvfp4_zero_block_scales_give_zero(tkg):
    # a block whose scale is 0 contributes nothing, whatever its e2m1 codes
    ops = synth.make_operands("nvfp4", 256, 256, 512, "normal", 21, 22)
    ops.sfa[:, 1::2] = 0
    g = run_gpu(ops)
    acc, c_ref = oracle.gemm(ops)
    check_against_oracle("nvfp4", g.c_bits(), acc, c_ref, ops.scale_a, ops.scale_b)


def test_nvfp4_repeated_calls_reuse_scratch(tkg):
    # the interleaved-scale scratch is stream-ordered and recycled between calls
    shapes = [(512, 384, 1024), (256, 256, 256), (768, 1024, 512)]
    for i, (M, N, K) in enumerate(shapes * 2):
        ops = synth.make_operands("nvfp4", M, N, K, "normal", 60 + i, 80 + i)
        g = run_gpu(ops)
        acc, c_ref = oracle.gemm(ops)
        check_against_oracle("nvfp4", g.c_bits(), acc, c_ref, ops.scale_a, ops.scale_b)


# ---- K order of a CTA's work items -------------------------------------------

@pytest.mark.parametrize("order", ["serpentine", "forward"])
@pytest.mark.parametrize("kind,variant", [("bf16", 2), ("bf16", 15), ("fp8", 15), ("nvfp4", 14)])
def test_k_order_keeps_results(tkg, kind, variant, order):
    """Two CTA pairs walk many tiles each, so half of every pair's tiles run their K blocks
    backwards in the serpentine order: exact on small integers, and within tolerance."""
    tkg.tkg_set_option(tkg.TKG_OPT_VARIANT, variant)
    tkg.tkg_set_option(tkg.TKG_OPT_K_ORDER,
                       tkg.TKG_K_ORDER_SERPENTINE if order == "serpentine" else tkg.TKG_K_ORDER_FORWARD)
    tkg.tkg_set_option(tkg.TKG_OPT_MAX_CTAS, 4)
    try:
        M, N, K = 1280, 1536, {"bf16": 640, "fp8": 768, "nvfp4": 1536}[kind]
        ops = synth.small_int_operands(kind, M, N, K, seed=K)
        g = run_gpu(ops)
        _, c_ref = oracle.gemm(ops)
        assert np.array_equal(g.c_bits(), c_ref)
        ops = synth.make_operands(kind, M, N, K, "normal_sqrtk" if kind == "bf16" else "normal", 12, 13)
        g = run_gpu(ops)
        acc, c_ref = oracle.gemm(ops)
        check_against_oracle(kind, g.c_bits(), acc, c_ref, ops.scale_a, ops.scale_b)
    finally:
        tkg.tkg_set_option(tkg.TKG_OPT_MAX_CTAS, 0)
        tkg.tkg_set_option(tkg.TKG_OPT_K_ORDER, 0)
        tkg.tkg_set_option(tkg.TKG_OPT_VARIANT, 0)
