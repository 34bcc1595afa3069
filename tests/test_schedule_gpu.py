"""Tile schedules and launch overlap on the GPU.

Every schedule (the persistent static grid, the dynamic one driven by cluster
launch control, one cluster per tile) must store every output tile exactly
once and give the oracle's result; GEMMs launched as programmatic dependents
must still see their predecessor's output (read after write) and must not
overwrite what the predecessor is still reading (write after read)."""
import numpy as np
import pytest

import oracle
from tiled_tensor_core_gb300 import synth

from gpu_util import check_against_oracle, run_gpu, sample_rows

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

SCHEDULES = {"static": 1, "dynamic": 2, "single": 3}


@pytest.fixture(scope="module")
def tkg():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from tiled_tensor_core_gb300 import tkg as mod
    yield mod
    mod.tkg_set_option(mod.TKG_OPT_SCHEDULE, 0)
    mod.tkg_set_option(mod.TKG_OPT_LAUNCH_OVERLAP, 0)
    mod.tkg_set_option(mod.TKG_OPT_VARIANT, 0)


@pytest.fixture
def schedule(tkg, request):
    tkg.tkg_set_option(tkg.TKG_OPT_SCHEDULE, SCHEDULES[request.param])
    yield request.param
    tkg.tkg_set_option(tkg.TKG_OPT_SCHEDULE, 0)


def tiles_of(tkg, kind, M, N, K):
    info = tkg.tkg_debug_variant_info({"bf16": 0, "fp8": 1, "nvfp4": 2}[kind],
                                      tkg.tkg_debug_pick_variant({"bf16": 0, "fp8": 1, "nvfp4": 2}[kind], M, N, K))
    tm = -(-M // info["tile_m"])
    tn = -(-N // info["tile_n"])
    return tm * tn


def run_counted(tkg, ops):
    """Run one GEMM with the tile-visit counter armed; returns (DeviceGemm, counts)."""
    from tiled_tensor_core_gb300.device import DeviceGemm
    g = DeviceGemm(ops, "cuda")
    g.c.fill_(float("nan"))
    counts = torch.zeros(tiles_of(tkg, ops.kind, ops.M, ops.N, ops.K), dtype=torch.int32, device="cuda")
    tkg.tkg_debug_set_visit_counter(counts)
    g.run()
    st = tkg.tkg_check_status()
    assert st == tkg.TKG_OK, tkg.status_string(st)
    return g, counts.cpu().numpy()


SHAPES = {
    "bf16": [(256, 256, 64), (300, 520, 200), (1000, 1000, 512), (2048, 1536, 64), (77, 100, 40)],
    "fp8": [(300, 520, 208), (1000, 1000, 512), (2048, 1536, 128)],
    "nvfp4": [(300, 520, 416), (1000, 1000, 1024), (2048, 1536, 256)],
}


@pytest.mark.parametrize("schedule", list(SCHEDULES), indirect=True)
@pytest.mark.parametrize("kind", ["bf16", "fp8", "nvfp4"])
def test_schedule_matches_oracle_and_visits_each_tile_once(tkg, schedule, kind):
    for i, (M, N, K) in enumerate(SHAPES[kind]):
        ops = synth.make_operands(kind, M, N, K, "normal_sqrtk" if kind == "bf16" else "normal", 90 + i, 95 + i)
        g, counts = run_counted(tkg, ops)
        assert (counts == 1).all(), (schedule, M, N, K, np.unique(counts, return_counts=True))
        acc, c_ref = oracle.gemm(ops)
        check_against_oracle(kind, g.c_bits(), acc, c_ref, ops.scale_a, ops.scale_b)


@pytest.mark.parametrize("schedule", list(SCHEDULES), indirect=True)
@pytest.mark.parametrize("kind", ["bf16", "fp8", "nvfp4"])
def test_schedule_small_integers_bit_exact(tkg, schedule, kind):
    ops = synth.small_int_operands(kind, 1280, 1024, 256, seed=7)
    g, counts = run_counted(tkg, ops)
    assert (counts == 1).all()
    _, c_ref = oracle.gemm(ops)
    assert np.array_equal(g.c_bits(), c_ref)


@pytest.mark.parametrize("schedule", list(SCHEDULES), indirect=True)
@pytest.mark.parametrize("K", [64, 256, 1024])
def test_k_sweep_shapes(tkg, schedule, K):
    # the persistent-vs-non-persistent study shape of "Persistent Grid Launch" (Table 2): M = N = 4096
    ops = synth.workload_operands(f"bf16_4096_k{K}")
    g, counts = run_counted(tkg, ops)
    assert (counts == 1).all()
    rows = sample_rows(ops.M, 16, seed=K)
    acc, c_ref = oracle.gemm(ops, rows=rows)
    c = g.c[torch.from_numpy(rows).cuda()].view(torch.int16).cpu().numpy().view(np.uint16)
    check_against_oracle("bf16", c, acc, c_ref)


@pytest.mark.parametrize("schedule", ["dynamic", "single"], indirect=True)
def test_schedule_full_size_nvfp4_sampled(tkg, schedule):
    ops = synth.workload_operands("nvfp4_16384")
    g, counts = run_counted(tkg, ops)
    assert (counts == 1).all()
    rows = sample_rows(ops.M, 8, seed=3)
    acc, c_ref = oracle.gemm(ops, rows=rows)
    c = g.c[torch.from_numpy(rows).cuda()].view(torch.int16).cpu().numpy().view(np.uint16)
    check_against_oracle("nvfp4", c, acc, c_ref, ops.scale_a, ops.scale_b)


def test_static_capped_grid_visits_each_tile_once(tkg):
    ops = synth.make_operands("bf16", 2048, 2048, 128, "normal_sqrtk", 12, 13)
    tkg.tkg_set_option(tkg.TKG_OPT_MAX_CTAS, 6)
    try:
        g, counts = run_counted(tkg, ops)
    finally:
        tkg.tkg_set_option(tkg.TKG_OPT_MAX_CTAS, 0)
    assert (counts == 1).all()
    acc, c_ref = oracle.gemm(ops)
    check_against_oracle("bf16", g.c_bits(), acc, c_ref)


# ---- the 256x512 pair tile ---------------------------------------------------

@pytest.fixture
def variant(tkg, request):
    tkg.tkg_set_option(tkg.TKG_OPT_VARIANT, request.param)
    yield request.param
    tkg.tkg_set_option(tkg.TKG_OPT_VARIANT, 0)


# odd and even numbers of 512-wide tile columns, one tile row, one column, ragged last rows and
# columns, and many tiles per cluster
WIDE_SHAPES = [(300, 520, 200), (256, 1024, 128), (1000, 1000, 512), (77, 100, 40), (2048, 1536, 64),
               (512, 2100, 128)]


@pytest.mark.parametrize("variant", [15], indirect=True)
@pytest.mark.parametrize("schedule", list(SCHEDULES), indirect=True)
@pytest.mark.parametrize("kind", ["bf16", "fp8"])
def test_wide_tile_matches_oracle_and_visits_each_tile_once(tkg, variant, schedule, kind):
    for i, (M, N, K) in enumerate(WIDE_SHAPES):
        if kind == "fp8":
            K = -(-K // 16) * 16
        ops = synth.make_operands(kind, M, N, K, "normal_sqrtk" if kind == "bf16" else "normal", 70 + i, 75 + i)
        g, counts = run_counted(tkg, ops)
        assert (counts == 1).all(), (variant, schedule, M, N, K, np.unique(counts, return_counts=True))
        acc, c_ref = oracle.gemm(ops)
        check_against_oracle(kind, g.c_bits(), acc, c_ref, ops.scale_a, ops.scale_b)


@pytest.mark.parametrize("variant", [15], indirect=True)
def test_wide_tile_one_cluster_walks_every_tile(tkg, variant):
    ops = synth.small_int_operands("bf16", 1280, 1600, 256, seed=11)
    tkg.tkg_set_option(tkg.TKG_OPT_MAX_CTAS, 2)
    try:
        g, counts = run_counted(tkg, ops)
    finally:
        tkg.tkg_set_option(tkg.TKG_OPT_MAX_CTAS, 0)
    assert (counts == 1).all()
    _, c_ref = oracle.gemm(ops)
    assert np.array_equal(g.c_bits(), c_ref)


# ---- launch overlap (programmatic dependent launch) -------------------------

def _chain(tkg, overlap, schedule, reps):
    """Back-to-back dependent GEMMs on one stream, with no other kernel between
    them.  Round r:  x1 = a[r]·b0ᵀ;  x2[r] = x1·b1ᵀ (reads x1: read after
    write);  x1 = a[r+1]·Iᵀ (overwrites x1 while the previous GEMM reads it:
    write after read);  x3[r] = x1·b1ᵀ.  Returns the x2 and x3 outputs."""
    tkg.tkg_set_option(tkg.TKG_OPT_LAUNCH_OVERLAP, overlap)
    tkg.tkg_set_option(tkg.TKG_OPT_SCHEDULE, schedule)
    try:
        n = 1024
        gen = torch.Generator(device="cpu").manual_seed(5)
        rnd = lambda: (torch.randn(n, n, generator=gen) / n ** 0.5).to(torch.bfloat16).cuda()
        a = [rnd() for _ in range(reps + 1)]
        b0, b1 = rnd(), rnd()
        ident = torch.eye(n, dtype=torch.bfloat16, device="cuda")
        x1 = torch.empty(n, n, dtype=torch.bfloat16, device="cuda")
        x2 = [torch.empty(n, n, dtype=torch.bfloat16, device="cuda") for _ in range(reps)]
        x3 = [torch.empty(n, n, dtype=torch.bfloat16, device="cuda") for _ in range(reps)]
        torch.cuda.synchronize()
        for r in range(reps):
            tkg.tkg_gemm_bf16(n, n, n, a[r], b0, x1)
            tkg.tkg_gemm_bf16(n, n, n, x1, b1, x2[r])
            tkg.tkg_gemm_bf16(n, n, n, a[r + 1], ident, x1)
            tkg.tkg_gemm_bf16(n, n, n, x1, b1, x3[r])
        st = tkg.tkg_check_status()
        assert st == tkg.TKG_OK, tkg.status_string(st)
        torch.cuda.synchronize()
        bits = lambda t: t.view(torch.int16).cpu().numpy()
        return [bits(t) for t in x2], [bits(t) for t in x3], a, b1
    finally:
        tkg.tkg_set_option(tkg.TKG_OPT_LAUNCH_OVERLAP, 0)
        tkg.tkg_set_option(tkg.TKG_OPT_SCHEDULE, 0)


@pytest.mark.parametrize("schedule", [1, 2, 3])
def test_overlapped_launches_keep_stream_order(tkg, schedule):
    p2, p3, _, _ = _chain(tkg, tkg.TKG_OVERLAP_OFF, schedule, reps=8)
    o2, o3, a, b1 = _chain(tkg, tkg.TKG_OVERLAP_ON, schedule, reps=8)
    for r in range(8):
        assert np.array_equal(p2[r], o2[r]), r
        assert np.array_equal(p3[r], o3[r]), r
    # x3[r] is a[r+1]·b1ᵀ: the identity GEMM copied a[r+1] exactly before x3 read it (the
    # reference runs in the same schedule, so that it splits K, or not, as the chain did)
    n = 1024
    ref = torch.empty(n, n, dtype=torch.bfloat16, device="cuda")
    tkg.tkg_set_option(tkg.TKG_OPT_SCHEDULE, schedule)
    try:
        for r in range(8):
            tkg.tkg_gemm_bf16(n, n, n, a[r + 1], b1, ref)
            assert tkg.tkg_check_status() == tkg.TKG_OK
            assert np.array_equal(ref.view(torch.int16).cpu().numpy(), o3[r]), r
    finally:
        tkg.tkg_set_option(tkg.TKG_OPT_SCHEDULE, 0)


def test_overlapped_chain_matches_oracle(tkg):
    # the first link of the chain against the oracle, with overlap on and a
    # predecessor still running when the dependent grid is launched
    ops = synth.make_operands("bf16", 2048, 2048, 1024, "normal_sqrtk", 40, 41)
    from tiled_tensor_core_gb300.device import DeviceGemm
    big = DeviceGemm(synth.make_operands("bf16", 4096, 4096, 4096, "normal_sqrtk", 42, 43), "cuda")
    g = DeviceGemm(ops, "cuda")
    g.c.fill_(float("nan"))
    tkg.tkg_set_option(tkg.TKG_OPT_LAUNCH_OVERLAP, tkg.TKG_OVERLAP_ON)
    try:
        big.run()
        g.run()
        assert tkg.tkg_check_status() == tkg.TKG_OK
    finally:
        tkg.tkg_set_option(tkg.TKG_OPT_LAUNCH_OVERLAP, 0)
    acc, c_ref = oracle.gemm(ops)
    check_against_oracle("bf16", g.c_bits(), acc, c_ref)
