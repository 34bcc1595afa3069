"""The split-K head of the static schedule on the GPU.

When the persistent grid's last round of tiles would be at most half full,
those tiles are cut along K into pieces that run first; the last piece of a
tile to finish adds the fp32 partials in piece order and stores the tile.
Small grids (TKG_OPT_MAX_CTAS) force every split factor on small shapes the
oracle checks in full, including ragged single tiles and the generic store
path; the results must be deterministic and every tile stored exactly once."""
import numpy as np
import pytest

import oracle
from tiled_tensor_core_gb300 import synth

from gpu_util import check_against_oracle, run_gpu

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

KIND_ID = {"bf16": 0, "fp8": 1, "nvfp4": 2}


@pytest.fixture(scope="module")
def tkg():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from tiled_tensor_core_gb300 import tkg as mod
    yield mod
    mod.tkg_set_option(mod.TKG_OPT_MAX_CTAS, 0)
    mod.tkg_set_option(mod.TKG_OPT_SPLIT_K, 0)
    mod.tkg_set_option(mod.TKG_OPT_VARIANT, 0)


def plan_for(tkg, kind, M, N, K, ctas):
    """The split plan the library will use for this shape on a grid capped at `ctas` CTAs."""
    kid = KIND_ID[kind]
    info = tkg.tkg_debug_variant_info(kid, tkg.tkg_debug_pick_variant(kid, M, N, K))
    cg = info["cta_group"]
    tiles = -(-M // info["tile_m"]) * -(-N // info["tile_n"])
    k_bytes = {"bf16": 2 * K, "fp8": K, "nvfp4": K // 2}[kind]
    num_kb = -(-k_bytes // 128)
    return tkg.tkg_debug_split_plan(tiles, ctas // cg, num_kb), tiles


def run_counted(tkg, ops, tiles):
    from tiled_tensor_core_gb300.device import DeviceGemm
    g = DeviceGemm(ops, "cuda")
    g.c.fill_(float("nan"))
    counts = torch.zeros(tiles, dtype=torch.int32, device="cuda")
    tkg.tkg_debug_set_visit_counter(counts)
    g.run()
    st = tkg.tkg_check_status()
    assert st == tkg.TKG_OK, tkg.status_string(st)
    torch.cuda.synchronize()
    return g, counts.cpu().numpy()


# (M, N, K, CTAs): 2-SM pairs, so CTAs / 2 clusters; the plan (split tiles, pieces) in comments
CASES = {
    "bf16": [(1280, 256, 4096, 8),    # 5 tiles on 4 pairs: (1, 4)
             (1280, 512, 512, 12),    # 10 tiles on 6 pairs: last round 4 of 6, no split
             (768, 256, 4096, 16),    # 3 tiles on 8 pairs: (3, 2)
             (100, 100, 4096, 8),     # one ragged tile, generic stores (N % 8 != 0): (1, 4)
             (300, 520, 4000, 48),    # ragged edges, 6 tiles on 24 pairs: (6, 3), 63 K stages (last partial)
             (2560, 1792, 2048, 32),  # 70 tiles on 16 pairs: (6, 2)
             (256, 256, 64, 8)],      # one tile of one K stage: no split
    "fp8": [(1280, 256, 4096, 8), (100, 112, 8192, 8), (2560, 1792, 4096, 32)],     # (1, 2), (1, 4), (6, 2)
    "nvfp4": [(1280, 256, 8192, 8), (100, 128, 16384, 8), (2560, 1792, 8192, 32)],  # (1, 2), (1, 4), (6, 2)
}


@pytest.mark.parametrize("kind", ["bf16", "fp8", "nvfp4"])
def test_split_matches_oracle_and_stores_each_tile_once(tkg, kind):
    split_seen = 0
    for i, (M, N, K, ctas) in enumerate(CASES[kind]):
        tkg.tkg_set_option(tkg.TKG_OPT_MAX_CTAS, ctas)
        (st, ss), tiles = plan_for(tkg, kind, M, N, K, ctas)
        split_seen += st > 0
        ops = synth.make_operands(kind, M, N, K, "normal_sqrtk" if kind == "bf16" else "normal", 300 + i, 310 + i)
        g, counts = run_counted(tkg, ops, tiles)
        assert (counts == 1).all(), (M, N, K, ctas, st, ss, np.unique(counts, return_counts=True))
        acc, c_ref = oracle.gemm(ops)
        check_against_oracle(kind, g.c_bits(), acc, c_ref, ops.scale_a, ops.scale_b)
        # deterministic: the partials are added in piece order whichever piece finishes last
        first = g.c_bits()
        g.c.fill_(float("nan"))
        g.run()
        assert tkg.tkg_check_status() == tkg.TKG_OK
        assert np.array_equal(g.c_bits(), first)
    assert split_seen >= 2


@pytest.mark.parametrize("kind", ["bf16", "fp8", "nvfp4"])
@pytest.mark.parametrize("ctas", [8, 16])
def test_split_small_integers_bit_exact(tkg, kind, ctas):
    # 8 CTAs: 5 tiles, two rounds; 16 CTAs: 3 tiles in one round, which needs 48 K stages a tile
    M, N = (1280, 256) if ctas == 8 else (768, 256)
    K = {"bf16": 4096, "fp8": 4096, "nvfp4": 8192}[kind] * (1 if ctas == 8 or kind == "bf16" else 2)
    tkg.tkg_set_option(tkg.TKG_OPT_MAX_CTAS, ctas)
    (st, ss), tiles = plan_for(tkg, kind, M, N, K, ctas)
    assert st > 0
    ops = synth.small_int_operands(kind, M, N, K, seed=ctas)
    g, counts = run_counted(tkg, ops, tiles)
    assert (counts == 1).all()
    _, c_ref = oracle.gemm(ops)
    assert np.array_equal(g.c_bits(), c_ref)


def test_split_off_runs_whole_tiles(tkg):
    M, N, K, ctas = 1280, 256, 4096, 8
    tkg.tkg_set_option(tkg.TKG_OPT_MAX_CTAS, ctas)
    ops = synth.make_operands("bf16", M, N, K, "normal_sqrtk", 5, 6)
    on = run_gpu(ops).c_bits()
    tkg.tkg_set_option(tkg.TKG_OPT_SPLIT_K, tkg.TKG_SPLIT_OFF)
    try:
        off = run_gpu(ops).c_bits()
    finally:
        tkg.tkg_set_option(tkg.TKG_OPT_SPLIT_K, 0)
    acc, c_ref = oracle.gemm(ops)
    check_against_oracle("bf16", on, acc, c_ref)
    check_against_oracle("bf16", off, acc, c_ref)


def test_split_on_two_streams_and_repeated_launches(tkg):
    # each stream has its own workspace; back-to-back launches on a stream reuse it (the
    # counters return to zero at the end of every launch)
    M, N, K, ctas = 1280, 256, 4096, 8
    tkg.tkg_set_option(tkg.TKG_OPT_MAX_CTAS, ctas)
    from tiled_tensor_core_gb300.device import DeviceGemm
    opsets = [synth.make_operands("bf16", M, N, K, "normal_sqrtk", 40 + i, 50 + i) for i in range(2)]
    gs = [DeviceGemm(o, "cuda") for o in opsets]
    streams = [torch.cuda.Stream() for _ in range(2)]
    for rep in range(3):
        for g, s in zip(gs, streams):
            g.c.fill_(float("nan"))
            with torch.cuda.stream(s):
                g.run(stream=s.cuda_stream)
        torch.cuda.synchronize()
        assert tkg.tkg_check_status() == tkg.TKG_OK
        for g, o in zip(gs, opsets):
            acc, c_ref = oracle.gemm(o)
            check_against_oracle("bf16", g.c_bits(), acc, c_ref)


def test_split_recovers_after_timeout_and_shutdown(tkg):
    # a launch that gives up may leave piece counts behind: tkg_check_status drops the
    # workspaces, and the next split launch (on fresh ones) is exact; so is one after
    # tkg_shutdown, which frees them too
    M, N, K, ctas = 1280, 256, 4096, 8
    tkg.tkg_set_option(tkg.TKG_OPT_MAX_CTAS, ctas)
    (st, ss), tiles = plan_for(tkg, "bf16", M, N, K, ctas)
    assert st > 0
    ops = synth.small_int_operands("bf16", M, N, K, seed=23)
    _, c_ref = oracle.gemm(ops)
    from tiled_tensor_core_gb300.device import DeviceGemm
    g = DeviceGemm(ops, "cuda")
    tkg.tkg_set_option(tkg.TKG_OPT_TIMEOUT_NS, 100_000_000)  # 0.1 s per wait
    try:
        tkg.tkg_debug_set_fault(1)
        g.run()
        assert tkg.tkg_check_status() == tkg.TKG_ERR_TIMEOUT
    finally:
        tkg.tkg_debug_set_fault(0)
        tkg.tkg_set_option(tkg.TKG_OPT_TIMEOUT_NS, 0)
    for _ in range(2):
        g2, counts = run_counted(tkg, ops, tiles)
        assert (counts == 1).all()
        assert np.array_equal(g2.c_bits(), c_ref)
    tkg.tkg_shutdown()
    tkg.tkg_set_option(tkg.TKG_OPT_MAX_CTAS, ctas)
    g3, counts = run_counted(tkg, ops, tiles)
    assert (counts == 1).all()
    assert np.array_equal(g3.c_bits(), c_ref)
