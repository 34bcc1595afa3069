"""C-ABI checks that need no GPU: the library loads, exports every function
the headers declare, rejects bad arguments before touching CUDA, and its
host-compiled scheduler / swizzle helpers agree with the definitions."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

from oracle import swizzle as sw

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def tkg():
    from tiled_tensor_core_gb300 import build
    build.build()
    from tiled_tensor_core_gb300 import tkg as mod
    return mod


def declared_functions():
    names = []
    for h in ("tkg.h", "tkg_debug.h"):
        text = open(os.path.join(ROOT, "include", h)).read()
        names += re.findall(r"TKG_API\s+[\w\s\*]+?\b(tkg_\w+)\s*\(", text)
    return sorted(set(names))


def test_headers_declare_the_boundary():
    names = declared_functions()
    for required in ("tkg_gemm_bf16", "tkg_gemm_fp8", "tkg_gemm_nvfp4", "tkg_check_status",
                     "tkg_status_string", "tkg_shutdown"):
        assert required in names


def test_library_exports_every_declared_symbol(tkg):
    out = subprocess.run(["nm", "-D", "--defined-only", tkg.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT\s+(tkg_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert hasattr(tkg.lib, n)


def test_library_links_no_torch_and_no_libcuda(tkg):
    out = subprocess.run(["ldd", tkg.LIB_PATH], capture_output=True, text=True).stdout
    assert "torch" not in out and "libcuda.so" not in out


def test_status_strings(tkg):
    for s in range(7):
        assert tkg.status_string(s)
    assert tkg.status_string(99) == "unknown status"


@pytest.mark.parametrize("fn", ["tkg_gemm_bf16", "tkg_gemm_fp8", "tkg_gemm_nvfp4"])
def test_invalid_sizes_rejected_before_any_cuda_call(tkg, fn):
    f = getattr(tkg.lib, fn)
    A = B = C = 1 << 20  # 16-byte aligned fake addresses: never dereferenced
    for M, N, K in [(0, 8, 256), (8, 0, 256), (8, 8, 0), (-1, 8, 256), (8, 8, 1 << 31)]:
        assert f(M, N, K, A, B, C, None, None) == tkg.TKG_ERR_INVALID_ARG
    assert f(8, 8, 256, 0, B, C, None, None) == tkg.TKG_ERR_INVALID_ARG


def test_k_alignment_rules(tkg):
    A = B = C = 1 << 20
    s = tkg.tkg_scales(1 << 12, 1 << 12, None, None)
    assert tkg.lib.tkg_gemm_bf16(8, 8, 12, A, B, C, None, None) == tkg.TKG_ERR_INVALID_ARG
    assert tkg.lib.tkg_gemm_fp8(8, 8, 24, A, B, C, s, None) == tkg.TKG_ERR_INVALID_ARG
    s4 = tkg.tkg_scales(1 << 12, 1 << 12, 1 << 14, 1 << 14)
    assert tkg.lib.tkg_gemm_nvfp4(8, 8, 48, A, B, C, s4, None) == tkg.TKG_ERR_INVALID_ARG


def test_scale_arguments_checked(tkg):
    A = B = C = 1 << 20
    s = tkg.tkg_scales(1 << 12, 1 << 12, None, None)
    assert tkg.lib.tkg_gemm_bf16(8, 8, 64, A, B, C, s, None) == tkg.TKG_ERR_INVALID_ARG
    assert tkg.lib.tkg_gemm_fp8(8, 8, 64, A, B, C, None, None) == tkg.TKG_ERR_INVALID_ARG
    assert tkg.lib.tkg_gemm_fp8(8, 8, 64, A, B, C, tkg.tkg_scales(1 << 12, None, None, None), None) \
        == tkg.TKG_ERR_INVALID_ARG
    assert tkg.lib.tkg_gemm_nvfp4(8, 8, 64, A, B, C, s, None) == tkg.TKG_ERR_INVALID_ARG


def test_misaligned_pointers_rejected(tkg):
    A = B = C = 1 << 20
    assert tkg.lib.tkg_gemm_bf16(8, 8, 64, A + 2, B, C, None, None) == tkg.TKG_ERR_MISALIGNED
    assert tkg.lib.tkg_gemm_bf16(8, 8, 64, A, B + 8, C, None, None) == tkg.TKG_ERR_MISALIGNED
    assert tkg.lib.tkg_gemm_bf16(8, 8, 64, A, B, C + 4, None, None) == tkg.TKG_ERR_MISALIGNED
    s = tkg.tkg_scales((1 << 12) + 2, 1 << 12, None, None)
    assert tkg.lib.tkg_gemm_fp8(8, 8, 64, A, B, C, s, None) == tkg.TKG_ERR_MISALIGNED
    s4 = tkg.tkg_scales(1 << 12, 1 << 12, (1 << 14) + 4, 1 << 14)
    assert tkg.lib.tkg_gemm_nvfp4(8, 8, 64, A, B, C, s4, None) == tkg.TKG_ERR_MISALIGNED


def test_options_roundtrip(tkg):
    assert tkg.tkg_get_option(tkg.TKG_OPT_GROUP_M) == 16
    tkg.tkg_set_option(tkg.TKG_OPT_GROUP_M, 12)
    assert tkg.tkg_get_option(tkg.TKG_OPT_GROUP_M) == 12
    tkg.tkg_set_option(tkg.TKG_OPT_GROUP_M, 0)
    assert tkg.tkg_get_option(tkg.TKG_OPT_GROUP_M) == 16
    assert tkg.tkg_get_option(tkg.TKG_OPT_TIMEOUT_NS) == 2_000_000_000
    with pytest.raises(tkg.TkgError):
        tkg.tkg_set_option(tkg.TKG_OPT_VARIANT, 99)
    with pytest.raises(tkg.TkgError):
        tkg.tkg_set_option(77, 1)


def test_k_order_option(tkg):
    assert tkg.tkg_get_option(tkg.TKG_OPT_K_ORDER) == tkg.TKG_K_ORDER_SERPENTINE
    tkg.tkg_set_option(tkg.TKG_OPT_K_ORDER, tkg.TKG_K_ORDER_FORWARD)
    assert tkg.tkg_get_option(tkg.TKG_OPT_K_ORDER) == tkg.TKG_K_ORDER_FORWARD
    tkg.tkg_set_option(tkg.TKG_OPT_K_ORDER, 0)
    assert tkg.tkg_get_option(tkg.TKG_OPT_K_ORDER) == tkg.TKG_K_ORDER_SERPENTINE
    with pytest.raises(tkg.TkgError):
        tkg.tkg_set_option(tkg.TKG_OPT_K_ORDER, 3)


def test_schedule_and_overlap_options(tkg):
    assert tkg.tkg_get_option(tkg.TKG_OPT_SCHEDULE) == tkg.TKG_SCHEDULE_STATIC
    assert tkg.tkg_get_option(tkg.TKG_OPT_LAUNCH_OVERLAP) == tkg.TKG_OVERLAP_ON
    for v in (tkg.TKG_SCHEDULE_STATIC, tkg.TKG_SCHEDULE_DYNAMIC, tkg.TKG_SCHEDULE_SINGLE):
        tkg.tkg_set_option(tkg.TKG_OPT_SCHEDULE, v)
        assert tkg.tkg_get_option(tkg.TKG_OPT_SCHEDULE) == v
    tkg.tkg_set_option(tkg.TKG_OPT_LAUNCH_OVERLAP, tkg.TKG_OVERLAP_OFF)
    assert tkg.tkg_get_option(tkg.TKG_OPT_LAUNCH_OVERLAP) == tkg.TKG_OVERLAP_OFF
    for key, bad in ((tkg.TKG_OPT_SCHEDULE, 4), (tkg.TKG_OPT_LAUNCH_OVERLAP, 3), (tkg.TKG_OPT_SCHEDULE, -1)):
        with pytest.raises(tkg.TkgError):
            tkg.tkg_set_option(key, bad)
    tkg.tkg_set_option(tkg.TKG_OPT_SCHEDULE, 0)
    tkg.tkg_set_option(tkg.TKG_OPT_LAUNCH_OVERLAP, 0)
    assert tkg.tkg_get_option(tkg.TKG_OPT_SCHEDULE) == tkg.TKG_SCHEDULE_STATIC
    assert tkg.tkg_get_option(tkg.TKG_OPT_LAUNCH_OVERLAP) == tkg.TKG_OVERLAP_ON


def test_split_option(tkg):
    assert tkg.tkg_get_option(tkg.TKG_OPT_SPLIT_K) == tkg.TKG_SPLIT_ON
    tkg.tkg_set_option(tkg.TKG_OPT_SPLIT_K, tkg.TKG_SPLIT_OFF)
    assert tkg.tkg_get_option(tkg.TKG_OPT_SPLIT_K) == tkg.TKG_SPLIT_OFF
    with pytest.raises(tkg.TkgError):
        tkg.tkg_set_option(tkg.TKG_OPT_SPLIT_K, 3)
    tkg.tkg_set_option(tkg.TKG_OPT_SPLIT_K, 0)
    assert tkg.tkg_get_option(tkg.TKG_OPT_SPLIT_K) == tkg.TKG_SPLIT_ON


def simulate_static(tkg, tiles, clusters, num_kb):
    """Plan the split-K head, walk the static schedule (cluster c takes items
    c, c + clusters, ...) and return (plan, per-tile K-block coverage, the
    busiest cluster's work in whole-tile units)."""
    st, ss = tkg.tkg_debug_split_plan(tiles, clusters, num_kb)
    items = tiles + st * (ss - 1)
    cover = np.zeros((tiles, num_kb), dtype=np.int32)
    load = np.zeros(clusters)
    pieces = []
    for w in range(items):
        tile, kb0, kb1, piece = tkg.tkg_debug_work_item(w, st, ss, num_kb)
        assert 0 <= tile < tiles and 0 <= kb0 < kb1 <= num_kb
        assert (piece >= 0) == (w < st * ss) and (piece < 0 or piece == w)
        cover[tile, kb0:kb1] += 1
        load[w % clusters] += (kb1 - kb0) / num_kb
        if piece >= 0:
            pieces.append((tile, piece % ss, kb0, kb1))
    return (st, ss), cover, load.max(), pieces


@pytest.mark.parametrize("tiles,clusters,num_kb", [
    (256, 76, 64),     # bf16 4096^3 on 76 CTA pairs: 3 rounds + 28 tail tiles
    (1024, 76, 64),    # FP8 8192^3
    (1024, 76, 128),   # bf16 8192^3
    (4096, 76, 128),   # NVFP4 16384^3: tail 68 of 76, no split
    (16, 76, 32), (16, 76, 64), (1, 76, 16), (1, 76, 3), (1, 76, 256), (77, 76, 64), (152, 76, 64),
    (190, 76, 8), (190, 76, 48), (5, 2, 40), (3, 1, 64), (100, 152, 64), (256, 76, 16), (256, 76, 24)])
def test_split_plan_covers_every_k_block_once_and_shortens_the_last_round(tkg, tiles, clusters, num_kb):
    (st, ss), cover, busiest, pieces = simulate_static(tkg, tiles, clusters, num_kb)
    assert (cover == 1).all()  # every tile's K blocks, exactly once
    rounds = -(-tiles // clusters)
    tail = tiles - (rounds - 1) * clusters
    if st:
        assert st == tail and 2 <= ss <= 4 and st * ss <= clusters and num_kb // ss >= 16
        assert busiest == pytest.approx(rounds - 1 + 1 / ss, abs=1e-9)
        # the pieces of one tile run side by side in the first round
        for tile, s, kb0, kb1 in pieces:
            assert kb0 == s * num_kb // ss and kb1 == (s + 1) * num_kb // ss
    else:
        assert ss == 1
        assert (2 * tail > clusters or min(clusters // tail, 4, num_kb // 16) < 2 or clusters < 2
                or (rounds == 1 and num_kb < 48))
        assert busiest == pytest.approx(rounds)


def test_split_plan_bf16_4096_example(tkg):
    # 4096^3 bf16 with 256x256 pair tiles: 256 tiles, 76 pairs, 64 K stages of 64
    assert tkg.tkg_debug_split_plan(256, 76, 64) == (28, 2)
    # pieces keep at least 16 K stages: K = 1024 (16 stages) is not split, K = 2048 is
    assert tkg.tkg_debug_split_plan(256, 76, 16) == (0, 1)
    assert tkg.tkg_debug_split_plan(256, 76, 32) == (28, 2)
    # one round of 16 tiles on 76 pairs: nothing hides the fix-up, so tiles need 48 stages
    assert tkg.tkg_debug_split_plan(16, 76, 32) == (0, 1)
    assert tkg.tkg_debug_split_plan(16, 76, 48) == (16, 3)
    assert tkg.tkg_debug_split_plan(16, 76, 64) == (16, 4)
    assert tkg.tkg_debug_work_item(0, 28, 2, 64) == (0, 0, 32, 0)
    assert tkg.tkg_debug_work_item(1, 28, 2, 64) == (0, 32, 64, 1)
    assert tkg.tkg_debug_work_item(56, 28, 2, 64) == (28, 0, 64, -1)
    assert tkg.tkg_debug_work_item(283, 28, 2, 64) == (255, 0, 64, -1)


@pytest.mark.parametrize("tiles_m,tiles_n,group_m", [(1, 1, 8), (16, 16, 8), (32, 32, 8), (64, 32, 12),
                                                     (13, 7, 8), (7, 13, 8), (5, 3, 1), (3, 5, 100), (33, 1, 8)])
def test_tile_order_visits_every_tile_once(tkg, tiles_m, tiles_n, group_m):
    seen = np.zeros((tiles_m, tiles_n), dtype=np.int32)
    for t in range(tiles_m * tiles_n):
        tm, tn = tkg.tkg_debug_tile_coord(t, tiles_m, tiles_n, group_m)
        assert 0 <= tm < tiles_m and 0 <= tn < tiles_n
        seen[tm, tn] += 1
    assert (seen == 1).all()


def test_tile_order_is_grouped(tkg):
    # inside a super-row the M index runs fastest: the first G tiles share tile-column 0
    G = 8
    coords = [tkg.tkg_debug_tile_coord(t, 32, 32, G) for t in range(2 * G)]
    assert [c[0] for c in coords[:G]] == list(range(G))
    assert all(c[1] == 0 for c in coords[:G]) and all(c[1] == 1 for c in coords[G:2 * G])
    # a persistent wave of 76 tile pairs touches 8 tile-rows and ~10 tile-columns, not 76 columns
    wave = {tkg.tkg_debug_tile_coord(t, 32, 32, G) for t in range(76)}
    assert len({m for m, _ in wave}) == 8 and len({n for _, n in wave}) <= 10


@pytest.mark.parametrize("s", [0, 32, 64, 128])
def test_device_swizzle_functor_matches_definition(tkg, s):
    for off in range(0, 4096, 4):
        assert tkg.tkg_debug_swizzle_offset(off, s) == sw.swizzle(off, s)


def test_swizzle_selection_matches_definition(tkg):
    for rb in range(16, 1040, 16):
        assert tkg.tkg_debug_select_swizzle(rb) == sw.select_swizzle(rb)


def test_compiled_variants_fit_the_sm(tkg):
    compiled = {0: (2, 15), 1: (2, 15), 2: (14,)}
    for kind in (0, 1, 2):
        for v in range(1, 17):
            if v not in compiled[kind]:
                with pytest.raises(tkg.TkgError):
                    tkg.tkg_debug_variant_info(kind, v)
                continue
            info = tkg.tkg_debug_variant_info(kind, v)
            assert info["smem_bytes"] <= 232448
            assert info["threads"] in (192, 512)
            assert info["cta_group"] == 2
            assert info["tile_m"] == 256
            assert info["tile_n"] == (512 if v == 15 else 256)


@pytest.mark.parametrize("sms", [152, 148, 132, 76])
def test_default_tile_follows_the_device_sm_count(tkg, sms):
    # bf16 / FP8 take the 256x512 tile for K >= 2048 once its tiles fill four rounds of the
    # device's CTA pairs (SMs / 2), else the 256x256 tile; NVFP4 always its one variant
    need = 4 * (sms // 2)
    for kind in (0, 1):
        for M, N in [(8192, 8192), (4096, 4096), (16384, 8192)]:
            wide = -(-M // 256) * -(-N // 512)
            want = 15 if wide >= need else 2
            assert tkg.tkg_debug_pick_variant(kind, M, N, 8192, sms) == want, (kind, M, N, sms)
            assert tkg.tkg_debug_pick_variant(kind, M, N, 2048, sms) == want, (kind, M, N, sms)
            assert tkg.tkg_debug_pick_variant(kind, M, N, 1024, sms) == 2
    assert tkg.tkg_debug_pick_variant(2, 16384, 16384, 16384, sms) == 14


def test_quantize_arguments_checked_before_any_gpu_work(tkg):
    x, q, sf, s = 4096, 8192, 12288, 16384  # never dereferenced: every call below fails validation
    for rows, cols in [(0, 16), (4, 0), (4, 24), (-1, 16)]:
        assert tkg.lib.tkg_quantize_fp8(rows, cols, x, q, s, None) == tkg.TKG_ERR_INVALID_ARG
        assert tkg.lib.tkg_quantize_nvfp4(rows, cols, x, q, sf, s, None) == tkg.TKG_ERR_INVALID_ARG
    assert tkg.lib.tkg_quantize_fp8(4, 16, None, q, s, None) == tkg.TKG_ERR_INVALID_ARG
    assert tkg.lib.tkg_quantize_nvfp4(4, 16, x, q, None, s, None) == tkg.TKG_ERR_INVALID_ARG
    assert tkg.lib.tkg_quantize_fp8(4, 16, x + 4, q, s, None) == tkg.TKG_ERR_MISALIGNED
    assert tkg.lib.tkg_quantize_nvfp4(4, 16, x, q + 8, sf, s, None) == tkg.TKG_ERR_MISALIGNED
    assert tkg.lib.tkg_quantize_fp8(4, 16, x, q, s + 2, None) == tkg.TKG_ERR_MISALIGNED


def test_attention_arguments_checked_before_any_gpu_work(tkg):
    f = tkg.lib.tkg_attention_fwd
    A = 1 << 12
    assert f(1, 1, 128, 128, 96, A, A, A, A, None, None) == tkg.TKG_ERR_INVALID_ARG    # head dim
    assert f(0, 1, 128, 128, 128, A, A, A, A, None, None) == tkg.TKG_ERR_INVALID_ARG   # empty batch
    assert f(1, 1, 0, 128, 128, A, A, A, A, None, None) == tkg.TKG_ERR_INVALID_ARG     # no queries
    assert f(1, 1, 128, 0, 128, A, A, A, A, None, None) == tkg.TKG_ERR_INVALID_ARG     # no keys
    assert f(256, 256, 128, 128, 64, A, A, A, A, None, None) == tkg.TKG_ERR_INVALID_ARG  # B*H > 65535
    assert f(1, 1, 128, 128, 64, None, A, A, A, None, None) == tkg.TKG_ERR_INVALID_ARG
    assert f(1, 1, 128, 128, 64, A + 8, A, A, A, None, None) == tkg.TKG_ERR_MISALIGNED
    assert f(1, 1, 128, 128, 64, A, A, A, A, A + 2, None) == tkg.TKG_ERR_MISALIGNED   # lse alignment
