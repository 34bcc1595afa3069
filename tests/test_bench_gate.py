"""The benchmark's parity gate (host logic, no GPU): sampled rows cover the tile
edges and every TMEM lane quarter, and the gate accepts the oracle's own output
but rejects an output with one wrong element, a NaN, or a dropped scale."""
import numpy as np
import pytest

import bench
import oracle
from tiled_tensor_core_gb300 import synth


def test_rows_cover_tile_edges_and_quarters():
    for M in (256, 4096, 16384):
        rows = bench.parity_rows(M, seed=1)
        assert len(rows) >= min(M, bench.PARITY_ROWS) and rows.max() < M and rows.min() == 0
        assert {0, 31, 32, 63, 64, 95, 96, 127, 128, 255} <= set(rows.tolist())
        assert M - 1 in rows


def _rows_of(ops, rows):
    acc, c_ref = oracle.gemm(ops, rows=rows)
    return acc, c_ref


@pytest.mark.parametrize("kind", ["bf16", "fp8", "nvfp4"])
def test_gate_accepts_the_oracle_output_and_rejects_a_wrong_one(kind):
    M, N, K = 300, 264, 256
    ops = synth.make_operands(kind, M, N, K, "normal_sqrtk" if kind == "bf16" else "normal", 5, 6)
    rows = bench.parity_rows(M, seed=2)
    _, c_ref = _rows_of(ops, rows)
    assert bench.parity_check(ops, c_ref.copy(), rows)["pass"]
    bad = c_ref.copy()
    # one element off by 0.25: bf16 fails elementwise (1e-2 (|ref| + 1)); FP8 / NVFP4 (Frobenius
    # only) get a whole row scaled instead
    if kind == "bf16":
        f = np.array([(bad[3, 7].astype(np.uint32) << 16)], dtype=np.uint32).view(np.float32) + np.float32(0.25)
        bad[3, 7] = np.uint16(f.view(np.uint32)[0] >> 16)
    else:
        f = (bad[3].astype(np.uint32) << 16).view(np.float32) * np.float32(1.5)
        bad[3] = (f.view(np.uint32) >> 16).astype(np.uint16)
    assert not bench.parity_check(ops, bad, rows)["pass"]
    nan = c_ref.copy()
    nan[0, 0] = 0x7FC0
    assert not bench.parity_check(ops, nan, rows)["pass"]


def test_gate_rejects_a_dropped_tensor_scale():
    ops = synth.make_operands("fp8", 256, 256, 256, "normal", 7, 8)
    rows = bench.parity_rows(256, seed=3)
    acc, _ = _rows_of(ops, rows)
    # the GPU forgot scale_b: bf16 of acc * scale_a only
    x = (acc.astype(np.float64) * ops.scale_a).astype(np.float32)
    u = x.view(np.uint32)
    wrong = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    assert not bench.parity_check(ops, wrong, rows)["pass"]


@pytest.mark.parametrize("name", bench.SUITE + ["bf16_4096_k64", "bf16_4096_k1024"])
def test_timed_launches_never_find_their_operands_in_l2(name):
    # the launches of a step rotate over copies whose combined footprint (operands in, C out) is at
    # least twice the 129 MB L2, so no launch reads what the previous use of its copy left there
    w = synth.WORKLOADS[name]
    a_b = {"bf16": 2 * (w.M + w.N) * w.K, "fp8": (w.M + w.N) * w.K + 8,
           "nvfp4": (w.M + w.N) * w.K // 2 + (w.M + w.N) * w.K // 16 + 8}[w.kind]
    footprint = a_b + 2 * w.M * w.N
    assert bench.operand_sets(footprint) * footprint >= 2 * bench.L2_BYTES
