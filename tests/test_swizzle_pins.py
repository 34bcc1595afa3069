"""Pins for the swizzle / bank-conflict model against the numbers the pages
print (tests/golden/bank_conflicts.txt) and against the swizzle's algebra."""
import os

import pytest

from oracle import swizzle as sw

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "bank_conflicts.txt")


def golden_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, degree = line.split()[:2]
        rows.append((name, int(degree)))
    return rows


@pytest.mark.parametrize("name,degree", golden_rows())
def test_conflict_degree_matches_pages(name, degree):
    s = 0 if name == "row_major" else int(name.split("_")[1][:-1])
    assert sw.row_load_conflict(128, s) == degree


def test_conflict_model_special_cases():
    # consecutive 16-byte words: every wavefront covers all 32 banks once
    assert sw.conflict_degree(16 * t for t in range(32)) == 1
    # every lane names the same 16 bytes: served together (broadcast)
    assert sw.conflict_degree([4096] * 32) == 1
    # two lanes per wavefront on the same group but different words: 2 passes
    assert sw.conflict_degree([0, 128] + [16 * t for t in range(2, 8)]) == 2
    # rows 256 B apart: all 8 lanes of a wavefront in bank group 0, 8 passes; the 128-byte
    # swizzle XORs the chunk index with address bits 7-9, and 256 t keeps bit 7 at 0, so it
    # reaches only the even groups 0, 2, 4, 6: two lanes each, 2 passes
    assert sw.row_load_conflict(256, 0) == 8
    assert sw.row_load_conflict(256, 128) == 2
    # rows 144 B apart (a padded 128 B row): the 16-byte offset alone spreads the groups
    assert sw.row_load_conflict(144, 0) == 1


def test_bank_definition():
    assert [sw.bank_of(a) for a in (0, 3, 4, 124, 128, 132)] == [0, 0, 1, 31, 0, 1]
    assert [sw.bank_group(a) for a in (0, 16, 112, 128, 144)] == [0, 1, 7, 0, 1]
    with pytest.raises(AssertionError):
        sw.bank_group(8)


def test_128B_form_equals_blog_form():
    for addr in range(0, 1 << 16, 2):
        assert sw.swizzle(addr, 128) == addr ^ (((addr >> 7) & 7) << 4)


@pytest.mark.parametrize("s", [32, 64, 128])
def test_swizzle_is_a_bijection_on_each_atom(s):
    atom = 8 * s if s else 128
    for base in (0, atom, 7 * atom):
        img = {sw.swizzle(base + a, s) for a in range(0, atom, 16)}
        assert img == set(range(base, base + atom, 16))
        for a in range(atom):  # bytes inside a 16-byte chunk keep their offset
            assert sw.swizzle(base + a, s) % 16 == a % 16


def test_selection_rule():
    # bf16 widths 64/32/16 -> 128/64/32-byte rows; fp8 width 128, fp4 width 256 -> 128 B
    assert sw.select_swizzle(64 * 2) == 128
    assert sw.select_swizzle(32 * 2) == 64
    assert sw.select_swizzle(16 * 2) == 32
    assert sw.select_swizzle(128 * 1) == 128
    assert sw.select_swizzle(256 // 2) == 128
    assert sw.select_swizzle(24) == 0
