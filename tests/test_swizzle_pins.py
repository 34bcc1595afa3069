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
    assert sw.max_conflict(128, s) == degree


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
