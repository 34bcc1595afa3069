"""Shared-memory swizzle and bank-conflict model — TEST INFRASTRUCTURE ONLY.

Restates, in plain Python, the three XOR swizzles of the ThunderKittens shared
tiles and the bank-conflict model used to justify them:

* Swizzle of a byte address for an S-byte swizzle (S in {32, 64, 128}):
  the 16-byte chunk index (address bits 4 and up) is XOR-ed with the row index
  taken from address bits 7 and up, modulo S/16 chunks — i.e.
  addr ^ (((addr mod 8S) >> 7) << 4).  (Paper summary, "Shared Memory Tiles:
  Automated Swizzling", the 32/64/128-byte list; the 128-byte case is the same
  as addr ^ (((addr >> 7) & 7) << 4) in the blog's model, "Warp level".)
* Selection: the widest of 128/64/32 bytes that the tile's row width in bytes
  is a multiple of (same section; blog "Warp level").
* Bank model: 32 banks of 4 bytes; a warp of 32 threads each supplies one
  16-byte row address, served in 4 phases of 8 threads; the conflict degree
  of a phase is the largest number of accesses landing in one bank (blog,
  "Warp level", the modelled load).
"""

BANKS = 32


def swizzle(addr: int, s_bytes: int) -> int:
    if s_bytes == 0:
        return addr
    assert s_bytes in (32, 64, 128)
    return addr ^ (((addr % (s_bytes * 8)) >> 7) << 4)


def select_swizzle(row_bytes: int) -> int:
    for s in (128, 64, 32):
        if row_bytes % s == 0:
            return s
    return 0


def bank(addr: int) -> int:
    return (addr // 4) % BANKS


def max_conflict(row_stride: int, s_bytes: int = 0) -> int:
    worst = 0
    for phase in range(4):
        counts = {}
        for t in range(phase * 8, phase * 8 + 8):
            a = swizzle(t * row_stride, s_bytes)
            for w in range(4):
                b = bank(a + 4 * w)
                counts[b] = counts.get(b, 0) + 1
        worst = max(worst, max(counts.values()))
    return worst
