"""Shared-memory swizzle and bank-conflict model — TEST INFRASTRUCTURE ONLY.

Restates, in plain Python, the three XOR swizzles of the ThunderKittens shared
tiles and a bank-conflict count written from the shared-memory bank
definition, to check the swizzles against the conflict degrees the pages print:

* Swizzle of a byte address for an S-byte swizzle (S in {32, 64, 128}):
  the 16-byte chunk index (address bits 4 and up) is XOR-ed with the row index
  taken from address bits 7 and up, modulo S/16 chunks — i.e.
  addr ^ (((addr mod 8S) >> 7) << 4).  (Paper summary "ThunderKittens: Simple,
  Fast, and Adorable AI Kernels", section "Shared Memory Tiles: Automated
  Swizzling", the 32/64/128-byte list; for S = 128 this is the XOR of bits 4-6
  with bits 7-9 in the blog "ThunderKittens: 16x16 Tiles, ...", section
  "Warp level".)
* Selection: the widest of 128/64/32 bytes that the tile's row width in bytes
  is a multiple of (same section; blog "Warp level").
* Bank conflicts, from the definition of the banks: shared memory is 32 banks
  of 4-byte words, word w living in bank w mod 32, so 128 consecutive bytes
  touch every bank once.  A 16-byte (128-bit) access that starts on a 16-byte
  boundary covers exactly one group of 4 adjacent banks, group
  (address / 16) mod 8.  The 32 lanes' 16-byte accesses are served 128 bytes
  at a time, i.e. in wavefronts of 8 lanes; inside a wavefront, lanes that
  name the same 16 bytes are served together, and distinct 16-byte words that
  fall in the same bank group are served one after another.  The conflict
  degree of the access is the largest such count in any wavefront (1 =
  conflict-free).  The access modelled is the one the blog uses: lane t reads
  the first 16 bytes of row t of a tile whose rows are `row_stride` bytes
  apart.
"""

NUM_BANKS = 32
BANK_WIDTH = 4                                   # bytes per bank word
ACCESS_BYTES = 16                                # one 128-bit access per lane
BANKS_PER_ACCESS = ACCESS_BYTES // BANK_WIDTH    # 4
BANK_GROUPS = NUM_BANKS // BANKS_PER_ACCESS      # 8 groups of 4 banks
LANES_PER_WAVEFRONT = BANK_GROUPS                # 8 lanes x 16 B = one pass over the banks
WARP_LANES = 32


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


def bank_of(byte_addr: int) -> int:
    """Bank holding the 4-byte word that contains `byte_addr`."""
    return (byte_addr // BANK_WIDTH) % NUM_BANKS


def bank_group(byte_addr: int) -> int:
    """The group of 4 adjacent banks a 16-byte-aligned 16-byte access covers."""
    assert byte_addr % ACCESS_BYTES == 0, "16-byte accesses start on 16-byte boundaries"
    return bank_of(byte_addr) // BANKS_PER_ACCESS


def conflict_degree(lane_addrs) -> int:
    """Worst number of serialised passes over one bank group, over the
    wavefronts of a warp whose lanes make the given 16-byte accesses."""
    lane_addrs = list(lane_addrs)
    worst = 1
    for w0 in range(0, len(lane_addrs), LANES_PER_WAVEFRONT):
        words_per_group = [set() for _ in range(BANK_GROUPS)]
        for a in lane_addrs[w0:w0 + LANES_PER_WAVEFRONT]:
            words_per_group[bank_group(a)].add(a)
        worst = max(worst, max(len(words) for words in words_per_group))
    return worst


def row_load_conflict(row_stride: int, s_bytes: int = 0) -> int:
    """Conflict degree of lane t reading the first 16 bytes of row t (t < 32)
    of a tile with `row_stride`-byte rows, stored with the S-byte swizzle."""
    return conflict_degree(swizzle(lane * row_stride, s_bytes) for lane in range(WARP_LANES))
