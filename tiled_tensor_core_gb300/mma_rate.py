"""Print the tensor-core issue rate of each MMA kind this library uses.

    python -m tiled_tensor_core_gb300.mma_rate

For every kind (bf16 K=16, e4m3 K=32, block-scaled e2m1 K=64; 32 bytes of K
per operand row each), CTA-group form (one CTA, or a CTA pair with
cta_group::2) and N, one thread issues 128 and then 1024 MMAs back to back
(tkg_debug_mma_rate); the difference gives the cost of one MMA in SM cycles,
and from it the dense rate per SM and, at a given clock, per GPU.  A second
table compares one accumulator with the 2x1 tile (pairs of MMAs sharing A,
two accumulators), with and without reuse of the A collector buffer; the last
compares the operand forms of the attention kernel's P·V product (B MN-major,
A read from tensor memory) with the GEMM's K-major shared operands.
"""
from __future__ import annotations

import argparse

KINDS = {0: ("bf16", 16), 1: ("e4m3", 32), 2: ("nvfp4", 64)}


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--clock-mhz", type=float, default=2070.0, help="SM clock for the per-GPU figure")
    args = ap.parse_args(argv)
    import torch

    from . import tkg

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    print(f"{sms} SMs, per-GPU figures at {args.clock_mhz:.0f} MHz")
    print("| kind | CTA group | MMA (M x N x K) | cycles per MMA | FMA per cycle per SM | TFLOP/s per GPU |")
    print("|---|---|---|---|---|---|")
    for kind, (name, k) in KINDS.items():
        for cg in (1, 2):
            for n in (256, 128):
                c0 = tkg.tkg_debug_mma_rate(kind, cg, n, 128)
                c1 = tkg.tkg_debug_mma_rate(kind, cg, n, 1024)
                per = (c1 - c0) / (1024 - 128)
                fma_sm = 128 * n * k / per  # each SM computes 128 rows of the (128*cg) x n tile
                tflops = 2 * fma_sm * sms * args.clock_mhz * 1e6 / 1e12
                print(f"| {name} | {cg} | {128 * cg} x {n} x {k} | {per:.1f} | {fma_sm:.0f} | {tflops:.0f} |")

    print()
    print("| kind | MMA (M x N x K), one CTA | one accumulator | 2x1: pairs sharing A | 2x1 + collector::a reuse |")
    print("|---|---|---|---|---|")
    for kind, (name, k) in KINDS.items():
        n = 128 if kind == 2 else 256
        cells = []
        for pattern in (0, 1, 2):
            c0 = tkg.tkg_debug_mma_rate(kind, 1, n, 128, pattern)
            c1 = tkg.tkg_debug_mma_rate(kind, 1, n, 1024, pattern)
            cells.append(f"{(c1 - c0) / (1024 - 128):.1f}")
        print(f"| {name} | 128 x {n} x {k} | " + " | ".join(cells) + " |")

    print()
    print("| kind | CTA group | MMA (M x N x K) | MMAs only | + per-stage sync work | commits only | waits only "
          "| fences only | waits, CTA-scope acquire | scale columns moving as in the GEMM | varied operand bits |")
    print("|---|---|---|---|---|---|---|---|---|---|---|")
    for kind, (name, k) in KINDS.items():
        for cg in (1, 2):
            cells = []
            for pattern in (0, 4, 5, 6, 7, 8, 3, 9):
                if pattern == 3 and kind != 2:
                    cells.append("—")
                    continue
                c0 = tkg.tkg_debug_mma_rate(kind, cg, 256, 128, pattern)
                c1 = tkg.tkg_debug_mma_rate(kind, cg, 256, 1024, pattern)
                cells.append(f"{(c1 - c0) / (1024 - 128):.1f}")
            print(f"| {name} | {cg} | {128 * cg} x 256 x {k} | " + " | ".join(cells) + " |")

    print()
    print("| kind | CTA group | cycles per MMA for N = 64, 96, ..., 256 (M = 128 x CTA group) |")
    print("|---|---|---|")
    for kind, (name, k) in KINDS.items():
        for cg in (1, 2):
            cells = []
            for n in range(64, 257, 32):
                c0 = tkg.tkg_debug_mma_rate(kind, cg, n, 128)
                c1 = tkg.tkg_debug_mma_rate(kind, cg, n, 1024)
                cells.append(f"{n}: {(c1 - c0) / (1024 - 128):.1f}")
            print(f"| {name} | {cg} | " + ", ".join(cells) + " |")

    print()
    print("| bf16, one CTA, MMA (M x N x K) | A, B K-major in shared memory | B MN-major | A from tensor memory "
          "| both (attention P·V) |")
    print("|---|---|---|---|---|")
    for n in (128, 256):
        cells = []
        for pattern in (0, 10, 11, 12):
            c0 = tkg.tkg_debug_mma_rate(0, 1, n, 128, pattern)
            c1 = tkg.tkg_debug_mma_rate(0, 1, n, 1024, pattern)
            cells.append(f"{(c1 - c0) / (1024 - 128):.1f}")
        print(f"| 128 x {n} x 16 | " + " | ".join(cells) + " |")
    c0 = tkg.tkg_debug_mma_rate(0, 1, 128, 128, 13)
    c1 = tkg.tkg_debug_mma_rate(0, 1, 128, 1024, 13)
    print()
    print(f"bf16 128 x 128 x 16, groups of 8 alternating between the two forms (as attention issues S and P·V): "
          f"{(c1 - c0) / (1024 - 128):.1f} cycles per MMA")


if __name__ == "__main__":
    main()
