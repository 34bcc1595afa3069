"""Seeded synthetic inputs for the dense tiled GEMM  C = A·Bᵀ.

This module only *makes operands*: random draws and their encoding into the
byte formats the GEMM consumes (bf16, FP8 e4m3 with a per-tensor scale, NVFP4
= e2m1 with an e4m3 scale per 16 K-elements plus an fp32 per-tensor scale).
It contains no GEMM arithmetic; both the CUDA path and the CPU oracle consume
exactly the bytes produced here.

Encodings follow the public format definitions:
  * bf16: the upper 16 bits of an IEEE fp32, rounded to nearest, ties to even.
  * e4m3 ("fn" variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits, no
    infinities, 0x7F/0xFF are NaN, largest finite magnitude 448 (0x7E).
  * e2m1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; magnitudes
    {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
Rounding into e4m3/e2m1 is round-to-nearest, ties to the even code, saturating
at the largest finite magnitude.

Workload shapes and value distributions are those of the ThunderKittens GEMM
study (square 4096-16384 problems, Table 1-3 of "ThunderKittens: Simple,
Fast, and Adorable AI Kernels") extended with the FP8 / NVFP4 block-scaled
variants the Rubin article describes ("ThunderKittens reaches 22.4 PFLOPS on
NVIDIA Rubin", NVFP4 paragraph).
"""
from __future__ import annotations

import dataclasses
import hashlib

import numpy as np

# --------------------------------------------------------------------------
# format value tables (built from the bit-field definitions)
# --------------------------------------------------------------------------


def _e4m3_positive_values() -> np.ndarray:
    """Values of the 127 non-negative finite e4m3 codes 0x00..0x7E (ascending)."""
    vals = np.empty(127, dtype=np.float64)
    for code in range(127):
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0:
            vals[code] = (m / 8.0) * 2.0 ** (1 - 7)
        else:
            vals[code] = (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


def _e2m1_positive_values() -> np.ndarray:
    vals = np.empty(8, dtype=np.float64)
    for code in range(8):
        e = (code >> 1) & 0x3
        m = code & 0x1
        vals[code] = (m / 2.0) if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1)
    return vals


E4M3_POS = _e4m3_positive_values()
E2M1_POS = _e2m1_positive_values()
E4M3_MAX = float(E4M3_POS[-1])  # 448
E2M1_MAX = float(E2M1_POS[-1])  # 6


def _encode_nearest_even(x: np.ndarray, table: np.ndarray, sign_bit: int, dtype) -> np.ndarray:
    """Round |x| to the nearest entry of an ascending magnitude table (ties to
    the even code, saturating at the last entry) and attach the sign bit."""
    x = np.asarray(x, dtype=np.float64)
    mag = np.abs(x)
    hi = np.searchsorted(table, mag, side="left")
    hi = np.clip(hi, 0, len(table) - 1)
    lo = np.clip(hi - 1, 0, len(table) - 1)
    d_lo = mag - table[lo]
    d_hi = table[hi] - mag
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((hi & 1) == 0))
    code = np.where(take_hi, hi, lo)
    code = np.where(mag >= table[-1], len(table) - 1, code)  # saturate
    neg = np.signbit(x) & (code != 0)
    return (code | (neg.astype(np.int64) << sign_bit)).astype(dtype)


def encode_e4m3_table(x: np.ndarray) -> np.ndarray:
    """fp values -> e4m3 codes by nearest-table-entry search (slow, plain)."""
    return _encode_nearest_even(x, E4M3_POS, 7, np.uint8)


def encode_e2m1_table(x: np.ndarray) -> np.ndarray:
    return _encode_nearest_even(x, E2M1_POS, 3, np.uint8)


_CHUNK = 1 << 22


def encode_e4m3(x: np.ndarray) -> np.ndarray:
    """fp values -> e4m3 codes (uint8), round to nearest even, saturating to ±448.

    Inside one binade [2^e, 2^(e+1)) the e4m3 grid is uniform with step
    2^(e-3) (2^-9 below 2^-6, the subnormal range), so rounding |x| / step to
    the nearest integer with ties to even (np.rint) is round-to-nearest-even on
    the grid; an integer of 16 is the first value of the next binade."""
    x = np.asarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    flat_in, flat_out = x.reshape(-1), out.reshape(-1)
    for s in range(0, flat_in.size, _CHUNK):
        a = np.abs(flat_in[s:s + _CHUNK])
        neg = np.signbit(flat_in[s:s + _CHUNK])
        a = np.minimum(a, np.float32(E4M3_MAX))
        e = ((a.view(np.int32) >> 23) & 0xFF) - 127
        e = np.maximum(e, -6)  # subnormals share the step of the first normal binade
        step_exp = (e - 3).astype(np.int32)
        r = np.rint(np.ldexp(a, -step_exp)).astype(np.int32)  # exact scaling by a power of two
        sub = e == -6
        # normal: r in [8, 16]; r == 16 carries into the next binade
        carry = r >= 16
        en = np.where(carry, e + 1, e)
        rn = np.where(carry, 8, r)
        code_norm = ((en + 7) << 3) | (rn - 8)
        code = np.where(sub & (r < 8), r, np.where(sub, 8 + (r - 8), code_norm))
        code = np.minimum(code, 0x7E)
        code = np.where(neg & (code != 0), code | 0x80, code)
        flat_out[s:s + _CHUNK] = code.astype(np.uint8)
    return out


_E2M1_FROM_HALVES = np.full(13, 255, dtype=np.uint8)
for _c, _v in enumerate([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]):
    _E2M1_FROM_HALVES[int(_v * 2)] = _c


def encode_e2m1(x: np.ndarray) -> np.ndarray:
    """fp values -> e2m1 codes (uint8 in 0..15), round to nearest even, saturating to ±6.

    Grid steps: 0.5 below 2, 1 in [2, 4), 2 from 4 up; as for e4m3 the rounded
    multiple of the step is the nearest-even grid value."""
    x = np.asarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    flat_in, flat_out = x.reshape(-1), out.reshape(-1)
    for s in range(0, flat_in.size, _CHUNK):
        v = flat_in[s:s + _CHUNK]
        a = np.abs(v)
        step = np.where(a < 2, np.float32(0.5), np.where(a < 4, np.float32(1.0), np.float32(2.0)))
        q = np.minimum(np.rint(a / step) * step, np.float32(E2M1_MAX))
        code = _E2M1_FROM_HALVES[(q * 2).astype(np.int32)]
        code = np.where(np.signbit(v) & (code != 0), code | 0x8, code)
        flat_out[s:s + _CHUNK] = code.astype(np.uint8)
    return out


def e4m3_value(codes: np.ndarray) -> np.ndarray:
    """Magnitude-with-sign of e4m3 codes (used to form block scales)."""
    codes = np.asarray(codes, dtype=np.int64)
    mag = E4M3_POS[np.minimum(codes & 0x7F, 126)]
    return np.where(codes & 0x80, -mag, mag)


def encode_bf16(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even. No NaN inputs."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def pack_fp4(codes: np.ndarray) -> np.ndarray:
    """[rows, K] e2m1 codes -> [rows, K/2] bytes; element 2j in the low nibble
    of byte j, element 2j+1 in the high nibble."""
    codes = np.asarray(codes, dtype=np.uint8)
    assert codes.shape[-1] % 2 == 0
    lo = codes[..., 0::2] & 0xF
    hi = codes[..., 1::2] & 0xF
    return (lo | (hi << 4)).astype(np.uint8)


def unpack_fp4(packed: np.ndarray) -> np.ndarray:
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out


# --------------------------------------------------------------------------
# quantisers (input encoding only)
# --------------------------------------------------------------------------


def _rowwise(x: np.ndarray, out_shapes, fn):
    """Apply fn(rows_in) -> tuple of row blocks to row chunks of x in parallel."""
    rows, K = x.shape
    outs = [np.empty(shape, dtype=dt) for shape, dt in out_shapes]
    ch = _chunk_rows(K)

    def work(c):
        r0, r1 = c * ch, min(rows, (c + 1) * ch)
        for o, v in zip(outs, fn(x[r0:r1])):
            o[r0:r1] = v

    with _pool() as ex:
        list(ex.map(work, range((rows + ch - 1) // ch)))
    return outs


def quantize_fp8(x: np.ndarray):
    """Per-tensor FP8: scale so max|x| maps to 448, cast to e4m3.

    Returns (codes uint8, dequant_scale float32) with dequant_scale = amax/448,
    so that value ≈ e4m3(code) * dequant_scale.
    """
    x = np.asarray(x, dtype=np.float32)
    amax = float(np.max(np.abs(x))) if x.size else 0.0
    if amax == 0.0:
        return encode_e4m3(x), np.float32(1.0)
    sq = np.float32(E4M3_MAX / amax)
    (codes,) = _rowwise(x, [(x.shape, np.uint8)], lambda xr: (encode_e4m3(xr * sq),))
    return codes, np.float32(amax / E4M3_MAX)


def _block_amax16(xb: np.ndarray) -> np.ndarray:
    a = np.abs(xb)
    a = np.maximum(a[..., :8], a[..., 8:])
    a = np.maximum(a[..., :4], a[..., 4:])
    a = np.maximum(a[..., :2], a[..., 2:])
    return np.maximum(a[..., 0], a[..., 1])


def quantize_nvfp4(x: np.ndarray):
    """NVFP4 two-level block scaling along the last (K) axis.

    g = amax_tensor / (6·448); per 16-element block sb = e4m3(amax_block/(6·g));
    q = e2m1(x / (e4m3(sb)·g)); a block whose scale decodes to 0 gets q = 0.
    Returns (packed uint8 [rows, K/2], block scales uint8 [rows, K/16], g float32).
    """
    x = np.asarray(x, dtype=np.float32)
    rows, K = x.shape
    assert K % 16 == 0
    amax = float(np.max(np.abs(x))) if x.size else 0.0
    g = np.float32(amax / (E2M1_MAX * E4M3_MAX)) if amax > 0 else np.float32(1.0)

    def block(xr):
        xb = xr.reshape(-1, K // 16, 16)
        sb = encode_e4m3(_block_amax16(xb) / np.float32(E2M1_MAX * float(g)))
        sbv = (e4m3_value(sb) * float(g)).astype(np.float32)[..., None]
        scaled = np.zeros_like(xb)
        np.divide(xb, sbv, out=scaled, where=sbv > 0)
        return pack_fp4(encode_e2m1(scaled).reshape(-1, K)), sb

    packed, sb_all = _rowwise(x, [((rows, K // 2), np.uint8), ((rows, K // 16), np.uint8)], block)
    return packed, sb_all, np.float32(g)


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    kind: str  # "bf16" | "fp8" | "nvfp4"
    M: int
    N: int
    K: int
    dist: str  # "uniform" | "normal_sqrtk" | "normal"
    seed_a: int
    seed_b: int
    description: str

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K


WORKLOADS = {
    w.name: w
    for w in [
        Workload("bf16_256", "bf16", 256, 256, 256, "uniform", 1001, 2001,
                 "bf16 GEMM M=N=K=256, U[-1,1] entries, fp32 accumulate, bf16 out"),
        Workload("bf16_4096", "bf16", 4096, 4096, 4096, "normal_sqrtk", 1002, 2002,
                 "bf16 GEMM M=N=K=4096, N(0,1)/sqrt(K) entries, fp32 accumulate, bf16 out"),
        Workload("bf16_8192", "bf16", 8192, 8192, 8192, "normal_sqrtk", 1003, 2003,
                 "bf16 GEMM M=N=K=8192, N(0,1)/sqrt(K) entries, fp32 accumulate, bf16 out"),
        Workload("bf16_skinny", "bf16", 16384, 8192, 2048, "normal_sqrtk", 1013, 2013,
                 "bf16 GEMM M=16384 N=8192 K=2048, N(0,1)/sqrt(K) entries, bf16 out"),
        Workload("fp8_8192", "fp8", 8192, 8192, 8192, "normal", 1004, 2004,
                 "FP8 e4m3 GEMM M=N=K=8192, per-tensor scale to amax=448, bf16 out"),
        Workload("nvfp4_16384", "nvfp4", 16384, 16384, 16384, "normal", 1005, 2005,
                 "NVFP4 GEMM M=N=K=16384, e2m1 + e4m3 per-16 scale + fp32 global, bf16 out"),
    ] + [
        # the K sweep of the persistent-grid study ("Persistent Grid Launch", Table 2): M = N = 4096
        Workload(f"bf16_4096_k{k}", "bf16", 4096, 4096, k, "normal_sqrtk", 1020 + i, 2020 + i,
                 f"bf16 GEMM M=N=4096 K={k}, N(0,1)/sqrt(K) entries, fp32 accumulate, bf16 out")
        for i, k in enumerate((64, 128, 256, 512, 1024))
    ]
}


def _chunk_rows(K: int) -> int:
    return max(1, (1 << 20) // max(K, 1))


def _pool():
    import concurrent.futures as cf
    import os
    return cf.ThreadPoolExecutor(max_workers=min(32, os.cpu_count() or 1))


def _draw(seed: int, rows: int, K: int, dist: str) -> np.ndarray:
    """Seeded draw of a [rows, K] fp32 matrix.  Row chunk c comes from the
    PCG64 stream of `seed` advanced by c jumps, so the result does not depend
    on how many threads fill it."""
    out = np.empty((rows, K), dtype=np.float32)
    ch = _chunk_rows(K)
    base = np.random.PCG64(seed)

    def fill(c):
        rng = np.random.Generator(base.jumped(c))
        r0, r1 = c * ch, min(rows, (c + 1) * ch)
        if dist == "uniform":
            out[r0:r1] = rng.uniform(-1.0, 1.0, size=(r1 - r0, K)).astype(np.float32)
        else:
            rng.standard_normal(size=(r1 - r0, K), dtype=np.float32, out=out[r0:r1])
            if dist == "normal_sqrtk":
                out[r0:r1] *= np.float32(1.0 / np.sqrt(K))

    n = (rows + ch - 1) // ch
    with _pool() as ex:
        list(ex.map(fill, range(n)))
    return out


def draw_fp32(seed: int, rows: int, cols: int, dist: str = "normal") -> np.ndarray:
    """Seeded fp32 [rows, cols] matrix ("uniform" U[-1,1], "normal" N(0,1) or
    "normal_sqrtk" N(0,1)/sqrt(cols)): the input of the FP8 / NVFP4 encoders."""
    return _draw(seed, rows, cols, dist)


@dataclasses.dataclass
class Operands:
    """Raw operand bytes for one GEMM.  a/b are [rows, K] (bf16 bits as uint16,
    e4m3 codes as uint8) or [rows, K/2] packed e2m1; sfa/sfb are [rows, K/16]
    e4m3 block scales (NVFP4 only); scale_a/scale_b are the fp32 per-tensor
    dequantisation scales (FP8, NVFP4; 1.0 for bf16)."""
    kind: str
    M: int
    N: int
    K: int
    a: np.ndarray
    b: np.ndarray
    sfa: np.ndarray | None = None
    sfb: np.ndarray | None = None
    scale_a: float = 1.0
    scale_b: float = 1.0

    def digest(self) -> str:
        h = hashlib.sha256()
        for arr in (self.a, self.b, self.sfa, self.sfb):
            if arr is not None:
                h.update(np.ascontiguousarray(arr).tobytes())
        h.update(np.float32(self.scale_a).tobytes())
        h.update(np.float32(self.scale_b).tobytes())
        return h.hexdigest()


def encode(kind: str, xa: np.ndarray, xb: np.ndarray) -> Operands:
    """Encode two fp32 operand matrices [M,K], [N,K] into the kind's format."""
    M, K = xa.shape
    N = xb.shape[0]
    if kind == "bf16":
        (a,) = _rowwise(xa, [(xa.shape, np.uint16)], lambda r: (encode_bf16(r),))
        (b,) = _rowwise(xb, [(xb.shape, np.uint16)], lambda r: (encode_bf16(r),))
        return Operands(kind, M, N, K, a, b)
    if kind == "fp8":
        a, sa = quantize_fp8(xa)
        b, sb = quantize_fp8(xb)
        return Operands(kind, M, N, K, a, b, scale_a=float(sa), scale_b=float(sb))
    if kind == "nvfp4":
        a, sfa, ga = quantize_nvfp4(xa)
        b, sfb, gb = quantize_nvfp4(xb)
        return Operands(kind, M, N, K, a, b, sfa, sfb, float(ga), float(gb))
    raise ValueError(kind)


def make_operands(kind: str, M: int, N: int, K: int, dist: str, seed_a: int, seed_b: int) -> Operands:
    xa = _draw(seed_a, M, K, dist)
    xb = _draw(seed_b, N, K, dist)
    return encode(kind, xa, xb)


def workload_operands(name: str) -> Operands:
    w = WORKLOADS[name]
    return make_operands(w.kind, w.M, w.N, w.K, w.dist, w.seed_a, w.seed_b)


def small_int_operands(kind: str, M: int, N: int, K: int, seed: int) -> Operands:
    """Operands whose every partial sum is a small integer (or a multiple of
    1/4 for NVFP4 with power-of-two block scales): exact in fp32 under any
    summation order, so GPU and oracle must agree bit for bit."""
    rng = np.random.default_rng(seed)
    if kind == "nvfp4":
        # e2m1 magnitudes {0,1,2} with random sign; block scales in {0.5,1,2}.
        mags = rng.choice(np.array([0.0, 1.0, 2.0]), size=(M, K))
        xa = mags * rng.choice(np.array([-1.0, 1.0]), size=(M, K))
        mags = rng.choice(np.array([0.0, 1.0, 2.0]), size=(N, K))
        xb = mags * rng.choice(np.array([-1.0, 1.0]), size=(N, K))
        sf_choices = encode_e4m3(np.array([0.5, 1.0, 2.0]))
        sfa = rng.choice(sf_choices, size=(M, K // 16)).astype(np.uint8)
        sfb = rng.choice(sf_choices, size=(N, K // 16)).astype(np.uint8)
        return Operands(kind, M, N, K, pack_fp4(encode_e2m1(xa)), pack_fp4(encode_e2m1(xb)),
                        sfa, sfb, 1.0, 1.0)
    xa = rng.integers(-2, 3, size=(M, K)).astype(np.float32)
    xb = rng.integers(-2, 3, size=(N, K)).astype(np.float32)
    if kind == "bf16":
        return Operands(kind, M, N, K, encode_bf16(xa), encode_bf16(xb))
    if kind == "fp8":
        return Operands(kind, M, N, K, encode_e4m3(xa), encode_e4m3(xb), scale_a=1.0, scale_b=1.0)
    raise ValueError(kind)


def permutation_operands(kind: str, M: int, K: int, seed: int, identity: bool = False) -> tuple[Operands, np.ndarray]:
    """A random (generic values), B = a permutation matrix P with B[n, perm[n]] = 1
    (N = K).  The exact product is C[m, n] = A[m, perm[n]]."""
    rng = np.random.default_rng(seed)
    N = K
    perm = np.arange(K) if identity else rng.permutation(K)
    xb = np.zeros((N, K), dtype=np.float32)
    xb[np.arange(N), perm] = 1.0
    if kind == "bf16":
        xa = rng.uniform(-4, 4, size=(M, K)).astype(np.float32)
        return Operands(kind, M, N, K, encode_bf16(xa), encode_bf16(xb)), perm
    if kind == "fp8":
        xa = rng.uniform(-400, 400, size=(M, K)).astype(np.float32)
        return Operands(kind, M, N, K, encode_e4m3(xa), encode_e4m3(xb), scale_a=1.0, scale_b=1.0), perm
    if kind == "nvfp4":
        # distinct magnitudes at even and odd k pin the nibble order
        xa = rng.choice(np.array([0.5, 1.5, 3.0, 6.0, -1.0, -2.0, -4.0]), size=(M, K))
        sfa = encode_e4m3(rng.choice(np.array([0.25, 1.0, 8.0, 96.0]), size=(M, K // 16)))
        sfb = np.full((N, K // 16), encode_e4m3(np.array([1.0]))[0], dtype=np.uint8)
        return Operands(kind, M, N, K, pack_fp4(encode_e2m1(xa)), pack_fp4(encode_e2m1(xb)),
                        sfa, sfb, 1.0, 1.0), perm
    raise ValueError(kind)


# ---------------------------------------------------------------- attention forward inputs

@dataclasses.dataclass(frozen=True)
class AttnWorkload:
    """Non-causal attention forward: Q [B, H, Nq, D], K and V [B, H, Nkv, D],
    bf16 N(0,1) entries (seeded), O [B, H, Nq, D] bf16."""
    name: str
    B: int
    H: int
    Nq: int
    Nkv: int
    D: int
    seed: int
    description: str

    @property
    def flops(self) -> float:
        # two matrix products (Q·Kᵀ and P·V), 2 flops per multiply-add
        return 4.0 * self.B * self.H * self.Nq * self.Nkv * self.D


# Shapes of the pages' attention study (batch 16, 16 heads, head dim 64 / 128,
# sequence lengths from about a thousand to several thousand).
ATTN_WORKLOADS = {
    w.name: w
    for w in [
        AttnWorkload("attn_n1024_d128", 16, 16, 1024, 1024, 128, 3001,
                     "non-causal attention forward B=16 H=16 N=1024 D=128, bf16 N(0,1) Q/K/V, bf16 O"),
        AttnWorkload("attn_n4096_d128", 16, 16, 4096, 4096, 128, 3002,
                     "non-causal attention forward B=16 H=16 N=4096 D=128, bf16 N(0,1) Q/K/V, bf16 O"),
        AttnWorkload("attn_n4096_d64", 16, 16, 4096, 4096, 64, 3003,
                     "non-causal attention forward B=16 H=16 N=4096 D=64, bf16 N(0,1) Q/K/V, bf16 O"),
    ]
}


@dataclasses.dataclass
class AttnInputs:
    """bf16 bit patterns (uint16) of Q [B, H, Nq, D], K and V [B, H, Nkv, D]."""
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray

    @property
    def shape(self):
        B, H, Nq, D = self.q.shape
        return B, H, Nq, self.k.shape[2], D


def attention_inputs(B: int, H: int, Nq: int, Nkv: int, D: int, seed: int, dist: str = "normal") -> AttnInputs:
    """Seeded bf16 Q, K, V (N(0,1) entries by default, rounded to bf16)."""
    def one(s, n):
        x = _draw(s, B * H * n, D, dist)
        (bits,) = _rowwise(x, [(x.shape, np.uint16)], lambda r: (encode_bf16(r),))
        return bits.reshape(B, H, n, D)
    return AttnInputs(one(seed, Nq), one(seed + 1, Nkv), one(seed + 2, Nkv))


def attn_workload_inputs(name: str) -> AttnInputs:
    w = ATTN_WORKLOADS[name]
    return attention_inputs(w.B, w.H, w.Nq, w.Nkv, w.D, w.seed)
