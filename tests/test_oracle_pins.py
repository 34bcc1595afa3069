"""Pins for the CPU oracle: each test checks it against something other than
itself — an independent decoder (torch's dtype casts), a literal format table,
exact integer arithmetic, the identity/permutation closed forms, or a float64
brute force bounded by the recursive-summation error bound.  A dropped term, a
wrong sign or index, a transposed operand, a swapped nibble or a misapplied
scale in the oracle fails at least one of these.
"""
import numpy as np
import pytest
import torch

from tiled_tensor_core_gb300 import synth

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")

# OCP Microscaling Formats (MX) v1.0, FP4 E2M1 element table: codes 0..7.
E2M1_LITERAL = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


# ---------------------------------------------------------------- decoders

def test_e4m3_spot_values(oracle_mod):
    d = oracle_mod.dec_e4m3(np.array([0x7E, 0x01, 0x38, 0x08, 0x07, 0x00, 0x80, 0xFE, 0x40, 0x30], dtype=np.uint8))
    assert d[0] == 448.0
    assert d[1] == 2.0 ** -9
    assert d[2] == 1.0
    assert d[3] == 2.0 ** -6          # smallest normal
    assert d[4] == 7 * 2.0 ** -9      # largest subnormal
    assert d[5] == 0.0 and d[6] == 0.0 and np.signbit(d[6])
    assert d[7] == -448.0
    assert d[8] == 2.0 and d[9] == 0.5
    nan = oracle_mod.dec_e4m3(np.array([0x7F, 0xFF], dtype=np.uint8))
    assert np.isnan(nan).all()


def test_e4m3_table_matches_torch(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle_mod.dec_e4m3(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    both_nan = np.isnan(mine) & np.isnan(ref)
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    assert np.array_equal(mine[~both_nan].view(np.uint32), ref[~both_nan].view(np.uint32))


def test_e2m1_table_matches_literal(oracle_mod):
    codes = np.arange(16, dtype=np.uint8)
    mine = oracle_mod.dec_e2m1(codes)
    ref = np.concatenate([E2M1_LITERAL, -E2M1_LITERAL]).astype(np.float32)
    assert np.array_equal(mine, ref)


def test_bf16_decode_matches_torch(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = oracle_mod.dec_bf16(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    ok = np.isnan(mine) & np.isnan(ref)
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    assert np.array_equal(mine[~ok].view(np.uint32), ref[~ok].view(np.uint32))


def test_rne_bf16_matches_torch(oracle_mod):
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 4000),
        # exact ties: low half exactly 0x8000, both parities of the kept bit
        (rng.integers(0, 2 ** 31, 2000, dtype=np.uint64).astype(np.uint32) & 0xFFFF0000 | 0x8000).view(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38, 1e-40, -1e-40], dtype=np.float32),
    ]).astype(np.float32)
    x = x[np.isfinite(x)]
    mine = oracle_mod.rne_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)


def test_nvfp4_decode_nibble_order_and_scale(oracle_mod):
    # byte 0x21 holds element 0 = code 1 (0.5) in the low nibble, element 1 = code 2 (1.0) high
    packed = np.array([[0x21] * 8], dtype=np.uint8)
    sf = np.array([synth.encode_e4m3(np.array([4.0]))[0]], dtype=np.uint8).reshape(1, 1)
    d = oracle_mod.dec_nvfp4(packed, sf, 16)
    assert np.array_equal(d[0, 0::2], np.full(8, 2.0, np.float32))   # 0.5 * 4
    assert np.array_equal(d[0, 1::2], np.full(8, 4.0, np.float32))   # 1.0 * 4


# ---------------------------------------------------------- independent decode

def ref_decode(ops):
    """Float64 decode of an Operands bundle without the oracle's tables."""
    if ops.kind == "bf16":
        f = lambda x: torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
        return f(ops.a), f(ops.b), 1.0, 1.0
    e4 = lambda x: torch.from_numpy(np.ascontiguousarray(x)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    if ops.kind == "fp8":
        return e4(ops.a), e4(ops.b), ops.scale_a, ops.scale_b
    table = np.concatenate([E2M1_LITERAL, -E2M1_LITERAL])

    def fp4(packed, sf):
        codes = synth.unpack_fp4(packed)
        return table[codes] * np.repeat(e4(sf), 16, axis=1)

    return fp4(ops.a, ops.sfa), fp4(ops.b, ops.sfb), ops.scale_a, ops.scale_b


def bf16_bits_to_f64(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


KINDS = ["bf16", "fp8", "nvfp4"]


# ---------------------------------------------------------- closed forms

@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("identity", [True, False])
def test_identity_and_permutation(oracle_mod, kind, identity):
    M, K = 48, 64
    ops, perm = synth.permutation_operands(kind, M, K, seed=11, identity=identity)
    acc, C = oracle_mod.gemm(ops)
    a64, _, _, _ = ref_decode(ops)
    expect = a64[:, perm]                       # C[m, n] = A[m, perm[n]]
    assert np.array_equal(acc.astype(np.float64), expect)
    # every such value is exactly representable in bf16
    assert np.array_equal(bf16_bits_to_f64(C), expect)


@pytest.mark.parametrize("kind", ["bf16", "fp8"])
def test_a_identity_gives_b_transposed(oracle_mod, kind):
    # A = I (M = K): C[m, n] = B[n, m]
    K = 32
    ops_b, _ = synth.permutation_operands(kind, 40, K, seed=5)
    b_vals = ops_b.a                              # generic [40, K] values become B
    eye = synth.encode_bf16(np.eye(K, dtype=np.float32)) if kind == "bf16" else synth.encode_e4m3(np.eye(K))
    ops = synth.Operands(kind, K, 40, K, eye, b_vals)
    acc, C = oracle_mod.gemm(ops)
    _, b64, _, _ = ref_decode(ops)
    assert np.array_equal(acc.astype(np.float64), b64.T)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("shape", [(16, 24, 32), (33, 17, 256), (64, 64, 128)])
def test_small_integers_exact(oracle_mod, kind, shape):
    M, N, K = shape
    ops = synth.small_int_operands(kind, M, N, K, seed=M * 1000 + N * 10 + K)
    acc, C = oracle_mod.gemm(ops)
    a64, b64, _, _ = ref_decode(ops)
    exact = a64 @ b64.T                           # exact: every term is a multiple of 1/4, |sum| < 2^13
    assert np.array_equal(acc.astype(np.float64), exact)
    ref_c = torch.from_numpy(exact).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(C, ref_c)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("shape", [(8, 8, 32), (31, 29, 64), (64, 48, 64)])
def test_f64_bruteforce_within_summation_bound(oracle_mod, kind, shape):
    M, N, K = shape
    ops = synth.make_operands(kind, M, N, K, "normal", 100 + M, 200 + N)
    acc, C = oracle_mod.gemm(ops)
    a64, b64, sa, sb = ref_decode(ops)
    exact = a64 @ b64.T
    absprod = np.abs(a64) @ np.abs(b64).T
    u = 2.0 ** -24
    gamma = K * u / (1 - K * u)
    err = np.abs(acc.astype(np.float64) - exact)
    assert np.all(err <= gamma * absprod), float((err / np.maximum(gamma * absprod, 1e-300)).max())
    # output: scaled, then rounded once to bf16 (half an ulp = 2^-8 relative)
    ref_out = exact * sa * sb
    out = bf16_bits_to_f64(C)
    bound = gamma * absprod * sa * sb + 2.0 ** -8 * np.abs(ref_out) + 4 * u * np.abs(ref_out) + 1e-30
    assert np.all(np.abs(out - ref_out) <= bound)
    # and the bf16 is exactly the nearest-even rounding of the scaled fp32 accumulator
    scaled = (acc * np.float32(sa)).astype(np.float32) * np.float32(sb)
    ref_c = torch.from_numpy(scaled.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(C, ref_c)


@pytest.mark.parametrize("kind", KINDS)
def test_row_subset_matches_full(oracle_mod, kind):
    ops = synth.make_operands(kind, 40, 24, 64, "normal", 3, 4)
    acc, C = oracle_mod.gemm(ops)
    rows = np.array([39, 0, 17, 17, 5])
    acc_r, C_r = oracle_mod.gemm(ops, rows=rows)
    assert np.array_equal(acc_r, acc[rows])
    assert np.array_equal(C_r, C[rows])


def test_nvfp4_scale_pins_block_index(oracle_mod):
    # Two blocks along K with scales 1 and 8; B = all ones with scale 1.
    # A's block-1 elements must be multiplied by 8, block-0 ones by 1.
    K = 32
    one, two = synth.encode_e2m1(np.array([1.0, 2.0]))
    codes = np.full((1, K), one, dtype=np.uint8)
    codes[0, 16:] = two
    sfa = synth.encode_e4m3(np.array([[1.0, 8.0]]))
    b = synth.pack_fp4(np.full((1, K), one, dtype=np.uint8))
    sfb = synth.encode_e4m3(np.array([[1.0, 1.0]]))
    acc, _ = oracle_mod.gemm_nvfp4(synth.pack_fp4(codes), b, sfa, sfb, 1.0, 1.0)
    assert acc[0, 0] == 16 * 1.0 + 16 * 16.0


def test_fp8_scales_applied_to_both_operands(oracle_mod):
    ops = synth.small_int_operands("fp8", 8, 8, 32, seed=3)
    acc, _ = oracle_mod.gemm_fp8(ops.a, ops.b, 1.0, 1.0)
    _, C = oracle_mod.gemm_fp8(ops.a, ops.b, 0.5, 4.0)
    ref = torch.from_numpy(acc.astype(np.float64) * 2.0).to(torch.float32).to(torch.bfloat16)
    assert np.array_equal(C, ref.view(torch.int16).numpy().view(np.uint16))
