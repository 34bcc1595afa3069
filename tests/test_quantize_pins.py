"""Pins for the oracle's FP8 / NVFP4 encoders (oracle/quantize.c), each against
something other than the encoder itself: torch's float8_e4m3fn cast, a brute
force nearest-value search over the format tables (which are pinned in
test_oracle_pins.py), closed forms for inputs that are exactly representable,
and the project's independent numpy encoder used to generate GEMM inputs
(synth.quantize_fp8 / quantize_nvfp4), which follows the same reading with
separately written code.  A wrong rounding direction, a lost sign, a missing
saturation, a swapped nibble, a misplaced block or a mis-ordered scale
operation fails one of these.
"""
import numpy as np
import pytest
import torch

from tiled_tensor_core_gb300 import synth

E2M1_LITERAL = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _e4m3_positive_values(oracle_mod):
    codes = np.arange(0, 0x7F, dtype=np.uint8)  # 0x00..0x7E, all finite non-negative codes
    return codes, oracle_mod.dec_e4m3(codes).astype(np.float64)


def test_e4m3_encoder_matches_torch_cast(oracle_mod):
    rng = np.random.default_rng(11)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(50.0),
        rng.uniform(-448, 448, 20000).astype(np.float32),
        (rng.standard_normal(5000) * 1e-3).astype(np.float32),
    ])
    ours = oracle_mod.e4m3_rne_sat(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    zero = (ours & 0x7F) == 0
    assert np.array_equal(ours[~zero], ref[~zero])
    assert np.all((ref[zero] & 0x7F) == 0)
    assert np.array_equal(ours[zero] >> 7, np.signbit(x[zero]).astype(np.uint8))


def test_e4m3_encoder_is_nearest_with_ties_to_even(oracle_mod):
    codes, vals = _e4m3_positive_values(oracle_mod)
    # every representable value maps to itself
    assert np.array_equal(oracle_mod.e4m3_rne_sat(vals.astype(np.float32)), codes)
    # midpoints of neighbours go to the even code; points just inside go to the nearer one
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    assert np.all(mids.astype(np.float64) == (vals[:-1] + vals[1:]) / 2)  # exact in fp32
    got = oracle_mod.e4m3_rne_sat(mids)
    want = np.where(codes[:-1] % 2 == 0, codes[:-1], codes[1:])
    assert np.array_equal(got, want)
    below = np.nextafter(mids, np.float32(0)).astype(np.float32)
    above = np.nextafter(mids, np.float32(np.inf)).astype(np.float32)
    assert np.array_equal(oracle_mod.e4m3_rne_sat(below), codes[:-1])
    assert np.array_equal(oracle_mod.e4m3_rne_sat(above), codes[1:])


def test_e4m3_encoder_saturates_and_keeps_sign(oracle_mod):
    x = np.array([448.0, 449.0, 464.0, 480.0, 1e30, -449.0, -1e30, -0.0, -1e-30, 1e-30], dtype=np.float32)
    assert list(oracle_mod.e4m3_rne_sat(x)) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x80, 0x80, 0x00]


def test_e2m1_encoder_against_brute_force(oracle_mod):
    x = np.concatenate([np.linspace(-7, 7, 2801), np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])]).astype(np.float32)
    got = oracle_mod.e2m1_rne_sat(x)
    a = np.abs(x.astype(np.float64))
    dist = np.abs(a[:, None] - E2M1_LITERAL[None, :])
    code = []
    for ai, di in zip(a, dist):
        idx = np.flatnonzero(di == di.min())       # the nearest magnitudes
        if ai >= 6.0:
            code.append(7)                         # saturate at 6
        elif idx.size > 1:
            code.append(idx[idx % 2 == 0][0])      # a tie goes to the even code
        else:
            code.append(idx[0])
    want = (np.array(code) | (np.signbit(x).astype(np.int64) << 3)).astype(np.uint8)
    assert np.array_equal(got, want)


def test_fp8_quantize_closed_forms(oracle_mod):
    # amax a power of two times 448: the scale is a power of two, products exact
    codes, vals = _e4m3_positive_values(oracle_mod)
    t = np.float32(2.0 ** -5)
    x = np.concatenate([vals, -vals[1:]]).astype(np.float32) * t
    x = x.reshape(1, -1)
    q, s = oracle_mod.quantize_fp8(x)
    assert s == np.float32(448.0) * t / np.float32(448.0)
    assert np.array_equal(q[0, :codes.size], codes)
    assert np.array_equal(q[0, codes.size:], codes[1:] | 0x80)
    # all zeros: scale 1, codes 0
    q0, s0 = oracle_mod.quantize_fp8(np.zeros((3, 16), np.float32))
    assert s0 == 1.0 and not q0.any()


def test_fp8_quantize_matches_independent_encoder(oracle_mod):
    x = synth.draw_fp32(4321, 64, 256, "normal")
    q, s = oracle_mod.quantize_fp8(x)
    q2, s2 = synth.quantize_fp8(x)
    assert s == s2
    # synth's encoder writes +0 where the sign of an underflowing value is negative
    same = (q == q2) | (((q & 0x7F) == 0) & ((q2 & 0x7F) == 0))
    assert same.all()
    # reconstruction within half a unit of the code's binade
    amax = np.abs(x).max()
    assert np.abs(oracle_mod.dec_e4m3(q).astype(np.float64) * s - x).max() <= amax * 2.0 ** -4


def test_nvfp4_quantize_closed_forms(oracle_mod):
    # one row, three blocks: zeros; exact e2m1 multiples of a power-of-two block scale; the tensor amax
    blk_exact = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -6, -4, -3, -2, -1.5, -1, -.5, -0.0], np.float32)
    x = np.concatenate([np.zeros(16, np.float32), blk_exact * np.float32(0.25), blk_exact * np.float32(0.25 * 448 / 1.0)])
    x = x.reshape(1, 48)
    q, sf, g = oracle_mod.quantize_nvfp4(x)
    amax = np.float32(6 * 0.25 * 448)
    assert g == amax / np.float32(2688.0)
    assert sf[0, 0] == 0 and not q[0, :8].any()
    # block 3 holds the tensor amax: its scale is 448 (0x7E) and its codes are exact
    assert sf[0, 2] == 0x7E
    codes = synth.unpack_fp4(q)[0]
    want = np.array([0, 1, 2, 3, 4, 5, 6, 7, 15, 14, 13, 12, 11, 10, 9, 8], np.uint8)
    assert np.array_equal(codes[32:48], want)
    # block 2: b = 1.5 -> b/(6g) = 1.5 * 2688 / (6 * 672) = 1.0 exactly -> scale 1 (0x38), codes exact
    assert sf[0, 1] == 0x38
    assert np.array_equal(codes[16:32], want)


def test_nvfp4_quantize_matches_independent_encoder(oracle_mod):
    x = synth.draw_fp32(9876, 48, 512, "normal")
    x[3, 32:48] = 0.0                       # an all-zero block
    x[5, 64:80] *= np.float32(1e-7)         # a block whose scale underflows to 0
    q, sf, g = oracle_mod.quantize_nvfp4(x)
    q2, sf2, g2 = synth.quantize_nvfp4(x)
    assert g == g2
    assert np.array_equal(sf, sf2)
    c, c2 = synth.unpack_fp4(q), synth.unpack_fp4(q2)
    same = (c == c2) | (((c & 7) == 0) & ((c2 & 7) == 0))
    assert same.all()
    assert sf[5, 4] == 0 and not (c[5, 64:80] & 7).any()


def test_nvfp4_codes_are_nearest_on_the_block_grid(oracle_mod):
    x = synth.draw_fp32(555, 16, 256, "normal")
    q, sf, g = oracle_mod.quantize_nvfp4(x)
    d = (oracle_mod.dec_e4m3(sf).astype(np.float32) * g).astype(np.float32)   # [16, 16]
    y = x.reshape(16, 16, 16) / d[..., None]
    c = synth.unpack_fp4(q).reshape(16, 16, 16)
    mag = E2M1_LITERAL[c & 7]
    err = np.abs(np.abs(y.astype(np.float64)) - mag)
    best = np.abs(np.abs(y.astype(np.float64))[..., None] - E2M1_LITERAL).min(axis=-1)
    assert np.all(err <= best + 1e-12)
