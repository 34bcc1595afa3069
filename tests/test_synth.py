"""Input generator checks: the fast encoders agree with the plain nearest-table
search and with torch's float8 cast; quantised operands reconstruct the draw
within half a grid step; generation is deterministic."""
import numpy as np
import torch

from tiled_tensor_core_gb300 import synth


def test_e4m3_fast_equals_table_and_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        (rng.standard_normal(300_000) * 10.0 ** rng.integers(-4, 4, 300_000)).astype(np.float32),
        synth.E4M3_POS.astype(np.float32), -synth.E4M3_POS.astype(np.float32),
        ((synth.E4M3_POS[1:] + synth.E4M3_POS[:-1]) / 2).astype(np.float32),  # exact ties
        np.array([448, 449, 460, 464, 470, 500, 1e6, 0.0, -0.0], np.float32)]).astype(np.float32)
    fast = synth.encode_e4m3(x)
    assert np.array_equal(fast, synth.encode_e4m3_table(x))
    inr = np.abs(x) <= 448
    ref = torch.from_numpy(x[inr]).to(torch.float8_e4m3fn).to(torch.float32).numpy()
    mine = synth.e4m3_value(fast[inr])
    assert np.array_equal(mine, ref)  # equal values (torch keeps -0 where this encoder writes +0)


def test_e2m1_fast_equals_table():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.uniform(-8, 8, 200_000), np.arange(-7, 7.01, 0.25)]).astype(np.float32)
    assert np.array_equal(synth.encode_e2m1(x), synth.encode_e2m1_table(x))


def test_nvfp4_quantisation_error_bounded():
    x = synth._draw(3, 64, 512, "normal")
    packed, sb, g = synth.quantize_nvfp4(x)
    codes = synth.unpack_fp4(packed)
    vals = np.concatenate([synth.E2M1_POS, -synth.E2M1_POS])[codes]
    scale = np.repeat(synth.e4m3_value(sb) * float(g), 16, axis=1)
    recon = vals * scale
    # inside a block the e2m1 grid step is at most 2 (times the block scale), so the error is at most 1 step
    assert np.all(np.abs(recon - x) <= 1.0 * scale + 1e-6)
    # the block scale is chosen so the block maximum lands near 6 (within e4m3's relative precision)
    bmax = np.abs(x).reshape(64, -1, 16).max(axis=2)
    assert np.all(bmax <= 6.0 * synth.e4m3_value(sb) * float(g) * (1 + 2 ** -3) + 1e-6)


def test_fp8_quantisation_maps_amax_to_448():
    x = synth._draw(4, 32, 256, "normal")
    codes, s = synth.quantize_fp8(x)
    assert synth.e4m3_value(codes).max() == 448.0 or synth.e4m3_value(codes).min() == -448.0
    recon = synth.e4m3_value(codes) * float(s)
    assert np.max(np.abs(recon - x) / np.maximum(np.abs(x), 2 ** -6 * float(s))) <= 2 ** -4 + 1e-6


def test_generation_is_deterministic():
    a = synth.make_operands("nvfp4", 300, 200, 512, "normal", 5, 6)
    b = synth.make_operands("nvfp4", 300, 200, 512, "normal", 5, 6)
    c = synth.make_operands("nvfp4", 300, 200, 512, "normal", 5, 7)
    assert a.digest() == b.digest() != c.digest()
