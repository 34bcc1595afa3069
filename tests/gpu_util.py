"""Helpers shared by the GPU tests: run a tkg GEMM on synthetic operands and
compare with the CPU oracle under the stated tolerances."""
import numpy as np
import torch

# Tolerances of the GEMM contract: bf16 output compared with the oracle's bf16
# output (relative Frobenius <= 1e-3 and |delta| <= 1e-2 (|ref| + 1)
# elementwise); FP8 / NVFP4 compared with the oracle's fp32 accumulation of the
# same decoded values times the per-tensor scales (relative Frobenius <= 2e-3).
BF16_REL_FRO = 1e-3
BF16_ELEM = 1e-2
SCALED_REL_FRO = 2e-3


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    u = bits.astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def rel_fro(x: np.ndarray, ref: np.ndarray) -> float:
    den = np.linalg.norm(ref)
    num = np.linalg.norm(x - ref)
    return float(num / den) if den > 0 else float(num)


def check_against_oracle(kind, c_bits, acc_ref, c_ref_bits, scale_a=1.0, scale_b=1.0):
    """Returns a dict of error metrics; asserts the contract's tolerance."""
    g = bf16_bits_to_f64(c_bits)
    assert np.isfinite(g).all(), "non-finite output"
    r_bf16 = bf16_bits_to_f64(c_ref_bits)
    out = {"rel_fro_vs_bf16": rel_fro(g, r_bf16)}
    if kind == "bf16":
        elem = np.abs(g - r_bf16) / (np.abs(r_bf16) + 1.0)
        out["max_elem"] = float(elem.max()) if elem.size else 0.0
        assert out["rel_fro_vs_bf16"] <= BF16_REL_FRO, out
        assert out["max_elem"] <= BF16_ELEM, out
    else:
        ref = acc_ref.astype(np.float64) * scale_a * scale_b
        out["rel_fro_vs_fp32"] = rel_fro(g, ref)
        assert out["rel_fro_vs_fp32"] <= SCALED_REL_FRO, out
    return out


def sample_rows(M: int, n_random: int, seed: int) -> np.ndarray:
    """Rows spanning tile and CTA-pair boundaries, every 32-row TMEM lane
    quarter, the last row, plus random rows."""
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 31, 32, 63, 64, 95, 96, 127, 128, 159, 191, 255, 256, 383, 511, 512, M // 2, M - 129, M - 2, M - 1]
    rows = [r for r in fixed if 0 <= r < M]
    rows += list(rng.integers(0, M, size=n_random))
    return np.unique(np.array(rows, dtype=np.int64))


def run_gpu(ops, device="cuda"):
    from tiled_tensor_core_gb300.device import DeviceGemm
    from tiled_tensor_core_gb300 import tkg
    g = DeviceGemm(ops, device)
    g.c.fill_(float("nan"))
    g.run()
    st = tkg.tkg_check_status()
    assert st == tkg.TKG_OK, tkg.status_string(st)
    torch.cuda.synchronize()
    return g
