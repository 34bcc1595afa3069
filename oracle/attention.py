"""CPU oracle for non-causal attention forward, O = softmax(Q·Kᵀ/√D)·V.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
benchmark's CPU-baseline leg.  The GPU library never imports it, and it shares
no code with the CUDA path.

What is computed follows the attention example of "ThunderKittens: Simple,
Fast, and Adorable AI Kernels" ("The Four Functions: Load, Compute, Store,
Finish": scores Q·Kᵀ, a softmax that subtracts the row maximum, exponentiates
and divides by the row sum, then the product with V; the final division by the
normaliser is the "finish" step) and the non-causal attention prefill of the
ThunderKittens DSL page ("Реальный пример: attention prefill").  The pages'
kernel reaches that result by an online (tiled) softmax; the oracle is the
plain definition, evaluated whole and in float64:

    S[i, j]   = (Σ_d q[i, d] · k[j, d]) · scale          scale = 1/√D
    m[i]      = max_j S[i, j]
    l[i]      = Σ_j exp(S[i, j] − m[i])
    O[i, :]   = Σ_j exp(S[i, j] − m[i]) · v[j, :] / l[i]
    lse[i]    = m[i] + ln l[i]                            (log of the softmax normaliser)

Inputs are bf16 bit patterns (uint16) laid out [B, H, N, D]; they are decoded
by the bf16 definition (the 16 bits are the high half of an IEEE binary32).
The output O is rounded once, from float64, to bf16 with round-to-nearest-even.
Readings where the pages are silent: the softmax scale is 1/√D; keys and
queries may differ in number (Nq rows of Q against Nkv rows of K and V).
"""
from __future__ import annotations

import numpy as np


def bf16_decode(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 values (bits are the top half of a binary32)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):  # NaN patterns stay NaN
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """float64 -> bf16 bit patterns, rounding the float64 value itself to the
    nearest bf16 (8 significant bits), ties to even.  Finite normal inputs and
    zero only (attention outputs are bounded by max |v|)."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                      # x = m · 2^e, 0.5 <= |m| < 1
    q = np.round(m * 256.0)                 # 8 significant bits; np.round is half-to-even
    y = np.ldexp(q, e - 8).astype(np.float32)  # exactly representable in binary32
    return (y.view(np.uint32) >> 16).astype(np.uint16)


def attention_forward(q_bits: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray, scale: float | None = None,
                      heads=None, rows=None):
    """Non-causal attention forward on [B, H, N, D] bf16 inputs.

    heads: optional list of (b, h) pairs to evaluate (default: all).
    rows:  optional array of query-row indices to evaluate in each head.
    Returns a dict with, per evaluated head (in the order of `heads`):
      "o"     float64 [n_heads, n_rows, D]  exact output before rounding
      "o_bf16" uint16 [n_heads, n_rows, D] the output rounded to bf16
      "lse"   float64 [n_heads, n_rows]     m + ln l
      "pv_abs" float64 [n_heads, n_rows, D] Σ_j p[i,j]·|v[j,:]| (the size of the terms
              summed into O, for error bounds that scale with it)
    """
    B, H, Nq, D = q_bits.shape
    Nkv = k_bits.shape[2]
    assert k_bits.shape == (B, H, Nkv, D) and v_bits.shape == (B, H, Nkv, D)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    rows = np.arange(Nq) if rows is None else np.asarray(rows, dtype=np.int64)
    out_o, out_lse, out_abs = [], [], []
    for b, h in heads:
        q = bf16_decode(q_bits[b, h][rows])          # [n_rows, D]
        k = bf16_decode(k_bits[b, h])                # [Nkv, D]
        v = bf16_decode(v_bits[b, h])                # [Nkv, D]
        s = (q @ k.T) * scale                        # scores
        m = s.max(axis=1, keepdims=True)             # row maxima
        p = np.exp(s - m)                            # unnormalised probabilities
        l = p.sum(axis=1, keepdims=True)             # normaliser
        out_o.append((p @ v) / l)
        out_abs.append((p @ np.abs(v)) / l)
        out_lse.append(m[:, 0] + np.log(l[:, 0]))
    o = np.stack(out_o)
    return {"o": o, "o_bf16": bf16_round(o), "lse": np.stack(out_lse), "pv_abs": np.stack(out_abs)}
