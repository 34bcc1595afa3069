"""Pins of the attention-forward oracle against things other than itself:
closed forms (uniform attention, a dominant key, two keys), invariants (rows of
the softmax sum to one, joint permutation of keys and values, a shift of every
score of a row), torch's bf16 conversions, and torch's own scaled-dot-product
attention evaluated in float64 on random inputs."""
import math

import numpy as np
import pytest

from oracle import attention as oa
from tiled_tensor_core_gb300 import synth

torch = pytest.importorskip("torch")


def bits_of(x: np.ndarray) -> np.ndarray:
    """float values exactly representable in bf16 -> bf16 bit patterns."""
    y = np.asarray(x, dtype=np.float32)
    b = y.view(np.uint32)
    assert (b & 0xFFFF == 0).all(), "value not exact in bf16"
    return (b >> 16).astype(np.uint16)


def test_bf16_decode_matches_torch_for_every_finite_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    got = oa.bf16_decode(bits)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])


def test_bf16_round_matches_torch_on_binary32_values_and_ties():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 20, 200000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oa.bf16_round(x.astype(np.float64)), ref)
    # exact ties round to the even significand: 1 + 2^-8 -> 1, 1 + 3*2^-8 -> 1 + 2^-6
    assert oa.bf16_round(np.array([1 + 2.0 ** -8]))[0] == 0x3F80
    assert oa.bf16_round(np.array([1 + 3 * 2.0 ** -8]))[0] == 0x3F82
    # just above a tie rounds up (a float64 value no binary32 can hold)
    assert oa.bf16_round(np.array([1 + 2.0 ** -8 + 2.0 ** -40]))[0] == 0x3F81
    assert oa.bf16_round(np.array([0.0, -2.0]))[0] == 0 and oa.bf16_round(np.array([-2.0]))[0] == 0xC000


@pytest.mark.parametrize("nq,nkv,d", [(5, 7, 64), (33, 129, 128), (1, 1, 64)])
def test_uniform_attention_is_the_mean_of_v(nq, nkv, d):
    x = synth.attention_inputs(1, 2, nq, nkv, d, seed=11)
    k0 = np.zeros_like(x.k)  # every score 0
    r = oa.attention_forward(x.q, k0, x.v)
    mean_v = oa.bf16_decode(x.v).mean(axis=2).reshape(2, 1, d)
    assert np.allclose(r["o"], np.broadcast_to(mean_v, r["o"].shape), rtol=0, atol=1e-14)
    assert np.allclose(r["lse"], math.log(nkv), rtol=0, atol=1e-12)


def test_dominant_key_selects_its_value():
    d, nkv, j = 64, 50, 17
    q = np.zeros((1, 1, 3, d), np.float32)
    q[..., 0] = 200.0                       # scores 200 * 2 / sqrt(64) = 50 for key j, 0 for the rest
    k = np.zeros((1, 1, nkv, d), np.float32)
    k[0, 0, j, 0] = 2.0
    v = synth.attention_inputs(1, 1, 1, nkv, d, seed=3).v
    r = oa.attention_forward(bits_of(q), bits_of(k), v)
    vj = oa.bf16_decode(v[0, 0, j])
    bound = nkv * math.exp(-50.0) * np.abs(oa.bf16_decode(v)).max()
    assert np.abs(r["o"][0] - vj).max() <= bound
    assert abs(r["lse"][0, 0] - 50.0) <= nkv * math.exp(-50.0)


@pytest.mark.parametrize("d", [64, 128])
def test_two_keys_sigmoid_closed_form(d):
    # scores s1 = q·k1/sqrt(d), s2 = q·k2/sqrt(d); weight of key 1 = 1/(1 + e^(s2 - s1))
    q = np.zeros((1, 1, 1, d), np.float32)
    q[..., :2] = [1.5, -0.75]
    k = np.zeros((1, 1, 2, d), np.float32)
    k[0, 0, 0, :2] = [2.0, 1.0]
    k[0, 0, 1, :2] = [-1.0, 0.5]
    v = np.zeros((1, 1, 2, d), np.float32)
    v[0, 0, 0] = 1.0
    v[0, 0, 1] = -3.0
    r = oa.attention_forward(bits_of(q), bits_of(k), bits_of(v))
    s1 = (1.5 * 2.0 - 0.75 * 1.0) / math.sqrt(d)
    s2 = (1.5 * -1.0 - 0.75 * 0.5) / math.sqrt(d)
    w1 = 1.0 / (1.0 + math.exp(s2 - s1))
    assert np.allclose(r["o"], w1 * 1.0 + (1 - w1) * -3.0, rtol=0, atol=1e-14)
    assert abs(r["lse"][0, 0] - np.logaddexp(s1, s2)) <= 1e-14


def test_softmax_rows_sum_to_one_even_for_huge_scores():
    x = synth.attention_inputs(1, 1, 40, 300, 64, seed=8)
    q = oa.bf16_decode(x.q) * 256.0         # scores of order 10^3: exp would overflow without the max shift
    ones = bits_of(np.ones((1, 1, 300, 64), np.float32))
    r = oa.attention_forward(bits_of(q.astype(np.float32)), x.k, ones)
    assert np.isfinite(r["lse"]).all()
    assert np.abs(r["o"] - 1.0).max() <= 1e-13
    assert (r["o_bf16"] == 0x3F80).all()


def test_joint_permutation_of_keys_and_values_and_row_shift():
    x = synth.attention_inputs(1, 1, 20, 90, 64, seed=9)
    r0 = oa.attention_forward(x.q, x.k, x.v)
    perm = np.random.default_rng(1).permutation(90)
    r1 = oa.attention_forward(x.q, x.k[:, :, perm], x.v[:, :, perm])
    assert np.allclose(r0["o"], r1["o"], rtol=0, atol=1e-13)
    # adding the same vector c to every key shifts row i's scores by q_i·c: O unchanged, lse shifted
    # (c = e_3, added to keys whose component 3 is zero, so the shifted keys stay exact in bf16)
    k0 = x.k.copy()
    k0[..., 3] = 0
    k1 = k0.copy()
    k1[..., 3] = 0x3F80  # 1.0
    r2 = oa.attention_forward(x.q, k0, x.v)
    r3 = oa.attention_forward(x.q, k1, x.v)
    assert np.allclose(r2["o"], r3["o"], rtol=0, atol=1e-12)
    shift = oa.bf16_decode(x.q)[0, 0, :, 3] / 8.0
    assert np.allclose(r3["lse"][0] - r2["lse"][0], shift, rtol=0, atol=1e-12)


@pytest.mark.parametrize("b,h,nq,nkv,d", [(2, 3, 64, 64, 64), (1, 2, 130, 257, 128), (1, 1, 1, 300, 64)])
def test_matches_torch_sdpa_in_float64(b, h, nq, nkv, d):
    x = synth.attention_inputs(b, h, nq, nkv, d, seed=nq + nkv)
    q, k, v = (torch.from_numpy(oa.bf16_decode(t)) for t in (x.q, x.k, x.v))
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v).numpy()
    lse_ref = torch.logsumexp((q @ k.transpose(-1, -2)) / math.sqrt(d), dim=-1).numpy()
    r = oa.attention_forward(x.q, x.k, x.v)
    assert np.allclose(r["o"].reshape(b, h, nq, d), ref, rtol=1e-12, atol=1e-13)
    assert np.allclose(r["lse"].reshape(b, h, nq), lse_ref, rtol=1e-13, atol=1e-12)
    assert (r["pv_abs"] >= np.abs(r["o"]) - 1e-15).all()


def test_head_and_row_subsets_are_slices_of_the_whole():
    x = synth.attention_inputs(2, 2, 50, 60, 64, seed=4)
    full = oa.attention_forward(x.q, x.k, x.v)
    rows = np.array([0, 7, 49])
    sub = oa.attention_forward(x.q, x.k, x.v, heads=[(1, 0), (0, 1)], rows=rows)
    assert np.array_equal(sub["o_bf16"][0], full["o_bf16"][2][rows])
    assert np.array_equal(sub["o_bf16"][1], full["o_bf16"][1][rows])
    assert np.allclose(sub["lse"][0], full["lse"][2][rows], rtol=0, atol=0)
