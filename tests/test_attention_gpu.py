"""Parity of the attention-forward kernel with the float64 oracle.

Error bound (derived from the arithmetic, u = 2^-9 the bf16 unit roundoff):
the probabilities enter P·V rounded to bf16 (relative error <= u each), so the
output moves by at most u·Σ_j p_j|v_j| / l (the oracle's `pv_abs`); the final
rounding of O to bf16 adds at most u·|O|; fp32 scores, sums and accumulation
add terms of order Nkv·2^-24 relative, far below those.  The test allows twice
the first two terms: |O_gpu - O| <= 2u·pv_abs + 2u·|O| + 1e-6, and relative
Frobenius error <= 4e-3.  The log-sum-exp is fp32 throughout:
|lse_gpu - lse| <= 4·Nkv·2^-24 + 1e-5.  Cases whose probabilities are exactly
0 or 1 in fp32 (one key dominating every row, a single key) are bit-exact."""
import numpy as np
import pytest

from oracle import attention as oa
from tiled_tensor_core_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

U = 2.0 ** -9


@pytest.fixture(scope="module")
def tkg():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from tiled_tensor_core_gb300 import tkg as mod
    return mod


def run_attn(tkg, q, k, v, with_lse=True):
    B, H, Nq, D = q.shape
    Nkv = k.shape[2]
    dev = torch.device("cuda")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)
    tq, tk, tv = t(q), t(k), t(v)
    o = torch.full((B, H, Nq, D), -1, dtype=torch.int16, device=dev)  # NaN-free poison: 0xFFFF is a NaN bf16
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device=dev) if with_lse else None
    tkg.tkg_attention_fwd(B, H, Nq, Nkv, D, tq, tk, tv, o, lse)
    st = tkg.tkg_check_status()
    assert st == tkg.TKG_OK, tkg.status_string(st)
    torch.cuda.synchronize()
    o_bits = o.cpu().numpy().view(np.uint16)
    return o_bits, (lse.cpu().numpy() if with_lse else None)


def check(o_bits, lse, ref, nkv):
    got = oa.bf16_decode(o_bits).reshape(ref["o"].shape)
    assert np.isfinite(got).all(), "non-finite output"
    err = np.abs(got - ref["o"])
    bound = 2 * U * ref["pv_abs"] + 2 * U * np.abs(ref["o"]) + 1e-6
    worst = float((err / bound).max())
    assert worst <= 1.0, f"elementwise bound exceeded: {worst:.3f}"
    rel = float(np.linalg.norm(got - ref["o"]) / np.linalg.norm(ref["o"]))
    assert rel <= 4e-3, rel
    if lse is not None:
        dl = np.abs(lse.reshape(ref["lse"].shape) - ref["lse"])
        assert float(dl.max()) <= 4 * nkv * 2.0 ** -24 + 1e-5, float(dl.max())
    return rel


SHAPES = [(1, 1, 128, 128, 128), (2, 3, 256, 384, 128), (1, 2, 200, 333, 64), (2, 2, 1, 77, 128),
          (1, 1, 1000, 1, 64), (1, 4, 513, 1025, 128), (3, 1, 640, 129, 64), (1, 1, 130, 2000, 64)]


@pytest.mark.parametrize("shape", SHAPES)
def test_matches_oracle(tkg, shape):
    B, H, Nq, Nkv, D = shape
    x = synth.attention_inputs(B, H, Nq, Nkv, D, seed=sum(shape))
    o, lse = run_attn(tkg, x.q, x.k, x.v)
    ref = oa.attention_forward(x.q, x.k, x.v)
    check(o, lse, ref, Nkv)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("tiles", [1, 2, 3])
def test_dominant_key_is_bit_exact_across_kv_tiles(tkg, D, tiles):
    # query i = 1024·e_{a_i}; key j = (1 + j // 128)·e_{j mod 128 mod D}: every row's scores are
    # 0 except one key per KV tile, and the key in the last tile dominates the others by more than
    # 90 nats, so every other probability underflows in fp32 and O_i = V[that key] exactly.  The
    # running maximum grows from tile to tile, so the O rescaling is exercised.
    Nq, Nkv = 256, 128 * tiles
    rng = np.random.default_rng(D + tiles)
    a = rng.integers(0, min(D, 128), size=Nq)
    q = np.zeros((1, 1, Nq, D), np.float32)
    q[0, 0, np.arange(Nq), a] = 1024.0
    k = np.zeros((1, 1, Nkv, D), np.float32)
    for j in range(Nkv):
        if j % 128 < D:
            k[0, 0, j, j % 128] = 1.0 + j // 128
    v = synth.attention_inputs(1, 1, 1, Nkv, D, seed=5).v
    bits = lambda z: (z.view(np.uint32) >> 16).astype(np.uint16)
    o, lse = run_attn(tkg, bits(q), bits(k), v)
    want = v[0, 0, a + 128 * (tiles - 1)]
    assert np.array_equal(o[0, 0], want)
    score = 1024.0 * tiles / np.sqrt(D)
    assert np.allclose(lse[0, 0], score, rtol=2e-6, atol=0)


def test_single_key_gives_its_value(tkg):
    x = synth.attention_inputs(2, 2, 300, 1, 128, seed=2)
    o, lse = run_attn(tkg, x.q, x.k, x.v)
    assert np.array_equal(o, np.broadcast_to(x.v, o.shape))
    s = (oa.bf16_decode(x.q) * oa.bf16_decode(x.k)).sum(-1) / np.sqrt(128)
    assert np.allclose(lse, s, rtol=0, atol=1e-4)


def test_huge_scores_stay_finite(tkg):
    x = synth.attention_inputs(1, 2, 256, 512, 64, seed=12)
    q = (oa.bf16_decode(x.q) * 64.0).astype(np.float32)
    qb = (q.view(np.uint32) >> 16).astype(np.uint16)  # exact: a power-of-two multiple
    o, lse = run_attn(tkg, qb, x.k, x.v)
    ref = oa.attention_forward(qb, x.k, x.v)
    check(o, lse, ref, 512)


def test_without_lse_and_repeatable(tkg):
    x = synth.attention_inputs(1, 2, 384, 640, 128, seed=21)
    o1, _ = run_attn(tkg, x.q, x.k, x.v, with_lse=False)
    o2, lse = run_attn(tkg, x.q, x.k, x.v)
    assert np.array_equal(o1, o2)


@pytest.mark.parametrize("name", ["attn_n1024_d128", "attn_n4096_d64"])
def test_workload_sampled_heads(tkg, name):
    w = synth.ATTN_WORKLOADS[name]
    x = synth.attn_workload_inputs(name)
    o, lse = run_attn(tkg, x.q, x.k, x.v)
    heads = [(0, 0), (w.B // 2, w.H - 1), (w.B - 1, w.H // 3)]
    rows = np.unique(np.concatenate([np.arange(0, w.Nq, 61), [w.Nq - 1]]))
    ref = oa.attention_forward(x.q, x.k, x.v, heads=heads, rows=rows)
    got = np.stack([o[b, h][rows] for b, h in heads])
    got_lse = np.stack([lse[b, h][rows] for b, h in heads])
    check(got, got_lse, ref, w.Nkv)
