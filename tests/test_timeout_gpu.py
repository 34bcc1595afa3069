"""Failure detection without a GPU fault: every pipeline wait in the kernels is
bounded.  Fault injection makes the producer skip the copies of its first ring
stage (no copy is in flight for it), so the compute role's wait on that stage
runs out; the kernel records the timeout in the status word, every role stops,
tensor memory is released, and the context stays usable for the next call.
Every compiled GEMM variant is stalled this way: the 256x256 pair tile with its
two accumulators, the 256x512 pair tile with a single accumulator and four
48 KB stages, and the NVFP4 kernel, whose four scale-copy issuers also wait
(for the stage's scales in shared memory) and must give up in turn, and then
wait for their own copies, as must its eight epilogue warps (in their own
warpgroups, with a register split)."""
import numpy as np
import pytest

import oracle
from tiled_tensor_core_gb300 import synth

from gpu_util import check_against_oracle, run_gpu

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def tkg():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from tiled_tensor_core_gb300 import tkg as mod
    yield mod
    mod.tkg_set_option(mod.TKG_OPT_TIMEOUT_NS, 0)
    mod.tkg_set_option(mod.TKG_OPT_VARIANT, 0)


@pytest.mark.parametrize("kind,variant,shape", [("bf16", 2, (512, 512, 512)), ("bf16", 15, (512, 1024, 4096)),
                                                ("fp8", 15, (512, 1024, 4096)), ("nvfp4", 14, (512, 512, 2048))])
def test_injected_stall_reports_timeout_then_recovers(tkg, kind, variant, shape):
    from tiled_tensor_core_gb300.device import DeviceGemm
    M, N, K = shape
    ops = synth.make_operands(kind, M, N, K, "normal_sqrtk" if kind == "bf16" else "normal", 1, 2)
    tkg.tkg_set_option(tkg.TKG_OPT_VARIANT, variant)
    tkg.tkg_set_option(tkg.TKG_OPT_TIMEOUT_NS, 100_000_000)  # 0.1 s per wait
    try:
        g = DeviceGemm(ops, "cuda")
        tkg.tkg_debug_set_fault(1)
        g.run()
        assert tkg.tkg_check_status() == tkg.TKG_ERR_TIMEOUT
        # the status word was cleared by the check, and the next call is healthy
        assert tkg.tkg_check_status() == tkg.TKG_OK
        tkg.tkg_set_option(tkg.TKG_OPT_TIMEOUT_NS, 0)
        g2 = run_gpu(ops)
        acc, c_ref = oracle.gemm(ops)
        check_against_oracle(kind, g2.c_bits(), acc, c_ref, ops.scale_a, ops.scale_b)
    finally:
        tkg.tkg_debug_set_fault(0)
        tkg.tkg_set_option(tkg.TKG_OPT_TIMEOUT_NS, 0)
        tkg.tkg_set_option(tkg.TKG_OPT_VARIANT, 0)


def test_attention_injected_stall_reports_timeout_then_recovers(tkg):
    from oracle import attention as oa
    x = synth.attention_inputs(1, 2, 256, 384, 128, seed=17)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
    q, k, v = t(x.q), t(x.k), t(x.v)
    o = torch.empty_like(q)
    tkg.tkg_set_option(tkg.TKG_OPT_TIMEOUT_NS, 100_000_000)  # 0.1 s per wait
    try:
        tkg.tkg_debug_set_fault(2)
        tkg.tkg_attention_fwd(1, 2, 256, 384, 128, q, k, v, o)
        assert tkg.tkg_check_status() == tkg.TKG_ERR_TIMEOUT
        assert tkg.tkg_check_status() == tkg.TKG_OK
        tkg.tkg_set_option(tkg.TKG_OPT_TIMEOUT_NS, 0)
        tkg.tkg_attention_fwd(1, 2, 256, 384, 128, q, k, v, o)
        assert tkg.tkg_check_status() == tkg.TKG_OK
        got = oa.bf16_decode(o.cpu().numpy().view(np.uint16))
        ref = oa.attention_forward(x.q, x.k, x.v)
        err = np.abs(got.reshape(ref["o"].shape) - ref["o"])
        assert (err <= 2 * 2.0 ** -9 * (ref["pv_abs"] + np.abs(ref["o"])) + 1e-6).all()
    finally:
        tkg.tkg_debug_set_fault(0)
        tkg.tkg_set_option(tkg.TKG_OPT_TIMEOUT_NS, 0)


def test_fault_modes_are_consumed_by_their_own_kind(tkg):
    # an armed attention fault is not taken by a GEMM launch (and the GEMM is correct)
    ops = synth.make_operands("bf16", 256, 256, 256, "normal_sqrtk", 3, 4)
    try:
        tkg.tkg_debug_set_fault(2)
        g = run_gpu(ops)
        acc, c_ref = oracle.gemm(ops)
        check_against_oracle("bf16", g.c_bits(), acc, c_ref)
    finally:
        tkg.tkg_debug_set_fault(0)
