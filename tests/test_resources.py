"""Register budget of the GEMM kernels (host only: nvcc cross-compiles, no GPU).

Every GEMM variant must fit its per-thread register budget without spilling:
the 448-thread NVFP4 kernels get 128 registers, and a spill there once came
from the split-K reduction holding a whole fp32 chunk.  ptxas reports the
registers and spill bytes of each kernel entry; this test compiles the three
GEMM translation units and checks them.
"""
import concurrent.futures as cf
import os
import shutil

import pytest

from tiled_tensor_core_gb300 import build as tkg_build

pytestmark = pytest.mark.skipif(
    not (shutil.which("nvcc") or os.path.exists("/usr/local/cuda/bin/nvcc")), reason="nvcc not available")

GEMM_UNITS = ("gemm_bf16.cu", "gemm_fp8.cu", "gemm_nvfp4.cu")


@pytest.fixture(scope="module")
def usage():
    srcs = [os.path.join(tkg_build.CSRC, f) for f in GEMM_UNITS]
    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        return dict(zip(GEMM_UNITS, ex.map(tkg_build.resource_usage, srcs)))


def test_every_gemm_variant_is_spill_free(usage):
    bad = []
    n = 0
    for unit, entries in usage.items():
        for e in entries:
            if "tkg_gemm_kernel" not in e["name"]:
                continue
            n += 1
            if e.get("spill_stores", 0) or e.get("spill_loads", 0):
                bad.append((unit, e["name"], e["registers"], e["spill_stores"], e["spill_loads"]))
    assert n >= 5, f"expected every compiled GEMM variant, found {n}"
    assert not bad, f"GEMM kernels spilling registers: {bad}"



def test_register_split_kernel_uses_its_launch_registers(usage):
    # the NVFP4 kernel's warpgroups trade registers with setmaxnreg out of what the block was
    # launched with: 512 threads x 128; fewer at launch would leave setmaxnreg.inc waiting (the
    # library refuses such a build at run time as well)
    nv = [e for e in usage["gemm_nvfp4.cu"] if "tkg_gemm_kernel" in e["name"]]
    assert nv and all(e["registers"] == 128 for e in nv), nv
