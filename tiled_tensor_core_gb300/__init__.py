"""GB300-native dense tiled tensor-core GEMM  C = A·Bᵀ  (bf16 / FP8 / NVFP4).

The compute path is the C-ABI library ``_tkg.so`` (hand-written sm_103a
kernels: TMA ring + tcgen05.mma into TMEM + TMA-store epilogue, persistent
L2-grouped tile order).  ``tkg`` is the thin ctypes binding with the same
names as the C entry points; ``synth`` makes seeded synthetic operands.
The binding is imported lazily so that ``synth`` works on machines without the
built library; any call into ``tkg`` raises if the library is missing.
"""
import importlib

__all__ = ["tkg", "synth"]


def __getattr__(name):
    if name in ("tkg", "synth", "build"):
        return importlib.import_module(f".{name}", __name__)
    tkg = importlib.import_module(".tkg", __name__)
    if hasattr(tkg, name):
        return getattr(tkg, name)
    raise AttributeError(name)
