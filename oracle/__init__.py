"""CPU oracle for the dense tiled GEMM C = A·Bᵀ (bf16 / FP8 e4m3 / NVFP4).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
benchmark's CPU-baseline leg.  The GPU library never imports or links it, and
it shares no code with the CUDA path.

The arithmetic lives in ``oracle.c`` (plain C, fp32 sequential-k accumulation,
table decoding, bf16 round-to-nearest-even output); this module only builds it
with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_SRCS = [_SRC, os.path.join(_HERE, "quantize.c")]
_LIB_PATH = os.path.join(_HERE, "_oracle.so")
_lock = threading.Lock()
_lib = None

# -O2 without -ffast-math; -ffp-contract=off keeps "multiply, round, add, round".
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile oracle.c and quantize.c into _oracle.so (gcc, a second or two)."""
    newest = max(os.path.getmtime(p) for p in _SRCS)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < newest:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, *_SRCS, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            i64, f32, vp = ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
            lib.oracle_init.restype = None
            lib.oracle_dec_bf16.argtypes = [ctypes.c_uint16]
            lib.oracle_dec_bf16.restype = f32
            lib.oracle_dec_e4m3.argtypes = [ctypes.c_uint8]
            lib.oracle_dec_e4m3.restype = f32
            lib.oracle_dec_e2m1.argtypes = [ctypes.c_uint8]
            lib.oracle_dec_e2m1.restype = f32
            lib.oracle_rne_bf16.argtypes = [f32]
            lib.oracle_rne_bf16.restype = ctypes.c_uint16
            lib.oracle_decode_bf16.argtypes = [vp, vp, i64]
            lib.oracle_decode_e4m3.argtypes = [vp, vp, i64]
            lib.oracle_decode_nvfp4.argtypes = [vp, vp, vp, i64, i64]
            lib.oracle_gemm_bf16_rows.argtypes = [i64, i64, i64, vp, vp, vp, i64, vp, vp]
            lib.oracle_gemm_bf16_rows.restype = ctypes.c_int
            lib.oracle_gemm_fp8_rows.argtypes = [i64, i64, i64, vp, vp, f32, f32, vp, i64, vp, vp]
            lib.oracle_gemm_fp8_rows.restype = ctypes.c_int
            lib.oracle_gemm_nvfp4_rows.argtypes = [i64, i64, i64, vp, vp, vp, vp, f32, f32, vp, i64, vp, vp]
            lib.oracle_gemm_nvfp4_rows.restype = ctypes.c_int
            lib.oracle_e4m3_rne_sat.argtypes = [f32]
            lib.oracle_e4m3_rne_sat.restype = ctypes.c_uint8
            lib.oracle_e2m1_rne_sat.argtypes = [f32]
            lib.oracle_e2m1_rne_sat.restype = ctypes.c_uint8
            lib.oracle_quantize_fp8.argtypes = [i64, i64, vp, vp, vp]
            lib.oracle_quantize_fp8.restype = None
            lib.oracle_quantize_nvfp4.argtypes = [i64, i64, vp, vp, vp, vp]
            lib.oracle_quantize_nvfp4.restype = None
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
            lib.oracle_init()
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


# ---- scalar / array decoders (exposed for the pins) -----------------------

def dec_bf16(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float32)
    _load().oracle_decode_bf16(_ptr(bits), _ptr(out), bits.size)
    return out


def dec_e4m3(codes: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape, dtype=np.float32)
    _load().oracle_decode_e4m3(_ptr(codes), _ptr(out), codes.size)
    return out


def dec_e2m1(codes: np.ndarray) -> np.ndarray:
    lib = _load()
    codes = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.oracle_dec_e2m1(int(c)) for c in codes.ravel()], dtype=np.float32).reshape(codes.shape)


def dec_nvfp4(packed: np.ndarray, sf: np.ndarray, K: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    rows = packed.shape[0]
    out = np.empty((rows, K), dtype=np.float32)
    _load().oracle_decode_nvfp4(_ptr(packed), _ptr(sf), _ptr(out), rows, K)
    return out


def rne_bf16(x: np.ndarray) -> np.ndarray:
    lib = _load()
    x = np.asarray(x, dtype=np.float32)
    return np.array([lib.oracle_rne_bf16(float(v)) for v in x.ravel()], dtype=np.uint16).reshape(x.shape)


# ---- GEMMs ----------------------------------------------------------------

def _rows_arg(M: int, rows):
    if rows is None:
        return None, M
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    if rows.size and (rows.min() < 0 or rows.max() >= M):
        raise ValueError("row index out of range")
    return rows, rows.size


def gemm_bf16(a: np.ndarray, b: np.ndarray, rows=None):
    """a: [M,K] uint16 bf16 bits, b: [N,K]. Returns (acc fp32 [R,N], C bf16 bits [R,N])."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    b = np.ascontiguousarray(b, dtype=np.uint16)
    M, K = a.shape
    N = b.shape[0]
    assert b.shape[1] == K
    r, nr = _rows_arg(M, rows)
    acc = np.empty((nr, N), dtype=np.float32)
    C = np.empty((nr, N), dtype=np.uint16)
    rc = _load().oracle_gemm_bf16_rows(M, N, K, _ptr(a), _ptr(b), _ptr(r), nr, _ptr(acc), _ptr(C))
    if rc:
        raise MemoryError("oracle allocation failed")
    return acc, C


def gemm_fp8(a: np.ndarray, b: np.ndarray, scale_a: float, scale_b: float, rows=None):
    """a: [M,K] e4m3 codes, b: [N,K] e4m3 codes, per-tensor dequant scales."""
    a = np.ascontiguousarray(a, dtype=np.uint8)
    b = np.ascontiguousarray(b, dtype=np.uint8)
    M, K = a.shape
    N = b.shape[0]
    assert b.shape[1] == K
    r, nr = _rows_arg(M, rows)
    acc = np.empty((nr, N), dtype=np.float32)
    C = np.empty((nr, N), dtype=np.uint16)
    rc = _load().oracle_gemm_fp8_rows(M, N, K, _ptr(a), _ptr(b), float(scale_a), float(scale_b),
                                      _ptr(r), nr, _ptr(acc), _ptr(C))
    if rc:
        raise MemoryError("oracle allocation failed")
    return acc, C


def gemm_nvfp4(a: np.ndarray, b: np.ndarray, sfa: np.ndarray, sfb: np.ndarray, g_a: float, g_b: float, rows=None):
    """a: [M,K/2] packed e2m1, b: [N,K/2], sfa: [M,K/16] e4m3, sfb: [N,K/16] e4m3."""
    a = np.ascontiguousarray(a, dtype=np.uint8)
    b = np.ascontiguousarray(b, dtype=np.uint8)
    sfa = np.ascontiguousarray(sfa, dtype=np.uint8)
    sfb = np.ascontiguousarray(sfb, dtype=np.uint8)
    M, K2 = a.shape
    K = 2 * K2
    N = b.shape[0]
    assert b.shape[1] == K2 and sfa.shape == (M, K // 16) and sfb.shape == (N, K // 16)
    r, nr = _rows_arg(M, rows)
    acc = np.empty((nr, N), dtype=np.float32)
    C = np.empty((nr, N), dtype=np.uint16)
    rc = _load().oracle_gemm_nvfp4_rows(M, N, K, _ptr(a), _ptr(b), _ptr(sfa), _ptr(sfb), float(g_a), float(g_b),
                                        _ptr(r), nr, _ptr(acc), _ptr(C))
    if rc:
        raise MemoryError("oracle allocation failed")
    return acc, C


def gemm(ops, rows=None):
    """Dispatch on an Operands bundle (see tiled_tensor_core_gb300.synth)."""
    if ops.kind == "bf16":
        return gemm_bf16(ops.a, ops.b, rows)
    if ops.kind == "fp8":
        return gemm_fp8(ops.a, ops.b, ops.scale_a, ops.scale_b, rows)
    if ops.kind == "nvfp4":
        return gemm_nvfp4(ops.a, ops.b, ops.sfa, ops.sfb, ops.scale_a, ops.scale_b, rows)
    raise ValueError(ops.kind)


# ---- input encodings (quantize.c) -------------------------------------------


def e4m3_rne_sat(x: np.ndarray) -> np.ndarray:
    """fp32 -> e4m3 code, round to nearest even, saturating at 448 (elementwise)."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    return np.fromiter((lib.oracle_e4m3_rne_sat(float(v)) for v in x), dtype=np.uint8, count=x.size)


def e2m1_rne_sat(x: np.ndarray) -> np.ndarray:
    """fp32 -> e2m1 code (0..15), round to nearest even, saturating at 6 (elementwise)."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    return np.fromiter((lib.oracle_e2m1_rne_sat(float(v)) for v in x), dtype=np.uint8, count=x.size)


def quantize_fp8(x: np.ndarray):
    """Per-tensor FP8 encoding of fp32 [rows][cols]: (codes uint8, dequantisation scale float32)."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, cols = x.shape
    q = np.empty((rows, cols), dtype=np.uint8)
    s = np.zeros(1, dtype=np.float32)
    lib.oracle_quantize_fp8(rows, cols, _ptr(x), _ptr(q), _ptr(s))
    return q, np.float32(s[0])


def quantize_nvfp4(x: np.ndarray):
    """NVFP4 encoding of fp32 [rows][cols] (cols % 16 == 0): (packed uint8 [rows][cols/2],
    block scales uint8 [rows][cols/16], global scale float32)."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, cols = x.shape
    assert cols % 16 == 0
    q = np.empty((rows, cols // 2), dtype=np.uint8)
    sf = np.empty((rows, cols // 16), dtype=np.uint8)
    g = np.zeros(1, dtype=np.float32)
    lib.oracle_quantize_nvfp4(rows, cols, _ptr(x), _ptr(q), _ptr(sf), _ptr(g))
    return q, sf, np.float32(g[0])
