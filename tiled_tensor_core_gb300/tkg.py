"""ctypes binding of the tkg C ABI (include/tkg.h, include/tkg_debug.h).

Argument marshalling only: every GEMM step runs in the CUDA library.  Matrix
arguments may be torch tensors (their data pointer is used) or raw integer
device addresses.  ``stream=None`` means torch's current stream on the current
device.  Importing this module raises if the library has not been built — there
is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_tkg.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"tkg CUDA library not built ({LIB_PATH} missing); run __graft_entry__.build()")

lib = ctypes.CDLL(LIB_PATH)

TKG_OK = 0
TKG_ERR_INVALID_ARG = 1
TKG_ERR_MISALIGNED = 2
TKG_ERR_UNSUPPORTED_DEVICE = 3
TKG_ERR_CUDA = 4
TKG_ERR_TIMEOUT = 5
TKG_ERR_INTERNAL = 6

TKG_OPT_TIMEOUT_NS = 1
TKG_OPT_GROUP_M = 2
TKG_OPT_VARIANT = 3
TKG_OPT_MAX_CTAS = 4
TKG_OPT_LAUNCH_OVERLAP = 5
TKG_OPT_SCHEDULE = 6
TKG_OPT_SPLIT_K = 7
TKG_OPT_K_ORDER = 8

TKG_OVERLAP_ON = 1
TKG_OVERLAP_OFF = 2
TKG_SCHEDULE_STATIC = 1
TKG_SCHEDULE_DYNAMIC = 2
TKG_SCHEDULE_SINGLE = 3
TKG_SPLIT_ON = 1
TKG_SPLIT_OFF = 2
TKG_K_ORDER_SERPENTINE = 1
TKG_K_ORDER_FORWARD = 2

KIND_BF16, KIND_FP8, KIND_NVFP4 = 0, 1, 2


class tkg_scales(ctypes.Structure):
    _fields_ = [
        ("a_scale", ctypes.c_void_p),
        ("b_scale", ctypes.c_void_p),
        ("a_block_scale", ctypes.c_void_p),
        ("b_block_scale", ctypes.c_void_p),
    ]


class TkgError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_i64, _vp, _i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
for _name in ("tkg_gemm_bf16", "tkg_gemm_fp8", "tkg_gemm_nvfp4", "tkg_gemm_nvfp4_noalloc"):
    _f = getattr(lib, _name)
    _f.argtypes = [_i64, _i64, _i64, _vp, _vp, _vp, ctypes.POINTER(tkg_scales), _vp]
    _f.restype = _i32
lib.tkg_attention_fwd.argtypes = [_i64, _i64, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp]
lib.tkg_attention_fwd.restype = _i32
lib.tkg_check_status.argtypes = [_vp]
lib.tkg_check_status.restype = _i32
lib.tkg_status_string.argtypes = [_i32]
lib.tkg_status_string.restype = ctypes.c_char_p
lib.tkg_shutdown.argtypes = []
lib.tkg_shutdown.restype = None
lib.tkg_set_option.argtypes = [_i32, _i64]
lib.tkg_set_option.restype = _i32
lib.tkg_get_option.argtypes = [_i32]
lib.tkg_get_option.restype = _i64
lib.tkg_debug_tile_coord.argtypes = [_i32, _i32, _i32, _i32, ctypes.POINTER(_i32), ctypes.POINTER(_i32)]
lib.tkg_debug_tile_coord.restype = _i32
lib.tkg_debug_swizzle_offset.argtypes = [ctypes.c_uint32, ctypes.c_uint32]
lib.tkg_debug_swizzle_offset.restype = ctypes.c_uint32
lib.tkg_debug_select_swizzle.argtypes = [ctypes.c_uint32]
lib.tkg_debug_select_swizzle.restype = ctypes.c_uint32
lib.tkg_debug_variant_info.argtypes = [_i32, _i32, ctypes.POINTER(ctypes.c_int32)]
lib.tkg_debug_variant_info.restype = _i32
lib.tkg_debug_pick_variant.argtypes = [_i32, _i64, _i64, _i64, _i32]
lib.tkg_debug_pick_variant.restype = _i32
lib.tkg_debug_split_plan.argtypes = [_i64, _i64, _i32, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]
lib.tkg_debug_split_plan.restype = _i32
lib.tkg_debug_work_item.argtypes = [_i32, _i32, _i32, _i32, ctypes.POINTER(ctypes.c_int32)]
lib.tkg_debug_work_item.restype = _i32
lib.tkg_debug_set_fault.argtypes = [_i32]
lib.tkg_debug_set_fault.restype = _i32
lib.tkg_debug_set_visit_counter.argtypes = [_vp]
lib.tkg_debug_set_visit_counter.restype = _i32
lib.tkg_debug_tma_swizzle_probe.argtypes = [_i32, _vp, _vp, _vp]
lib.tkg_debug_tma_swizzle_probe.restype = _i32
lib.tkg_debug_mma_probe.argtypes = [_i32, _i32, _i32, _vp, _vp, _vp, _vp, ctypes.POINTER(ctypes.c_int32), _vp, _vp]
lib.tkg_debug_mma_probe.restype = _i32
lib.tkg_quantize_fp8.argtypes = [_i64, _i64, _vp, _vp, _vp, _vp]
lib.tkg_quantize_fp8.restype = _i32
lib.tkg_quantize_nvfp4.argtypes = [_i64, _i64, _vp, _vp, _vp, _vp, _vp]
lib.tkg_quantize_nvfp4.restype = _i32


def _addr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def status_string(status: int) -> str:
    return lib.tkg_status_string(int(status)).decode()


def _scales(scales):
    if scales is None:
        return None
    if isinstance(scales, tkg_scales):
        return ctypes.byref(scales)
    if isinstance(scales, dict):
        s = tkg_scales(*(_addr(scales.get(k)) for k in ("a_scale", "b_scale", "a_block_scale", "b_block_scale")))
    else:
        s = tkg_scales(*(_addr(v) for v in scales))
    return ctypes.byref(s)


def _check(status: int, where: str) -> int:
    if status != TKG_OK:
        raise TkgError(status, where)
    return status


def tkg_gemm_bf16(M, N, K, A, B, C, scales=None, stream=None, check=True) -> int:
    st = lib.tkg_gemm_bf16(M, N, K, _addr(A), _addr(B), _addr(C), _scales(scales), _stream(stream))
    return _check(st, "tkg_gemm_bf16") if check else st


def tkg_gemm_fp8(M, N, K, A, B, C, scales, stream=None, check=True) -> int:
    st = lib.tkg_gemm_fp8(M, N, K, _addr(A), _addr(B), _addr(C), _scales(scales), _stream(stream))
    return _check(st, "tkg_gemm_fp8") if check else st


def tkg_gemm_nvfp4(M, N, K, A, B, C, scales, stream=None, check=True) -> int:
    st = lib.tkg_gemm_nvfp4(M, N, K, _addr(A), _addr(B), _addr(C), _scales(scales), _stream(stream))
    return _check(st, "tkg_gemm_nvfp4") if check else st


def tkg_gemm_nvfp4_noalloc(M, N, K, A, B, C, scales, stream=None, check=True) -> int:
    """NVFP4 GEMM whose scale re-layout scratch is a fixed array inside the
    library instead of a pool allocation, for callers that must not allocate
    device memory during the call.  Calls that overlap on the GPU share that
    array and race; the first call on a device must precede any capture."""
    st = lib.tkg_gemm_nvfp4_noalloc(M, N, K, _addr(A), _addr(B), _addr(C), _scales(scales), _stream(stream))
    return _check(st, "tkg_gemm_nvfp4_noalloc") if check else st


def tkg_attention_fwd(B, H, Nq, Nkv, D, Q, K, V, O, lse=None, stream=None, check=True) -> int:
    """O = softmax(Q·Kᵀ/√D)·V per (batch, head); Q/O bf16 [B,H,Nq,D], K/V bf16
    [B,H,Nkv,D]; lse (optional) fp32 [B,H,Nq] receives each row's log-sum-exp."""
    st = lib.tkg_attention_fwd(B, H, Nq, Nkv, D, _addr(Q), _addr(K), _addr(V), _addr(O), _addr(lse),
                               _stream(stream))
    return _check(st, "tkg_attention_fwd") if check else st


def tkg_check_status(stream=None) -> int:
    return lib.tkg_check_status(_stream(stream))


def tkg_shutdown() -> None:
    lib.tkg_shutdown()


def tkg_set_option(key: int, value: int) -> None:
    _check(lib.tkg_set_option(key, int(value)), "tkg_set_option")


def tkg_get_option(key: int) -> int:
    return int(lib.tkg_get_option(key))


# ---- debug entry points ---------------------------------------------------

def tkg_debug_tile_coord(t, tiles_m, tiles_n, group_m):
    tm, tn = ctypes.c_int(), ctypes.c_int()
    rc = lib.tkg_debug_tile_coord(t, tiles_m, tiles_n, group_m, ctypes.byref(tm), ctypes.byref(tn))
    if rc != 0:
        raise ValueError("tile id out of range")
    return tm.value, tn.value


def tkg_debug_swizzle_offset(off, s_bytes) -> int:
    return int(lib.tkg_debug_swizzle_offset(off, s_bytes))


def tkg_debug_select_swizzle(row_bytes) -> int:
    return int(lib.tkg_debug_select_swizzle(row_bytes))


def tkg_debug_variant_info(kind, variant):
    info = (ctypes.c_int32 * 7)()
    _check(lib.tkg_debug_variant_info(kind, variant, info), "tkg_debug_variant_info")
    return dict(zip(("cta_group", "tile_n", "stages", "epilogue_warps", "threads", "smem_bytes", "tile_m"),
                    list(info)))


def tkg_debug_pick_variant(kind, M, N, K, sm_count=0) -> int:
    """Variant the GEMM of this shape launches on a device of sm_count SMs (0: the current device)."""
    return int(lib.tkg_debug_pick_variant(kind, M, N, K, sm_count))


def tkg_debug_split_plan(tiles, clusters, num_kb):
    """(split_tiles, split_s) of the split-K head for this grid."""
    t, s = ctypes.c_int32(), ctypes.c_int32()
    if lib.tkg_debug_split_plan(tiles, clusters, num_kb, ctypes.byref(t), ctypes.byref(s)) != 0:
        raise ValueError("tkg_debug_split_plan: invalid arguments")
    return t.value, s.value


def tkg_debug_work_item(w, split_tiles, split_s, num_kb):
    """(tile, first K stage, end K stage, piece or -1) of work item w."""
    out = (ctypes.c_int32 * 4)()
    if lib.tkg_debug_work_item(w, split_tiles, split_s, num_kb, out) != 0:
        raise ValueError("tkg_debug_work_item: invalid arguments")
    return tuple(out)


def tkg_debug_set_fault(mode: int) -> None:
    _check(lib.tkg_debug_set_fault(mode), "tkg_debug_set_fault")


def tkg_debug_set_visit_counter(counts) -> None:
    """Count tile visits of the next GEMM launch into `counts` (zeroed
    uint32/int32 device array, one word per output tile); None disables."""
    _check(lib.tkg_debug_set_visit_counter(_addr(counts)), "tkg_debug_set_visit_counter")


def tkg_debug_tma_swizzle_probe(s_bytes, src, dst, stream=None) -> int:
    return lib.tkg_debug_tma_swizzle_probe(s_bytes, _addr(src), _addr(dst), _stream(stream))


def tkg_debug_mma_probe(kind, n, ksteps, a_tile, b_tile, sfa=None, sfb=None, sf_cols=None, d_out=None,
                        stream=None) -> int:
    cols = None
    if sf_cols is not None:
        cols = (ctypes.c_int32 * len(sf_cols))(*[int(c) for c in sf_cols])
    return lib.tkg_debug_mma_probe(kind, n, ksteps, _addr(a_tile), _addr(b_tile), _addr(sfa), _addr(sfb), cols,
                                   _addr(d_out), _stream(stream))


def tkg_quantize_fp8(rows, cols, x, q, dequant_scale, stream=None, check=True) -> int:
    st = lib.tkg_quantize_fp8(rows, cols, _addr(x), _addr(q), _addr(dequant_scale), _stream(stream))
    return _check(st, "tkg_quantize_fp8") if check else st


def tkg_quantize_nvfp4(rows, cols, x, q_packed, block_scales, global_scale, stream=None, check=True) -> int:
    st = lib.tkg_quantize_nvfp4(rows, cols, _addr(x), _addr(q_packed), _addr(block_scales), _addr(global_scale),
                                _stream(stream))
    return _check(st, "tkg_quantize_nvfp4") if check else st

