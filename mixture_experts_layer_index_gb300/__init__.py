"""Python binding of libmoe_gb300.so, the GB300 (sm_103a) routed MoE FFN forward.

Argument marshalling only: every step of the forward runs in the library's
CUDA kernels.  Functions carry the C ABI's names (include/moe.h) and take
torch CUDA tensors for device memory (plus the current torch stream by
default); each raises MoeError when the library returns a non-OK status.

The library must have been built (``build.build()`` or
``__graft_entry__.build()``); the first call into it raises RuntimeError if it
is missing - there is no other implementation to fall back on.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_gb300.so")

# moe_status
MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_DEVICE_TIMEOUT = 5
MOE_ERR_DEVICE_BOUNDS = 6
# moe_quant
MOE_BF16 = 0
MOE_FP8_PER_TENSOR = 1
MOE_FP8_BLOCK128 = 2
MOE_MXFP8 = 3
# moe_path
MOE_PATH_AUTO = 0
MOE_PATH_GROUPED = 1
MOE_PATH_ROUTE_DIRECT = 2

QUANT_BY_NAME = {"bf16": MOE_BF16, "fp8_tensor": MOE_FP8_PER_TENSOR, "fp8_block": MOE_FP8_BLOCK128,
                 "mxfp8": MOE_MXFP8}
GEMM_BM = 128  # row-tile height of the grouped GEMMs (tile map of moe_forward)


class moe_problem(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("E", ctypes.c_int), ("k", ctypes.c_int), ("H", ctypes.c_int),
                ("I", ctypes.c_int), ("quant", ctypes.c_int), ("path", ctypes.c_int)]


class moe_views(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("ids", "w", "counts", "offsets", "perm", "inv", "tiles", "num_tiles", "xs", "x_scale",
                 "amax_x")]


class moe_forward_options(ctypes.Structure):
    _fields_ = [("n_shared", ctypes.c_int), ("w1_shared", ctypes.c_void_p), ("w2_shared", ctypes.c_void_p),
                ("w1_shared_scale", ctypes.c_void_p), ("w2_shared_scale", ctypes.c_void_p), ("y_fp32", ctypes.c_int),
                ("mx_weight_scales_blocked", ctypes.c_int)]


class moe_stage_time(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("total_ms", ctypes.c_double), ("launches", ctypes.c_int)]


_vp, _sz, _i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
_P = ctypes.POINTER(moe_problem)
_O = ctypes.POINTER(moe_forward_options)
_SIGS = {
    "moe_route": (_i, [_vp, _i, _i, _i, _vp, _vp, _vp]),
    "moe_shuffle_workspace_size": (_sz, [_i, _i, _i]),
    "moe_shuffle": (_i, [_vp, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_shuffle_noalloc": (_i, [_vp, _i, _i, _i, _vp, _vp, _vp, _vp, _vp]),
    "moe_tile_map": (_i, [_vp, _i, _i, _vp, _vp, _i, _vp, _sz, _vp]),
    "moe_select_path": (_i, [_P]),
    "moe_workspace_size": (_sz, [_P]),
    "moe_forward": (_i, [_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_forward_views": (_i, [_P, _vp, _sz, ctypes.POINTER(moe_views)]),
    "moe_workspace_size_ex": (_sz, [_P, _O]),
    "moe_forward_ex": (_i, [_P, _O, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_forward_views_ex": (_i, [_P, _O, _vp, _sz, ctypes.POINTER(moe_views)]),
    "moe_round_bf16": (_i, [_vp, _vp, _sz, _vp]),
    "moe_mx_blocked_bytes": (_sz, [_i, _i, _i]),
    "moe_mx_weight_scales_bytes": (_sz, [_i, _i, _i, _i]),
    "moe_mx_weight_scales": (_i, [_vp, _vp, _i, _i, _i, _vp, _vp, _vp]),
    "moe_mx_blocked_workspace_size": (_sz, [_i, _i]),
    "moe_mx_blocked_scales": (_i, [_vp, _i, _i, _vp, _i, _vp, _sz, _vp, _vp, _sz, _vp]),
    "moe_read_device_status": (_i, [_vp, _vp]),
    "moe_profile_start": (_i, []),
    "moe_profile_start_stage": (_i, [ctypes.c_char_p]),
    "moe_profile_stop": (_i, [ctypes.POINTER(moe_stage_time), _i]),
    "moe_status_string": (ctypes.c_char_p, [_i]),
}
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with mixture_experts_layer_index_gb300.build.build() "
                "(the CUDA library is the only implementation)")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(handle, name)
            f.restype = res
            f.argtypes = args
        _lib = handle
    return _lib


EXPORTED = tuple(_SIGS)


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {moe_status_string(status)} (status {status})")


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != MOE_OK:
        raise MoeError(status, where)


def _ptr(t) -> Optional[int]:
    """Device pointer of a contiguous CUDA tensor (None -> NULL; ints pass through)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def problem(T: int, E: int, k: int, H: int, I: int, quant=MOE_BF16, path=MOE_PATH_AUTO) -> moe_problem:
    if isinstance(quant, str):
        quant = QUANT_BY_NAME[quant]
    return moe_problem(T, E, k, H, I, int(quant), int(path))


def moe_route(scores, T, E, k, ids, w, stream=None) -> None:
    _check(lib().moe_route(_ptr(scores), T, E, k, _ptr(ids), _ptr(w), _stream(stream)), "moe_route")


def moe_shuffle_workspace_size(T, E, k) -> int:
    return int(lib().moe_shuffle_workspace_size(T, E, k))


def moe_shuffle(ids, T, E, k, counts, offsets, perm, inv, ws, ws_bytes=None, stream=None) -> None:
    nb = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(lib().moe_shuffle(_ptr(ids), T, E, k, _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv), _ptr(ws), nb,
                            _stream(stream)), "moe_shuffle")


def moe_shuffle_noalloc(ids, T, E, k, counts, offsets, perm, inv, stream=None) -> None:
    """moe_shuffle with the library's fixed scratch array instead of a workspace
    (for callers that cannot allocate device memory; see include/moe.h)."""
    _check(lib().moe_shuffle_noalloc(_ptr(ids), T, E, k, _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv),
                                     _stream(stream)), "moe_shuffle_noalloc")


def moe_tile_map(counts, E, BM, tiles, num_tiles, max_tiles, ws, ws_bytes=None, stream=None) -> None:
    nb = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(lib().moe_tile_map(_ptr(counts), E, BM, _ptr(tiles), _ptr(num_tiles), max_tiles, _ptr(ws), nb,
                             _stream(stream)), "moe_tile_map")


def moe_select_path(p: moe_problem) -> int:
    return int(lib().moe_select_path(ctypes.byref(p)))


def moe_workspace_size(p: moe_problem) -> int:
    return int(lib().moe_workspace_size(ctypes.byref(p)))


def moe_forward(p: moe_problem, x, scores, w1, w2, w1_scale, w2_scale, y, ws, ws_bytes=None, stream=None) -> None:
    nb = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(lib().moe_forward(ctypes.byref(p), _ptr(x), _ptr(scores), _ptr(w1), _ptr(w2), _ptr(w1_scale),
                            _ptr(w2_scale), _ptr(y), _ptr(ws), nb, _stream(stream)), "moe_forward")


def forward_options(n_shared=0, w1_shared=None, w2_shared=None, w1_shared_scale=None, w2_shared_scale=None,
                    y_fp32=False, mx_weight_scales_blocked=False) -> moe_forward_options:
    return moe_forward_options(int(n_shared), _ptr(w1_shared), _ptr(w2_shared), _ptr(w1_shared_scale),
                               _ptr(w2_shared_scale), 1 if y_fp32 else 0, 1 if mx_weight_scales_blocked else 0)


def _opt_ref(opt):
    return None if opt is None else ctypes.byref(opt)


def moe_workspace_size_ex(p: moe_problem, opt: Optional[moe_forward_options]) -> int:
    return int(lib().moe_workspace_size_ex(ctypes.byref(p), _opt_ref(opt)))


def moe_forward_ex(p: moe_problem, opt: Optional[moe_forward_options], x, scores, w1, w2, w1_scale, w2_scale, y, ws,
                   ws_bytes=None, stream=None) -> None:
    nb = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(lib().moe_forward_ex(ctypes.byref(p), _opt_ref(opt), _ptr(x), _ptr(scores), _ptr(w1), _ptr(w2),
                               _ptr(w1_scale), _ptr(w2_scale), _ptr(y), _ptr(ws), nb, _stream(stream)),
           "moe_forward_ex")


def moe_forward_views_ex(p: moe_problem, opt: Optional[moe_forward_options], ws, ws_bytes=None) -> moe_views:
    nb = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    v = moe_views()
    _check(lib().moe_forward_views_ex(ctypes.byref(p), _opt_ref(opt), _ptr(ws), nb, ctypes.byref(v)),
           "moe_forward_views_ex")
    return v


def moe_round_bf16(y32, y, n=None, stream=None) -> None:
    n = y32.numel() if n is None else n
    _check(lib().moe_round_bf16(_ptr(y32), _ptr(y), n, _stream(stream)), "moe_round_bf16")


def moe_mx_weight_scales_bytes(E: int, H: int, I: int, which: int) -> int:
    return int(lib().moe_mx_weight_scales_bytes(E, H, I, which))


def moe_mx_weight_scales(w1_scale, w2_scale, E, H, I, w1_blocked, w2_blocked, stream=None) -> None:
    """MXFP8 weight scales converted once into the forward's blocked layouts."""
    _check(lib().moe_mx_weight_scales(_ptr(w1_scale), _ptr(w2_scale), E, H, I, _ptr(w1_blocked), _ptr(w2_blocked),
                                     _stream(stream)), "moe_mx_weight_scales")


def moe_mx_blocked_bytes(rows: int, cols: int, groups: int) -> int:
    return int(lib().moe_mx_blocked_bytes(rows, cols, groups))


def moe_mx_blocked_workspace_size(rows: int, groups: int) -> int:
    return int(lib().moe_mx_blocked_workspace_size(rows, groups))


def moe_mx_blocked_scales(scales, rows, cols, group_offsets, groups, out, group_starts, ws, out_bytes=None,
                          ws_bytes=None, stream=None) -> None:
    """Per-group blocked layout of MX scales (see include/moe.h)."""
    ob = out.numel() * out.element_size() if out_bytes is None else out_bytes
    nb = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(lib().moe_mx_blocked_scales(_ptr(scales), rows, cols, _ptr(group_offsets), groups, _ptr(out), ob,
                                      _ptr(group_starts), _ptr(ws), nb, _stream(stream)), "moe_mx_blocked_scales")


def moe_forward_views(p: moe_problem, ws, ws_bytes=None) -> moe_views:
    nb = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    v = moe_views()
    _check(lib().moe_forward_views(ctypes.byref(p), _ptr(ws), nb, ctypes.byref(v)), "moe_forward_views")
    return v


def moe_read_device_status(ws, stream=None) -> int:
    return int(lib().moe_read_device_status(_ptr(ws), _stream(stream)))


def moe_profile_start() -> None:
    lib().moe_profile_start()


def moe_profile_start_stage(stage: str) -> None:
    """Profile only the launches of one stage (e.g. "gateup_gemm")."""
    lib().moe_profile_start_stage(stage.encode() if stage else None)


def moe_profile_stop(max_stages: int = 32) -> dict:
    """Stops stage timing; returns {stage name: (total_ms, launches)} in launch order."""
    arr = (moe_stage_time * max_stages)()
    n = int(lib().moe_profile_stop(arr, max_stages))
    if n < 0:
        raise MoeError(MOE_ERR_CUDA, "moe_profile_stop")
    return {arr[i].name.decode(): (float(arr[i].total_ms), int(arr[i].launches)) for i in range(min(n, max_stages))}


def raw_status(fn_name: str, *args) -> int:
    """Call an entry point with raw arguments and return its status code
    (used by boundary tests that pass NULL or misaligned pointers)."""
    return int(getattr(lib(), fn_name)(*args))
