"""Thin Python binding of libmc2moe (ctypes).

Argument marshalling only: every step of the block runs in the library's
CUDA kernels.  PyTorch supplies device memory and the current stream.  The
functions carry the C entry points' names and argument order; tensors are
passed as raw pointers (``None`` -> NULL).  If the shared library is missing
the binding raises -- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmc2moe.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "mc2moe.h")

MC2_OK, MC2_ERR_INVALID_ARG, MC2_ERR_UNSUPPORTED, MC2_ERR_CUDA = 0, 1, 2, 3
MC2_ERR_DEVICE_TIMEOUT, MC2_ERR_BAD_EXPERT_ID = 4, 5
MC2_DEV_BAD_EXPERT_ID, MC2_DEV_TIMEOUT, MC2_DEV_INTERNAL = 0x1, 0x2, 0x4
DTYPE = {"f32": 0, "bf16": 1, "i8": 2, "i32": 3}


class Mc2Error(RuntimeError):
    def __init__(self, fn, status, text):
        super().__init__(f"{fn}: {text} (status {status})")
        self.status = status


class Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("T", "H", "I", "E", "k", "W", "act", "out")]

    @classmethod
    def make(cls, T, H, I, E, k, W, act="bf16", out=None):
        if out is None:
            out = {"f32": "f32", "bf16": "bf16", "i8": "bf16"}[act]
        return cls(T, H, I, E, k, W, DTYPE[act], DTYPE[out])


_lib = None
_P = ctypes.c_void_p
_SP = ctypes.POINTER(Shape)

_SIGS = {
    "mc2_check_shape": (ctypes.c_int, [_SP]),
    "mc2_workspace_bytes": (ctypes.c_size_t, [_SP]),
    "mc2_moe_counts": (ctypes.c_int, [_SP] + [_P] * 9),
    "mc2_moe_counts_static": (ctypes.c_int, [_SP] + [_P] * 8),
    "mc2_alltoallv_gmm": (ctypes.c_int, [_SP] + [_P] * 11),
    "mc2_gmm_alltoallv": (ctypes.c_int, [_SP] + [_P] * 12),
    "mc2_moe_forward": (ctypes.c_int, [_SP] + [_P] * 19),
    "mc2_permute_rows": (ctypes.c_int, [_SP] + [_P] * 4),
    "mc2_backward_workspace_bytes": (ctypes.c_size_t, [_SP]),
    "mc2_transpose_weights": (ctypes.c_int, [_SP] + [_P] * 5),
    "mc2_moe_backward": (ctypes.c_int, [_SP] + [_P] * 17),
    "mc2_alltoallv_gmm_keep": (ctypes.c_int, [_SP] + [_P] * 8),
    "mc2_mm_reduce_scatter_workspace_bytes": (ctypes.c_size_t, [ctypes.c_void_p]),
    "mc2_mm_reduce_scatter_i8": (ctypes.c_int, [ctypes.c_void_p] + [_P] * 8),
    "mc2_gmm_swiglu": (ctypes.c_int, [_SP] + [_P] * 6),
    "mc2_prepack_weights": (ctypes.c_int, [_SP] + [_P] * 4),
    "mc2_selftest_wait": (ctypes.c_int, [ctypes.c_uint64, _P, _P]),
    "mc2_set_wait_limit_ns": (None, [ctypes.c_uint64]),
    "mc2_set_tile_pairing": (None, [ctypes.c_int32]),
    "mc2_set_launch_overlap": (None, [ctypes.c_int32]),
    "mc2_set_counts_path": (None, [ctypes.c_int32]),
    "mc2_set_mmrs_path": (None, [ctypes.c_int32]),
    "mc2_set_combine_path": (None, [ctypes.c_int32]),
    "mc2_set_gemm_events": (None, [ctypes.c_void_p, ctypes.c_void_p]),
    "mc2_last_launch_count": (ctypes.c_int32, []),
    "mc2_status_str": (ctypes.c_char_p, [ctypes.c_int]),
}


def header_functions():
    """Names of the functions include/mc2moe.h declares."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mc2_\w+)\s*\(", src)))


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libmc2moe.so is not built ({LIB_PATH}); run "
                "moe_expert_dispatch_histc_gb300.build.build() -- there is no fallback path")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, st):
    if st != MC2_OK:
        raise Mc2Error(fn, st, lib().mc2_status_str(st).decode())


def status_str(st: int) -> str:
    return lib().mc2_status_str(st).decode()


def mc2_check_shape(shape: Shape) -> int:
    return lib().mc2_check_shape(ctypes.byref(shape))


def mc2_workspace_bytes(shape: Shape) -> int:
    return lib().mc2_workspace_bytes(ctypes.byref(shape))


def mc2_moe_counts(shape, sel, cnt, recv, offsets, permute_src, unpermute_dst, ws,
                   dev_status=None, stream=None, check=True):
    st = lib().mc2_moe_counts(ctypes.byref(shape), _p(sel), _p(cnt), _p(recv), _p(offsets),
                              _p(permute_src), _p(unpermute_dst), _p(ws), _p(dev_status),
                              _stream(stream))
    if check:
        _check("mc2_moe_counts", st)
    return st


def mc2_moe_counts_static(shape, sel, cnt, recv, offsets, permute_src, unpermute_dst,
                          dev_status=None, stream=None, check=True):
    """mc2_moe_counts without a workspace, for callers that cannot allocate
    device memory; its scratch is a fixed array inside the library."""
    st = lib().mc2_moe_counts_static(ctypes.byref(shape), _p(sel), _p(cnt), _p(recv),
                                     _p(offsets), _p(permute_src), _p(unpermute_dst),
                                     _p(dev_status), _stream(stream))
    if check:
        _check("mc2_moe_counts_static", st)
    return st


def mc2_alltoallv_gmm(shape, x, x_scale, w1, w1_scale, offsets, permute_src, ws, h, h_scale,
                      dev_status=None, stream=None, check=True):
    st = lib().mc2_alltoallv_gmm(ctypes.byref(shape), _p(x), _p(x_scale), _p(w1), _p(w1_scale),
                                 _p(offsets), _p(permute_src), _p(ws), _p(h), _p(h_scale),
                                 _p(dev_status), _stream(stream))
    if check:
        _check("mc2_alltoallv_gmm", st)
    return st


def mc2_gmm_alltoallv(shape, h, h_scale, w2, w2_scale, offsets, permute_src, unpermute_dst,
                      probs, ws, out, dev_status=None, stream=None, check=True):
    st = lib().mc2_gmm_alltoallv(ctypes.byref(shape), _p(h), _p(h_scale), _p(w2), _p(w2_scale),
                                 _p(offsets), _p(permute_src), _p(unpermute_dst), _p(probs),
                                 _p(ws), _p(out), _p(dev_status), _stream(stream))
    if check:
        _check("mc2_gmm_alltoallv", st)
    return st


def mc2_backward_workspace_bytes(shape) -> int:
    return int(lib().mc2_backward_workspace_bytes(ctypes.byref(shape)))


def mc2_transpose_weights(shape, w1, w2, w1t, w2t, stream=None, check=True):
    st = lib().mc2_transpose_weights(ctypes.byref(shape), _p(w1), _p(w2), _p(w1t), _p(w2t),
                                     _stream(stream))
    if check:
        _check("mc2_transpose_weights", st)
    return st


def mc2_alltoallv_gmm_keep(shape, x, w1, offsets, permute_src, h, g, dev_status=None,
                           stream=None, check=True):
    st = lib().mc2_alltoallv_gmm_keep(ctypes.byref(shape), _p(x), _p(w1), _p(offsets),
                                      _p(permute_src), _p(h), _p(g), _p(dev_status),
                                      _stream(stream))
    if check:
        _check("mc2_alltoallv_gmm_keep", st)
    return st


def mc2_moe_backward(shape, x, probs, w1, w1t, w2t, dout, offsets, permute_src, unpermute_dst,
                     dx, dw1, dw2, dprobs, ws, dev_status=None, stream=None, check=True, g=None):
    st = lib().mc2_moe_backward(ctypes.byref(shape), _p(x), _p(probs), _p(w1), _p(g), _p(w1t),
                                _p(w2t),
                                _p(dout), _p(offsets), _p(permute_src), _p(unpermute_dst),
                                _p(dx), _p(dw1), _p(dw2), _p(dprobs), _p(ws), _p(dev_status),
                                _stream(stream))
    if check:
        _check("mc2_moe_backward", st)
    return st


class MmrsShape(ctypes.Structure):
    """mc2_mmrs_shape_t: quantised matmul + reduce-scatter over W logical ranks."""
    _fields_ = [("m", ctypes.c_int32), ("k", ctypes.c_int32), ("n", ctypes.c_int32),
                ("W", ctypes.c_int32)]


def mc2_mm_reduce_scatter_workspace_bytes(shape) -> int:
    return int(lib().mc2_mm_reduce_scatter_workspace_bytes(ctypes.byref(shape)))


def mc2_mm_reduce_scatter_i8(shape, x1, x1_scale, x2, x2_scale, out, ws, dev_status=None,
                             stream=None, check=True):
    st = lib().mc2_mm_reduce_scatter_i8(ctypes.byref(shape), _p(x1), _p(x1_scale), _p(x2),
                                        _p(x2_scale), _p(out), _p(ws), _p(dev_status),
                                        _stream(stream))
    if check:
        _check("mc2_mm_reduce_scatter_i8", st)
    return st


def mc2_permute_rows(shape, x, permute_src, xp, stream=None, check=True):
    st = lib().mc2_permute_rows(ctypes.byref(shape), _p(x), _p(permute_src), _p(xp),
                                _stream(stream))
    if check:
        _check("mc2_permute_rows", st)
    return st


def mc2_gmm_swiglu(shape, xp, w1, offsets, h, dev_status=None, stream=None, check=True):
    st = lib().mc2_gmm_swiglu(ctypes.byref(shape), _p(xp), _p(w1), _p(offsets), _p(h),
                              _p(dev_status), _stream(stream))
    if check:
        _check("mc2_gmm_swiglu", st)
    return st


def mc2_moe_forward(shape, x, x_scale, sel, probs, w1, w1_scale, w2, w2_scale, cnt, recv,
                    offsets, permute_src, unpermute_dst, h, h_scale, out, ws,
                    dev_status=None, stream=None, check=True):
    st = lib().mc2_moe_forward(ctypes.byref(shape), _p(x), _p(x_scale), _p(sel), _p(probs),
                               _p(w1), _p(w1_scale), _p(w2), _p(w2_scale), _p(cnt), _p(recv),
                               _p(offsets), _p(permute_src), _p(unpermute_dst), _p(h),
                               _p(h_scale), _p(out), _p(ws), _p(dev_status), _stream(stream))
    if check:
        _check("mc2_moe_forward", st)
    return st


def mc2_prepack_weights(shape, w1, w2, ws, stream=None, check=True):
    st = lib().mc2_prepack_weights(ctypes.byref(shape), _p(w1), _p(w2), _p(ws), _stream(stream))
    if check:
        _check("mc2_prepack_weights", st)
    return st


def mc2_selftest_wait(limit_ns, dev_status, stream=None, check=True):
    st = lib().mc2_selftest_wait(int(limit_ns), _p(dev_status), _stream(stream))
    if check:
        _check("mc2_selftest_wait", st)
    return st


def mc2_set_wait_limit_ns(limit_ns: int) -> None:
    lib().mc2_set_wait_limit_ns(int(limit_ns))


def mc2_set_tile_pairing(mode: int) -> None:
    lib().mc2_set_tile_pairing(int(mode))


def mc2_set_launch_overlap(enabled: int) -> None:
    lib().mc2_set_launch_overlap(int(enabled))


def mc2_set_counts_path(mode: int) -> None:
    lib().mc2_set_counts_path(int(mode))


def mc2_set_mmrs_path(mode: int) -> None:
    lib().mc2_set_mmrs_path(int(mode))


def mc2_set_combine_path(mode: int) -> None:
    """0: the weighted combine in its own kernel (default); 1: inside the fc2 kernel."""
    lib().mc2_set_combine_path(int(mode))


def mc2_set_gemm_events(before, after) -> None:
    """CUDA events recorded around the fc1 / fc2 kernel of later calls of this
    thread (torch.cuda.Event objects, already recorded once so that they exist,
    or None); mc2_set_gemm_events(None, None) stops it."""
    def handle(ev):
        if ev is None:
            return None
        h = int(ev.cuda_event)
        if h == 0:  # torch creates the CUDA event at its first record
            raise ValueError("mc2_set_gemm_events: record the event once before passing it")
        return ctypes.c_void_p(h)
    hb, ha = handle(before), handle(after)
    lib().mc2_set_gemm_events(hb, ha)


def mc2_last_launch_count() -> int:
    return lib().mc2_last_launch_count()
