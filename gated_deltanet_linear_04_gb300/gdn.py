"""Thin Python binding of the C ABI in include/gdn.h (ctypes).

Argument marshalling only: every function here checks tensor dtypes, devices,
contiguity and element counts, passes raw device pointers and the current CUDA stream to the
library, and raises ``GdnError`` on a non-zero status.  All arithmetic runs in
the CUDA kernels of libgdn.so; there is no fallback.  PyTorch provides device
memory and streams.

The functions named like the ABI (``gdn_conv_update`` ...) take
caller-allocated outputs; the short names (``conv_update`` ...) allocate
outputs with torch and return them.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libgdn.so")

GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_CUDA, GDN_ERR_TIMEOUT = range(5)

# batch rows gdn_prefill_noalloc accepts (GDN_NOALLOC_MAX_ROWS in gdn.h)
GDN_NOALLOC_MAX_ROWS = 4096


class GdnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s" % (where, status_string(status)))


class GdnDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("Hk", ctypes.c_int32), ("Hv", ctypes.c_int32),
                ("Dk", ctypes.c_int32), ("Dv", ctypes.c_int32), ("K", ctypes.c_int32), ("eps_qk", ctypes.c_float)]


_lib = None

_P = ctypes.c_void_p
_SIGS = {
    "gdn_conv_update": (ctypes.c_int, [ctypes.POINTER(GdnDims), _P, _P, _P, _P, _P, _P, _P, _P]),
    "gdn_gating": (ctypes.c_int, [ctypes.POINTER(GdnDims), _P, _P, _P, _P, _P, _P, _P]),
    "gdn_recurrent_decode": (ctypes.c_int, [ctypes.POINTER(GdnDims), _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "gdn_prefill": (ctypes.c_int, [ctypes.POINTER(GdnDims), _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_int, _P,
                                   ctypes.c_size_t, _P]),
    "gdn_recurrent_decode_gated": (ctypes.c_int, [ctypes.POINTER(GdnDims)] + [_P] * 11 +
                                   [ctypes.c_float, _P, _P]),
    "gdn_prefill_gated": (ctypes.c_int, [ctypes.POINTER(GdnDims)] + [_P] * 10 +
                          [ctypes.c_float, _P, ctypes.c_int, _P, ctypes.c_size_t, _P]),
    "gdn_prefill_backward_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(GdnDims)]),
    "gdn_prefill_backward": (ctypes.c_int, [ctypes.POINTER(GdnDims)] + [_P] * 16 + [ctypes.c_size_t, _P]),
    "gdn_prefill_backward_chunked_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(GdnDims)]),
    "gdn_prefill_backward_chunked": (ctypes.c_int, [ctypes.POINTER(GdnDims)] + [_P] * 16 + [ctypes.c_size_t, _P]),
    "gdn_prefill_vec": (ctypes.c_int, [ctypes.POINTER(GdnDims), _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "gdn_prefill_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(GdnDims), ctypes.c_int]),
    "gdn_prefill_noalloc": (ctypes.c_int, [ctypes.POINTER(GdnDims)] + [ctypes.c_void_p] * 9 +
                            [ctypes.c_int, ctypes.c_void_p]),
    "gdn_decode_window": (ctypes.c_int, [ctypes.POINTER(GdnDims), _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "gdn_recurrent_decode_host_steps": (ctypes.c_int, [ctypes.POINTER(GdnDims), ctypes.c_int] + [_P] * 11 +
                                        [ctypes.c_size_t, _P]),
    "gdn_decode_host_staging_size": (ctypes.c_size_t, [ctypes.POINTER(GdnDims)]),
    "gdn_rmsnorm_gated": (ctypes.c_int, [ctypes.POINTER(GdnDims), _P, _P, _P, ctypes.c_float, _P, _P]),
    "gdn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "gdn_device_status": (ctypes.c_int, [_P]),
    "gdn_selftest_timeout": (ctypes.c_int, [_P]),
    "gdn_abi_version": (ctypes.c_int, []),
}


def lib():
    """The loaded libgdn.so.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libgdn.so is not built (%s); run __graft_entry__.build() first" % LIB_PATH)
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib = l
    return _lib


def status_string(status: int) -> str:
    return lib().gdn_status_string(int(status)).decode()


def make_dims(d) -> GdnDims:
    return GdnDims(int(d.B), int(d.T), int(d.Hk), int(d.Hv), int(d.Dk), int(d.Dv), int(d.K),
                   float(getattr(d, "eps_qk", 1e-6)))


def _ptr(t: Optional[torch.Tensor], dtype: torch.dtype, name: str):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor or None" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if t.numel() > 0 and not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr() or None


def _host_ptr(t: torch.Tensor, dtype: torch.dtype, name: str):
    """A contiguous CPU tensor's address (page-locked ones copy asynchronously)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if t.is_cuda:
        raise ValueError("%s must be a host (CPU) tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr() or None


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream or None
    return int(stream) or None


def _check(status: int, where: str):
    if status != GDN_OK:
        raise GdnError(status, where)


class _Counts:
    """Element counts of every buffer of the ABI for given dims (the layouts
    of include/gdn.h); the library sees only addresses, so the binding
    compares each tensor's size with these before passing it on."""

    def __init__(self, d: GdnDims):
        B, T, Hk, Hv, Dk, Dv, K = d.B, d.T, d.Hk, d.Hv, d.Dk, d.Dv, d.K
        C = 2 * Hk * Dk + Hv * Dv
        self.qkv, self.conv_w, self.conv_state = B * T * C, C * K, B * (K - 1) * C
        self.mask, self.qk, self.v, self.gate = B * T, B * T * Hk * Dk, B * T * Hv * Dv, B * T * Hv
        self.head, self.state, self.row, self.norm_w = Hv, B * Hv * Dv * Dk, B, Dv
        self.g_vec = B * T * Hv * Dk


def _sizes(where: str, *items):
    """Raises if a given tensor's element count differs from the expected one
    (items: (name, tensor or None, count))."""
    for name, t, n in items:
        if isinstance(t, torch.Tensor) and t.numel() != n:
            raise ValueError("%s: %s must hold %d elements for these dims, got %d" % (where, name, n, t.numel()))


BF16, F32, U8 = torch.bfloat16, torch.float32, torch.uint8


# ---------------------------------------------------------------------------
# ABI-named calls (caller-allocated outputs)
# ---------------------------------------------------------------------------
def gdn_conv_update(dims, qkv, conv_w, conv_state, mask, q, k, v, stream=None):
    d = make_dims(dims)
    n = _Counts(d)
    _sizes("gdn_conv_update", ("qkv", qkv, n.qkv), ("conv_w", conv_w, n.conv_w),
           ("conv_state", conv_state, n.conv_state), ("mask", mask, n.mask), ("q", q, n.qk), ("k", k, n.qk),
           ("v", v, n.v))
    _check(lib().gdn_conv_update(ctypes.byref(d), _ptr(qkv, BF16, "qkv"), _ptr(conv_w, BF16, "conv_w"),
                                 _ptr(conv_state, BF16, "conv_state"), _ptr(mask, U8, "mask"), _ptr(q, BF16, "q"),
                                 _ptr(k, BF16, "k"), _ptr(v, BF16, "v"), _stream(stream)), "gdn_conv_update")


def gdn_gating(dims, a, b, A_log, dt_bias, g, beta, stream=None):
    d = make_dims(dims)
    n = _Counts(d)
    _sizes("gdn_gating", ("a", a, n.gate), ("b", b, n.gate), ("A_log", A_log, n.head), ("dt_bias", dt_bias, n.head),
           ("g", g, n.gate), ("beta", beta, n.gate))
    _check(lib().gdn_gating(ctypes.byref(d), _ptr(a, BF16, "a"), _ptr(b, BF16, "b"), _ptr(A_log, F32, "A_log"),
                            _ptr(dt_bias, F32, "dt_bias"), _ptr(g, F32, "g"), _ptr(beta, F32, "beta"),
                            _stream(stream)), "gdn_gating")


def gdn_recurrent_decode(dims, qkv, conv_w, conv_state, a, b, A_log, dt_bias, state, row_mask, y, stream=None):
    d = make_dims(dims)
    n = _Counts(d)
    _sizes("gdn_recurrent_decode", ("qkv", qkv, n.qkv), ("conv_w", conv_w, n.conv_w),
           ("conv_state", conv_state, n.conv_state), ("a", a, n.gate), ("b", b, n.gate), ("A_log", A_log, n.head),
           ("dt_bias", dt_bias, n.head), ("state", state, n.state), ("row_mask", row_mask, n.row), ("y", y, n.v))
    _check(lib().gdn_recurrent_decode(ctypes.byref(d), _ptr(qkv, BF16, "qkv"), _ptr(conv_w, BF16, "conv_w"),
                                      _ptr(conv_state, BF16, "conv_state"), _ptr(a, BF16, "a"), _ptr(b, BF16, "b"),
                                      _ptr(A_log, F32, "A_log"), _ptr(dt_bias, F32, "dt_bias"),
                                      _ptr(state, F32, "state"), _ptr(row_mask, U8, "row_mask"),
                                      _ptr(y, BF16, "y"), _stream(stream)), "gdn_recurrent_decode")


def gdn_decode_window(dims, qkv, conv_w, conv_state, a, b, A_log, dt_bias, state, keep, y, stream=None):
    d = make_dims(dims)
    n = _Counts(d)
    _sizes("gdn_decode_window", ("qkv", qkv, n.qkv), ("conv_w", conv_w, n.conv_w),
           ("conv_state", conv_state, n.conv_state), ("a", a, n.gate), ("b", b, n.gate), ("A_log", A_log, n.head),
           ("dt_bias", dt_bias, n.head), ("state", state, n.state), ("keep", keep, n.row), ("y", y, n.v))
    _check(lib().gdn_decode_window(ctypes.byref(d), _ptr(qkv, BF16, "qkv"), _ptr(conv_w, BF16, "conv_w"),
                                   _ptr(conv_state, BF16, "conv_state"), _ptr(a, BF16, "a"), _ptr(b, BF16, "b"),
                                   _ptr(A_log, F32, "A_log"), _ptr(dt_bias, F32, "dt_bias"),
                                   _ptr(state, F32, "state"), _ptr(keep, torch.int32, "keep"), _ptr(y, BF16, "y"),
                                   _stream(stream)), "gdn_decode_window")


def gdn_decode_host_staging_size(dims) -> int:
    d = make_dims(dims)
    return int(lib().gdn_decode_host_staging_size(ctypes.byref(d)))


def gdn_recurrent_decode_host_steps(dims, n_steps, qkv_h, a_h, b_h, y_h, conv_w, conv_state, A_log, dt_bias, state,
                                    row_mask, staging, stream=None):
    d = make_dims(dims)
    n1 = _Counts(d)
    _sizes("gdn_recurrent_decode_host_steps", ("conv_w", conv_w, n1.conv_w),
           ("conv_state", conv_state, n1.conv_state), ("A_log", A_log, n1.head), ("dt_bias", dt_bias, n1.head),
           ("state", state, n1.state), ("row_mask", row_mask, n1.row))
    n = int(n_steps)
    for name, t, shape in (("qkv_h", qkv_h, (n, dims.B, d.Hk * d.Dk * 2 + d.Hv * d.Dv)),
                           ("a_h", a_h, (n, dims.B, d.Hv)), ("b_h", b_h, (n, dims.B, d.Hv)),
                           ("y_h", y_h, (n, dims.B, d.Hv, d.Dv))):
        if tuple(t.shape[:len(shape)]) != shape or t.numel() != _numel(shape):
            raise ValueError("%s must have shape %s, got %s" % (name, shape, tuple(t.shape)))
    _check(lib().gdn_recurrent_decode_host_steps(
        ctypes.byref(d), n, _host_ptr(qkv_h, BF16, "qkv_h"), _host_ptr(a_h, BF16, "a_h"),
        _host_ptr(b_h, BF16, "b_h"), _host_ptr(y_h, BF16, "y_h"), _ptr(conv_w, BF16, "conv_w"),
        _ptr(conv_state, BF16, "conv_state"), _ptr(A_log, F32, "A_log"), _ptr(dt_bias, F32, "dt_bias"),
        _ptr(state, F32, "state"), _ptr(row_mask, U8, "row_mask"), _ptr(staging, torch.uint8, "staging"),
        staging.numel(), _stream(stream)), "gdn_recurrent_decode_host_steps")


def _numel(shape) -> int:
    n = 1
    for x in shape:
        n *= x
    return n


def gdn_prefill_workspace_size(dims, chunk: int) -> int:
    d = make_dims(dims)
    return int(lib().gdn_prefill_workspace_size(ctypes.byref(d), int(chunk)))


def gdn_prefill(dims, q, k, v, g, beta, state_in, state_out, mask, y, chunk=0, workspace=None, stream=None):
    d = make_dims(dims)
    n = _Counts(d)
    _sizes("gdn_prefill", ("q", q, n.qk), ("k", k, n.qk), ("v", v, n.v), ("g", g, n.gate), ("beta", beta, n.gate),
           ("state_in", state_in, n.state), ("state_out", state_out, n.state), ("mask", mask, n.mask),
           ("y", y, n.v))
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    ws_ptr = None if workspace is None else (workspace.data_ptr() or None)
    _check(lib().gdn_prefill(ctypes.byref(d), _ptr(q, BF16, "q"), _ptr(k, BF16, "k"), _ptr(v, BF16, "v"),
                             _ptr(g, F32, "g"), _ptr(beta, F32, "beta"), _ptr(state_in, F32, "state_in"),
                             _ptr(state_out, F32, "state_out"), _ptr(mask, U8, "mask"), _ptr(y, BF16, "y"),
                             int(chunk), ws_ptr, ws_bytes, _stream(stream)), "gdn_prefill")


def gdn_recurrent_decode_gated(dims, qkv, conv_w, conv_state, a, b, A_log, dt_bias, state, row_mask, z, norm_w,
                               norm_eps, out, stream=None):
    d = make_dims(dims)
    n = _Counts(d)
    _sizes("gdn_recurrent_decode_gated", ("qkv", qkv, n.qkv), ("conv_w", conv_w, n.conv_w),
           ("conv_state", conv_state, n.conv_state), ("a", a, n.gate), ("b", b, n.gate), ("A_log", A_log, n.head),
           ("dt_bias", dt_bias, n.head), ("state", state, n.state), ("row_mask", row_mask, n.row), ("z", z, n.v),
           ("norm_w", norm_w, n.norm_w), ("out", out, n.v))
    _check(lib().gdn_recurrent_decode_gated(ctypes.byref(d), _ptr(qkv, BF16, "qkv"), _ptr(conv_w, BF16, "conv_w"),
                                            _ptr(conv_state, BF16, "conv_state"), _ptr(a, BF16, "a"),
                                            _ptr(b, BF16, "b"), _ptr(A_log, F32, "A_log"),
                                            _ptr(dt_bias, F32, "dt_bias"), _ptr(state, F32, "state"),
                                            _ptr(row_mask, U8, "row_mask"), _ptr(z, BF16, "z"),
                                            _ptr(norm_w, F32, "norm_w"), float(norm_eps), _ptr(out, BF16, "out"),
                                            _stream(stream)), "gdn_recurrent_decode_gated")


def gdn_prefill_gated(dims, q, k, v, g, beta, state_in, state_out, mask, z, norm_w, norm_eps, out, chunk=0,
                      workspace=None, stream=None):
    d = make_dims(dims)
    n = _Counts(d)
    _sizes("gdn_prefill_gated", ("q", q, n.qk), ("k", k, n.qk), ("v", v, n.v), ("g", g, n.gate),
           ("beta", beta, n.gate), ("state_in", state_in, n.state), ("state_out", state_out, n.state),
           ("mask", mask, n.mask), ("z", z, n.v), ("norm_w", norm_w, n.norm_w), ("out", out, n.v))
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    ws_ptr = None if workspace is None else (workspace.data_ptr() or None)
    _check(lib().gdn_prefill_gated(ctypes.byref(d), _ptr(q, BF16, "q"), _ptr(k, BF16, "k"), _ptr(v, BF16, "v"),
                                   _ptr(g, F32, "g"), _ptr(beta, F32, "beta"), _ptr(state_in, F32, "state_in"),
                                   _ptr(state_out, F32, "state_out"), _ptr(mask, U8, "mask"), _ptr(z, BF16, "z"),
                                   _ptr(norm_w, F32, "norm_w"), float(norm_eps), _ptr(out, BF16, "out"),
                                   int(chunk), ws_ptr, ws_bytes, _stream(stream)), "gdn_prefill_gated")


def gdn_prefill_backward_workspace_size(dims) -> int:
    d = make_dims(dims)
    return int(lib().gdn_prefill_backward_workspace_size(ctypes.byref(d)))


def _backward_call(name, dims, q, k, v, g, beta, state_in, mask, dy, dstate_out, dq, dk, dv, dg, dbeta, dstate_in,
                   workspace, stream):
    d = make_dims(dims)
    n = _Counts(d)
    _sizes(name, ("q", q, n.qk), ("k", k, n.qk), ("v", v, n.v), ("g", g, n.gate),
           ("beta", beta, n.gate), ("state_in", state_in, n.state), ("mask", mask, n.mask), ("dy", dy, n.v),
           ("dstate_out", dstate_out, n.state), ("dq", dq, n.qk), ("dk", dk, n.qk), ("dv", dv, n.v),
           ("dg", dg, n.gate), ("dbeta", dbeta, n.gate), ("dstate_in", dstate_in, n.state))
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    ws_ptr = None if workspace is None else (workspace.data_ptr() or None)
    _check(getattr(lib(), name)(ctypes.byref(d), _ptr(q, BF16, "q"), _ptr(k, BF16, "k"), _ptr(v, BF16, "v"),
                                _ptr(g, F32, "g"), _ptr(beta, F32, "beta"), _ptr(state_in, F32, "state_in"),
                                _ptr(mask, U8, "mask"), _ptr(dy, BF16, "dy"),
                                _ptr(dstate_out, F32, "dstate_out"), _ptr(dq, F32, "dq"), _ptr(dk, F32, "dk"),
                                _ptr(dv, F32, "dv"), _ptr(dg, F32, "dg"), _ptr(dbeta, F32, "dbeta"),
                                _ptr(dstate_in, F32, "dstate_in"), ws_ptr, ws_bytes, _stream(stream)), name)


def gdn_prefill_backward(dims, q, k, v, g, beta, state_in, mask, dy, dstate_out, dq, dk, dv, dg, dbeta, dstate_in,
                         workspace, stream=None):
    _backward_call("gdn_prefill_backward", dims, q, k, v, g, beta, state_in, mask, dy, dstate_out, dq, dk, dv, dg,
                   dbeta, dstate_in, workspace, stream)


def gdn_prefill_backward_chunked_workspace_size(dims) -> int:
    d = make_dims(dims)
    return int(lib().gdn_prefill_backward_chunked_workspace_size(ctypes.byref(d)))


def gdn_prefill_backward_chunked(dims, q, k, v, g, beta, state_in, mask, dy, dstate_out, dq, dk, dv, dg, dbeta,
                                 dstate_in, workspace, stream=None):
    _backward_call("gdn_prefill_backward_chunked", dims, q, k, v, g, beta, state_in, mask, dy, dstate_out, dq, dk,
                   dv, dg, dbeta, dstate_in, workspace, stream)


def gdn_prefill_noalloc(dims, q, k, v, g, beta, state_in, state_out, mask, y, chunk=0, stream=None):
    """gdn_prefill with the library's own fixed scratch (no workspace, no
    allocation); for callers that cannot allocate device memory."""
    d = make_dims(dims)
    n = _Counts(d)
    _sizes("gdn_prefill_noalloc", ("q", q, n.qk), ("k", k, n.qk), ("v", v, n.v), ("g", g, n.gate),
           ("beta", beta, n.gate), ("state_in", state_in, n.state), ("state_out", state_out, n.state),
           ("mask", mask, n.mask), ("y", y, n.v))
    _check(lib().gdn_prefill_noalloc(ctypes.byref(d), _ptr(q, BF16, "q"), _ptr(k, BF16, "k"), _ptr(v, BF16, "v"),
                                     _ptr(g, F32, "g"), _ptr(beta, F32, "beta"), _ptr(state_in, F32, "state_in"),
                                     _ptr(state_out, F32, "state_out"), _ptr(mask, U8, "mask"),
                                     _ptr(y, BF16, "y"), int(chunk), _stream(stream)), "gdn_prefill_noalloc")


def gdn_rmsnorm_gated(dims, y, z, norm_w, norm_eps, out, stream=None):
    d = make_dims(dims)
    n = _Counts(d)
    _sizes("gdn_rmsnorm_gated", ("y", y, n.v), ("z", z, n.v), ("norm_w", norm_w, n.norm_w), ("out", out, n.v))
    _check(lib().gdn_rmsnorm_gated(ctypes.byref(d), _ptr(y, BF16, "y"), _ptr(z, BF16, "z"),
                                   _ptr(norm_w, F32, "norm_w"), float(norm_eps), _ptr(out, BF16, "out"),
                                   _stream(stream)), "gdn_rmsnorm_gated")


def gdn_prefill_vec(dims, q, k, v, g_vec, beta, state_in, state_out, mask, y, stream=None):
    d = make_dims(dims)
    n = _Counts(d)
    _sizes("gdn_prefill_vec", ("q", q, n.qk), ("k", k, n.qk), ("v", v, n.v), ("g_vec", g_vec, n.g_vec),
           ("beta", beta, n.gate), ("state_in", state_in, n.state), ("state_out", state_out, n.state),
           ("mask", mask, n.mask), ("y", y, n.v))
    _check(lib().gdn_prefill_vec(ctypes.byref(d), _ptr(q, BF16, "q"), _ptr(k, BF16, "k"), _ptr(v, BF16, "v"),
                                 _ptr(g_vec, F32, "g_vec"), _ptr(beta, F32, "beta"), _ptr(state_in, F32, "state_in"),
                                 _ptr(state_out, F32, "state_out"), _ptr(mask, U8, "mask"), _ptr(y, BF16, "y"),
                                 _stream(stream)), "gdn_prefill_vec")


def gdn_device_status(stream=None) -> int:
    return int(lib().gdn_device_status(_stream(stream)))


def gdn_selftest_timeout(stream=None) -> int:
    return int(lib().gdn_selftest_timeout(_stream(stream)))


def gdn_abi_version() -> int:
    return int(lib().gdn_abi_version())


# ---------------------------------------------------------------------------
# allocating conveniences
# ---------------------------------------------------------------------------
def conv_update(dims, qkv, conv_w, conv_state=None, mask=None, stream=None):
    """Returns (q, k, v); conv_state (if given) is updated in place."""
    dev = qkv.device
    q = torch.empty((dims.B, dims.T, dims.Hk, dims.Dk), dtype=BF16, device=dev)
    k = torch.empty_like(q)
    v = torch.empty((dims.B, dims.T, dims.Hv, dims.Dv), dtype=BF16, device=dev)
    gdn_conv_update(dims, qkv, conv_w, conv_state, mask, q, k, v, stream)
    return q, k, v


def gating(dims, a, b, A_log, dt_bias, stream=None):
    g = torch.empty((dims.B, dims.T, dims.Hv), dtype=F32, device=a.device)
    beta = torch.empty_like(g)
    gdn_gating(dims, a, b, A_log, dt_bias, g, beta, stream)
    return g, beta


def shard_rows(B: int, world: int, rank: int):
    """Rows [start, stop) of a batch of B rows that rank `rank` of `world`
    takes when one call is split across ranks by batch row: contiguous, the
    sizes differing by at most one.  Every (b, head) owns its state, conv
    channels and outputs, so the ranks exchange nothing: each runs the same
    call on its rows (dims with B = stop - start, every per-row tensor sliced
    on its batch dimension) and the results are those of the whole batch."""
    if world < 1 or not 0 <= rank < world or B < 0:
        raise ValueError("shard_rows: need world >= 1, 0 <= rank < world, B >= 0")
    q, r = divmod(B, world)
    start = rank * q + min(rank, r)
    return start, start + q + (1 if rank < r else 0)


def recurrent_decode(dims, qkv, conv_w, conv_state, a, b, A_log, dt_bias, state, row_mask=None, stream=None):
    """One token; conv_state and state are updated in place.  Returns y [B, Hv, Dv]."""
    y = torch.empty((dims.B, dims.Hv, dims.Dv), dtype=BF16, device=qkv.device)
    gdn_recurrent_decode(dims, qkv, conv_w, conv_state, a, b, A_log, dt_bias, state, row_mask, y, stream)
    return y


def recurrent_decode_host_steps(dims, qkv_h, a_h, b_h, conv_w, conv_state, A_log, dt_bias, state, row_mask=None,
                                y_h=None, staging=None, stream=None):
    """len(qkv_h) decode steps with inputs in host memory ([n, B, ...], pinned
    for overlapped copies); conv_state and state advance in place.  Returns
    the host tensor y_h [n, B, Hv, Dv], valid once `stream` has completed."""
    n = qkv_h.shape[0]
    if y_h is None:
        y_h = torch.empty((n, dims.B, dims.Hv, dims.Dv), dtype=BF16).pin_memory()
    if staging is None:
        staging = torch.empty(gdn_decode_host_staging_size(dims), dtype=torch.uint8, device=conv_state.device)
    gdn_recurrent_decode_host_steps(dims, n, qkv_h, a_h, b_h, y_h, conv_w, conv_state, A_log, dt_bias, state,
                                    row_mask, staging, stream)
    return y_h


def decode_window(dims, qkv, conv_w, conv_state, a, b, A_log, dt_bias, state, keep=None, stream=None):
    """dims.T tokens per row; conv_state and state advance by keep[b] (default
    all) tokens in place.  Returns y [B, T, Hv, Dv]."""
    y = torch.empty((dims.B, dims.T, dims.Hv, dims.Dv), dtype=BF16, device=qkv.device)
    gdn_decode_window(dims, qkv, conv_w, conv_state, a, b, A_log, dt_bias, state, keep, y, stream)
    return y


def prefill(dims, q, k, v, g, beta, state_in=None, mask=None, chunk=0, state_out=None, stream=None,
            use_workspace=True):
    """Returns (y, state_out).  With use_workspace, the workspace the sizes ask
    for is passed (row order for masked batches; the two-pass chunked form
    for few heads); the results are the same either way."""
    dev = q.device
    y = torch.empty((dims.B, dims.T, dims.Hv, dims.Dv), dtype=BF16, device=dev)
    if state_out is None:
        state_out = torch.empty((dims.B, dims.Hv, dims.Dv, dims.Dk), dtype=F32, device=dev)
    ws = None
    if use_workspace:
        nws = gdn_prefill_workspace_size(dims, chunk)
        ws = torch.empty(nws, dtype=torch.uint8, device=dev) if nws > 0 else None
    gdn_prefill(dims, q, k, v, g, beta, state_in, state_out, mask, y, chunk, ws, stream)
    return y, state_out


def recurrent_decode_gated(dims, qkv, conv_w, conv_state, a, b, A_log, dt_bias, state, z, norm_w, norm_eps=1e-6,
                           row_mask=None, stream=None):
    """One token with the gated norm fused; returns out [B, Hv, Dv]."""
    out = torch.empty((dims.B, dims.Hv, dims.Dv), dtype=BF16, device=qkv.device)
    gdn_recurrent_decode_gated(dims, qkv, conv_w, conv_state, a, b, A_log, dt_bias, state, row_mask, z, norm_w,
                               norm_eps, out, stream)
    return out


def prefill_gated(dims, q, k, v, g, beta, z, norm_w, norm_eps=1e-6, state_in=None, mask=None, chunk=0,
                  state_out=None, stream=None):
    """Returns (out, state_out), out the gated norm of y."""
    dev = q.device
    out = torch.empty((dims.B, dims.T, dims.Hv, dims.Dv), dtype=BF16, device=dev)
    if state_out is None:
        state_out = torch.empty((dims.B, dims.Hv, dims.Dv, dims.Dk), dtype=F32, device=dev)
    nws = gdn_prefill_workspace_size(dims, chunk)
    ws = torch.empty(nws, dtype=torch.uint8, device=dev) if nws > 0 else None
    gdn_prefill_gated(dims, q, k, v, g, beta, state_in, state_out, mask, z, norm_w, norm_eps, out, chunk, ws, stream)
    return out, state_out


def prefill_backward(dims, q, k, v, g, beta, dy, state_in=None, mask=None, dstate_out=None, stream=None, chunk=0):
    """Gradients of the recurrence; returns a dict dq, dk [B,T,Hk,Dk], dv
    [B,T,Hv,Dv], dg, dbeta [B,T,Hv], dstate_in [B,Hv,Dv,Dk] (float32).
    chunk = 0: sequential form; 64: chunked form on the tensor cores."""
    if chunk not in (0, 64):
        raise ValueError("prefill_backward: chunk must be 0 or 64")
    dev = q.device
    B, T = dims.B, dims.T
    out = {"dq": torch.empty((B, T, dims.Hk, dims.Dk), dtype=F32, device=dev),
           "dk": torch.empty((B, T, dims.Hk, dims.Dk), dtype=F32, device=dev),
           "dv": torch.empty((B, T, dims.Hv, dims.Dv), dtype=F32, device=dev),
           "dg": torch.empty((B, T, dims.Hv), dtype=F32, device=dev),
           "dbeta": torch.empty((B, T, dims.Hv), dtype=F32, device=dev),
           "dstate_in": torch.empty((B, dims.Hv, dims.Dv, dims.Dk), dtype=F32, device=dev)}
    size_fn, call = ((gdn_prefill_backward_chunked_workspace_size, gdn_prefill_backward_chunked) if chunk
                     else (gdn_prefill_backward_workspace_size, gdn_prefill_backward))
    nws = size_fn(dims)
    ws = torch.empty(nws, dtype=torch.uint8, device=dev) if nws > 0 else None
    call(dims, q, k, v, g, beta, state_in, mask, dy, dstate_out, out["dq"], out["dk"], out["dv"], out["dg"],
         out["dbeta"], out["dstate_in"], ws, stream)
    return out


def rmsnorm_gated(dims, y, z, norm_w, norm_eps=1e-6, stream=None):
    """Returns out = bf16(silu(z) * w * rms_normalize(y)) shaped like y."""
    out = torch.empty_like(y)
    gdn_rmsnorm_gated(dims, y, z, norm_w, norm_eps, out, stream)
    return out


def prefill_vec(dims, q, k, v, g_vec, beta, state_in=None, mask=None, stream=None):
    """Vectorized gating (g_vec [B, T, Hv, Dk]); returns (y, state_out)."""
    y = torch.empty((dims.B, dims.T, dims.Hv, dims.Dv), dtype=BF16, device=q.device)
    state_out = torch.empty((dims.B, dims.Hv, dims.Dv, dims.Dk), dtype=F32, device=q.device)
    gdn_prefill_vec(dims, q, k, v, g_vec, beta, state_in, state_out, mask, y, stream)
    return y, state_out


def core_prefill(dims, qkv, conv_w, a, b, A_log, dt_bias, conv_state=None, state_in=None, mask=None, chunk=0,
                 stream=None, use_workspace=True):
    """conv -> gates -> recurrence; returns (y, state_out).  conv_state (if
    given) is updated in place."""
    q, k, v = conv_update(dims, qkv, conv_w, conv_state, mask, stream)
    g, beta = gating(dims, a, b, A_log, dt_bias, stream)
    return prefill(dims, q, k, v, g, beta, state_in, mask, chunk, None, stream, use_workspace)
