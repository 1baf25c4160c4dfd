"""Python binding of the GB300 mixture-of-experts layer library (include/moe.h).

Argument marshalling only: every step of the layer runs in the CUDA kernels of
``libmoe_gb300.so``.  Functions take torch tensors (or raw device pointers as
ints, or None for NULL) and a stream (default: torch's current stream) and
return the library's status code; :func:`check` turns a non-zero code into an
exception.  There is no CPU fallback: importing the binding without the built
library raises.
"""
import ctypes
import os

from . import build as _build

# MOE_GB300_LIB names another build of the library (e.g. the bounds-checked
# debug build, build.build(debug=True)) for this process.
LIB_PATH = os.environ.get("MOE_GB300_LIB") or _build.LIB

MOE_BF16, MOE_MXFP8, MOE_NVFP4 = 0, 1, 2
DTYPES = {"bf16": MOE_BF16, "mxfp8": MOE_MXFP8, "nvfp4": MOE_NVFP4}
MOE_FLAG_BACKWARD = 1
MOE_FLAG_DEBUG_STARVE = 2
MOE_FLAG_DEBUG_DUMP = 4
STATUS = {0: "ok", -1: "invalid argument", -2: "unsupported shape", -3: "pointer not 16-byte aligned",
          -4: "CUDA error", -5: "device is not sm_103", -6: "a device-side wait timed out",
          -7: "a device-side bounds check failed (debug build)"}

WEIGHT_FIELDS = ["gu", "gu_scale", "dn", "dn_scale", "gu_t", "gu_t_scale", "dn_t", "dn_t_scale",
                 "s_gu", "s_dn", "s_gu_t", "s_dn_t", "gu_gscale", "dn_gscale"]


class MoeConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("T", "d", "m", "E", "k", "m_shared", "dtype", "flags",
                                              "ring_rows", "gather_sms")] + [("aux_alpha", ctypes.c_float)]


class MoeWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in WEIGHT_FIELDS]


_lib = None
EXPORTS = ["moe_workspace_bytes", "moe_saved_bytes", "moe_buffer_info", "moe_padded_rows",
           "moe_quantize_weights", "moe_quantize_mx", "moe_quantize_mx_both", "moe_prepare_weights",
           "moe_prepare_scales",
           "moe_canonical_scales", "moe_transpose_bf16", "moe_route",
           "moe_forward", "moe_backward",
           "moe_get_status", "moe_status_string", "moe_trace_enable", "moe_trace_clear", "moe_trace_count",
           "moe_trace_name", "moe_trace_ms", "moe_route_noalloc", "moe_router_forward", "moe_router_backward"]


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libmoe_gb300.so is not built (run __graft_entry__.build() or "
                               "python -m mixture_experts_layer_device_gb300.build)")
        L = ctypes.CDLL(LIB_PATH)
        P, I, Z, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
        cfgp = ctypes.POINTER(MoeConfig)
        L.moe_workspace_bytes.argtypes, L.moe_workspace_bytes.restype = [cfgp], Z
        L.moe_saved_bytes.argtypes, L.moe_saved_bytes.restype = [cfgp], Z
        L.moe_buffer_info.argtypes = [cfgp, I, ctypes.c_char_p, ctypes.POINTER(Z), ctypes.POINTER(Z)]
        L.moe_buffer_info.restype = I
        L.moe_padded_rows.argtypes, L.moe_padded_rows.restype = [cfgp], ctypes.c_int64
        L.moe_quantize_weights.argtypes, L.moe_quantize_weights.restype = [cfgp, P, I, I, I, P, P, S], I
        L.moe_quantize_mx.argtypes, L.moe_quantize_mx.restype = [P, I, I, I, I, P, P, S], I
        L.moe_quantize_mx_both.argtypes, L.moe_quantize_mx_both.restype = [P, I, I, I, P, P, P, P, S], I
        L.moe_prepare_weights.argtypes = [cfgp, P, P, P, P, P, P, P, P, P, P, P, P, S]
        L.moe_prepare_weights.restype = I
        L.moe_prepare_scales.argtypes, L.moe_prepare_scales.restype = [P, ctypes.c_int64, ctypes.c_int32, P, S], I
        L.moe_canonical_scales.argtypes = [P, ctypes.c_int64, ctypes.c_int32, P, S]
        L.moe_canonical_scales.restype = I
        L.moe_transpose_bf16.argtypes, L.moe_transpose_bf16.restype = [P, I, I, I, P, S], I
        L.moe_route.argtypes, L.moe_route.restype = [cfgp, P, P, P, P, P, P, P, S], I
        L.moe_forward.argtypes = [cfgp, P, P, ctypes.POINTER(MoeWeights), P, P, P, S]
        L.moe_forward.restype = I
        L.moe_backward.argtypes = [cfgp, P, P, ctypes.POINTER(MoeWeights), P, P, P, P, P, P, P, P, S]
        L.moe_backward.restype = I
        L.moe_get_status.argtypes, L.moe_get_status.restype = [P, S], I
        L.moe_status_string.argtypes, L.moe_status_string.restype = [I], ctypes.c_char_p
        L.moe_route_noalloc.argtypes, L.moe_route_noalloc.restype = [cfgp, P, P, P, P, P, P, S], I
        L.moe_router_forward.argtypes, L.moe_router_forward.restype = [cfgp, P, P, P, P, S], I
        L.moe_router_backward.argtypes, L.moe_router_backward.restype = [cfgp, P, P, P, P, P, P, S], I
        L.moe_trace_enable.argtypes, L.moe_trace_enable.restype = [I], I
        L.moe_trace_clear.argtypes, L.moe_trace_clear.restype = [], None
        L.moe_trace_count.argtypes, L.moe_trace_count.restype = [], I
        L.moe_trace_name.argtypes, L.moe_trace_name.restype = [I], ctypes.c_char_p
        L.moe_trace_ms.argtypes, L.moe_trace_ms.restype = [I], ctypes.c_float
        _lib = L
    return _lib


def _ptr(t):
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


def config(T, d, m, E, k, m_shared=0, dtype=MOE_BF16, flags=0, ring_rows=0, gather_sms=0, aux_alpha=0.0):
    if isinstance(dtype, str):
        dtype = DTYPES[dtype]
    return MoeConfig(T, d, m, E, k, m_shared, dtype, flags, ring_rows, gather_sms, aux_alpha)


def moe_router_forward(cfg, x, W_r, logits, ws, stream=None):
    return lib().moe_router_forward(ctypes.byref(cfg), _ptr(x), _ptr(W_r), _ptr(logits), _ptr(ws), _stream(stream))


def moe_router_backward(cfg, dlogits, x, W_r, dx, dW_r, ws, stream=None):
    return lib().moe_router_backward(ctypes.byref(cfg), _ptr(dlogits), _ptr(x), _ptr(W_r), _ptr(dx), _ptr(dW_r),
                                     _ptr(ws), _stream(stream))


def weights(**kw):
    """MoeWeights from keyword tensors (names as in moe_weights)."""
    w = MoeWeights()
    for n in WEIGHT_FIELDS:
        setattr(w, n, _ptr(kw.get(n)))
    return w


def check(rc):
    if rc != 0:
        raise RuntimeError("moe library error %d: %s" % (rc, STATUS.get(rc, "unknown")))
    return rc


def moe_workspace_bytes(cfg):
    return lib().moe_workspace_bytes(ctypes.byref(cfg))


def moe_saved_bytes(cfg):
    return lib().moe_saved_bytes(ctypes.byref(cfg))


def moe_padded_rows(cfg):
    return lib().moe_padded_rows(ctypes.byref(cfg))


def moe_buffer_info(cfg, which, name):
    off, nb = ctypes.c_size_t(), ctypes.c_size_t()
    check(lib().moe_buffer_info(ctypes.byref(cfg), which, name.encode(), ctypes.byref(off), ctypes.byref(nb)))
    return off.value, nb.value


def moe_quantize_mx_both(src, batch, rows, cols, codes, scales, codes_t, scales_t, stream=None):
    return lib().moe_quantize_mx_both(_ptr(src), batch, rows, cols, _ptr(codes), _ptr(scales), _ptr(codes_t),
                                      _ptr(scales_t), _stream(stream))


def moe_quantize_weights(cfg, w_bf16, rows, cols, blocks_along_rows, codes, scales, stream=None):
    return lib().moe_quantize_weights(ctypes.byref(cfg), _ptr(w_bf16), rows, cols, int(blocks_along_rows),
                                      _ptr(codes), _ptr(scales), _stream(stream))


def moe_quantize_mx(src, batch, rows, cols, transpose, codes, scales, stream=None):
    return lib().moe_quantize_mx(_ptr(src), batch, rows, cols, int(transpose), _ptr(codes), _ptr(scales),
                                 _stream(stream))


def moe_prepare_weights(cfg, w_gu, w_dn, gu, gu_scale, dn, dn_scale, gu_t=None, gu_t_scale=None, dn_t=None,
                        dn_t_scale=None, gu_gscale=None, dn_gscale=None, stream=None):
    return lib().moe_prepare_weights(ctypes.byref(cfg), _ptr(w_gu), _ptr(w_dn), _ptr(gu), _ptr(gu_scale), _ptr(dn),
                                     _ptr(dn_scale), _ptr(gu_t), _ptr(gu_t_scale), _ptr(dn_t), _ptr(dn_t_scale),
                                     _ptr(gu_gscale), _ptr(dn_gscale), _stream(stream))


def moe_prepare_scales(scales, rows, K, prepared, stream=None):
    return lib().moe_prepare_scales(_ptr(scales), rows, K, _ptr(prepared), _stream(stream))


def moe_canonical_scales(prepared, rows, K, scales, stream=None):
    return lib().moe_canonical_scales(_ptr(prepared), rows, K, _ptr(scales), _stream(stream))


def moe_transpose_bf16(src, batch, rows, cols, dst, stream=None):
    return lib().moe_transpose_bf16(_ptr(src), batch, rows, cols, _ptr(dst), _stream(stream))


def moe_route(cfg, logits, idx, w, counts, offsets, perm, ws, stream=None):
    return lib().moe_route(ctypes.byref(cfg), _ptr(logits), _ptr(idx), _ptr(w), _ptr(counts), _ptr(offsets),
                           _ptr(perm), _ptr(ws), _stream(stream))


def moe_route_noalloc(cfg, logits, idx, w, counts, offsets, perm, stream=None):
    return lib().moe_route_noalloc(ctypes.byref(cfg), _ptr(logits), _ptr(idx), _ptr(w), _ptr(counts),
                                   _ptr(offsets), _ptr(perm), _stream(stream))


def moe_forward(cfg, x, logits, W, y, saved, ws, stream=None):
    return lib().moe_forward(ctypes.byref(cfg), _ptr(x), _ptr(logits), ctypes.byref(W), _ptr(y), _ptr(saved),
                             _ptr(ws), _stream(stream))


def moe_backward(cfg, dy, x, W, saved, dx, dlogits, dW_gu, dW_dn, dWs_gu, dWs_dn, ws, stream=None):
    return lib().moe_backward(ctypes.byref(cfg), _ptr(dy), _ptr(x), ctypes.byref(W), _ptr(saved), _ptr(dx),
                              _ptr(dlogits), _ptr(dW_gu), _ptr(dW_dn), _ptr(dWs_gu), _ptr(dWs_dn), _ptr(ws),
                              _stream(stream))


def moe_get_status(ws, stream=None):
    return lib().moe_get_status(_ptr(ws), _stream(stream))


def moe_trace_enable(capacity):
    return lib().moe_trace_enable(capacity)


def moe_trace_clear():
    lib().moe_trace_clear()


def moe_trace_records():
    """[(kernel name, milliseconds)] of the launches recorded since the last clear."""
    L = lib()
    return [(L.moe_trace_name(i).decode(), L.moe_trace_ms(i)) for i in range(L.moe_trace_count())]
