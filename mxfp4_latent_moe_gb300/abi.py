"""ctypes binding of libmoe.so (include/moe.h): the same entry-point names,
torch tensors in, argument marshalling only. Every step of the layer runs in
the library's CUDA kernels; nothing here computes any part of it.

The library is loaded on first use. If it has not been built, or no CUDA
device is present, calls raise instead of falling back to anything else.
"""
import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe.so")

STATUS_BYTES = 256
OK, INVALID_ARGUMENT, UNSUPPORTED, WORKSPACE_TOO_SMALL, CUDA, DEVICE_TIMEOUT, DEVICE_BAD_INPUT = range(7)
GEMM_AUTO, GEMM_TOKEN_TILES, GEMM_WEIGHT_TILES, GEMM_PAIR_TILES = range(4)
SCALES_TILED128, SCALES_GROUP32 = range(2)
EPI_F32, EPI_BF16, EPI_SWIGLU_BF16 = range(3)


class MoeError(RuntimeError):
    def __init__(self, fn, code, text):
        super().__init__("%s failed: status %d (%s)" % (fn, code, text))
        self.code = code


_lib = None
_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t


class _Dims(ctypes.Structure):
    _fields_ = [("T", _i32), ("d", _i32), ("E", _i32), ("k", _i32), ("I", _i32)]


class _Weights(ctypes.Structure):
    _fields_ = [("w13", _vp), ("w13_sf", _vp), ("w2", _vp), ("w2_sf", _vp)]


class _BlockDims(ctypes.Structure):
    _fields_ = [("T", _i32), ("hidden", _i32), ("d", _i32), ("E", _i32), ("k", _i32),
                ("I", _i32), ("shared_I", _i32)]


class _BlockWeights(ctypes.Structure):
    _fields_ = [("w_down", _vp), ("w_router", _vp), ("w_shared13", _vp), ("w_out", _vp),
                ("routed", _Weights)]


_SIGS = {
    "moe_status_string": (ctypes.c_char_p, [_i32]),
    "moe_abi_version": (_i32, []),
    "moe_tiled_scale_bytes": (_sz, [_i64, _i32]),
    "moe_activation_scale_bytes": (_sz, [_i64, _i32, _i32]),
    "moe_rows_capacity": (_i64, [_i32, _i32, _i32, _i32]),
    "moe_default_kernel": (_i32, [_i32, _i32, _i32]),
    "moe_prepack_scales": (_i32, [_vp, _i64, _i32, _vp, _vp]),
    "moe_prepack_weights": (_i32, [_vp, _i64, _i32, _vp, _vp]),
    "moe_route_topk": (_i32, [_vp, _i32, _i32, _i32, _vp, _vp, _vp]),
    "moe_permute_workspace_size": (_sz, [_i32, _i32]),
    "moe_permute": (_i32, [_vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _i64, _vp, _sz, _vp]),
    "moe_permute_noalloc": (_i32, [_vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _i64, _vp, _vp]),
    "moe_quant_mxfp8": (_i32, [_vp, _i32, _i32, _vp, _i32, _vp, _vp, _i32, _i64, _vp]),
    "moe_grouped_gemm_w13_glu": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp,
                                        _vp, _i64, _vp, _sz, _vp]),
    "moe_grouped_gemm_w2": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _i64,
                                   _vp, _sz, _vp]),
    "moe_unpermute_combine": (_i32, [_vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp]),
    "moe_workspace_size": (_i32, [ctypes.POINTER(_Dims), ctypes.POINTER(_sz)]),
    "moe_forward": (_i32, [ctypes.POINTER(_Dims), _i32, _vp, _vp, ctypes.POINTER(_Weights), _vp,
                           _vp, _vp, _vp, _sz, _vp]),
    "moe_quant_mxfp4": (_i32, [_vp, _i32, _i32, _vp, _i32, _vp, _vp, _i32, _i64, _vp]),
    "moe_grouped_gemm_w13_glu_a4w4": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp,
                                             _vp, _vp, _i64, _vp, _sz, _vp]),
    "moe_forward_a4w4": (_i32, [ctypes.POINTER(_Dims), _i32, _vp, _vp, ctypes.POINTER(_Weights),
                                _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_gemm_bf16": (_i32, [_vp, _vp, _i64, _i32, _i32, _i32, _vp, _vp, _sz, _vp]),
    "moe_router_logits": (_i32, [_vp, _vp, _i32, _i32, _i32, _vp, _vp, _sz, _vp]),
    "moe_gemm_bf16_workspace_size": (_sz, [_i64, _i32, _i32, _i32]),
    "moe_gemm_bf16_cat": (_i32, [_vp, _i32, _vp, _i32, _vp, _i64, _i32, _i32, _vp, _vp, _sz,
                                 _vp]),
    "moe_block_workspace_size": (_i32, [ctypes.POINTER(_BlockDims), ctypes.POINTER(_sz)]),
    "moe_block_forward": (_i32, [ctypes.POINTER(_BlockDims), _i32, _vp,
                                 ctypes.POINTER(_BlockWeights), _vp, _vp, _sz, _vp, _vp]),
    "moe_check_device_status": (_i32, [_vp, _vp]),
    "moe_clear_device_status": (_i32, [_vp, _vp]),
    "moe_selftest_wait_timeout": (_i32, [_vp, _sz, ctypes.c_uint32, _vp]),
}

EXPORTED = tuple(_SIGS)


def lib():
    """The loaded library (raises if it is missing)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libmoe.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_string(code):
    return lib().moe_status_string(int(code)).decode()


def _check(name, code):
    if code != OK:
        raise MoeError(name, code, status_string(code))


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch tensor")
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _call(name, *args):
    _check(name, getattr(lib(), name)(*args))


# ---------------------------------------------------------------- sizes

def moe_abi_version():
    return lib().moe_abi_version()


def moe_tiled_scale_bytes(rows, K):
    return lib().moe_tiled_scale_bytes(rows, K)


def moe_activation_scale_bytes(rows, K, layout):
    return lib().moe_activation_scale_bytes(rows, K, layout)


def moe_rows_capacity(T, E, k, pad_m):
    return lib().moe_rows_capacity(T, E, k, pad_m)


def moe_default_kernel(T, E, k):
    return lib().moe_default_kernel(T, E, k)


def moe_permute_workspace_size(T, E):
    return lib().moe_permute_workspace_size(T, E)


def moe_workspace_size(T, d, E, k, I):
    out = _sz(0)
    _check("moe_workspace_size", lib().moe_workspace_size(ctypes.byref(_Dims(T, d, E, k, I)),
                                                          ctypes.byref(out)))
    return out.value


# ---------------------------------------------------------------- entry points

def moe_prepack_scales(src, rows, K, dst, stream=None):
    _call("moe_prepack_scales", _ptr(src), rows, K, _ptr(dst), _stream(stream))


def moe_prepack_weights(src, rows, K, dst, stream=None):
    _call("moe_prepack_weights", _ptr(src), rows, K, _ptr(dst), _stream(stream))


def moe_route_topk(logits, T, E, k, topk_ids, topk_w, stream=None):
    _call("moe_route_topk", _ptr(logits), T, E, k, _ptr(topk_ids), _ptr(topk_w), _stream(stream))


def moe_permute(topk_ids, T, E, k, pad_m, counts, offsets, slot_to_row, row_to_slot,
                rows_capacity, ws, stream=None):
    _call("moe_permute", _ptr(topk_ids), T, E, k, pad_m, _ptr(counts), _ptr(offsets),
          _ptr(slot_to_row), _ptr(row_to_slot), rows_capacity, _ptr(ws), ws.numel() * ws.element_size(),
          _stream(stream))


def moe_permute_noalloc(topk_ids, T, E, k, pad_m, counts, offsets, slot_to_row, row_to_slot,
                        rows_capacity, status=None, stream=None):
    """moe_permute without a workspace (for callers that cannot allocate one)."""
    _call("moe_permute_noalloc", _ptr(topk_ids), T, E, k, pad_m, _ptr(counts), _ptr(offsets),
          _ptr(slot_to_row), _ptr(row_to_slot), rows_capacity, _ptr(status), _stream(stream))


def moe_quant_mxfp8(x, T, d, slot_to_row, k, codes, scales, rows_capacity, scale_layout=0,
                    stream=None):
    _call("moe_quant_mxfp8", _ptr(x), T, d, _ptr(slot_to_row), k, _ptr(codes), _ptr(scales),
          scale_layout, rows_capacity, _stream(stream))


def moe_grouped_gemm_w13_glu(xq, xs, counts, offsets, E, d, I, kernel, w13, w13_sf, hq, hs,
                             rows_capacity, ws, stream=None):
    _call("moe_grouped_gemm_w13_glu", _ptr(xq), _ptr(xs), _ptr(counts), _ptr(offsets), E, d, I,
          kernel, _ptr(w13), _ptr(w13_sf), _ptr(hq), _ptr(hs), rows_capacity, _ptr(ws),
          ws.numel() * ws.element_size(), _stream(stream))


def moe_grouped_gemm_w2(hq, hs, counts, offsets, E, I, d, kernel, w2, w2_sf, yp, rows_capacity, ws,
                        stream=None):
    _call("moe_grouped_gemm_w2", _ptr(hq), _ptr(hs), _ptr(counts), _ptr(offsets), E, I, d, kernel,
          _ptr(w2), _ptr(w2_sf), _ptr(yp), rows_capacity, _ptr(ws), ws.numel() * ws.element_size(),
          _stream(stream))


def moe_unpermute_combine(yp, slot_to_row, topk_w, T, k, d, y, stream=None):
    _call("moe_unpermute_combine", _ptr(yp), _ptr(slot_to_row), _ptr(topk_w), T, k, d, _ptr(y),
          _stream(stream))


def moe_forward(T, d, E, k, I, kernel, x, logits, w13, w13_sf, w2, w2_sf, y, ws,
                topk_ids_out=None, topk_w_out=None, stream=None):
    W = _Weights(_ptr(w13), _ptr(w13_sf), _ptr(w2), _ptr(w2_sf))
    _call("moe_forward", ctypes.byref(_Dims(T, d, E, k, I)), kernel, _ptr(x), _ptr(logits),
          ctypes.byref(W), _ptr(y), _ptr(topk_ids_out), _ptr(topk_w_out), _ptr(ws),
          ws.numel() * ws.element_size(), _stream(stream))


def moe_quant_mxfp4(x, T, d, slot_to_row, k, codes, scales, rows_capacity, scale_layout=0,
                    stream=None):
    """MXFP4 activations: codes packed [rows_capacity][d/2]."""
    _call("moe_quant_mxfp4", _ptr(x), T, d, _ptr(slot_to_row), k, _ptr(codes), _ptr(scales),
          scale_layout, rows_capacity, _stream(stream))


def moe_grouped_gemm_w13_glu_a4w4(xq, xs, counts, offsets, E, d, I, hs_layout, w13, w13_sf, hq,
                                  hs, rows_capacity, ws, stream=None):
    _call("moe_grouped_gemm_w13_glu_a4w4", _ptr(xq), _ptr(xs), _ptr(counts), _ptr(offsets), E, d,
          I, hs_layout, _ptr(w13), _ptr(w13_sf), _ptr(hq), _ptr(hs), rows_capacity, _ptr(ws),
          ws.numel() * ws.element_size(), _stream(stream))


def moe_forward_a4w4(T, d, E, k, I, kernel, x, logits, w13, w13_sf, w2, w2_sf, y, ws,
                     topk_ids_out=None, topk_w_out=None, stream=None):
    W = _Weights(_ptr(w13), _ptr(w13_sf), _ptr(w2), _ptr(w2_sf))
    _call("moe_forward_a4w4", ctypes.byref(_Dims(T, d, E, k, I)), kernel, _ptr(x), _ptr(logits),
          ctypes.byref(W), _ptr(y), _ptr(topk_ids_out), _ptr(topk_w_out), _ptr(ws),
          ws.numel() * ws.element_size(), _stream(stream))


def moe_gemm_bf16(a, b, M, N, K, epilogue, c, ws, stream=None):
    """C = A . B^T for bf16 a [M][K], b [N][K]; c fp32 / bf16 per the epilogue."""
    _call("moe_gemm_bf16", _ptr(a), _ptr(b), M, N, K, epilogue, _ptr(c), _ptr(ws),
          ws.numel() * ws.element_size(), _stream(stream))


def moe_gemm_bf16_workspace_size(M, N, K, epilogue):
    return lib().moe_gemm_bf16_workspace_size(M, N, K, epilogue)


def moe_router_logits(x, w_router, T, d_in, E, logits, ws, stream=None):
    _call("moe_router_logits", _ptr(x), _ptr(w_router), T, d_in, E, _ptr(logits), _ptr(ws),
          ws.numel() * ws.element_size(), _stream(stream))


def moe_gemm_bf16_cat(a1, K1, a2, K2, b, M, N, epilogue, c, ws, stream=None):
    """C = [A1 | A2] . B^T: a1 bf16 [M][K1], a2 bf16 [M][K2], b [N][K1 + K2]."""
    _call("moe_gemm_bf16_cat", _ptr(a1), K1, _ptr(a2), K2, _ptr(b), M, N, epilogue, _ptr(c),
          _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))


def moe_block_workspace_size(T, hidden, d, E, k, I, shared_I):
    n = _sz(0)
    _call("moe_block_workspace_size", ctypes.byref(_BlockDims(T, hidden, d, E, k, I, shared_I)),
          ctypes.byref(n))
    return n.value


def moe_block_forward(T, hidden, d, E, k, I, shared_I, kernel, h, w_down, w_router, w_shared13,
                      w_out, w13, w13_sf, w2, w2_sf, out, ws, stream=None, shared_stream=None):
    """The composed block; shared_stream None runs everything on `stream`."""
    W = _BlockWeights(_ptr(w_down), _ptr(w_router), _ptr(w_shared13), _ptr(w_out),
                      _Weights(_ptr(w13), _ptr(w13_sf), _ptr(w2), _ptr(w2_sf)))
    st = _stream(stream)
    side = st if shared_stream is None else _stream(shared_stream)
    _call("moe_block_forward", ctypes.byref(_BlockDims(T, hidden, d, E, k, I, shared_I)), kernel,
          _ptr(h), ctypes.byref(W), _ptr(out), _ptr(ws), ws.numel() * ws.element_size(), st,
          side)


def moe_check_device_status(ws, stream=None):
    """Synchronises the stream; returns the device status code (0 = ok)."""
    return lib().moe_check_device_status(_ptr(ws), _stream(stream))


def moe_clear_device_status(ws, stream=None):
    _call("moe_clear_device_status", _ptr(ws), _stream(stream))


def moe_selftest_wait_timeout(ws, limit_us, stream=None):
    _call("moe_selftest_wait_timeout", _ptr(ws), ws.numel() * ws.element_size(), limit_us,
          _stream(stream))
