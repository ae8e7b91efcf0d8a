"""Host-side checks of the C-ABI library (no GPU needed, no CUDA call made):
it loads, exports every entry point include/moe.h declares, and rejects bad
arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

from mxfp4_latent_moe_gb300 import abi
from mxfp4_latent_moe_gb300.build import build_library

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe.h")


@pytest.fixture(scope="module")
def L():
    build_library()
    return abi.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_entry_point(L):
    names = _declared()
    assert len(names) >= 17
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(abi.EXPORTED)


def test_status_strings_and_version(L):
    assert abi.moe_abi_version() == 1
    for code in range(7):
        assert abi.status_string(code)
    assert abi.status_string(99) == "unknown status"


def test_size_helpers():
    # tiled scales: rows rounded up to 128, one byte per 32 inputs
    assert abi.moe_tiled_scale_bytes(1, 3584) == 128 * 112
    assert abi.moe_tiled_scale_bytes(896 * 6144, 3584) == 896 * 6144 * 112
    assert abi.moe_tiled_scale_bytes(10, 100) == 0       # K not a multiple of 128
    assert abi.moe_activation_scale_bytes(1, 3584, abi.SCALES_TILED128) == 128 * 112
    assert abi.moe_activation_scale_bytes(1, 3584, abi.SCALES_GROUP32) == 32 * 3584 // 8
    assert abi.moe_activation_scale_bytes(64, 256, abi.SCALES_GROUP32) == 2 * 512 * 2
    assert abi.moe_activation_scale_bytes(64, 256, 5) == 0
    # T*k + min(E, T*k)*(pad_m - 1), rounded up to 128
    assert abi.moe_rows_capacity(64, 896, 16, 128) == (1024 + 896 * 127 + 127) // 128 * 128
    assert abi.moe_rows_capacity(8, 32, 4, 128) == (32 + 32 * 127 + 127) // 128 * 128
    assert abi.moe_rows_capacity(8, 32, 4, 100) == -1    # not a power of two
    assert abi.moe_default_kernel(64, 896, 16) == abi.GEMM_WEIGHT_TILES
    assert abi.moe_default_kernel(3136, 896, 16) == abi.GEMM_WEIGHT_TILES
    assert abi.moe_default_kernel(3137, 896, 16) == abi.GEMM_TOKEN_TILES
    assert abi.moe_default_kernel(8192, 896, 16) == abi.GEMM_TOKEN_TILES
    assert abi.moe_default_kernel(8, 896, 33) == -1
    assert abi.moe_permute_workspace_size(0, 896) == 256
    assert abi.moe_permute_workspace_size(300, 896) == 256 + ((2 * 896 * 4 + 255) // 256) * 256
    ws = abi.moe_workspace_size(32768, 3584, 896, 16, 3072)
    rows = abi.moe_rows_capacity(32768, 896, 16, 128)
    assert ws > rows * (3584 * 2 + 3584 + 3072)          # Yp + Xq + hq at least


def _rc(L, name, *args):
    return getattr(L, name)(*args)


def test_host_validation_rejects_before_any_launch(L):
    E, k = 896, 16
    # routing: k > E, E too large, negative T, null pointers
    assert _rc(L, "moe_route_topk", None, 4, 8, 9, None, None, None) == abi.UNSUPPORTED
    assert _rc(L, "moe_route_topk", None, 4, 2048, 4, None, None, None) == abi.UNSUPPORTED
    assert _rc(L, "moe_route_topk", None, -1, E, k, None, None, None) == abi.INVALID_ARGUMENT
    assert _rc(L, "moe_route_topk", None, 4, E, k, None, None, None) == abi.INVALID_ARGUMENT
    assert _rc(L, "moe_route_topk", None, 0, E, k, None, None, None) == abi.OK   # nothing to do
    # permute: bad pad, short row capacity, short workspace
    fake = ctypes.c_void_p(4096)
    assert _rc(L, "moe_permute", fake, 4, E, k, 100, fake, fake, fake, fake, 10 ** 6, fake, 10 ** 6,
               None) == abi.UNSUPPORTED
    assert _rc(L, "moe_permute", fake, 4, E, k, 128, fake, fake, fake, fake, 64, fake, 10 ** 6,
               None) == abi.WORKSPACE_TOO_SMALL
    assert _rc(L, "moe_permute", fake, 4, E, k, 128, fake, fake, fake, fake, 10 ** 6, fake, 16,
               None) == abi.WORKSPACE_TOO_SMALL
    # quant: d not a multiple of 128, misaligned x
    assert _rc(L, "moe_quant_mxfp8", fake, 4, 100, None, 0, fake, fake, 0, 128, None) == \
        abi.UNSUPPORTED
    assert _rc(L, "moe_quant_mxfp8", fake, 4, 256, None, 0, fake, fake, 2, 128, None) == \
        abi.UNSUPPORTED                                     # unknown scale layout
    assert _rc(L, "moe_quant_mxfp8", ctypes.c_void_p(4098), 4, 256, None, 0, fake, fake, 1, 128,
               None) == abi.INVALID_ARGUMENT
    # GEMMs: unknown kernel, capacity not a multiple of 128, misaligned weights, no workspace
    args = [fake, fake, fake, fake, E, 3584, 3072]
    assert _rc(L, "moe_grouped_gemm_w13_glu", *args, 0, fake, fake, fake, fake, 1024, fake, 256,
               None) == abi.UNSUPPORTED
    assert _rc(L, "moe_grouped_gemm_w13_glu", *args, 1, fake, fake, fake, fake, 1000, fake, 256,
               None) == abi.UNSUPPORTED
    assert _rc(L, "moe_grouped_gemm_w13_glu", *args, 2, ctypes.c_void_p(4096 + 16), fake, fake,
               fake, 1024, fake, 256, None) == abi.INVALID_ARGUMENT
    assert _rc(L, "moe_grouped_gemm_w13_glu", *args, 1, fake, fake, fake, fake, 1024, fake, 8,
               None) == abi.WORKSPACE_TOO_SMALL
    assert _rc(L, "moe_grouped_gemm_w13_glu", fake, fake, None, fake, E, 3584, 3072, 1, fake, fake,
               fake, fake, 1024, fake, 256, None) == abi.INVALID_ARGUMENT   # counts required
    assert _rc(L, "moe_grouped_gemm_w2", fake, fake, fake, fake, E, 3072, 3584, 1, fake, fake, None,
               1024, fake, 256, None) == abi.INVALID_ARGUMENT
    # combine: null output
    assert _rc(L, "moe_unpermute_combine", fake, fake, fake, 4, k, 3584, None, None) == \
        abi.INVALID_ARGUMENT
    # forward: dims null / unsupported
    assert _rc(L, "moe_forward", None, 0, fake, fake, None, fake, None, None, fake, 10, None) == \
        abi.INVALID_ARGUMENT
    dims = abi._Dims(4, 3584, 896, 33, 3072)
    assert _rc(L, "moe_forward", ctypes.byref(dims), 0, fake, fake, None, fake, None, None, fake,
               10, None) == abi.UNSUPPORTED
    dims = abi._Dims(4, 3584, 896, 16, 3072)
    W = abi._Weights(4096, 4096, 4096, 4096)
    assert _rc(L, "moe_forward", ctypes.byref(dims), 7, fake, fake, ctypes.byref(W), fake, None,
               None, fake, 10 ** 9, None) == abi.UNSUPPORTED
    assert _rc(L, "moe_forward", ctypes.byref(dims), 0, fake, fake, ctypes.byref(W), fake, None,
               None, fake, 10, None) == abi.WORKSPACE_TOO_SMALL
    # A4W4: quant layout, d not a multiple of 256, bad hs layout, misaligned codes
    assert _rc(L, "moe_quant_mxfp4", fake, 4, 256, None, 0, fake, fake, 3, 128, None) == \
        abi.UNSUPPORTED
    assert _rc(L, "moe_quant_mxfp4", fake, 4, 256, None, 0, ctypes.c_void_p(4098), fake, 0, 128,
               None) == abi.INVALID_ARGUMENT
    assert _rc(L, "moe_grouped_gemm_w13_glu_a4w4", fake, fake, fake, fake, E, 384, 3072, 0, fake,
               fake, fake, fake, 1024, fake, 256, None) == abi.UNSUPPORTED      # d % 256
    assert _rc(L, "moe_grouped_gemm_w13_glu_a4w4", fake, fake, fake, fake, E, 3584, 3072, 2, fake,
               fake, fake, fake, 1024, fake, 256, None) == abi.UNSUPPORTED      # hs layout
    assert _rc(L, "moe_grouped_gemm_w13_glu_a4w4", fake, fake, fake, fake, E, 3584, 3072, 0, fake,
               fake, fake, fake, 1024, fake, 8, None) == abi.WORKSPACE_TOO_SMALL
    dims_a4 = abi._Dims(4, 384, 896, 16, 3072)
    assert _rc(L, "moe_forward_a4w4", ctypes.byref(dims_a4), 0, fake, fake, ctypes.byref(W), fake,
               None, None, fake, 10 ** 9, None) == abi.UNSUPPORTED               # d % 256
    assert _rc(L, "moe_forward_a4w4", ctypes.byref(dims), 0, fake, fake, ctypes.byref(W), fake,
               None, None, fake, 10, None) == abi.WORKSPACE_TOO_SMALL
    # BF16 GEMMs: K not a multiple of 64, N not a multiple of 8, SwiGLU N % 256, bad epilogue,
    # misaligned operands, short workspace, E too large for the router
    assert _rc(L, "moe_gemm_bf16", fake, fake, 64, 256, 96, 1, fake, fake, 256, None) == \
        abi.UNSUPPORTED
    assert _rc(L, "moe_gemm_bf16", fake, fake, 64, 100, 128, 1, fake, fake, 256, None) == \
        abi.UNSUPPORTED
    assert _rc(L, "moe_gemm_bf16", fake, fake, 64, 384, 128, 2, fake, fake, 256, None) == \
        abi.UNSUPPORTED
    assert _rc(L, "moe_gemm_bf16", fake, fake, 64, 256, 128, 3, fake, fake, 256, None) == \
        abi.UNSUPPORTED
    assert _rc(L, "moe_gemm_bf16", ctypes.c_void_p(4104), fake, 64, 256, 128, 1, fake, fake, 256,
               None) == abi.INVALID_ARGUMENT
    assert _rc(L, "moe_gemm_bf16", fake, fake, 64, 256, 128, 1, fake, fake, 8, None) == \
        abi.WORKSPACE_TOO_SMALL
    assert _rc(L, "moe_gemm_bf16", fake, fake, 0, 256, 128, 1, None, None, 0, None) == abi.OK
    assert _rc(L, "moe_router_logits", fake, fake, 4, 7168, 2048, fake, fake, 256, None) == \
        abi.UNSUPPORTED
    # status helpers
    assert _rc(L, "moe_check_device_status", None, None) == abi.INVALID_ARGUMENT
    assert _rc(L, "moe_selftest_wait_timeout", fake, 8, 100, None) == abi.WORKSPACE_TOO_SMALL


def test_block_sizes_and_host_validation(L):
    full = (64, 7168, 3584, 896, 16, 3072, 6144)
    n = abi.moe_block_workspace_size(*full)
    layer = abi.moe_workspace_size(64, 3584, 896, 16, 3072)
    # status + x + logits + routed output + shared h + two GEMM workspaces + the layer's
    assert n >= layer + 64 * (3584 * 2 * 2 + 896 * 4 + 6144 * 2)
    for bad, code in (((64, 7168, 3584, 900, 16, 3072, 6144), abi.UNSUPPORTED),   # E % 8
                      ((64, 7100, 3584, 896, 16, 3072, 6144), abi.UNSUPPORTED),   # hidden % 64
                      ((64, 7168, 3584, 896, 16, 3072, 6000), abi.UNSUPPORTED),   # shared_I % 128
                      ((64, 7168, 3500, 896, 16, 3072, 6144), abi.UNSUPPORTED),   # d % 128
                      ((-1, 7168, 3584, 896, 16, 3072, 6144), abi.INVALID_ARGUMENT)):
        with pytest.raises(abi.MoeError) as err:
            abi.moe_block_workspace_size(*bad)
        assert err.value.code == code
    # null pointers are refused on the host, before any launch
    dims = abi._BlockDims(*full)
    W = abi._BlockWeights(None, None, None, None, abi._Weights(None, None, None, None))
    rc = L.moe_block_forward(ctypes.byref(dims), 0, None, ctypes.byref(W), None, None, 0, None,
                             None)
    assert rc == abi.INVALID_ARGUMENT
    rc = L.moe_gemm_bf16_cat(None, 64, None, 64, None, 8, 8, 1, None, None, 0, None)
    assert rc == abi.INVALID_ARGUMENT
    rc = L.moe_gemm_bf16_cat(None, 32, None, 64, None, 8, 8, 1, None, None, 0, None)
    assert rc == abi.UNSUPPORTED    # K1 below one 64-input stage
