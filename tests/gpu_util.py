"""Helpers for the GPU parity tests: library loading, the TILED scale layout
written out in numpy (from its definition in include/moe.h), tolerances."""
import numpy as np
import pytest
import torch


def cuda_lib():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for tests marked gpu")
    from mxfp4_latent_moe_gb300 import abi
    from mxfp4_latent_moe_gb300.build import build_library
    build_library()
    abi.lib()
    return abi


def tiled_index(rows, K):
    """Byte offsets of scale (r, b) in the TILED layout, shape [rows][K/32]."""
    r = np.arange(rows, dtype=np.int64)[:, None]
    b = np.arange(K // 32, dtype=np.int64)[None, :]
    return ((r // 128) * (K // 128) + b // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + b % 4


def group32_index(rows, K):
    """Byte offsets of scale (r, b) in the GROUP32 layout, shape [rows][K/32]."""
    r = np.arange(rows, dtype=np.int64)[:, None]
    b = np.arange(K // 32, dtype=np.int64)[None, :]
    return ((r // 32) * (K // 128) + b // 4) * 512 + (r % 32) * 16 + b % 4


def scale_offsets(rows, K, layout):
    """Byte offsets, as a torch tensor on rows' device, of the scales of the
    given rows (int64 tensor [n]) in layout 0 (TILED) or 1 (GROUP32): [n][K/32]."""
    r = rows.to(torch.int64)[:, None]
    b = torch.arange(K // 32, dtype=torch.int64, device=rows.device)[None, :]
    if layout:
        return ((r // 32) * (K // 128) + b // 4) * 512 + (r % 32) * 16 + b % 4
    return ((r // 128) * (K // 128) + b // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + b % 4


def untile_g32(buf, rows, K):
    return buf.reshape(-1)[group32_index(rows, K)]


def tile_g32(canon, K):
    rows = canon.shape[0]
    out = np.zeros((rows + 31) // 32 * 32 * K // 8, np.uint8)
    out[group32_index(rows, K)] = canon
    return out


def untile(tiled, rows, K):
    flat = tiled.reshape(-1)
    return flat[tiled_index(rows, K)]


def tile(canon, K, rows_padded=None):
    rows = canon.shape[0]
    rp = rows_padded or (rows + 127) // 128 * 128
    out = np.zeros(rp * (K // 32), np.uint8)
    out[tiled_index(rows, K)] = canon
    return out


def e4m3(codes):
    c = torch.from_numpy(np.ascontiguousarray(codes, np.uint8))
    return c.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def dequant_mxfp8(codes, scales):
    return e4m3(codes) * np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), 32, axis=-1)


def bf16_to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def bf16_half_ulp(v):
    """Half the spacing of bf16 values at |v| (2^(floor(log2|v|) - 8); 0 at 0):
    the most that rounding the exact value to the bf16 output moves it."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.ldexp(1.0, (e - 8).astype(np.int64)), 0.0)


def assert_layer_close(got, ref, what="y"):
    """The layer's output bar: |gpu - oracle| <= 2e-2 * rms(oracle row) + 1e-3,
    on top of the rounding to the bf16 output format itself.

    ref is the oracle's exact (fp64) output. Any bf16 result, the exact value
    rounded once included, differs from it by up to half a bf16 ulp,
    2^-8 |y| at the top of a binade: more than 2e-2 * rms for elements above
    5.12 rms. The bound is therefore applied to the error beyond that half
    ulp: |gpu - ref| <= 2e-2 * rms + 1e-3 + half_ulp_bf16(ref)."""
    rms = np.sqrt((ref ** 2).mean(axis=-1, keepdims=True))
    err = np.abs(got - ref)
    bound = 2e-2 * rms + 1e-3 + bf16_half_ulp(ref)
    bad = err > bound
    worst = np.unravel_index(np.argmax(err / bound), err.shape)
    assert not bad.any(), (
        "%s: %d of %d elements outside tolerance; worst at %s: |err| %.3g, bound %.3g, "
        "|ref| %.3g, row rms %.3g" % (what, int(bad.sum()), bad.size, tuple(int(i) for i in worst),
                                      float(err[worst]), float(bound[worst]),
                                      float(abs(ref[worst])), float(np.broadcast_to(rms, err.shape)[worst])))
