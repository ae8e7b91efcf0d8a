"""A second, independent statement of the MX formats for the oracle pins.

It decodes E2M1 from the OCP value list in tests/golden, E8M0 with numpy's
ldexp and E4M3 with torch's float8_e4m3fn type, and quantises with numpy's
frexp plus torch's RNE float8 cast (after clamping to +-448, since torch does
not saturate). Nothing here comes from the oracle or from the CUDA library.
"""
import os

import numpy as np
import torch

_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e2m1_values.txt")


def e2m1_table():
    vals = []
    with open(_GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                vals.extend(float(t) for t in line.split())
    return np.array(vals, np.float64)


def e4m3_decode(codes):
    c = torch.from_numpy(np.ascontiguousarray(codes, np.uint8))
    return c.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def e8m0_decode(codes):
    return np.ldexp(1.0, np.asarray(codes, np.int64) - 127)


def decode_mxfp4(packed, scales):
    """packed u8 [..., R, K/2], scales u8 [..., R, K/32] -> fp64 [..., R, K]."""
    packed = np.asarray(packed, np.uint8)
    lo, hi = packed & 0xF, packed >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(*packed.shape[:-1], packed.shape[-1] * 2)
    vals = e2m1_table()[codes]
    sc = np.repeat(e8m0_decode(scales), 32, axis=-1)
    return vals * sc


def decode_mxfp8(codes, scales):
    return e4m3_decode(codes) * np.repeat(e8m0_decode(scales), 32, axis=-1)


def quant_mxfp8(v):
    """fp32 [rows][K] -> (codes, scales) by the OCP MX rule with saturation."""
    v = np.asarray(v, np.float32)
    rows, K = v.shape
    b = v.astype(np.float64).reshape(rows, K // 32, 32)
    amax = np.abs(b).max(axis=2)
    _, ex = np.frexp(amax)
    sc = np.clip(ex - 1 - 8 + 127, 0, 254)
    sc[amax == 0] = 0
    q = np.clip(b / np.ldexp(1.0, sc - 127)[:, :, None], -448.0, 448.0)
    codes = torch.from_numpy(np.ascontiguousarray(q)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return codes.reshape(rows, K), sc.astype(np.uint8)


def bf16_bits_to_f64(bits):
    b = np.asarray(bits, np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def e2m1_rne_sat(v):
    """Round to E2M1 by arithmetic, independent of any table search: below 1
    the step is 0.5 (subnormals), in [2^e, 2^(e+1)) it is 2^(e-1); v/step is
    rounded half-to-even by numpy (an even multiple of the step is an even
    code), then magnitudes above 6 saturate. Returns fp64 values, sign kept."""
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    _, ex = np.frexp(a)                       # a = m * 2^ex, m in [0.5, 1)
    e = np.maximum(ex - 1, 0)                 # exponent of the binade, 0 for a < 1
    step = np.ldexp(1.0, e - 1)
    q = np.minimum(np.round(a / step) * step, 6.0)
    return np.copysign(q, v)


def e2m1_code_of(vals):
    """E2M1 codes of exactly representable values (sign of zero kept), by
    lookup in the OCP value list."""
    vals = np.asarray(vals, np.float64)
    table = e2m1_table()[:8]
    mag = np.abs(vals)
    idx = np.array([int(np.flatnonzero(table == m)[0]) for m in mag.reshape(-1)]).reshape(mag.shape)
    return (idx | (np.signbit(vals).astype(np.int64) << 3)).astype(np.uint8)


def quant_mxfp4(v):
    """fp32 [rows][K] -> (packed E2M1 [rows][K/2], scales) by the OCP MX rule
    with E2M1 elements (shared exponent floor(log2 amax) - 2), saturation to 6."""
    v = np.asarray(v, np.float32)
    rows, K = v.shape
    b = v.astype(np.float64).reshape(rows, K // 32, 32)
    amax = np.abs(b).max(axis=2)
    _, ex = np.frexp(amax)
    sc = np.clip(ex - 1 - 2 + 127, 0, 254)
    sc[amax == 0] = 0
    q = e2m1_rne_sat(b / np.ldexp(1.0, sc - 127)[:, :, None])
    codes = e2m1_code_of(q).reshape(rows, K)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, sc.astype(np.uint8)
