"""Pins of the oracle's element formats and roundings.

Each check compares the oracle with a source other than the oracle itself:
the OCP value list, torch's float8 conversions (library routines), or closed
forms with exactly known answers.
"""
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_floats(name):
    vals = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                vals.extend(float(tok) for tok in line.split())
    return vals


def _golden_kv(name):
    kv = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, val = line.split()
                kv[key] = float(val)
    return kv


def test_e2m1_table_matches_ocp_value_list(orc):
    expect = _golden_floats("e2m1_values.txt")
    assert len(expect) == 16
    for code, v in enumerate(expect):
        got = orc.e2m1_value(code)
        assert got == v and math.copysign(1.0, got) == math.copysign(1.0, v), (code, got, v)


def test_e4m3_table_matches_torch_float8_e4m3fn(orc):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = orc.e4m3_value(c)
        if np.isnan(ref[c]):
            assert math.isnan(got) and c in (0x7F, 0xFF)
        else:
            assert got == ref[c] and math.copysign(1, got) == math.copysign(1, ref[c]), c
    assert orc.e4m3_value(0x7E) == 448.0
    assert orc.e4m3_value(0x01) == 2.0 ** -9


def test_e8m0_table_matches_torch_float8_e8m0fnu(orc):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    for c in range(256):
        got = orc.e8m0_value(c)
        if c == 255:
            assert math.isnan(got) and math.isnan(ref[c])
        else:
            assert got == ref[c] == 2.0 ** (c - 127), c


def test_e4m3_encode_matches_torch_rne_in_range(orc):
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.normal(0, 1, 3000), rng.normal(0, 60, 3000), rng.uniform(-448, 448, 2000),
        rng.uniform(-2.0 ** -6, 2.0 ** -6, 2000),           # subnormal range
    ])
    # exact midpoints between neighbouring codes (ties to even)
    mags = [orc.e4m3_value(c) for c in range(0x7F)]
    mids = [(a + b) / 2 for a, b in zip(mags[:-1], mags[1:])]
    vals = np.concatenate([vals, mids, [-m for m in mids]]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(float(v)) for v in vals], np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_encode_saturates_and_keeps_zero_sign(orc):
    assert orc.e4m3_encode(448.0) == 0x7E
    assert orc.e4m3_encode(463.99) == 0x7E
    assert orc.e4m3_encode(464.0) == 0x7E      # tie between 448 and (absent) 480
    assert orc.e4m3_encode(511.0) == 0x7E
    assert orc.e4m3_encode(1e9) == 0x7E
    assert orc.e4m3_encode(-1e9) == 0xFE
    assert orc.e4m3_encode(0.0) == 0x00
    assert orc.e4m3_encode(-0.0) == 0x80
    assert orc.e4m3_encode(-1e-30) == 0x80     # rounds to -0
    assert orc.e4m3_encode(2.0 ** -10) == 0x00  # tie between 0 and 2^-9 -> even (0)
    assert orc.e4m3_encode(1.5 * 2.0 ** -10) == 0x01


def test_bf16_rounding_single_step_from_fp64(orc):
    # closed forms: 1 + 2^-8 is the midpoint of 1 and 1 + 2^-7
    assert orc.bf16_rne(1.0 + 2.0 ** -8) == 0x3F80               # tie -> even (1.0)
    assert orc.bf16_rne(1.0 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81  # just above the tie
    assert orc.bf16_rne(1.0 + 3 * 2.0 ** -8) == 0x3F82            # tie -> even (1+2^-6)
    assert orc.bf16_rne(-2.0) == 0xC000
    assert orc.bf16_rne(-0.0) == 0x8000
    assert orc.bf16_rne(3.0e38) == 0x7F62
    assert orc.bf16_rne(1e39) == 0x7F80
    assert orc.bf16_rne(2.0 ** -133) == 0x0001                    # smallest subnormal
    # against torch's fp32 -> bf16 rounding on values exact in fp32
    rng = np.random.default_rng(2)
    v = np.concatenate([rng.normal(0, 1, 4000), rng.normal(0, 1e-3, 1000) * 1e-36]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.bf16_rne(float(a)) for a in v], np.uint16)
    assert np.array_equal(got, ref)


def test_storage_pins_from_weight_distribution_table(orc):
    g = _golden_kv("storage_pins.txt")
    per_expert = orc.expert_bytes(int(g["latent"]), int(g["intermediate"]))
    assert per_expert == 17_547_264
    total = per_expert * int(g["experts"]) * int(g["moe_layers"])
    assert total == 1_446_456_066_048
    assert round(total / 1e9, 3) == g["routed_expert_full_gb"]
    assert round(total / g["tp"] / 1e9, 3) == g["routed_expert_tp8_gb"]


def test_index_key_pin_fixes_four_bit_codes_and_one_scale_per_32(orc):
    g = _golden_kv("storage_pins.txt")
    K = int(g["index_key_dims"])
    # one expert-sized matrix of 1 row x K: packed codes + scales
    mx4 = orc.expert_bytes(K, 32) // 3 // 32 * 1  # bytes of a 32 x K matrix / 32 rows
    assert mx4 == g["index_key_mxfp4_bytes"]
    fp8 = K + K // 32
    assert fp8 == g["index_key_fp8_bytes"]
    assert round(100 * (1 - mx4 / fp8), 1) == g["index_key_saving_pct"]
