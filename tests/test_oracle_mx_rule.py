"""Pins of the oracle's MX quantisation rule (MXFP8: E4M3 elements, one E8M0
scale per 32).

Hand-built blocks with exactly known answers, the scaling invariance that the
outlier workload relies on, exact round trips, and an independent restatement
of the rule through numpy's frexp and torch's float8_e4m3fn conversion.
"""
import numpy as np
import torch


def _block(vals):
    b = np.zeros(32, np.float32)
    b[: len(vals)] = vals
    return b


def _q(orc, block):
    codes, scales = orc.mx_quant_rows(np.asarray(block, np.float32).reshape(1, 32))
    return codes[0], int(scales[0, 0])


def test_powers_of_two(orc):
    for s in (-20, -3, 0, 5, 40):
        vals = np.array([2.0 ** (s - j) for j in range(32)], np.float32)
        codes, scale = _q(orc, vals)
        # amax = 2^s -> shared exponent s - 8 -> element value 2^(8 - j)
        assert scale == s - 8 + 127
        for j in range(32):
            expect = 2.0 ** (8 - j)
            got = orc.e4m3_value(codes[j])
            if expect >= 2.0 ** -9:
                assert got == expect, (s, j)
            elif expect > 2.0 ** -10:
                assert got == 2.0 ** -9
            else:
                assert got == 0.0


def test_amax_448_times_power_of_two_is_not_saturated(orc):
    for s in (-5, 0, 7):
        codes, scale = _q(orc, _block([448.0 * 2.0 ** s, -3.0 * 2.0 ** s]))
        assert scale == 127 + s and codes[0] == 0x7E
        assert orc.e4m3_value(codes[1]) == -3.0


def test_amax_511_saturates_to_448(orc):
    codes, scale = _q(orc, _block([511.0, 500.0, 464.0, 463.0, -511.0]))
    assert scale == 127  # floor(log2(511)) = 8 -> X = 2^0
    assert list(codes[:5]) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE]


def test_midpoints_round_to_even_code(orc):
    # amax 256 -> X = 1, so the other elements are rounded as given
    codes, scale = _q(orc, _block([256.0, 1.0625, 1.1875, -1.0625, 2.5 * 2.0 ** -9, 3.5 * 2.0 ** -9]))
    assert scale == 127
    assert codes[1] == 0x38          # 1.0625 between 1.0 (0x38) and 1.125 (0x39)
    assert codes[2] == 0x3A          # 1.1875 between 1.125 (0x39) and 1.25 (0x3A)
    assert codes[3] == 0xB8
    assert codes[4] == 0x02          # subnormal tie 2.5 * 2^-9 -> 2 * 2^-9
    assert codes[5] == 0x04          # subnormal tie 3.5 * 2^-9 -> 4 * 2^-9


def test_single_nonzero_element_and_subnormal_codes(orc):
    codes, scale = _q(orc, _block([0.0] * 5 + [256.0] + [0.0] * 3 + [2.0 ** -8, 2.0 ** -9 * 3]))
    assert scale == 127
    assert codes[5] == 0x78                    # 256 = 2^8
    assert codes[9] == 0x02                    # 2^-8 = 2 * 2^-9
    assert codes[10] == 0x03
    assert all(codes[i] == 0 for i in range(32) if i not in (5, 9, 10))


def test_all_zero_block_and_negative_zero(orc):
    codes, scale = _q(orc, np.zeros(32, np.float32))
    assert scale == 0 and not codes.any()
    b = np.zeros(32, np.float32)
    b[3] = -0.0
    codes, scale = _q(orc, b)
    assert scale == 0 and codes[3] == 0x80 and codes.sum() == 0x80


def test_tiny_amax_clamps_scale_code_to_zero(orc):
    v = np.float32(2.0 ** -130)  # fp32 subnormal; floor(log2) - 8 + 127 < 0
    codes, scale = _q(orc, _block([v, -v]))
    assert scale == 0
    assert orc.e4m3_value(codes[0]) * 2.0 ** -127 == float(v)
    assert orc.e4m3_value(codes[1]) * 2.0 ** -127 == -float(v)


def test_scaling_invariance_codes_equal_scale_shifts(orc):
    """quant(2^s * v) has the same codes and scale + s: the x64 outlier rows
    of the long-prefill workload must give the unscaled row's codes, scales + 6."""
    rng = np.random.default_rng(3)
    v = rng.normal(0, 1, (64, 32)).astype(np.float32)
    c0, s0 = orc.mx_quant_rows(v)
    for s in (6, -6, 20):
        c1, s1 = orc.mx_quant_rows((v * np.float32(2.0 ** s)).astype(np.float32))
        assert np.array_equal(c0, c1)
        assert np.array_equal(s1.astype(int), s0.astype(int) + s)


def test_round_trip_of_representable_blocks(orc):
    rng = np.random.default_rng(4)
    for _ in range(200):
        codes = rng.integers(0, 0x7F, 32).astype(np.uint8) | (rng.integers(0, 2, 32) * 0x80).astype(np.uint8)
        codes[rng.integers(0, 32)] = 0x78 + rng.integers(0, 7)   # one element in [256, 448]
        s = int(rng.integers(20, 230))
        vals = np.array([orc.e4m3_value(c) * 2.0 ** (s - 127) for c in codes], np.float32)
        c2, s2 = _q(orc, vals)
        assert s2 == s
        back = np.array([orc.e4m3_value(c) for c in c2]) * 2.0 ** (s - 127)
        assert np.array_equal(back, vals.astype(np.float64))


def test_rule_matches_frexp_and_torch_cast_restatement(orc):
    """An independent statement of the rule: the scale from numpy's frexp of
    amax, the elements from torch's RNE float8_e4m3fn cast after clamping to
    +-448 (torch does not saturate)."""
    rng = np.random.default_rng(5)
    v = np.concatenate([
        rng.normal(0, 1, (200, 32)), rng.normal(0, 1, (50, 32)) * 64.0,
        rng.standard_cauchy((50, 32)), rng.normal(0, 1e-30, (20, 32)),
    ]).astype(np.float32)
    codes, scales = orc.mx_quant_rows(v)
    amax = np.abs(v.astype(np.float64)).max(axis=1)
    _, ex = np.frexp(amax)
    sc = np.clip(ex - 1 - 8 + 127, 0, 254)
    sc[amax == 0] = 0
    q = v.astype(np.float64) / np.ldexp(1.0, sc - 127)[:, None]
    q = np.clip(q, -448.0, 448.0)
    ref = torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(scales[:, 0], sc.astype(np.uint8))
    assert np.array_equal(codes, ref)


def test_bf16_rows_equal_fp32_rows(orc):
    rng = np.random.default_rng(6)
    x = torch.from_numpy(rng.normal(0, 1, (16, 256)).astype(np.float32)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    c1, s1 = orc.mx_quant_rows_bf16(bits)
    c2, s2 = orc.mx_quant_rows(x.float().numpy())
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2)
