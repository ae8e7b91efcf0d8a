"""Pins of the oracle's A4W4 stage 1 (MXFP4 activations).

- E2M1 round-to-nearest-even with saturation against hand-derived cases
  (tests/golden/e2m1_rne_cases.txt) and against an arithmetic restatement
  (numpy round-half-even on v / step) on random values and every midpoint.
- The MX rule with E2M1 elements: powers of two, amax = 6 * 2^s (exact),
  amax just below 8 * 2^s (saturates), all zeros, scaling invariance, exact
  round trips, and an independent numpy restatement.
- Stage 1 with MXFP4 activations against the dense fp64 restatement.
- The A4W4 layer: sparse oracle = dense brute force; E = k = 1 is a textbook
  gated MLP with MXFP4 activations; k = 0 gives zeros; it differs from the
  MXFP8 layer (the activation format is really switched).
"""
import os

import numpy as np
import pytest
import torch
from scipy.special import expit

from mxfp4_latent_moe_gb300 import synth
from tests import mx_numpy as mx

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e2m1_rne_cases.txt")


def _golden_cases():
    out = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                v, c = line.split()
                out.append((float(v), int(c, 16)))
    return out


@pytest.mark.parametrize("v,code", _golden_cases())
def test_e2m1_encode_golden(orc, v, code):
    assert orc.e2m1_encode(v) == code


def test_e2m1_encode_matches_arithmetic_rounding(orc):
    g = np.random.default_rng(11)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    v = np.concatenate([g.uniform(-8, 8, 20000), g.normal(0, 1, 5000) * 10.0 ** g.integers(-3, 2, 5000),
                        mids, -mids, mx.e2m1_table()])
    got = np.array([orc.e2m1_encode(x) for x in v], np.uint8)
    ref = mx.e2m1_code_of(mx.e2m1_rne_sat(v))
    assert np.array_equal(got, ref)


def _blocks(values32):
    return np.asarray(values32, np.float32).reshape(1, 32)


def test_mxfp4_rule_hand_blocks(orc):
    # amax = 6 * 2^s: scale 2^s, exact, no saturation
    for s in (-10, 0, 7):
        v = np.zeros(32, np.float32)
        v[3], v[4] = 6.0 * 2.0 ** s, -1.5 * 2.0 ** s
        p, sc = orc.mxfp4_quant_rows(_blocks(v))
        assert sc[0, 0] == 127 + s
        codes = np.stack([p[0] & 0xF, p[0] >> 4], axis=-1).reshape(32)
        assert codes[3] == 0x7 and codes[4] == 0xB and not codes[np.arange(32) > 4].any()
    # amax just below 8 * 2^s: same scale, saturates to 6
    v = np.zeros(32, np.float32)
    v[0] = 7.96875
    p, sc = orc.mxfp4_quant_rows(_blocks(v))
    assert sc[0, 0] == 127 and (p[0, 0] & 0xF) == 0x7
    # amax = 4: floor(log2 4) - 2 = 0 -> scale 2^0, 4 -> code 6
    v[0] = 4.0
    p, sc = orc.mxfp4_quant_rows(_blocks(v))
    assert sc[0, 0] == 127 and (p[0, 0] & 0xF) == 0x6
    # all zeros (and -0): scale code 0, codes keep the sign of zero
    v = np.zeros(32, np.float32)
    v[1] = -0.0
    p, sc = orc.mxfp4_quant_rows(_blocks(v))
    assert sc[0, 0] == 0 and p[0, 0] == 0x80 and not p[0, 1:].any()


def test_mxfp4_scaling_invariance_and_round_trip(orc):
    g = np.random.default_rng(3)
    x = (g.standard_normal((16, 128)) * 3).astype(np.float32)
    p0, s0 = orc.mxfp4_quant_rows(x)
    for s in (-20, 6, 40):
        p, sc = orc.mxfp4_quant_rows((x * 2.0 ** s).astype(np.float32))
        assert np.array_equal(p, p0) and np.array_equal(sc.astype(int), s0.astype(int) + s)
    # representable blocks (E2M1 values x 2^s with amax in {4, 6} x 2^s) round-trip exactly
    table = mx.e2m1_table()
    for s in (-3, 0, 5):
        vals = table[g.integers(0, 16, (8, 64))] * 2.0 ** s
        vals[:, ::32] = 6.0 * 2.0 ** s
        p, sc = orc.mxfp4_quant_rows(vals.astype(np.float32))
        np.testing.assert_array_equal(mx.decode_mxfp4(p, sc), vals)


def test_mxfp4_rows_match_numpy_restatement(orc):
    g = np.random.default_rng(5)
    x = g.standard_normal((64, 256)).astype(np.float32)
    x[3] *= 2.0 ** 40
    x[7, :32] = 0.0
    x[9] = np.round(x[9] * 4) / 4      # many exact midpoints after scaling
    p, sc = orc.mxfp4_quant_rows(x)
    rp, rsc = mx.quant_mxfp4(x)
    assert np.array_equal(p, rp) and np.array_equal(sc, rsc)
    # the bf16 entry point quantises the decoded bf16 values
    xb = synth.bf16_bits(torch.from_numpy(x).to(torch.bfloat16))
    pb, sb = orc.mxfp4_quant_rows_bf16(xb)
    rpb, rsb = mx.quant_mxfp4(mx.bf16_bits_to_f64(xb).astype(np.float32))
    assert np.array_equal(pb, rpb) and np.array_equal(sb, rsb)


def test_stage1_a4_matches_dense_restatement(orc):
    wl = synth.shape("stages", T=6, d=128, E=2, k=1, I=64)
    L = synth.make_layer(wl, seed=5)
    w13, w13s = L["w13"].numpy()[1], L["w13_s"].numpy()[1]
    xq = (synth.random_e4m3_codes((6, 64), seed=7).numpy())          # any bytes: packed E2M1
    xs = synth.random_scale_codes((6, 4), lo=120, hi=130, seed=8).numpy()
    W13 = mx.decode_mxfp4(w13, w13s)
    for r in range(6):
        xd = mx.decode_mxfp4(xq[r:r + 1], xs[r:r + 1])[0]
        g, u = W13[:64] @ xd, W13[64:] @ xd
        h = orc.expert_stage1_a4(xq[r], xs[r], w13, w13s)
        np.testing.assert_allclose(h, g * expit(g) * u, rtol=1e-12, atol=1e-300)


def _dense_layer_a4(x_bits, logits, k, w13, w13s, w2, w2s):
    """Every expert on every token in fp64 with MXFP4 stage-1 activations."""
    T, d = x_bits.shape
    E = logits.shape[1]
    I = w13.shape[1] // 2
    xp, xs = mx.quant_mxfp4(mx.bf16_bits_to_f64(x_bits).astype(np.float32))
    Xd = mx.decode_mxfp4(xp, xs)
    ids = np.stack([np.lexsort((np.arange(E), -logits[t].astype(np.float64)))[:k]
                    for t in range(T)]) if k > 0 else np.zeros((T, 0), np.int64)
    sel = np.take_along_axis(logits.astype(np.float64), ids, axis=1)
    s = expit(sel)
    w = (s / s.sum(axis=1, keepdims=True)).astype(np.float32) if k > 0 else s
    gate = np.zeros((T, E))
    for t in range(T):
        gate[t, ids[t]] = w[t]
    y = np.zeros((T, d))
    for e in range(E):
        W13 = mx.decode_mxfp4(w13[e], w13s[e])
        G, U = Xd @ W13[:I].T, Xd @ W13[I:].T
        H = (G * expit(G) * U).astype(np.float32)
        hc, hs = mx.quant_mxfp8(H)
        y += gate[:, e:e + 1].astype(np.float64) * (mx.decode_mxfp8(hc, hs) @ mx.decode_mxfp4(w2[e], w2s[e]).T)
    return y, ids


@pytest.mark.parametrize("wl", [
    synth.workload("tiny"),
    synth.shape("ragged", T=13, d=128, E=9, k=3, I=96),
    synth.shape("outliers", T=20, d=64, E=6, k=2, I=32, outlier_frac=0.1),
])
def test_a4w4_layer_equals_dense_brute_force(orc, wl):
    L = synth.make_layer(wl, seed=0)
    xb = synth.bf16_bits(L["x"])
    lg = L["logits"].numpy()
    W = {n: L[n].numpy() for n in ("w13", "w13_s", "w2", "w2_s")}
    out = orc.moe_forward(xb, lg, wl.k, W["w13"], W["w13_s"], W["w2"], W["w2_s"], want_y64=True,
                          a4w4=True)
    ref, ids = _dense_layer_a4(xb, lg, wl.k, W["w13"], W["w13_s"], W["w2"], W["w2_s"])
    assert np.array_equal(out["ids"], ids)
    rms = np.sqrt((ref ** 2).mean(axis=1, keepdims=True))
    assert np.all(np.abs(out["y64"] - ref) <= 1e-12 * rms + 1e-300)
    # really a different layer from the MXFP8 one
    out8 = orc.moe_forward(xb, lg, wl.k, W["w13"], W["w13_s"], W["w2"], W["w2_s"], want_y64=True)
    assert not np.allclose(out8["y64"], out["y64"], rtol=1e-3, atol=0)


def test_a4w4_one_expert_is_a_textbook_gated_mlp(orc):
    wl = synth.shape("one", T=10, d=256, E=1, k=1, I=128)
    L = synth.make_layer(wl, seed=3)
    xb = synth.bf16_bits(L["x"])
    out = orc.moe_forward(xb, L["logits"].numpy(), 1, L["w13"].numpy(), L["w13_s"].numpy(),
                          L["w2"].numpy(), L["w2_s"].numpy(), want_y64=True, a4w4=True)
    xp, xs = mx.quant_mxfp4(mx.bf16_bits_to_f64(xb).astype(np.float32))
    X = torch.from_numpy(mx.decode_mxfp4(xp, xs))
    W13 = torch.from_numpy(mx.decode_mxfp4(L["w13"].numpy()[0], L["w13_s"].numpy()[0]))
    W2 = torch.from_numpy(mx.decode_mxfp4(L["w2"].numpy()[0], L["w2_s"].numpy()[0]))
    H = torch.nn.functional.silu(X @ W13[:128].T) * (X @ W13[128:].T)
    hc, hs = mx.quant_mxfp8(H.float().numpy())
    ref = (torch.from_numpy(mx.decode_mxfp8(hc, hs)) @ W2.T).numpy()
    rms = np.sqrt((ref ** 2).mean(axis=1, keepdims=True))
    assert np.all(np.abs(out["y64"] - ref) <= 1e-12 * rms)


def test_a4w4_k_zero_gives_zeros(orc):
    wl = synth.shape("k0", T=4, d=64, E=5, k=0, I=32)
    L = synth.make_layer(wl, seed=1)
    out = orc.moe_forward(synth.bf16_bits(L["x"]), L["logits"].numpy(), 0, L["w13"].numpy(),
                          L["w13_s"].numpy(), L["w2"].numpy(), L["w2_s"].numpy(), want_y64=True,
                          a4w4=True)
    assert not out["y"].any() and not out["y64"].any()
