"""Pins of the oracle's whole layer.

- A dense brute force in numpy/torch (every expert on every token, then masked
  with the routing weights) must equal the oracle's sparse per-token layer.
- One expert with k = 1 reduces to a textbook gated MLP (torch fp64 matmuls).
- k = 0 gives zeros.
- The stage functions agree with the same dense restatement.
"""
import numpy as np
import pytest
import torch
from scipy.special import expit

from mxfp4_latent_moe_gb300 import synth
from tests import mx_numpy as mx


def _dense_layer(x_bits, logits, k, w13, w13s, w2, w2s):
    """Every expert on every token in fp64, masked by the routing."""
    T, d = x_bits.shape
    E = logits.shape[1]
    I = w13.shape[1] // 2
    xc, xs = mx.quant_mxfp8(mx.bf16_bits_to_f64(x_bits).astype(np.float32))
    Xd = mx.decode_mxfp8(xc, xs)                                   # [T][d]
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
        W13 = mx.decode_mxfp4(w13[e], w13s[e])                     # [2I][d]
        G = Xd @ W13[:I].T
        U = Xd @ W13[I:].T
        H = (G * expit(G) * U).astype(np.float32)
        hc, hs = mx.quant_mxfp8(H)
        Hd = mx.decode_mxfp8(hc, hs)
        Y = Hd @ mx.decode_mxfp4(w2[e], w2s[e]).T                  # [T][d]
        y += gate[:, e:e + 1].astype(np.float64) * Y
    return y, ids


def _np(layer):
    return {k: (v.numpy() if isinstance(v, torch.Tensor) and v.dtype != torch.bfloat16 else v)
            for k, v in layer.items()}


@pytest.mark.parametrize("wl", [
    synth.workload("tiny"),
    synth.shape("ragged", T=13, d=128, E=9, k=3, I=96),
    synth.shape("skewed", T=16, d=128, E=12, k=5, I=64, skew=True),
    synth.shape("outliers", T=20, d=64, E=6, k=2, I=32, outlier_frac=0.1),
])
def test_sparse_layer_equals_dense_brute_force(orc, wl):
    L = synth.make_layer(wl, seed=0)
    xb = synth.bf16_bits(L["x"])
    lg = L["logits"].numpy()
    W = {n: L[n].numpy() for n in ("w13", "w13_s", "w2", "w2_s")}
    out = orc.moe_forward(xb, lg, wl.k, W["w13"], W["w13_s"], W["w2"], W["w2_s"], want_y64=True)
    ref, ids = _dense_layer(xb, lg, wl.k, W["w13"], W["w13_s"], W["w2"], W["w2_s"])
    assert np.array_equal(out["ids"], ids)
    rms = np.sqrt((ref ** 2).mean(axis=1, keepdims=True))
    assert np.all(np.abs(out["y64"] - ref) <= 1e-12 * rms + 1e-300)
    # the bf16 output is the fp64 sum rounded once
    yb = mx.bf16_bits_to_f64(out["y"])
    assert np.all(np.abs(yb - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-38)


def test_one_expert_top1_is_a_textbook_gated_mlp(orc):
    wl = synth.shape("one", T=10, d=256, E=1, k=1, I=128)
    L = synth.make_layer(wl, seed=3)
    xb = synth.bf16_bits(L["x"])
    out = orc.moe_forward(xb, L["logits"].numpy(), 1, L["w13"].numpy(), L["w13_s"].numpy(),
                          L["w2"].numpy(), L["w2_s"].numpy(), want_y64=True)
    assert np.all(out["w"] == 1.0) and np.all(out["ids"] == 0)
    xc, xs = mx.quant_mxfp8(mx.bf16_bits_to_f64(xb).astype(np.float32))
    X = torch.from_numpy(mx.decode_mxfp8(xc, xs))
    W13 = torch.from_numpy(mx.decode_mxfp4(L["w13"].numpy()[0], L["w13_s"].numpy()[0]))
    W2 = torch.from_numpy(mx.decode_mxfp4(L["w2"].numpy()[0], L["w2_s"].numpy()[0]))
    G, U = X @ W13[:128].T, X @ W13[128:].T
    H = torch.nn.functional.silu(G) * U
    hc, hs = mx.quant_mxfp8(H.float().numpy())
    Y = torch.from_numpy(mx.decode_mxfp8(hc, hs)) @ W2.T
    ref = Y.numpy()
    rms = np.sqrt((ref ** 2).mean(axis=1, keepdims=True))
    assert np.all(np.abs(out["y64"] - ref) <= 1e-12 * rms)


def test_k_zero_gives_zeros(orc):
    wl = synth.shape("k0", T=4, d=64, E=5, k=0, I=32)
    L = synth.make_layer(wl, seed=1)
    out = orc.moe_forward(synth.bf16_bits(L["x"]), L["logits"].numpy(), 0, L["w13"].numpy(),
                          L["w13_s"].numpy(), L["w2"].numpy(), L["w2_s"].numpy(), want_y64=True)
    assert not out["y"].any() and not out["y64"].any()


def test_stage_functions_match_dense_restatement(orc):
    wl = synth.shape("stages", T=6, d=128, E=2, k=1, I=64)
    L = synth.make_layer(wl, seed=5)
    w13, w13s = L["w13"].numpy()[1], L["w13_s"].numpy()[1]
    w2, w2s = L["w2"].numpy()[1], L["w2_s"].numpy()[1]
    xq = synth.random_e4m3_codes((6, 128), seed=7).numpy()
    xs = synth.random_scale_codes((6, 4), lo=120, hi=130, seed=8).numpy()
    hq = synth.random_e4m3_codes((6, 64), seed=9).numpy()
    hs = synth.random_scale_codes((6, 2), lo=120, hi=130, seed=10).numpy()
    W13 = mx.decode_mxfp4(w13, w13s)
    W2 = mx.decode_mxfp4(w2, w2s)
    for r in range(6):
        xd = mx.decode_mxfp8(xq[r:r + 1], xs[r:r + 1])[0]
        g, u = W13[:64] @ xd, W13[64:] @ xd
        h = orc.expert_stage1(xq[r], xs[r], w13, w13s)
        np.testing.assert_allclose(h, g * expit(g) * u, rtol=1e-12, atol=1e-300)
        y = orc.expert_stage2(hq[r], hs[r], w2, w2s)
        np.testing.assert_allclose(y, W2 @ mx.decode_mxfp8(hq[r:r + 1], hs[r:r + 1])[0], rtol=1e-12)
