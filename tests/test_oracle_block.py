"""Pins of the oracle's composed block (oracle.block_forward), on CPU.

The block is a composition of pinned steps (the BF16 products, bf16
rounding, the routed layer). What is pinned here is the composition itself,
against a restatement that shares none of its code: numpy fp64 products of the
decoded bf16 operands, a numpy round-half-even to bf16, and the routed layer
taken as given (its own pins are in test_oracle_layer.py). Special cases fix
which operand feeds which product: with the latent-up columns of w_out zero the
block is the shared experts alone; with the shared gate rows zero it is the
latent up projection of the routed output alone. Also checked: the block
inputs' power-of-two grid makes every fp32 sum of the router exact.
"""
import numpy as np
import pytest
import torch

from mxfp4_latent_moe_gb300 import synth

BW = synth.block_shape("tiny_block", T=6, hidden=256, d=128, E=16, k=4, I=128, shared_I=128)


def _f64(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16) \
        .float().numpy().astype(np.float64)


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _bf16_round(v):
    """Round-half-even of fp64 values to bf16 (8 significant bits), numpy only."""
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    step = np.ldexp(1.0, (e - 7).astype(np.int64))
    return np.where(a > 0, np.round(v / step) * step, v)


def _inputs(seed=0):
    B = synth.make_block(BW, seed=seed)
    return B, {n: _bits(B[n]) for n in ("h", "w_down", "w_router", "w_shared13", "w_out")}, \
        {n: B[n].numpy() for n in ("w13", "w13_s", "w2", "w2_s")}


def _block(orc, hb, W):
    return orc.block_forward(hb["h"], BW.k, hb["w_down"], hb["w_router"], hb["w_shared13"],
                             hb["w_out"], W["w13"], W["w13_s"], W["w2"], W["w2_s"], threads=2)


def test_block_equals_numpy_composition(orc):
    B, hb, W = _inputs()
    got = _block(orc, hb, W)
    h = _f64(hb["h"])
    x = _bf16_round(h @ _f64(hb["w_down"]).T)
    logits = (h @ _f64(hb["w_router"]).T).astype(np.float32)
    assert np.array_equal(_f64(got["x"]), x)
    assert np.array_equal(got["logits"], logits)
    routed = orc.moe_forward(_bits(torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)),
                             logits, BW.k, W["w13"], W["w13_s"], W["w2"], W["w2_s"])
    assert np.array_equal(got["y_lat"], routed["y"])
    Is = BW.shared_I
    ws13 = _f64(hb["w_shared13"])
    g, u = h @ ws13[:Is].T, h @ ws13[Is:].T
    hs = _bf16_round(g / (1.0 + np.exp(-g)) * u)
    assert np.array_equal(_f64(got["hs"]), hs)
    y64 = np.concatenate([_f64(routed["y"]), hs], axis=1) @ _f64(hb["w_out"]).T
    np.testing.assert_allclose(got["y64"], y64, rtol=1e-12, atol=1e-12)
    assert np.array_equal(_f64(got["y"]), _bf16_round(got["y64"]))


def test_block_without_latent_up_is_the_shared_experts(orc):
    B, hb, W = _inputs(seed=1)
    w_out = _f64(hb["w_out"]).copy()
    w_out[:, :BW.d] = 0.0
    hb["w_out"] = _bits(torch.from_numpy(w_out.astype(np.float32)).to(torch.bfloat16))
    got = _block(orc, hb, W)
    ref = _f64(got["hs"]) @ w_out[:, BW.d:].T
    np.testing.assert_allclose(got["y64"], ref, rtol=1e-12, atol=1e-12)


def test_block_without_shared_gate_is_the_routed_output(orc):
    B, hb, W = _inputs(seed=2)
    ws13 = _f64(hb["w_shared13"]).copy()
    ws13[:BW.shared_I] = 0.0                 # silu(0) = 0: hs is exactly zero
    hb["w_shared13"] = _bits(torch.from_numpy(ws13.astype(np.float32)).to(torch.bfloat16))
    got = _block(orc, hb, W)
    assert not _f64(got["hs"]).any()
    ref = _f64(got["y_lat"]) @ _f64(hb["w_out"])[:, :BW.d].T
    np.testing.assert_allclose(got["y64"], ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("hidden", [256, 7168])
def test_block_grid_makes_router_sums_exact_in_fp32(orc, hidden):
    """Every product of the grid is a multiple of 2^-11 below 2^11 in sum:
    an fp32 accumulation in any order equals the exact sum."""
    bw = synth.block_shape("grid", T=8, hidden=hidden, d=128, E=64, k=4, I=128, shared_I=128)
    B = synth.make_block(bw, seed=3)
    h = B["h"].float().numpy().astype(np.float64)
    w = B["w_router"].float().numpy().astype(np.float64)
    exact = h @ w.T
    prods = h[:, None, :] * w[None, :, :]
    fwd = np.cumsum(prods.astype(np.float32), axis=2, dtype=np.float32)[:, :, -1]
    rev = np.cumsum(prods[:, :, ::-1].astype(np.float32), axis=2, dtype=np.float32)[:, :, -1]
    assert np.array_equal(fwd.astype(np.float64), exact)
    assert np.array_equal(rev.astype(np.float64), exact)
    assert np.array_equal(orc.gemm_bf16(_bits(B["h"]), _bits(B["w_router"])), exact)
