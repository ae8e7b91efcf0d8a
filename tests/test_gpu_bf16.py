"""GPU parity of the dense BF16 steps (moe_gemm_bf16, moe_router_logits)
against the oracle's fp64 products.

Bars (fp32 accumulation of bf16 products, then the output rounding):
  fp32 out:  |gpu - ref| <= 1e-5 * sum_k |a_k b_k| + 1e-30
  bf16 out:  |gpu - ref| <= 2^-8 * |ref| + 1e-5 * sum_k |a_k b_k| + 1e-30
Shapes cover ragged M and N tails, several raster groups, K from one stage
to many, calls that split K over the SMs (few tiles) and calls that do not,
the router at the layer's sizes, and the SwiGLU epilogue.
"""
import numpy as np
import pytest
import torch
from scipy.special import expit

from mxfp4_latent_moe_gb300 import synth
from tests import gpu_util as gu
from tests import mx_numpy as mx

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def abi():
    return gu.cuda_lib()


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _operands(M, N, K, seed, scale_b=0.05):
    g = torch.Generator().manual_seed(seed)
    a = torch.randn(M, K, generator=g).to(torch.bfloat16)
    b = (torch.randn(N, K, generator=g) * scale_b).to(torch.bfloat16)
    return a, b


def _absdot(a, b):
    A = np.abs(a.float().numpy().astype(np.float64))
    B = np.abs(b.float().numpy().astype(np.float64))
    return A @ B.T


@pytest.mark.parametrize("M,N,K", [(1, 8, 64), (200, 904, 192), (1100, 520, 128),
                                   (64, 896, 3584), (300, 256, 7168)])
@pytest.mark.parametrize("epi", [0, 1])
def test_gemm_bf16_matches_oracle(abi, orc, M, N, K, epi):
    a, b = _operands(M, N, K, seed=M + N + K)
    c = torch.full((M, N), 7.0, dtype=torch.float32 if epi == 0 else torch.bfloat16, device="cuda")
    ws = torch.zeros(abi.moe_gemm_bf16_workspace_size(M, N, K, epi), dtype=torch.uint8,
                     device="cuda")
    abi.moe_gemm_bf16(a.cuda(), b.cuda(), M, N, K, epi, c, ws)
    assert abi.moe_check_device_status(ws) == 0
    ref = orc.gemm_bf16(_bits(a), _bits(b))
    got = c.float().cpu().numpy().astype(np.float64)
    bound = 1e-5 * _absdot(a, b) + 1e-30
    if epi == 1:
        bound += 2.0 ** -8 * np.abs(ref)
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) / bound))


@pytest.mark.parametrize("M,Nh,K", [(130, 128, 256), (1000, 384, 192), (16, 3072, 7168)])
def test_gemm_bf16_swiglu_matches_oracle(abi, orc, M, Nh, K):
    a, b = _operands(M, 2 * Nh, K, seed=M + Nh, scale_b=0.02)
    h = torch.full((M, Nh), 7.0, dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(abi.moe_gemm_bf16_workspace_size(M, 2 * Nh, K, 2), dtype=torch.uint8,
                     device="cuda")
    abi.moe_gemm_bf16(a.cuda(), b.cuda(), M, 2 * Nh, K, 2, h, ws)
    assert abi.moe_check_device_status(ws) == 0
    ref = orc.gemm_bf16_swiglu(_bits(a), _bits(b))
    G = orc.gemm_bf16(_bits(a), _bits(b[:Nh]))
    U = orc.gemm_bf16(_bits(a), _bits(b[Nh:]))
    np.testing.assert_allclose(ref, G * expit(G) * U, rtol=1e-12, atol=1e-30)
    got = h.float().cpu().numpy().astype(np.float64)
    # perturbation of silu(g)*u by the fp32 sums of g and u, then bf16 rounding
    ag = 1e-5 * _absdot(a, b[:Nh])
    au = 1e-5 * _absdot(a, b[Nh:])
    dsilu = np.abs(expit(G) * (1 + G * (1 - expit(G))))
    bound = 2.0 ** -8 * np.abs(ref) + dsilu * np.abs(U) * ag + np.abs(G * expit(G)) * au + 1e-6 * (np.abs(ref).max() + 1e-30)
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) / bound))


@pytest.mark.parametrize("T", [64, 512])
def test_router_logits_feed_the_routing(abi, orc, T):
    """The router at the layer's sizes on the composed block's power-of-two
    input grid, where every fp32 sum is exact: the GPU logits equal the
    oracle's bit for bit, and routing them on the GPU gives the oracle's
    routing of its own logits."""
    d_in, E, k = 7168, 896, 16
    B = synth.make_block(synth.block_shape("router", T=T, hidden=d_in, d=128, E=E, k=k, I=128,
                                           shared_I=128), seed=T)
    x, w = B["h"], B["w_router"]
    logits = torch.empty(T, E, dtype=torch.float32, device="cuda")
    ws = torch.zeros(abi.moe_gemm_bf16_workspace_size(T, E, d_in, 0), dtype=torch.uint8,
                     device="cuda")
    abi.moe_router_logits(x.cuda(), w.cuda(), T, d_in, E, logits, ws)
    assert abi.moe_check_device_status(ws) == 0
    ref = orc.gemm_bf16(_bits(x), _bits(w), threads=0)
    got = logits.cpu().numpy().astype(np.float64)
    assert np.array_equal(got, ref)
    ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
    wts = torch.empty(T, k, dtype=torch.float32, device="cuda")
    abi.moe_route_topk(logits, T, E, k, ids, wts)
    rids, rw = orc.route_topk(ref.astype(np.float32), k)
    assert np.array_equal(ids.cpu().numpy(), rids)
    np.testing.assert_allclose(wts.cpu().numpy(), rw, rtol=2e-6, atol=1e-7)
