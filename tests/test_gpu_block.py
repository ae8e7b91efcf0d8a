"""GPU parity of the composed latent-MoE block (moe_block_forward) and of the
two-part-A BF16 GEMM it ends with (moe_gemm_bf16_cat), against the oracle.

The block's inputs sit on the power-of-two grid of synth.make_block, where
the router logits and the latent x are exact in fp32, so the GPU and the
oracle route every token alike; the output is held to the layer's bar
(|gpu - oracle| <= 2e-2 * rms(oracle row) + 1e-3 on top of the bf16 output's
own half ulp). The shared experts run on a second stream; the same call with
one stream must give the same bits.
"""
import numpy as np
import pytest
import torch

from mxfp4_latent_moe_gb300 import synth
from mxfp4_latent_moe_gb300.layer import MoeBlock
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def abi():
    return gu.cuda_lib()


def _bits(t):
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _absdot(a, b):
    A = np.abs(a.float().cpu().numpy().astype(np.float64))
    B = np.abs(b.float().cpu().numpy().astype(np.float64))
    return A @ B.T


@pytest.mark.parametrize("M,K1,K2,N,epi", [(64, 3584, 6144, 7168, 1),   # the block's, split K
                                           (300, 256, 128, 520, 1),
                                           (200, 128, 0, 256, 0),
                                           (129, 192, 64, 512, 2),
                                           (1000, 64, 448, 264, 1)])
def test_gemm_bf16_cat_matches_oracle(abi, orc, M, K1, K2, N, epi):
    g = torch.Generator().manual_seed(M + K1 + K2 + N)
    a1 = torch.randn(M, K1, generator=g).to(torch.bfloat16)
    a2 = torch.randn(M, max(K2, 1), generator=g).to(torch.bfloat16)[:, :K2].contiguous()
    b = (torch.randn(N, K1 + K2, generator=g) * 0.03).to(torch.bfloat16)
    n_out = N // 2 if epi == 2 else N
    c = torch.full((M, n_out), 7.0, dtype=torch.float32 if epi == 0 else torch.bfloat16,
                   device="cuda")
    ws = torch.zeros(abi.moe_gemm_bf16_workspace_size(M, N, K1 + K2, epi), dtype=torch.uint8,
                     device="cuda")
    abi.moe_gemm_bf16_cat(a1.cuda(), K1, a2.cuda() if K2 else None, K2, b.cuda(), M, N, epi, c,
                          ws)
    assert abi.moe_check_device_status(ws) == 0
    a = torch.cat([a1, a2], dim=1)
    got = c.float().cpu().numpy().astype(np.float64)
    if epi == 2:
        Nh = N // 2
        ref = orc.gemm_bf16_swiglu(_bits(a), _bits(b), threads=0)
        G = orc.gemm_bf16(_bits(a), _bits(b[:Nh]), threads=0)
        U = orc.gemm_bf16(_bits(a), _bits(b[Nh:]), threads=0)
        s = 1.0 / (1.0 + np.exp(-G))
        dsilu = np.abs(s * (1 + G * (1 - s)))
        bound = (2.0 ** -8 * np.abs(ref) + dsilu * np.abs(U) * 1e-5 * _absdot(a, b[:Nh])
                 + np.abs(G * s) * 1e-5 * _absdot(a, b[Nh:]) + 1e-6 * (np.abs(ref).max() + 1e-30))
    else:
        ref = orc.gemm_bf16(_bits(a), _bits(b), threads=0)
        bound = 1e-5 * _absdot(a, b) + 1e-30
        if epi == 1:
            bound += 2.0 ** -8 * np.abs(ref)
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) / bound))


def _make(bw, device="cuda"):
    B = synth.make_block(bw, seed=0, device=device)
    blk = MoeBlock(B["w_down"], B["w_router"], B["w_shared13"], B["w_out"], B["w13"], B["w13_s"],
                   B["w2"], B["w2_s"], k=bw.k)
    return B, blk


def _oracle(orc, bw, B, tok):
    W = {n: B[n].cpu().numpy() for n in ("w13", "w13_s", "w2", "w2_s")}
    return orc.block_forward(_bits(B["h"][tok]), bw.k, _bits(B["w_down"]), _bits(B["w_router"]),
                             _bits(B["w_shared13"]), _bits(B["w_out"]), W["w13"], W["w13_s"],
                             W["w2"], W["w2_s"], threads=0)


def _run(abi, blk, h, two_streams):
    ws = blk.workspace(h.shape[0])
    side = torch.cuda.Stream() if two_streams else None
    out = blk.forward(h, ws=ws, shared_stream=side)
    assert abi.moe_check_device_status(ws) == 0
    return out


@pytest.mark.parametrize("bw", [
    synth.block_shape("small", T=40, hidden=256, d=128, E=16, k=4, I=128, shared_I=128),
    synth.block_shape("ragged", T=300, hidden=512, d=256, E=40, k=6, I=384, shared_I=256),
    synth.block_shape("one_token", T=1, hidden=192, d=128, E=8, k=2, I=128, shared_I=384),
])
def test_block_small_all_outputs(abi, orc, bw):
    B, blk = _make(bw)
    out2 = _run(abi, blk, B["h"], True)
    out1 = _run(abi, blk, B["h"], False)
    assert torch.equal(out1, out2)          # one stream or two: the same bits
    ref = _oracle(orc, bw, B, slice(None))
    gu.assert_layer_close(gu.bf16_to_f64(out2), ref["y64"], bw.name)


@pytest.mark.parametrize("name", ["block_decode_t64", "block_prefill_t8192"])
def test_block_full_size(abi, orc, name):
    """Every token of the decode batch; 512 seeded tokens of the prefill batch."""
    bw = synth.block_workload(name)
    B, blk = _make(bw)
    out = _run(abi, blk, B["h"], True)
    if bw.T <= 512:
        tok = np.arange(bw.T)
    else:
        tok = np.sort(np.random.default_rng(99).choice(bw.T, size=512, replace=False))
    ref = _oracle(orc, bw, B, torch.from_numpy(tok).cuda())
    gu.assert_layer_close(gu.bf16_to_f64(out[torch.from_numpy(tok).cuda()]), ref["y64"], name)
    out1 = _run(abi, blk, B["h"], False)
    assert torch.equal(out, out1)


def test_block_graph_capture_replays_both_streams(abi):
    """The block captured as one CUDA graph (the side stream forks from and
    joins the capturing stream) replays to the eager result."""
    bw = synth.block_shape("graph", T=64, hidden=512, d=256, E=32, k=4, I=256, shared_I=256)
    B, blk = _make(bw)
    ws = blk.workspace(bw.T)
    side = torch.cuda.Stream()
    ref = blk.forward(B["h"], ws=ws, shared_stream=side).clone()   # first call: events made
    torch.cuda.synchronize()
    out = torch.empty_like(ref)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        blk.forward(B["h"], ws=ws, out=out, shared_stream=side)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    assert abi.moe_check_device_status(ws) == 0
