"""The layer step captured as one CUDA graph (MoeLayer.capture): replays on
refilled input buffers give bit-for-bit the eager moe_forward /
moe_forward_a4w4 results (every kernel of the step is deterministic), for
both GEMM families, with the device status clean after each replay."""
import pytest
import torch

from mxfp4_latent_moe_gb300 import synth
from mxfp4_latent_moe_gb300.layer import MoeLayer
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def abi():
    return gu.cuda_lib()


@pytest.mark.parametrize("a4w4", [False, True])
@pytest.mark.parametrize("wl,kernel", [
    (synth.shape("small", T=40, d=512, E=24, k=4, I=384), 0),
    (synth.shape("small", T=40, d=512, E=24, k=4, I=384), 1),
    (synth.workload("decode_t64"), 0),
])
def test_graph_replay_matches_eager(abi, wl, kernel, a4w4):
    L = synth.make_layer(wl, seed=0, device="cuda")
    layer = MoeLayer(L["w13"], L["w13_s"], L["w2"], L["w2_s"], k=wl.k, kernel=kernel)
    x = L["x"].clone()
    logits = L["logits"].clone()
    ids = torch.empty(wl.T, wl.k, dtype=torch.int32, device="cuda")
    graph, y, ws = layer.capture(x, logits, topk_ids=ids, a4w4=a4w4)
    g = torch.Generator(device="cuda").manual_seed(5)
    for step in range(3):
        xn = torch.randn(wl.T, wl.d, generator=g, device="cuda").to(torch.bfloat16)
        ln = torch.randn(wl.T, wl.E, generator=g, device="cuda")
        x.copy_(xn)
        logits.copy_(ln)
        graph.replay()
        torch.cuda.synchronize()
        assert abi.moe_check_device_status(ws) == abi.OK
        got, got_ids = y.clone(), ids.clone()
        ref = layer.forward(xn, ln, a4w4=a4w4)
        ref_ids = torch.empty_like(ids)
        layer.forward(xn, ln, topk_ids=ref_ids, a4w4=a4w4)
        torch.cuda.synchronize()
        assert torch.equal(got_ids, ref_ids)
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), step
