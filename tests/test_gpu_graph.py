"""The layer step captured as one CUDA graph (MoeLayer.capture): replays on
refilled input buffers give bit-for-bit the eager moe_forward /
moe_forward_a4w4 results (every kernel of the step is deterministic), for
both GEMM families (token tiles also with CTA pairs of m-tiles), with the
device status clean after each replay."""
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
    # 4-5 m-tiles per expert: token tiles mostly as CTA pairs of m-tiles
    (synth.shape("even_mtiles", T=2048, d=256, E=8, k=2, I=256), 1),
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


def test_host_pipeline_matches_forward(abi):
    """Batches through HostPipeline (copies on their own streams, two device
    buffer sets rotating) give bit-identical outputs to eager forwards, in
    order, for more batches than buffer sets."""
    from mxfp4_latent_moe_gb300.layer import HostPipeline
    wl = synth.shape("pipe", T=24, d=256, E=16, k=4, I=256)
    L = synth.make_layer(wl, seed=5, device="cuda")
    layer = MoeLayer(L["w13"], L["w13_s"], L["w2"], L["w2_s"], k=wl.k)
    n = 5
    xs = [synth.make_activations(wl, seed=100 + i) for i in range(n)]
    want = [layer.forward(x.cuda(), lg.cuda()).cpu() for x, lg in xs]
    pipe = HostPipeline(layer, wl.T)
    outs = [torch.empty(wl.T, wl.d, dtype=torch.bfloat16).pin_memory() for _ in range(n)]
    for (x, lg), y_h in zip(xs, outs):
        pipe.submit(x.pin_memory(), lg.pin_memory(), y_h)
    pipe.synchronize()
    assert abi.moe_check_device_status(pipe.ws) == 0
    for got, ref in zip(outs, want):
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("name,n,a4w4", [("decode_t64", 60, False), ("decode_t64", 30, True),
                                         ("prefill_skewed_t8192", 10, False),
                                         ("uniform_t2048", 20, False),    # 64-token chunks
                                         ("uniform_t12288", 10, False)])  # all CTA pairs
def test_repeated_forwards_bit_identical(abi, name, n, a4w4):
    """Back-to-back forwards, eager and replayed as a graph, give the first
    forward's output bit for bit. Consecutive kernels overlap through
    programmatic dependent launch; a missing wait would show up here as a
    difference between repetitions."""
    wl = (synth.full_dims(int(name[len("uniform_t"):])) if name.startswith("uniform_t")
          else synth.workload(name))
    L = synth.make_layer(wl, seed=3, device="cuda")
    layer = MoeLayer(L["w13"], L["w13_s"], L["w2"], L["w2_s"], k=wl.k)
    ws = layer.workspace(wl.T)
    ref = layer.forward(L["x"], L["logits"], ws=ws, a4w4=a4w4).clone()
    y = torch.empty_like(ref)
    diffs = 0
    for _ in range(n):
        layer.forward(L["x"], L["logits"], ws=ws, y=y, a4w4=a4w4)
        diffs += int(not torch.equal(y.view(torch.int16), ref.view(torch.int16)))
    graph, yg, wsg = layer.capture(L["x"], L["logits"], a4w4=a4w4)
    for _ in range(n):
        graph.replay()
        diffs += int(not torch.equal(yg.view(torch.int16), ref.view(torch.int16)))
    assert diffs == 0
    assert abi.moe_check_device_status(ws) == 0 and abi.moe_check_device_status(wsg) == 0
