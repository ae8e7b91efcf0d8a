"""GPU parity of the whole layer (moe_forward, the call bench.py times)
against the CPU oracle.

Small shapes: every output element. The five workloads at full size, in the
configuration the benchmark runs and through the other GEMM family:
routing bit-exact on every token, grouping bit-exact on every slot, MXFP8
codes and scales of x bit-exact on every grouped row, and the bf16 output
within |gpu - oracle| <= 2e-2 * rms(oracle row) + 1e-3 on every token of the
decode batches (64, 512) and on 512 seeded tokens plus every outlier token of
the prefill batches (8192, 32768).
"""
import numpy as np
import pytest
import torch

from mxfp4_latent_moe_gb300 import synth
from mxfp4_latent_moe_gb300.layer import MoeLayer
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def abi():
    return gu.cuda_lib()


def _run_forward(abi, wl, L, kernel=0):
    layer = MoeLayer(L["w13"], L["w13_s"], L["w2"], L["w2_s"], k=wl.k, kernel=kernel)
    ws = layer.workspace(wl.T)
    ids = torch.empty(wl.T, max(wl.k, 1), dtype=torch.int32, device="cuda")
    w = torch.empty(wl.T, max(wl.k, 1), dtype=torch.float32, device="cuda")
    y = layer.forward(L["x"], L["logits"], ws=ws, topk_ids=ids, topk_w=w)
    assert abi.moe_check_device_status(ws) == 0
    return y, ids[:, : wl.k], w[:, : wl.k]


def _host_layer(L):
    return {n: L[n].cpu().numpy() for n in ("w13", "w13_s", "w2", "w2_s")}


@pytest.mark.parametrize("wl", [
    synth.workload("tiny"),
    synth.shape("ragged", T=200, d=512, E=40, k=6, I=384),
    synth.shape("skewed", T=300, d=256, E=64, k=8, I=256, skew=True),
    synth.shape("outliers", T=100, d=384, E=16, k=4, I=128, outlier_frac=0.05),
    synth.shape("one_expert", T=130, d=256, E=1, k=1, I=256),
    synth.shape("all_experts", T=20, d=128, E=8, k=8, I=128),
    # the top-ranked experts hold 8 or more m-tiles (CTA pairs of m-tiles and
    # an odd last one on a single CTA)
    synth.shape("heavy_experts", T=1500, d=256, E=16, k=4, I=256, skew=True),
    # the largest expert count and top-k the library accepts
    synth.shape("max_e_max_k", T=64, d=128, E=1024, k=32, I=128),
    # about 512 tokens for each of 8 experts: 4 (or 5) m-tiles each, token
    # tiles mostly as CTA pairs
    synth.shape("even_mtiles", T=2048, d=256, E=8, k=2, I=256),
])
@pytest.mark.parametrize("kernel", [1, 2])
def test_forward_small_all_outputs(abi, orc, wl, kernel):
    L = synth.make_layer(wl, seed=0, device="cuda")
    y, ids, w = _run_forward(abi, wl, L, kernel)
    H = _host_layer(L)
    ref = orc.moe_forward(synth.bf16_bits(L["x"]), L["logits"].cpu().numpy(), wl.k, H["w13"],
                          H["w13_s"], H["w2"], H["w2_s"], want_y64=True)
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    np.testing.assert_allclose(w.cpu().numpy(), ref["w"], rtol=2e-6, atol=1e-7)
    gu.assert_layer_close(gu.bf16_to_f64(y), ref["y64"])


@pytest.mark.parametrize("wl", [
    synth.shape("pair_small", T=300, d=512, E=24, k=6, I=512),
    synth.shape("pair_skewed", T=700, d=256, E=16, k=4, I=256, skew=True),
    synth.shape("pair_one_expert", T=300, d=256, E=1, k=1, I=256),
    synth.shape("pair_outliers", T=200, d=256, E=8, k=8, I=512, outlier_frac=0.05),
])
def test_forward_pair_tiles_small_all_outputs(abi, orc, wl):
    """The CTA-pair family (weights on the M side of a 2-CTA MMA) on shapes
    whose experts hold several 128- and 256-token chunks and a ragged last
    chunk, every output element."""
    L = synth.make_layer(wl, seed=0, device="cuda")
    y, ids, w = _run_forward(abi, wl, L, abi.GEMM_PAIR_TILES)
    H = _host_layer(L)
    ref = orc.moe_forward(synth.bf16_bits(L["x"]), L["logits"].cpu().numpy(), wl.k, H["w13"],
                          H["w13_s"], H["w2"], H["w2_s"], want_y64=True)
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    gu.assert_layer_close(gu.bf16_to_f64(y), ref["y64"], wl.name)


def test_forward_k0_gives_zeros_and_t0_is_a_noop(abi):
    wl = synth.shape("k0", T=16, d=128, E=4, k=0, I=128)
    L = synth.make_layer(wl, seed=0, device="cuda")
    layer = MoeLayer(L["w13"], L["w13_s"], L["w2"], L["w2_s"], k=0)
    y = torch.full((16, 128), 3.0, dtype=torch.bfloat16, device="cuda")
    layer.forward(L["x"], L["logits"], y=y)
    torch.cuda.synchronize()
    assert not y.float().abs().sum().item()
    wl0 = synth.shape("t0", T=0, d=128, E=4, k=2, I=128)
    L0 = synth.make_layer(wl0, seed=0, device="cuda")
    layer0 = MoeLayer(L0["w13"], L0["w13_s"], L0["w2"], L0["w2_s"], k=2)
    layer0.forward(L0["x"], L0["logits"], y=torch.empty(0, 128, dtype=torch.bfloat16,
                                                        device="cuda"))
    torch.cuda.synchronize()


# One workload's device tensors and oracle results at a time: the tests of a
# workload (one per GEMM family) are adjacent and share them.
_CACHE = {}


def _workload_state(orc, name):
    if name in _CACHE:
        return _CACHE[name]
    _CACHE.clear()
    torch.cuda.empty_cache()
    wl = (synth.full_dims(int(name[len("uniform_t"):])) if name.startswith("uniform_t")
          else synth.workload(name))
    L = synth.make_layer(wl, seed=0, device="cuda")
    tok = _compared_tokens(wl, L)
    xb = synth.bf16_bits(L["x"])
    logits = L["logits"].cpu().numpy()
    H = _host_layer(L)
    ref = orc.moe_forward(xb[tok], logits[tok], wl.k, H["w13"], H["w13_s"], H["w2"], H["w2_s"],
                          want_y64=True)
    del H
    rids, rw = orc.route_topk(logits, wl.k)
    ref_c, ref_s = _quant_all_rows(orc, xb)             # every token's MXFP8 codes and scales
    _CACHE[name] = dict(wl=wl, L=L, tok=tok, y64=ref["y64"], rids=rids, rw=rw,
                        ref_c=torch.from_numpy(ref_c).cuda(), ref_s=torch.from_numpy(ref_s).cuda())
    return _CACHE[name]


def _quant_all_rows(orc, xb):
    """The oracle's MX rule on every row, in row chunks on the host's cores
    (the oracle call releases the interpreter lock)."""
    import concurrent.futures as cf
    import os
    parts = np.array_split(np.arange(xb.shape[0]), max(1, min(os.cpu_count() or 1, 32)))
    with cf.ThreadPoolExecutor(len(parts)) as ex:
        res = list(ex.map(lambda p: orc.mx_quant_rows_bf16(xb[p]), [p for p in parts if len(p)]))
    return np.concatenate([c for c, _ in res]), np.concatenate([s for _, s in res])


def _compared_tokens(wl, L):
    """Every token up to 512; above that 512 seeded tokens plus every outlier
    token (the rows the workload scaled by 64)."""
    if wl.T <= 512:
        return np.arange(wl.T)
    g = np.random.default_rng(1234)
    idx = set(g.choice(wl.T, size=512, replace=False).tolist())
    if wl.outlier_frac > 0:
        amax = L["x"].float().abs().amax(dim=1).cpu().numpy()
        out = np.nonzero(amax > 32.0)[0]    # N(0,1) rows stay far below; x64 rows far above
        assert len(out) == int(round(wl.outlier_frac * wl.T))
        idx |= set(out.tolist())
    return np.array(sorted(idx))


@pytest.mark.parametrize("name,kernel", [("decode_t64", 0), ("decode_t64", 1),
                                         ("decode_t512", 0), ("decode_t512", 1),
                                         ("decode_t512", 3),
                                         ("prefill_skewed_t8192", 0), ("prefill_skewed_t8192", 2),
                                         ("prefill_skewed_t8192", 1), ("prefill_skewed_t8192", 3),
                                         ("prefill_outlier_t32768", 0),
                                         ("prefill_outlier_t32768", 2),
                                         ("prefill_outlier_t32768", 1),
                                         ("prefill_outlier_t32768", 3),
                                         # uniform routing at the full dims, 2 m-tiles for
                                         # most experts: token tiles mostly as CTA pairs
                                         ("uniform_t8192", 0)])
def test_forward_full_size_workloads(abi, orc, name, kernel):
    """The benchmark's configuration (kernel family 0 = moe_default_kernel:
    weight tiles at decode, token tiles at prefill), and each workload through
    the other family too. Routing on every token, grouping on every slot and
    the MXFP8 codes and scales of x on every grouped row, all bit-exact, with
    the padding and scale layout the forward itself uses; the bf16 output on
    every token of the decode batches and on 512 seeded tokens plus every
    outlier token of the prefill batches."""
    st = _workload_state(orc, name)
    wl, L, tok = st["wl"], st["L"], st["tok"]
    y, ids, w = _run_forward(abi, wl, L, kernel)
    # routing: every token
    assert np.array_equal(ids.cpu().numpy(), st["rids"])
    np.testing.assert_allclose(w.cpu().numpy(), st["rw"], rtol=2e-6, atol=1e-7)
    # the forward's family, padding and scale layout
    family = kernel or abi.moe_default_kernel(wl.T, wl.E, wl.k)
    pad = 32 if family == abi.GEMM_WEIGHT_TILES else 128
    layout = abi.SCALES_GROUP32 if family == abi.GEMM_WEIGHT_TILES else abi.SCALES_TILED128
    # grouping: every slot, through the step entry point
    rc = abi.moe_rows_capacity(wl.T, wl.E, wl.k, pad)
    counts = torch.empty(wl.E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(wl.E + 1, dtype=torch.int32, device="cuda")
    s2r = torch.empty(wl.T * wl.k, dtype=torch.int32, device="cuda")
    r2s = torch.empty(rc, dtype=torch.int32, device="cuda")
    pws = torch.zeros(abi.moe_permute_workspace_size(wl.T, wl.E), dtype=torch.uint8, device="cuda")
    abi.moe_permute(ids.contiguous(), wl.T, wl.E, wl.k, pad, counts, offsets, s2r, r2s, rc, pws)
    assert abi.moe_check_device_status(pws) == 0
    rperm = orc.permute(st["rids"], wl.E, pad)
    assert np.array_equal(counts.cpu().numpy(), rperm["counts"])
    assert np.array_equal(offsets.cpu().numpy(), rperm["offsets"])
    assert np.array_equal(s2r.cpu().numpy(), rperm["slot_to_row"])
    n = int(rperm["offsets"][wl.E])
    r2s_h = r2s.cpu().numpy()
    assert np.array_equal(r2s_h[:n], rperm["row_to_slot"]) and (r2s_h[n:] == -1).all()
    # MXFP8 codes and scales of x: every grouped row, full width
    xq = torch.zeros(rc, wl.d, dtype=torch.uint8, device="cuda")
    xs = torch.zeros(abi.moe_activation_scale_bytes(rc, wl.d, layout), dtype=torch.uint8,
                     device="cuda")
    abi.moe_quant_mxfp8(L["x"], wl.T, wl.d, s2r, wl.k, xq, xs, rc, layout)
    torch.cuda.synchronize()
    rows = s2r.view(wl.T, wl.k).long()
    for j in range(wl.k):
        r = rows[:, j]
        assert torch.equal(xq[r], st["ref_c"]), "x codes, slot %d" % j
        assert torch.equal(xs[gu.scale_offsets(r, wl.d, layout)], st["ref_s"]), "x scales, slot %d" % j
    # the layer's output
    gu.assert_layer_close(gu.bf16_to_f64(y[torch.from_numpy(tok).cuda()]), st["y64"],
                          "%s (%d tokens)" % (name, len(tok)))


def test_zz_release_full_size_state():
    _CACHE.clear()
    torch.cuda.empty_cache()
