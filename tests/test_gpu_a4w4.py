"""GPU parity of the A4W4 stage 1 (MXFP4 activations) against the oracle.

- moe_quant_mxfp4: packed E2M1 codes and E8M0 scales bit-exact, both scale
  layouts, dense and scattered to the k grouped rows, special values.
- moe_grouped_gemm_w13_glu_a4w4: requantised h within one E4M3 step of the
  oracle's (same bar as the MXFP8 stage 1), both h-scale layouts, ragged
  groups, padding rows untouched.
- moe_forward_a4w4: every output on small shapes through both stage-2
  families, and sampled tokens of full-size workloads, within
  |gpu - oracle| <= 2e-2 * rms(oracle row) + 1e-3.
"""
import numpy as np
import pytest
import torch

from mxfp4_latent_moe_gb300 import synth
from mxfp4_latent_moe_gb300.layer import MoeLayer
from tests import gpu_util as gu
from tests.test_gpu_gemm import _boxed, _check_mxfp8_rows, _dev, _groups, _prepacked

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def abi():
    return gu.cuda_lib()


def _quant4_gpu(abi, x_bf16, slot_to_row=None, k=0, rows_capacity=None, layout=0):
    T, d = x_bf16.shape
    rc = rows_capacity or (T + 127) // 128 * 128
    codes = torch.zeros(rc, d // 2, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(abi.moe_activation_scale_bytes(rc, d, layout), dtype=torch.uint8,
                         device="cuda")
    s2r = None if slot_to_row is None else torch.from_numpy(slot_to_row).cuda()
    abi.moe_quant_mxfp4(x_bf16.cuda(), T, d, s2r, k, codes, scales, rc, layout)
    torch.cuda.synchronize()
    sc = scales.cpu().numpy()
    return codes.cpu().numpy(), (gu.untile_g32(sc, rc, d) if layout else gu.untile(sc, rc, d))


def _special_rows(d):
    rng = np.random.default_rng(5)
    rows = np.zeros((9, d), np.float32)
    rows[1] = -0.0                                                    # signed zeros
    rows[2] = rng.normal(0, 1, d) * 2.0 ** -130                       # bf16 subnormals
    rows[3] = rng.normal(0, 1, d) * 1e37                              # near the top of bf16
    rows[4, ::32] = 7.5                                               # saturates to 6
    rows[4, 1::32] = 0.25                                             # tie -> 0
    rows[4, 2::32] = -0.75                                            # tie -> -1
    rows[4, 3::32] = 2.5                                              # tie -> 2
    rows[4, 4::32] = 5.0                                              # tie -> 4
    rows[5] = rng.normal(0, 1, d)
    rows[5, 7::32] = -0.0
    rows[6] = rng.standard_cauchy(d)                                  # heavy tails
    rows[7] = rng.normal(0, 1, d) * 64.0                              # outlier rows
    rows[8] = np.round(rng.normal(0, 2, d) * 4) / 4                   # many exact midpoints
    return torch.from_numpy(rows).to(torch.bfloat16)


@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("T,d", [(300, 3584), (8, 256), (1, 128),
                                 (1000, 3584), (1500, 2048)])   # the last two: 16 inputs a thread
def test_quant_mxfp4_dense_bit_exact(abi, orc, T, d, layout):
    x = torch.randn(T, d, generator=torch.Generator().manual_seed(T)).to(torch.bfloat16)
    codes, scales = _quant4_gpu(abi, x, layout=layout)
    rc, rs = orc.mxfp4_quant_rows_bf16(synth.bf16_bits(x))
    assert np.array_equal(scales[:T], rs)
    assert np.array_equal(codes[:T], rc)


def test_quant_mxfp4_special_values_bit_exact(abi, orc):
    x = _special_rows(512)
    codes, scales = _quant4_gpu(abi, x)
    rc, rs = orc.mxfp4_quant_rows_bf16(synth.bf16_bits(x))
    assert np.array_equal(scales[:9], rs)
    assert np.array_equal(codes[:9], rc)
    assert np.all(codes[1] == 0x88) and np.all(scales[0] == 0)


def test_quant_mxfp4_special_values_large_batch_bit_exact(abi, orc):
    x = _special_rows(4096).repeat(80, 1)    # 720 rows x 4096: 16 inputs a thread
    codes, scales = _quant4_gpu(abi, x)
    rc, rs = orc.mxfp4_quant_rows_bf16(synth.bf16_bits(x))
    assert np.array_equal(scales[:720], rs)
    assert np.array_equal(codes[:720], rc)


@pytest.mark.parametrize("pad,layout", [(128, 0), (32, 1)])
def test_quant_mxfp4_scattered_to_grouped_rows(abi, orc, pad, layout):
    T, d, E, k = 700, 3584, 896, 16
    rng = np.random.default_rng(8)
    ids, _ = orc.route_topk(rng.normal(0, 1, (T, E)).astype(np.float32), k)
    perm = orc.permute(ids, E, pad)
    rc = abi.moe_rows_capacity(T, E, k, pad)
    x = torch.randn(T, d, generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    codes, scales = _quant4_gpu(abi, x, perm["slot_to_row"], k, rc, layout)
    ref_c, ref_s = orc.mxfp4_quant_rows_bf16(synth.bf16_bits(x))
    rows = perm["slot_to_row"].reshape(T, k)
    for j in range(k):
        assert np.array_equal(codes[rows[:, j]], ref_c)
        assert np.array_equal(scales[rows[:, j]], ref_s)


CASES = [
    ([0, 1, 15, 16, 17, 127, 128, 129, 300], 256, 256),
    ([3, 0, 250, 130, 33, 64, 96, 65], 512, 384),
    (list(np.random.default_rng(0).integers(0, 300, 40)), 256, 512),
    # CTA pairs of m-tiles (even counts, and odd ones of at least 8, with 1-
    # and 20-row last tiles) beside single-CTA experts (7 m-tiles)
    ([1100, 0, 1024, 896, 897, 129, 1300], 256, 256),
    # every expert with an even m-tile count: all CTA pairs, no single-CTA work
    ([256, 200, 512, 129, 0], 256, 256),
]


@pytest.mark.parametrize("hs_layout", [0, 1])
@pytest.mark.parametrize("sizes,d,I", CASES)
def test_w13_glu_a4w4_matches_oracle_stage1(abi, orc, sizes, d, I, hs_layout):
    counts, offsets, rows, rc = _groups(sizes, 1)              # token tiles: groups of 128
    E = len(sizes)
    W = synth.make_weights(synth.shape("g", T=1, d=d, E=E, k=1, I=I), seed=1)
    g = torch.Generator().manual_seed(2)
    xq = torch.randint(0, 256, (rc, d // 2), generator=g, dtype=torch.uint8).numpy()  # E2M1 pairs
    xs = synth.random_scale_codes((rc, d // 32), lo=118, hi=130, seed=3).numpy()
    hq = torch.full((rc, I), 0x5A, dtype=torch.uint8, device="cuda")
    hs = torch.full((abi.moe_activation_scale_bytes(rc, I, hs_layout),), 0x5A, dtype=torch.uint8,
                    device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    abi.moe_grouped_gemm_w13_glu_a4w4(_dev(xq), _dev(gu.tile(xs, d)), _dev(counts), _dev(offsets),
                                      E, d, I, hs_layout,
                                      _boxed(abi, W["w13"].numpy(), E * 2 * I, d),
                                      _prepacked(abi, W["w13_s"].numpy(), E * 2 * I, d),
                                      hq, hs, rc, ws)
    assert abi.moe_check_device_status(ws) == 0
    got_c = hq.cpu().numpy()
    hsh = hs.cpu().numpy()
    got_s = gu.untile_g32(hsh, rc, I) if hs_layout else gu.untile(hsh, rc, I)
    w13, w13s = W["w13"].numpy(), W["w13_s"].numpy()
    idx = [r for _, r in rows]
    ref = np.stack([orc.expert_stage1_a4(xq[r], xs[r], w13[e], w13s[e]) for e, r in rows])
    ref_c, ref_s = orc.mx_quant_rows(ref.astype(np.float32))
    _check_mxfp8_rows(got_c[idx], got_s[idx], ref_c, ref_s)
    pad_rows = np.setdiff1d(np.arange(rc), idx)      # never written
    assert np.all(got_c[pad_rows] == 0x5A) and np.all(got_s[pad_rows] == 0x5A)


def _run_a4w4(abi, wl, L, kernel=0):
    layer = MoeLayer(L["w13"], L["w13_s"], L["w2"], L["w2_s"], k=wl.k, kernel=kernel)
    ws = layer.workspace(wl.T)
    ids = torch.empty(wl.T, max(wl.k, 1), dtype=torch.int32, device="cuda")
    w = torch.empty(wl.T, max(wl.k, 1), dtype=torch.float32, device="cuda")
    y = layer.forward(L["x"], L["logits"], ws=ws, topk_ids=ids, topk_w=w, a4w4=True)
    assert abi.moe_check_device_status(ws) == 0
    return y, ids[:, : wl.k], w[:, : wl.k]


def _host_layer(L):
    return {n: L[n].cpu().numpy() for n in ("w13", "w13_s", "w2", "w2_s")}


@pytest.mark.parametrize("wl", [
    synth.workload("tiny"),
    synth.shape("ragged", T=200, d=512, E=40, k=6, I=384),
    synth.shape("skewed", T=300, d=256, E=64, k=8, I=256, skew=True),
    synth.shape("outliers", T=100, d=512, E=16, k=4, I=128, outlier_frac=0.05),
    synth.shape("one_expert", T=130, d=256, E=1, k=1, I=256),
    # the top-ranked experts hold 8 or more m-tiles (CTA pairs of m-tiles and
    # an odd last one on a single CTA)
    synth.shape("heavy_experts", T=1500, d=256, E=16, k=4, I=256, skew=True),
    # 4 or 5 m-tiles per expert: stage 1 mostly as CTA pairs of m-tiles
    synth.shape("even_mtiles", T=2048, d=256, E=8, k=2, I=256),
])
@pytest.mark.parametrize("kernel", [1, 2, 3])
def test_forward_a4w4_small_all_outputs(abi, orc, wl, kernel):
    if kernel == 3 and (wl.d % 256 or wl.I % 256):
        pytest.skip("pair tiles need d and I multiples of 256")
    L = synth.make_layer(wl, seed=0, device="cuda")
    y, ids, w = _run_a4w4(abi, wl, L, kernel)
    H = _host_layer(L)
    ref = orc.moe_forward(synth.bf16_bits(L["x"]), L["logits"].cpu().numpy(), wl.k, H["w13"],
                          H["w13_s"], H["w2"], H["w2_s"], want_y64=True, a4w4=True)
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    gu.assert_layer_close(gu.bf16_to_f64(y), ref["y64"])


@pytest.mark.parametrize("name", ["decode_t64", "prefill_skewed_t8192", "prefill_outlier_t32768",
                                  "uniform_t8192"])
def test_forward_a4w4_full_size_sampled(abi, orc, name):
    """Routing on every token; the output on 128 seeded tokens plus, at
    T = 32,768, every outlier token (rows scaled by 64). uniform_t8192: most
    experts hold 2 m-tiles, so stage 1 runs mostly as CTA pairs."""
    wl = (synth.full_dims(int(name[len("uniform_t"):])) if name.startswith("uniform_t")
          else synth.workload(name))
    L = synth.make_layer(wl, seed=0, device="cuda")
    y, ids, _ = _run_a4w4(abi, wl, L)
    logits = L["logits"].cpu().numpy()
    rids, _ = orc.route_topk(logits, wl.k)
    assert np.array_equal(ids.cpu().numpy(), rids)
    tok = set(np.random.default_rng(77).choice(wl.T, size=min(128, wl.T), replace=False).tolist())
    if wl.outlier_frac > 0:
        amax = L["x"].float().abs().amax(dim=1).cpu().numpy()
        out = np.nonzero(amax > 32.0)[0]    # N(0,1) rows stay far below; x64 rows far above
        assert len(out) == int(round(wl.outlier_frac * wl.T))
        tok |= set(out.tolist())
    tok = np.array(sorted(tok))
    H = _host_layer(L)
    ref = orc.moe_forward(synth.bf16_bits(L["x"][torch.from_numpy(tok).cuda()]), logits[tok],
                          wl.k, H["w13"], H["w13_s"], H["w2"], H["w2_s"], want_y64=True,
                          a4w4=True)
    gu.assert_layer_close(gu.bf16_to_f64(y[torch.from_numpy(tok).cuda()]), ref["y64"], name)
