"""GPU parity of the two grouped GEMMs (tcgen05 block-scaled MMA) against the
oracle's per-expert stage functions, on ragged expert groups: empty groups,
groups of 1, 15..17, 127..129 and several hundred rows, K not a multiple of the
pipeline depth, and more tiles than SMs. All three kernel families: token
tiles (tokens on the MMA's M side, groups padded to 128, TILED activation
scales; experts with an even number of m-tiles or at least 8 as 2-CTA
pairs of m-tiles), weight tiles (weights on the M side, tokens as N = 32 or 64 per
tile by the groups' size, groups padded to 32, GROUP32 activation scales) and pair tiles (weights on the
M side of a 2-CTA MMA, tokens as N in chunks of 128 / 256 with a ragged last
chunk, groups padded to 128, TILED scales; d and I multiples of 256)."""
import numpy as np
import pytest
import torch

from mxfp4_latent_moe_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def abi():
    return gu.cuda_lib()


def _layout(kernel):
    return 1 if kernel == 2 else 0       # GROUP32 for weight tiles, else TILED


def _groups(sizes, kernel):
    pad = 32 if kernel == 2 else 128
    offsets = [0]
    for c in sizes:
        offsets.append(offsets[-1] + (c + pad - 1) // pad * pad)
    rows = [(e, offsets[e] + i) for e, c in enumerate(sizes) for i in range(c)]
    return (np.array(sizes, np.int32), np.array(offsets, np.int32), rows,
            max((offsets[-1] + 127) // 128 * 128, 128))


def _act_scales(canon, K, kernel):
    return gu.tile_g32(canon, K) if kernel == 2 else gu.tile(canon, K)


def _act_untile(buf, rows, K, kernel):
    return gu.untile_g32(buf, rows, K) if kernel == 2 else gu.untile(buf, rows, K)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _boxed(abi, codes, rows, K):
    dst = torch.empty(rows * K // 2, dtype=torch.uint8, device="cuda")
    abi.moe_prepack_weights(_dev(codes.reshape(rows, K // 2)), rows, K, dst)
    return dst


def _prepacked(abi, scales, rows, K):
    dst = torch.empty(abi.moe_tiled_scale_bytes(rows, K), dtype=torch.uint8, device="cuda")
    abi.moe_prepack_scales(_dev(scales.reshape(rows, K // 32)), rows, K, dst)
    return dst


def _check_mxfp8_rows(got_c, got_s, ref_c, ref_s):
    """Codes of a requantised fp32 result: GPU (fp32 sums) vs oracle (fp64 sums
    rounded to fp32). Codes may differ by one E4M3 step where the two sums
    straddle a rounding boundary; scales by one where amax straddles a power
    of two."""
    assert np.all(np.abs(got_s.astype(int) - ref_s.astype(int)) <= 1)
    assert (got_s != ref_s).mean() < 0.01
    g = gu.dequant_mxfp8(got_c, got_s)
    r = gu.dequant_mxfp8(ref_c, ref_s)
    X = np.repeat(np.ldexp(1.0, np.maximum(got_s, ref_s).astype(int) - 127), 32, axis=-1)
    step = np.maximum(np.abs(g), np.abs(r)) * 2.0 ** -3 + X * 2.0 ** -9
    assert np.all(np.abs(g - r) <= step * 1.0001)
    assert (got_c != ref_c).mean() < 0.01
    rel = np.linalg.norm(g - r, axis=-1) / (np.linalg.norm(r, axis=-1) + 1e-300)
    assert rel.max() < 0.02


CASES = [
    # few tokens per expert: weight tiles in 32-token chunks (the larger
    # groups below take 64-token chunks)
    ([1, 0, 5, 31, 32, 33, 2, 17], 256, 384),
    ([0, 1, 15, 16, 17, 127, 128, 129, 300], 256, 256),
    ([3, 0, 250, 130, 33, 64, 96, 65], 384, 384),
    (list(np.random.default_rng(0).integers(0, 300, 40)), 256, 512),
    # several token chunks per expert for the pair tiles (128 / 256 wide)
    ([0, 255, 256, 257, 1, 600, 383, 384, 31], 512, 512),
    # token tiles: experts with an even number of m-tiles of 128 rows, or at
    # least 8, run their full pairs of m-tiles over CTA pairs, the rest one
    # CTA per m-tile: 9 m-tiles (odd, the last with 76 rows), 8 (even, full),
    # 7 (odd, below 8: single CTAs), 8 with a 1-row last tile, 2 with a
    # 1-row last tile, 11 with a 20-row last tile
    ([1100, 0, 1024, 896, 897, 129, 1300], 256, 256),
    # every expert with an even m-tile count: all CTA pairs, no single-CTA work
    ([256, 200, 512, 129, 0], 256, 256),
]


def _supported(kernel, d, I):
    if kernel == 3 and (d % 256 or I % 256):
        pytest.skip("pair tiles need d and I multiples of 256")


@pytest.mark.parametrize("out_off", [0, 16])   # bytes: 32-byte-aligned output, or 16 only
@pytest.mark.parametrize("kernel", [1, 2, 3])
@pytest.mark.parametrize("sizes,d,I", CASES)
def test_w13_glu_matches_oracle_stage1(abi, orc, sizes, d, I, kernel, out_off):
    _supported(kernel, d, I)
    counts, offsets, rows, rc = _groups(sizes, kernel)
    E = len(sizes)
    W = synth.make_weights(synth.shape("g", T=1, d=d, E=E, k=1, I=I), seed=1)
    xq = synth.random_e4m3_codes((rc, d), seed=2).numpy()
    xs = synth.random_scale_codes((rc, d // 32), lo=118, hi=130, seed=3).numpy()
    hq = torch.full((rc * I + out_off,), 0x5A, dtype=torch.uint8, device="cuda")[out_off:]
    hq = hq.view(rc, I)
    hs = torch.full((abi.moe_activation_scale_bytes(rc, I, _layout(kernel)),), 0x5A,
                    dtype=torch.uint8, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    abi.moe_grouped_gemm_w13_glu(_dev(xq), _dev(_act_scales(xs, d, kernel)), _dev(counts),
                                 _dev(offsets), E, d,
                                 I, kernel,
                                 _boxed(abi, W["w13"].numpy(), E * 2 * I, d),
                                 _prepacked(abi, W["w13_s"].numpy(), E * 2 * I, d),
                                 hq, hs, rc, ws)
    assert abi.moe_check_device_status(ws) == 0
    got_c = hq.cpu().numpy()
    got_s = _act_untile(hs.cpu().numpy(), rc, I, kernel)
    w13, w13s = W["w13"].numpy(), W["w13_s"].numpy()
    idx = [r for _, r in rows]
    ref = np.stack([orc.expert_stage1(xq[r], xs[r], w13[e], w13s[e]) for e, r in rows])
    ref_c, ref_s = orc.mx_quant_rows(ref.astype(np.float32))
    _check_mxfp8_rows(got_c[idx], got_s[idx], ref_c, ref_s)
    pad_rows = np.setdiff1d(np.arange(rc), idx)      # never written
    assert np.all(got_c[pad_rows] == 0x5A) and np.all(got_s[pad_rows] == 0x5A)


@pytest.mark.parametrize("out_off", [0, 16])   # bytes: 32-byte-aligned output, or 16 only
@pytest.mark.parametrize("kernel", [1, 2, 3])
@pytest.mark.parametrize("sizes,d,I", CASES)
def test_w2_matches_oracle_stage2(abi, orc, sizes, d, I, kernel, out_off):
    _supported(kernel, d, I)
    counts, offsets, rows, rc = _groups(sizes, kernel)
    E = len(sizes)
    W = synth.make_weights(synth.shape("g", T=1, d=d, E=E, k=1, I=I), seed=4)
    hq = synth.random_e4m3_codes((rc, I), seed=5).numpy()
    hs = synth.random_scale_codes((rc, I // 32), lo=118, hi=130, seed=6).numpy()
    yp = torch.full((rc * d + out_off // 2,), 7.0, dtype=torch.bfloat16, device="cuda")
    yp = yp[out_off // 2:].view(rc, d)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    abi.moe_grouped_gemm_w2(_dev(hq), _dev(_act_scales(hs, I, kernel)), _dev(counts),
                            _dev(offsets), E, I, d,
                            kernel,
                            _boxed(abi, W["w2"].numpy(), E * d, I),
                            _prepacked(abi, W["w2_s"].numpy(), E * d, I), yp, rc,
                            ws)
    assert abi.moe_check_device_status(ws) == 0
    got = gu.bf16_to_f64(yp)
    w2, w2s = W["w2"].numpy(), W["w2_s"].numpy()
    idx = [r for _, r in rows]
    ref = np.stack([orc.expert_stage2(hq[r], hs[r], w2[e], w2s[e]) for e, r in rows])
    rms = np.sqrt((ref ** 2).mean(axis=1, keepdims=True))
    err = np.abs(got[idx] - ref)
    assert np.all(err <= np.abs(ref) * 2.0 ** -8 + 1e-5 * rms), float((err / (rms + 1e-30)).max())
    pad_rows = np.setdiff1d(np.arange(rc), idx)      # never written
    assert np.all(got[pad_rows] == 7.0)


def test_gemm_refuses_bad_groups(abi):
    d = I = 256
    W = synth.make_weights(synth.shape("g", T=1, d=d, E=2, k=1, I=I), seed=1)
    rc = 256
    xq = torch.zeros(rc, d, dtype=torch.uint8, device="cuda")
    xs = torch.zeros(abi.moe_tiled_scale_bytes(rc, d), dtype=torch.uint8, device="cuda")
    hq = torch.full((rc, I), 0x5A, dtype=torch.uint8, device="cuda")
    hs = torch.zeros(abi.moe_tiled_scale_bytes(rc, I), dtype=torch.uint8, device="cuda")
    w13_sf = _prepacked(abi, W["w13_s"].numpy(), 2 * 2 * I, d)
    w13_boxed = _boxed(abi, W["w13"].numpy(), 2 * 2 * I, d)
    bad = [(np.array([48, 48], np.int32), np.array([0, 48, 96], np.int32)),     # not padded
           (np.array([130, 0], np.int32), np.array([0, 128, 256], np.int32)),   # count > group
           (np.array([1, 1], np.int32), np.array([0, 128, 384], np.int32))]     # past the capacity
    for counts, offsets in bad:
        for kernel in (1, 2, 3):
            ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
            abi.moe_grouped_gemm_w13_glu(xq, xs, _dev(counts), _dev(offsets), 2, d, I, kernel,
                                         w13_boxed, w13_sf, hq, hs, rc, ws)
            assert abi.moe_check_device_status(ws) == 6       # MOE_ERR_DEVICE_BAD_INPUT
    assert bool((hq == 0x5A).all())                           # nothing written


def test_pair_tiles_refuse_widths_not_multiples_of_256(abi):
    d, I, E, rc = 384, 256, 2, 256
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    z = lambda n: torch.zeros(n, dtype=torch.uint8, device="cuda")
    counts = torch.zeros(E, dtype=torch.int32, device="cuda")
    offsets = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
    with pytest.raises(abi.MoeError) as err:
        abi.moe_grouped_gemm_w13_glu(z(rc * d), z(abi.moe_tiled_scale_bytes(rc, d)), counts,
                                     offsets, E, d, I, 3, z(E * 2 * I * d // 2),
                                     z(abi.moe_tiled_scale_bytes(E * 2 * I, d)), z(rc * I),
                                     z(abi.moe_tiled_scale_bytes(rc, I)), rc, ws)
    assert err.value.code == abi.UNSUPPORTED
