"""GPU parity of the SIMT steps of the layer against the CPU oracle, through
the C-ABI: routing and grouping bit-exact, MXFP8 codes and scales bit-exact,
the combine within bf16 rounding; plus the scale prepack and the device
status word (bounded-wait self-test)."""
import numpy as np
import pytest
import torch

from mxfp4_latent_moe_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def abi():
    return gu.cuda_lib()


def _route_gpu(abi, logits, k):
    T, E = logits.shape
    lg = torch.from_numpy(logits).cuda()
    ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    abi.moe_route_topk(lg, T, E, k, ids, w)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("T,E,k", [(64, 896, 16), (1000, 896, 16), (37, 32, 4), (5, 33, 5),
                                   (3, 1024, 32), (4, 1, 1), (9, 16, 16), (300, 200, 7)])
def test_route_bit_exact(abi, orc, T, E, k):
    rng = np.random.default_rng(T + E)
    logits = rng.normal(0, 1, (T, E)).astype(np.float32)
    ids, w = _route_gpu(abi, logits, k)
    rids, rw = orc.route_topk(logits, k)
    assert np.array_equal(ids, rids)
    np.testing.assert_allclose(w, rw, rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("lane_of_top", [0, 5, 31])
def test_route_top_experts_in_one_lane(abi, orc, lane_of_top):
    """All of the largest logits on experts e = lane (mod 32): the lane that
    holds them gives up every pick, so it rescans its values many times."""
    rng = np.random.default_rng(lane_of_top)
    T, E, k = 96, 896, 16
    logits = rng.normal(0, 1, (T, E)).astype(np.float32)
    logits[:, lane_of_top::32] += 10.0
    logits[::4, lane_of_top::64] = 20.0                        # ties inside that lane too
    ids, w = _route_gpu(abi, logits, k)
    rids, rw = orc.route_topk(logits, k)
    assert np.array_equal(ids, rids)
    np.testing.assert_allclose(w, rw, rtol=2e-6, atol=1e-7)


def test_route_ties_signed_zero_and_saturation(abi, orc):
    rng = np.random.default_rng(11)
    T, E, k = 512, 896, 16
    logits = np.round(rng.normal(0, 1, (T, E)) * 4) / 4          # many exact ties
    logits[::3, ::2] = 0.0
    logits[1::3, 1::2] = -0.0
    logits[2::7] = np.where(rng.random((len(logits[2::7]), E)) < 0.5, 30.0, -30.0)
    logits = logits.astype(np.float32)
    ids, w = _route_gpu(abi, logits, k)
    rids, rw = orc.route_topk(logits, k)
    assert np.array_equal(ids, rids)
    np.testing.assert_allclose(w, rw, rtol=2e-6, atol=1e-7)


def _permute_gpu(abi, ids, E, pad_m, rows_capacity=None):
    T, k = ids.shape
    rc = rows_capacity or max(abi.moe_rows_capacity(T, E, k, pad_m), 128)
    d_ids = torch.from_numpy(ids).cuda()
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    s2r = torch.empty(max(T * k, 1), dtype=torch.int32, device="cuda")
    r2s = torch.full((rc,), -7, dtype=torch.int32, device="cuda")
    ws = torch.zeros(abi.moe_permute_workspace_size(T, E), dtype=torch.uint8, device="cuda")
    abi.moe_permute(d_ids, T, E, k, pad_m, counts, offsets, s2r, r2s, rc, ws)
    status = abi.moe_check_device_status(ws)
    return dict(counts=counts.cpu().numpy(), offsets=offsets.cpu().numpy(),
                slot_to_row=s2r.cpu().numpy()[: T * k], row_to_slot=r2s.cpu().numpy(),
                status=status)


@pytest.mark.parametrize("pad_m", [1, 16, 128])
@pytest.mark.parametrize("T,E,k", [(1000, 896, 16), (64, 896, 16), (513, 64, 8), (1, 5, 2),
                                   (256, 1024, 32), (257, 896, 16)])
def test_permute_bit_exact(abi, orc, T, E, k, pad_m):
    rng = np.random.default_rng(T * 7 + pad_m)
    ids, _ = orc.route_topk(rng.normal(0, 1, (T, E)).astype(np.float32), k)
    got = _permute_gpu(abi, ids, E, pad_m)
    ref = orc.permute(ids, E, pad_m)
    assert got["status"] == 0
    for key in ("counts", "offsets", "slot_to_row"):
        assert np.array_equal(got[key], ref[key]), key
    n = int(ref["offsets"][-1])
    assert np.array_equal(got["row_to_slot"][:n], ref["row_to_slot"])
    assert np.all(got["row_to_slot"][n:] == -1)            # rows past the groups hold no slot


def test_permute_one_hot_expert_and_empty_experts(abi, orc):
    T, E, k = 2000, 896, 4
    rng = np.random.default_rng(3)
    ids = np.stack([np.concatenate([[7], 100 + rng.permutation(20)[: k - 1]]) for _ in range(T)])
    ids = ids.astype(np.int32)
    got = _permute_gpu(abi, ids, E, 128)
    ref = orc.permute(ids, E, 128)
    for key in ("counts", "offsets", "slot_to_row"):
        assert np.array_equal(got[key], ref[key]), key
    assert got["counts"][7] == T and (got["counts"] > 0).sum() == 21


@pytest.mark.parametrize("noalloc", [False, True])
def test_permute_back_to_back_calls_on_shared_buffers(abi, orc, noalloc):
    """One-block grouping calls (T <= 256) enqueued back to back on the same
    output buffers, a large batch then a small one, with no synchronisation
    between them: the second call's -1 fill of row_to_slot must not start
    before the first call's scatter is done, so every row past the second
    call's groups reads -1 and its groups match the oracle."""
    E, k, pad = 896, 16, 32
    rng = np.random.default_rng(21)
    big, _ = orc.route_topk(rng.normal(0, 1, (256, E)).astype(np.float32), k)
    small, _ = orc.route_topk(rng.normal(0, 1, (8, E)).astype(np.float32), k)
    rc = abi.moe_rows_capacity(256, E, k, pad)
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    s2r = torch.empty(256 * k, dtype=torch.int32, device="cuda")
    r2s = torch.full((rc,), -7, dtype=torch.int32, device="cuda")
    ws = torch.zeros(abi.moe_permute_workspace_size(256, E), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = orc.permute(small, E, pad)
    n = int(ref["offsets"][E])
    d_big, d_small = torch.from_numpy(big).cuda(), torch.from_numpy(small).cuda()
    for _ in range(10):
        for ids, T in ((d_big, 256), (d_small, 8)):
            if noalloc:
                abi.moe_permute_noalloc(ids, T, E, k, pad, counts, offsets, s2r, r2s, rc, status)
            else:
                abi.moe_permute(ids, T, E, k, pad, counts, offsets, s2r, r2s, rc, ws)
        torch.cuda.synchronize()
        got = r2s.cpu().numpy()
        assert np.array_equal(got[:n], ref["row_to_slot"])
        assert (got[n:] == -1).all()
        assert np.array_equal(offsets.cpu().numpy(), ref["offsets"])
        assert np.array_equal(s2r.cpu().numpy()[: 8 * k], ref["slot_to_row"])
    assert abi.moe_check_device_status(ws) == 0 and int(status.item()) == 0


def test_permute_flags_bad_ids_on_device(abi):
    ids = np.array([[0, 1], [2, 2], [3, 900]], np.int32)
    got = _permute_gpu(abi, ids, 8, 1, rows_capacity=128)
    assert got["status"] == 6  # MOE_ERR_DEVICE_BAD_INPUT


def _quant_gpu(abi, x_bf16, slot_to_row=None, k=0, rows_capacity=None, layout=0, codes_offset=0):
    T, d = x_bf16.shape
    rc = rows_capacity or (T + 127) // 128 * 128
    codes = torch.zeros(rc * d + codes_offset, dtype=torch.uint8,
                        device="cuda")[codes_offset:].view(rc, d)
    scales = torch.zeros(abi.moe_activation_scale_bytes(rc, d, layout), dtype=torch.uint8,
                         device="cuda")
    s2r = None if slot_to_row is None else torch.from_numpy(slot_to_row).cuda()
    abi.moe_quant_mxfp8(x_bf16.cuda(), T, d, s2r, k, codes, scales, rc, layout)
    torch.cuda.synchronize()
    sc = scales.cpu().numpy()
    return codes.cpu().numpy(), (gu.untile_g32(sc, rc, d) if layout else gu.untile(sc, rc, d))


def _special_rows(d):
    rows = np.zeros((8, d), np.float32)
    rng = np.random.default_rng(5)
    rows[1] = -0.0                                                    # signed zeros
    rows[2] = rng.normal(0, 1, d) * 2.0 ** -130                       # bf16 subnormals
    rows[3] = rng.normal(0, 1, d) * 1e37                              # near the top of bf16
    rows[4, ::32] = 510.0                                             # saturates to 448
    rows[4, 1::32] = 1.0
    rows[5] = rng.normal(0, 1, d)
    rows[5, 7::32] = 0.0
    rows[6] = rng.standard_cauchy(d)                                  # heavy tails
    rows[7] = rng.normal(0, 1, d) * 64.0                              # outlier rows
    return torch.from_numpy(rows).to(torch.bfloat16)


@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("T,d", [(300, 3584), (8, 256), (1, 128),
                                 (1000, 3584), (1500, 2048)])   # the last two: 16 inputs a thread
def test_quant_dense_bit_exact(abi, orc, T, d, layout):
    x = torch.randn(T, d, generator=torch.Generator().manual_seed(T)).to(torch.bfloat16)
    codes, scales = _quant_gpu(abi, x, layout=layout)
    rc, rs = orc.mx_quant_rows_bf16(synth.bf16_bits(x))
    assert np.array_equal(codes[:T], rc)
    assert np.array_equal(scales[:T], rs)


def test_quant_large_batch_codes_only_8_byte_aligned(abi, orc):
    """A large batch into a code buffer 8 but not 16 bytes aligned takes the
    8-inputs-a-thread kernel and gives the same bits."""
    x = torch.randn(1000, 3584, generator=torch.Generator().manual_seed(12)).to(torch.bfloat16)
    codes, scales = _quant_gpu(abi, x, codes_offset=8)
    rc, rs = orc.mx_quant_rows_bf16(synth.bf16_bits(x))
    assert np.array_equal(codes[:1000], rc)
    assert np.array_equal(scales[:1000], rs)


def test_quant_special_values_large_batch_bit_exact(abi, orc):
    x = _special_rows(4096).repeat(90, 1)    # 720 rows x 4096: 16 inputs a thread
    codes, scales = _quant_gpu(abi, x)
    rc, rs = orc.mx_quant_rows_bf16(synth.bf16_bits(x))
    assert np.array_equal(scales[:720], rs)
    assert np.array_equal(codes[:720], rc)


def test_quant_special_values_bit_exact(abi, orc):
    x = _special_rows(512)
    codes, scales = _quant_gpu(abi, x)
    rc, rs = orc.mx_quant_rows_bf16(synth.bf16_bits(x))
    assert np.array_equal(scales[:8], rs)
    assert np.array_equal(codes[:8], rc)
    assert np.all(codes[1] == 0x80) and np.all(scales[0] == 0)


def test_quant_outlier_rows_keep_codes_and_shift_scales(abi):
    x = torch.randn(64, 3584, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    x64 = (x.float() * 64).to(torch.bfloat16)
    c0, s0 = _quant_gpu(abi, x)
    c1, s1 = _quant_gpu(abi, x64)
    assert np.array_equal(c0, c1)
    assert np.array_equal(s1[:64].astype(int), s0[:64].astype(int) + 6)


@pytest.mark.parametrize("pad,layout", [(128, 0), (32, 1)])
def test_quant_scattered_to_grouped_rows(abi, orc, pad, layout):
    T, d, E, k = 700, 3584, 896, 16
    rng = np.random.default_rng(8)
    ids, _ = orc.route_topk(rng.normal(0, 1, (T, E)).astype(np.float32), k)
    perm = orc.permute(ids, E, pad)
    rc = abi.moe_rows_capacity(T, E, k, pad)
    x = torch.randn(T, d, generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    codes, scales = _quant_gpu(abi, x, perm["slot_to_row"], k, rc, layout)
    ref_c, ref_s = orc.mx_quant_rows_bf16(synth.bf16_bits(x))
    rows = perm["slot_to_row"].reshape(T, k)
    for j in range(k):
        assert np.array_equal(codes[rows[:, j]], ref_c)
        assert np.array_equal(scales[rows[:, j]], ref_s)


def test_prepack_scales_matches_layout_definition(abi):
    rng = np.random.default_rng(4)
    for rows, K in ((300, 3584), (6144, 256), (5, 128)):
        canon = rng.integers(0, 255, (rows, K // 32)).astype(np.uint8)
        dst = torch.full((abi.moe_tiled_scale_bytes(rows, K),), 0xAB, dtype=torch.uint8,
                         device="cuda")
        abi.moe_prepack_scales(torch.from_numpy(canon).cuda(), rows, K, dst)
        assert np.array_equal(dst.cpu().numpy(), gu.tile(canon, K))


def test_prepack_weights_matches_layout_definition(abi):
    rng = np.random.default_rng(6)
    for rows, K in ((256, 3584), (384, 256), (128, 128)):
        canon = rng.integers(0, 256, (rows, K // 2)).astype(np.uint8)
        dst = torch.full((rows * K // 2,), 0xAB, dtype=torch.uint8, device="cuda")
        abi.moe_prepack_weights(torch.from_numpy(canon).cuda(), rows, K, dst)
        # box (r/128, c/128) at index (r/128)*(K/128) + c/128, 64 bytes per box row
        ref = canon.reshape(rows // 128, 128, K // 128, 64).transpose(0, 2, 1, 3).reshape(-1)
        assert np.array_equal(dst.cpu().numpy(), ref)


@pytest.mark.parametrize("T,k,d", [(100, 16, 3584), (33, 4, 256), (5, 0, 128)])
def test_combine_matches_weighted_sum(abi, T, k, d):
    rng = np.random.default_rng(T)
    rows = T * k + 37
    yp = torch.randn(rows, d, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    s2r = np.stack([rng.permutation(rows)[:k] for _ in range(T)]).astype(np.int32).reshape(-1)
    w = rng.random((T, k)).astype(np.float32)
    y = torch.full((T, d), 7.0, dtype=torch.bfloat16, device="cuda")
    abi.moe_unpermute_combine(yp.cuda(), torch.from_numpy(s2r).cuda() if k else None,
                              torch.from_numpy(w).cuda() if k else None, T, k, d, y)
    got = gu.bf16_to_f64(y)
    ypf = yp.double().numpy()
    ref = np.zeros((T, d))
    for j in range(k):
        ref += w[:, j:j + 1].astype(np.float64) * ypf[s2r.reshape(T, k)[:, j]]
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-5 * (np.abs(ref).max() + 1e-30))


def test_bounded_wait_times_out_without_hanging(abi):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    abi.moe_selftest_wait_timeout(ws, 20000)      # 20 ms
    assert abi.moe_check_device_status(ws) == 5   # MOE_ERR_DEVICE_TIMEOUT
    abi.moe_clear_device_status(ws)
    assert abi.moe_check_device_status(ws) == 0
    # the context is still usable
    ids, _ = _route_gpu(abi, np.arange(64, dtype=np.float32).reshape(2, 32), 3)
    assert ids.tolist() == [[31, 30, 29], [31, 30, 29]]
