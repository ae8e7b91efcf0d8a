"""The allocation-free grouping entry point, moe_permute_noalloc.

It serves callers that cannot give the library device memory for a workspace
(a framework that owns all device memory and forbids library allocations, or a
serving path that must not call cudaMalloc). It must give exactly what the CPU
oracle's grouping gives, and what moe_permute gives with a caller-allocated
workspace, on consecutive calls that share its built-in scratch array: the
one-block path (T <= 256), the multi-chunk path, and the largest batch its
1 MiB array accepts. This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from tests import gpu_util as gu


@pytest.fixture(scope="module")
def abi():
    return gu.cuda_lib()


def _ids(T, E, k, seed):
    """k distinct expert ids per token, seeded (the first k of a random order)."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    keys = torch.rand(T, E, generator=g, device="cuda")
    return keys.argsort(dim=1)[:, :k].to(torch.int32).contiguous()


def _outputs(T, E, k, rc):
    return (torch.full((E,), -5, dtype=torch.int32, device="cuda"),
            torch.full((E + 1,), -5, dtype=torch.int32, device="cuda"),
            torch.full((max(T * k, 1),), -5, dtype=torch.int32, device="cuda"),
            torch.full((rc,), -5, dtype=torch.int32, device="cuda"))


def _check_against_oracle(orc, ids, E, pad, out):
    ref = orc.permute(ids.cpu().numpy(), E, pad)
    counts, offsets, s2r, r2s = (t.cpu().numpy() for t in out)
    n = int(ref["offsets"][E])
    assert np.array_equal(counts, ref["counts"])
    assert np.array_equal(offsets, ref["offsets"])
    assert np.array_equal(s2r, ref["slot_to_row"])
    assert np.array_equal(r2s[:n], ref["row_to_slot"])
    assert (r2s[n:] == -1).all()


@pytest.mark.gpu
def test_permute_noalloc_matches_oracle_and_permute_on_calls_in_a_row(abi, orc):
    """Multi-chunk, then one-block, then multi-chunk again: each call reuses
    the scratch the previous one left behind."""
    E, k, pad = 896, 16, 128
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for T, seed in ((1000, 1), (200, 2), (300, 3)):
        ids = _ids(T, E, k, seed)
        rc = abi.moe_rows_capacity(T, E, k, pad)
        a = _outputs(T, E, k, rc)
        b = _outputs(T, E, k, rc)
        ws = torch.zeros(abi.moe_permute_workspace_size(T, E), dtype=torch.uint8, device="cuda")
        abi.moe_permute(ids, T, E, k, pad, a[0], a[1], a[2], a[3], rc, ws)
        abi.moe_permute_noalloc(ids, T, E, k, pad, b[0], b[1], b[2], b[3], rc, status)
        torch.cuda.synchronize()
        assert abi.moe_check_device_status(ws) == 0
        assert int(status.item()) == 0
        for x, y in zip(a, b):          # integer outputs: bit-exact
            assert torch.equal(x, y)
        _check_against_oracle(orc, ids, E, pad, b)


@pytest.mark.gpu
def test_permute_noalloc_largest_accepted_batch(abi, orc):
    """T = 74,752 at E = 896: ceil(T/256) * E * 4 = 1,046,528 bytes, the most
    the 1 MiB array holds in whole chunks; one chunk more is refused."""
    E, k, pad = 896, 16, 128
    T = 74752
    assert (T + 255) // 256 * E * 4 <= 1 << 20 < ((T + 255) // 256 + 1) * E * 4
    ids = _ids(T, E, k, 7)
    rc = abi.moe_rows_capacity(T, E, k, pad)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = _outputs(T, E, k, rc)
    b = _outputs(T, E, k, rc)
    ws = torch.zeros(abi.moe_permute_workspace_size(T, E), dtype=torch.uint8, device="cuda")
    abi.moe_permute(ids, T, E, k, pad, a[0], a[1], a[2], a[3], rc, ws)
    abi.moe_permute_noalloc(ids, T, E, k, pad, b[0], b[1], b[2], b[3], rc, status)
    torch.cuda.synchronize()
    assert abi.moe_check_device_status(ws) == 0
    assert int(status.item()) == 0
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    _check_against_oracle(orc, ids, E, pad, b)
    T1 = T + 256
    big = torch.zeros(T1, k, dtype=torch.int32, device="cuda")
    rc1 = abi.moe_rows_capacity(T1, E, k, pad)
    out = _outputs(T1, E, k, rc1)
    with pytest.raises(abi.MoeError) as err:
        abi.moe_permute_noalloc(big, T1, E, k, pad, out[0], out[1], out[2], out[3], rc1, None)
    assert err.value.code == abi.WORKSPACE_TOO_SMALL


@pytest.mark.gpu
def test_permute_noalloc_reports_bad_ids(abi):
    E, k = 8, 2
    ids = torch.tensor([[0, 1], [3, 3]], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _outputs(2, E, k, 128)
    abi.moe_permute_noalloc(ids, 2, E, k, 1, out[0], out[1], out[2], out[3], 128, status)
    torch.cuda.synchronize()
    assert int(status.item()) == abi.DEVICE_BAD_INPUT
