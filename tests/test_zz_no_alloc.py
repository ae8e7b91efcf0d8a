"""The allocation-free grouping entry point, moe_permute_noalloc.

It serves callers that cannot give the library device memory for a workspace
(a framework that owns all device memory and forbids library allocations, or a
serving path that must not call cudaMalloc). It must give exactly what
moe_permute gives with a caller-allocated workspace, on consecutive calls that
share its built-in scratch array. This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from tests import gpu_util as gu


@pytest.fixture(scope="module")
def abi():
    return gu.cuda_lib()


def _ids(T, E, k, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)


def _outputs(T, E, rc):
    return (torch.full((E,), -5, dtype=torch.int32, device="cuda"),
            torch.full((E + 1,), -5, dtype=torch.int32, device="cuda"),
            torch.full((max(T, 1) * 16,), -5, dtype=torch.int32, device="cuda"),
            torch.full((rc,), -5, dtype=torch.int32, device="cuda"))


@pytest.mark.gpu
def test_permute_noalloc_matches_permute_on_two_calls_in_a_row(abi):
    E, k, pad = 896, 16, 128
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for T, seed in ((1000, 1), (300, 2)):       # the second call reuses the scratch of the first
        ids = _ids(T, E, k, seed).cuda()
        rc = abi.moe_rows_capacity(T, E, k, pad)
        a = _outputs(T, E, rc)
        b = _outputs(T, E, rc)
        ws = torch.zeros(abi.moe_permute_workspace_size(T, E), dtype=torch.uint8, device="cuda")
        abi.moe_permute(ids, T, E, k, pad, a[0], a[1], a[2], a[3], rc, ws)
        abi.moe_permute_noalloc(ids, T, E, k, pad, b[0], b[1], b[2], b[3], rc, status)
        torch.cuda.synchronize()
        assert abi.moe_check_device_status(ws) == 0
        assert int(status.item()) == 0
        for x, y in zip(a, b):          # integer outputs: bit-exact
            assert torch.equal(x, y)


@pytest.mark.gpu
def test_permute_noalloc_reports_bad_ids_and_refuses_oversize(abi):
    E, k = 8, 2
    ids = torch.tensor([[0, 1], [3, 3]], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _outputs(2, E, 128)
    abi.moe_permute_noalloc(ids, 2, E, k, 1, out[0], out[1], out[2], out[3], 128, status)
    torch.cuda.synchronize()
    assert int(status.item()) == abi.DEVICE_BAD_INPUT
    # ceil(T/256) * E * 4 bytes above the 1 MiB built-in array: refused on the host
    T = 256 * 293
    big = torch.zeros(T, 16, dtype=torch.int32, device="cuda")
    rc = abi.moe_rows_capacity(T, 896, 16, 128)
    with pytest.raises(abi.MoeError) as err:
        abi.moe_permute_noalloc(big, T, 896, 16, 128, out[0], out[1], out[2], out[3], rc, None)
    assert err.value.code == abi.WORKSPACE_TOO_SMALL
