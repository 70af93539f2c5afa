"""moe_permute_noalloc: the dispatch for callers that cannot allocate device memory.

Some users of this library only hold the layer's input and output buffers (a plug-in or
fixed-signature callback that receives tensors but no allocator, or a process whose device
memory belongs to another allocator), so they cannot pass the workspace moe_permute needs.
moe_permute_noalloc keeps that scratch in a fixed array owned by the library. This file is
collected last so that a run stopping at its first failure has run every other test.
"""
import numpy as np
import pytest
import torch

from pretraining_sigmoid_softmax_gb300 import ops

from gpu_common import dev, randn_bf16, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()


def _outputs(T, d, E, k):
    R = ops.moe_padded_rows(T, k, E)
    return dict(counts=torch.empty(E, dtype=torch.int32, device="cuda"),
                offsets=torch.empty(E + 1, dtype=torch.int64, device="cuda"),
                row_offsets=torch.empty(E + 1, dtype=torch.int64, device="cuda"),
                perm_token=torch.full((R,), -7, dtype=torch.int32, device="cuda"),
                slot_to_row=torch.empty(T, k, dtype=torch.int32, device="cuda"),
                X_perm=torch.full((R, d), float("nan"), dtype=torch.bfloat16, device="cuda"))


def _compare(a, b):
    ro = a["row_offsets"].cpu()
    assert torch.equal(ro, b["row_offsets"].cpu())
    used = int(ro[-1])
    for key in ("counts", "offsets", "slot_to_row"):
        assert torch.equal(a[key], b[key]), key
    assert torch.equal(a["perm_token"][:used], b["perm_token"][:used])
    # bit-exact rows (the dispatch copies bf16 rows; same tolerance as moe_permute's tests)
    assert torch.equal(a["X_perm"][:used].view(torch.int16), b["X_perm"][:used].view(torch.int16))


@pytest.mark.parametrize("T,d,E,k", [(3000, 256, 64, 8), (700, 128, 16, 4)])
def test_noalloc_matches_moe_permute_on_two_calls_in_a_row(T, d, E, k):
    g = torch.Generator().manual_seed(T + E)
    w = torch.tensor([1.0 / (i + 1) for i in range(E)])
    idx = torch.stack([torch.multinomial(w, k, replacement=False, generator=g)
                       for _ in range(T)]).to(torch.int32)
    x = randn_bf16((T, d), g)
    idx_d, x_d = dev(idx), dev(x)
    ref = _outputs(T, d, E, k)
    ws = torch.empty(ops.moe_workspace_bytes(T, d, E, k), dtype=torch.uint8, device="cuda")
    ops.moe_permute(idx_d, x_d, E, ref["counts"], ref["offsets"], ref["row_offsets"],
                    ref["perm_token"], ref["slot_to_row"], ref["X_perm"], ws)
    for _ in range(2):  # the static scratch keeps the previous call's contents
        out = _outputs(T, d, E, k)
        ops.moe_permute_noalloc(idx_d, x_d, E, out["counts"], out["offsets"],
                                out["row_offsets"], out["perm_token"], out["slot_to_row"],
                                out["X_perm"])
        torch.cuda.synchronize()
        _compare(ref, out)
    assert ops.moe_device_status()[0] == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    from pretraining_sigmoid_softmax_gb300 import _lib
    lib = _lib.load()
    E, k, d = 256, 8, 128
    T = 256 * (1048576 // E + 1)  # one chunk of counts more than the static array holds
    small = torch.zeros(16, dtype=torch.int32, device="cuda")
    rc = lib.moe_permute_noalloc(small.data_ptr(), small.data_ptr(), T, d, E, k,
                                 small.data_ptr(), small.data_ptr(), small.data_ptr(),
                                 small.data_ptr(), small.data_ptr(), small.data_ptr(), None)
    assert rc == 7  # MOE_ERR_TOO_LARGE, returned before any device work
