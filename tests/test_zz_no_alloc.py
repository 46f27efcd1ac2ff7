"""moe_permute_noalloc: the permutation for callers that cannot allocate device
memory (a pool or arena owns all of it, a serving loop may not allocate after
start-up, or a plug-in is handed only its input and output buffers).  It must
give exactly what moe_permute gives with a caller workspace, on consecutive
calls that reuse the library's built-in scratch array, and refuse sizes that do
not fit that array.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def lib():
    from moe_layer_bit_gb300 import _lib, build
    build.build()
    _lib.load()
    return _lib


def _outputs(T, H, E, k):
    n = T * k
    return (torch.empty(E, dtype=torch.int32, device=DEV), torch.empty(E + 1, dtype=torch.int32, device=DEV),
            torch.empty(max(n, 1), dtype=torch.int32, device=DEV), torch.empty(max(n, 1), dtype=torch.int32, device=DEV),
            torch.empty(max(n, 1), H, dtype=torch.bfloat16, device=DEV))


@pytest.mark.parametrize("T,H,E,k", [
    (32, 2048, 128, 8),     # one chunk: no scratch needed
    (1100, 256, 16, 4),     # 5 chunks
    (4096, 128, 256, 8),    # 32 chunks
    (8192, 128, 1024, 8),   # 64 chunks x 1024 experts: exactly the built-in capacity
])
def test_noalloc_permute_equals_workspace_permute(lib, T, H, E, k):
    g = torch.Generator().manual_seed(T + E)
    ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32).to(DEV)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16).to(DEV)
    d = lib.dims(T, H, 64, E, k)
    ws_bytes = lib.moe_stage_workspace_bytes(d)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=DEV)
    ref = _outputs(T, H, E, k)
    lib.moe_permute(ids, x, d, *ref, ws, ws_bytes)
    torch.cuda.synchronize()
    n = T * k
    for call in range(2):                   # two calls in a row share the scratch array
        got = _outputs(T, H, E, k)
        lib.moe_permute_noalloc(ids, x, d, *got)
        torch.cuda.synchronize()
        for a, b, name in zip(got[:4], ref[:4], ["counts", "offsets", "sorted_token", "inv_perm"]):
            m = n if name in ("sorted_token", "inv_perm") else a.numel()
            assert torch.equal(a[:m], b[:m]), (call, name)
        assert torch.equal(got[4][:n].view(torch.int16), ref[4][:n].view(torch.int16)), (call, "x_perm")


def test_noalloc_permute_refuses_sizes_beyond_its_scratch(lib):
    T, H, E, k = 16384, 128, 1024, 8        # 128 chunks x 1024 experts > 65536 entries
    d = lib.dims(T, H, 64, E, k)
    ids = torch.zeros(T, k, dtype=torch.int32, device=DEV)
    x = torch.zeros(T, H, dtype=torch.bfloat16, device=DEV)
    outs = _outputs(T, H, E, k)
    with pytest.raises(lib.MoeError) as exc:
        lib.moe_permute_noalloc(ids, x, d, *outs)
    assert exc.value.status == lib.MOE_ERR_UNSUPPORTED_SHAPE
