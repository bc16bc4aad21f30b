"""moe_dispatch_layout_noalloc against moe_dispatch_layout.

The no-alloc variant serves callers that cannot allocate device memory
(a plugin whose host engine owns the whole device pool, or a service that
forbids cudaMalloc after start-up because an allocation can synchronise the
device).  It must give the same layout as the workspace variant: these are
integer results, so the comparison is exact.  Two calls run back to back on
different inputs, so the second also shows that the histograms a previous
call left in the shared static scratch do not leak into the next result.

This file is collected last on purpose: it runs after every other test in
a full run, and also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from combine_router_gemm_top_b300 import _lib as L

pytestmark = pytest.mark.gpu

DEV = "cuda"
SCRATCH_BYTES = 1 << 20      # MOE_NOALLOC_LAYOUT_SCRATCH_BYTES


def _outputs(T, k, E, R):
    P = max(T * k, 1)
    i32 = dict(dtype=torch.int32, device=DEV)
    return [torch.full((E,), -5, **i32), torch.full((E + 1,), -5, **i32),
            torch.full((P,), -5, **i32), torch.full((P,), -5, **i32),
            torch.full((1,), -5, **i32), torch.full((1,), -5, **i32),
            torch.full((R,), -5, **i32), torch.full((R,), -5, **i32)]


def _with_workspace(idx, T, k, E, R, cap):
    out = _outputs(T, k, E, R)
    ws = torch.empty(L.moe_dispatch_layout_workspace_size(T, k, E),
                     dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.moe_dispatch_layout(T, k, E, R, cap, idx, *out, ws, st)
    return out, st


def _no_alloc(idx, T, k, E, R, cap):
    out = _outputs(T, k, E, R)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.moe_dispatch_layout_noalloc(T, k, E, R, cap, idx, *out, st)
    return out, st


def _idx(T, k, E, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, E, (T, k), generator=g,
                         dtype=torch.int32).to(DEV)


@pytest.mark.parametrize("calls", [
    # (T, k, E, R, capacity) for two calls in a row
    [(65536, 8, 128, 8, 0), (2048, 2, 8, 8, 0)],
    [(3000, 4, 64, 16, 150), (700, 2, 16, 4, 40)],
    # both calls on the three-kernel path that uses the scratch, the second
    # with fewer chunks (16 against 256) and fewer experts (64 against 128):
    # cells the first call wrote and the second does not must not leak in
    [(65536, 8, 128, 8, 0), (4096, 8, 64, 8, 0)],
    # the largest request the 1 MiB scratch holds: 256 chunks x 1024 experts
    [(65536, 8, 1024, 32, 0), (65536, 8, 1024, 32, 300)],
])
def test_no_alloc_matches_workspace_variant(calls):
    for n, (T, k, E, R, cap) in enumerate(calls):
        idx = _idx(T, k, E, seed=17 * n + E)
        ref, st_ref = _with_workspace(idx, T, k, E, R, cap)
        got, st_got = _no_alloc(idx, T, k, E, R, cap)
        torch.cuda.synchronize()
        assert st_ref.item() == 0 and st_got.item() == 0
        P = T * k
        names = ["counts", "offsets", "dst_row", "src_pair", "n_kept",
                 "n_dropped", "rank_send_counts", "rank_send_displs"]
        n_kept = int(ref[4].item())
        for name, a, b in zip(names, ref, got):
            if name == "src_pair":
                a, b = a[:n_kept], b[:n_kept]
            elif name == "dst_row":
                a, b = a[:P], b[:P]
            assert torch.equal(a, b), name


def test_no_alloc_rejects_requests_beyond_the_scratch():
    T, k, E, R = 65793, 8, 1024, 32          # 258 chunks x 1024 > 1 MiB
    assert -(-T * k // 2048) * E * 4 > SCRATCH_BYTES
    idx = torch.zeros((T, k), dtype=torch.int32, device=DEV)
    out = _outputs(T, k, E, R)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    with pytest.raises(L.MoeError) as e:
        L.moe_dispatch_layout_noalloc(T, k, E, R, 0, idx, *out, st)
    assert e.value.code == L.MOE_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert int(out[0][0].item()) == -5       # nothing was launched
