"""ep_dispatch_layout_noalloc: the routing layout for callers that cannot
allocate device memory (C or embedded hosts without a device allocator, and
latency-critical paths that must not call cudaMalloc, which blocks the host and
synchronises the device).  It keeps its workspace in a device array built into
the library, so these tests check that its outputs equal those of
ep_dispatch_layout (caller-provided workspace) and those of the CPU oracle's
layout bit for bit, over two calls in a row: the array keeps the previous
call's contents, which must not leak into the next result.  Collected last so
that a run stopping at its first failure has already run every other test."""
import numpy as np
import pytest
import torch

import combine_ep_dispatch_gb300 as ep
import oracle
from combine_ep_dispatch_gb300.inputs import make_routing

pytestmark = pytest.mark.gpu

SENT = -987654321


@pytest.fixture(scope="module", autouse=True)
def _library():
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)


def _outputs(T, E, W):
    i32 = dict(dtype=torch.int32, device="cuda")
    return {"num_tokens_per_expert": torch.full((E,), SENT, **i32),
            "num_tokens_per_rank": torch.full((W,), SENT, **i32),
            "rank_offset": torch.full((W + 1,), SENT, **i32),
            "slot": torch.full((T, W), SENT, **i32),
            "status": torch.zeros(1, **i32)}


def _with_workspace(idx, E, W):
    o = _outputs(idx.shape[0], E, W)
    ws = torch.empty(max(ep.ep_layout_workspace_bytes(idx.shape[0], W, E), 16), dtype=torch.uint8,
                     device="cuda")
    ep.ep_dispatch_layout(idx, E, W, o["num_tokens_per_expert"], o["num_tokens_per_rank"],
                          o["rank_offset"], o["slot"], ws, o["status"])
    return o


def _noalloc(idx, E, W):
    o = _outputs(idx.shape[0], E, W)
    ep.ep_dispatch_layout_noalloc(idx, E, W, o["num_tokens_per_expert"], o["num_tokens_per_rank"],
                                  o["rank_offset"], o["slot"], o["status"])
    return o


def _routing(T, E, k, seed, invalid=0.0):
    rng = np.random.default_rng(seed)
    idx = make_routing(rng, T, E, k, "zipf" if seed % 2 else "uniform")
    if invalid:
        idx[rng.random(idx.shape) < invalid] = E + 1
    return torch.from_numpy(idx).cuda()


@pytest.mark.parametrize("first,second", [
    ((40000, 256, 8, 8, 0.0), (12000, 96, 5, 3, 0.05)),   # large call, then a smaller ragged one
    ((9000, 64, 6, 8, 0.02), (60000, 128, 8, 8, 0.0)),    # smaller call, then a larger one
    ((4096, 256, 8, 8, 0.0), (20000, 256, 8, 8, 0.01)),   # the DeepSeek-V3 batch, then a large one
    ((0, 16, 4, 4, 0.0), (128, 16, 4, 4, 0.0)),           # empty call, then the tiny workload
])
def test_noalloc_matches_workspace_layout_two_calls_in_a_row(first, second):
    for n, (T, E, k, W, bad) in enumerate((first, second)):
        idx = _routing(T, E, k, seed=17 + n, invalid=bad)
        want = _with_workspace(idx, E, W)
        got = _noalloc(idx, E, W)
        torch.cuda.synchronize()
        for key in want:
            assert torch.equal(got[key], want[key]), (n, key)
        ref = oracle.layout(idx.cpu().numpy(), E, W)
        for key in ("num_tokens_per_expert", "num_tokens_per_rank", "rank_offset", "slot"):
            np.testing.assert_array_equal(got[key].cpu().numpy(), ref[key], err_msg=f"{n} {key}")
        assert int(got["status"].item()) == ref["status"], n


def test_noalloc_rejects_sizes_beyond_its_array():
    T, E, k, W = 130000, 256, 8, 8
    assert ep.ep_layout_workspace_bytes(T, W, E) > ep._lib.EP_LAYOUT_NOALLOC_SCRATCH_BYTES
    idx = torch.zeros(T, k, dtype=torch.int32, device="cuda")
    o = _outputs(T, E, W)
    with pytest.raises(ep.EPError) as e:
        ep.ep_dispatch_layout_noalloc(idx, E, W, o["num_tokens_per_expert"],
                                      o["num_tokens_per_rank"], o["rank_offset"], o["slot"],
                                      o["status"])
    assert e.value.code == ep.EP_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert int((o["slot"] != SENT).sum().item()) == 0    # nothing was launched
