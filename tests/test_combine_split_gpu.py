"""The combine's work split against the oracle, bit for bit.

With NW warps in the grid, the first floor(T / NW) * NW tokens are summed
whole (one token per warp and pass) and the rounds of the other tokens are
shared out in contiguous ranges, so that a warp's range may start or end
inside a token.  The batches here sit just below, on and just above multiples
of the grid's warp count for one to four CTAs of 8 warps per SM (the count
depends on the device's SM count and the kernel's occupancy), with rows whose
last round is whole or partial; unweighted and weighted combine, one buffer
and per-rank regions."""
import numpy as np
import pytest
import torch

import combine_ep_dispatch_gb300 as ep
import oracle
from combine_ep_dispatch_gb300.inputs import make_bf16, make_routing

from gpu_util import SENT_BF16, assert_rows_equal, to_dev_bf16, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    import __graft_entry__

    __graft_entry__.build()


def _batches():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    out = set()
    for per_sm in (1, 2, 3, 4):
        nw = sms * per_sm * 8
        out.update({nw - 1, nw, nw + 1})
    return sorted(out)


def _case(T, H, E=64, k=6, W=8, seed=0):
    rng = np.random.default_rng(seed * 7919 + T * 31 + H)
    idx = make_routing(rng, T, E, k, "zipf" if seed % 2 else "uniform")
    lay = oracle.layout(idx, E, W)
    R = int(lay["rank_offset"][-1])
    y = make_bf16(rng, (R, H))
    return rng, lay, y


@pytest.mark.parametrize("H", [1024, 264, 7168])
def test_combine_around_warp_count_multiples(H):
    Ts = _batches() if H != 7168 else _batches()[:4]
    for i, T in enumerate(Ts):
        _, lay, y = _case(T, H, seed=i)
        want = oracle.combine(y, lay["slot"])["out"]
        out = torch.full((T, H), SENT_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        ep.ep_combine(to_dev_bf16(y), torch.from_numpy(lay["slot"]).cuda(), out, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert_rows_equal(u16(out), want, f"combine T={T} H={H}")


def test_weighted_combine_around_warp_count_multiples():
    H, k = 520, 5   # 65 pieces: two rounds, the second with one piece
    for i, T in enumerate(_batches()):
        rng = np.random.default_rng(1000 + T)
        E = 40
        idx = make_routing(rng, T, E, k, "uniform")
        lay = oracle.layout_experts(idx, E)
        R = int(lay["expert_offset"][-1])
        y = make_bf16(rng, (R, H))
        w = rng.standard_normal((T, k), dtype=np.float32)
        want = oracle.combine_weighted(y, lay["slot"], w)["out"]
        out = torch.full((T, H), SENT_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        ep.ep_combine_weighted(to_dev_bf16(y), torch.from_numpy(lay["slot"]).cuda(),
                               torch.from_numpy(w).cuda(), out, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert_rows_equal(u16(out), want, f"weighted combine T={T}")


def test_region_combine_around_warp_count_multiples():
    H, W = 1024, 8
    for i, T in enumerate(_batches()[::2]):
        _, lay, y = _case(T, H, W=W, seed=i)
        off = lay["rank_offset"]
        y_regs = [to_dev_bf16(y[int(off[r]):int(off[r + 1])]) for r in range(W)]
        want = oracle.combine(y, lay["slot"])["out"]
        out = torch.full((T, H), SENT_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        ep.ep_combine_regions(y_regs, torch.from_numpy(lay["slot"]).cuda(),
                              torch.from_numpy(off).cuda(), out, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert_rows_equal(u16(out), want, f"region combine T={T}")
