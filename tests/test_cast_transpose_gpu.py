"""ep_cast_transpose_experts against the oracle, bit for bit: the row-major
FP8 cast, the per-expert transposed cast (padding included), and the amax,
on ragged expert sizes, wide scale ranges (saturating products included) and
the full expert-major DeepSeek-V3 step."""
import numpy as np
import pytest
import torch

import combine_ep_dispatch_gb300 as ep
import oracle
from combine_ep_dispatch_gb300.inputs import make_bf16, make_inputs
from gpu_util import assert_rows_equal, run_dispatch, to_dev_bf16

pytestmark = pytest.mark.gpu

SENT = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _library():
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)


def _run(y, off, scale, amax0, cap=None):
    R_buf, H = y.shape
    cap = R_buf if cap is None else cap
    E = off.size - 1
    yd = to_dev_bf16(y)[:cap].contiguous() if cap < R_buf else to_dev_bf16(y)
    out_c = torch.full((cap, H), SENT, dtype=torch.uint8, device="cuda")
    tb = ep.ep_cast_transpose_t_bytes(cap, E, H)
    out_t = torch.full((max(tb, 16),), SENT, dtype=torch.uint8, device="cuda")
    amax = torch.from_numpy(amax0.copy()).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ep_cast_transpose_experts(yd, torch.from_numpy(off.astype(np.int32)).cuda(),
                                 torch.from_numpy(scale).cuda(), out_c, out_t, amax, st)
    torch.cuda.synchronize()
    return out_c.cpu().numpy(), out_t.cpu().numpy(), amax.cpu().numpy(), int(st.item())


def _check(y, off, scale, amax0):
    want = oracle.cast_transpose(y, off, scale, amax0)
    got_c, got_t, got_amax, st = _run(y, off, scale, amax0)
    R = int(off[-1])
    assert st == 0
    assert_rows_equal(got_c[:R], want["out_c"], "out_c")
    assert np.all(got_c[R:] == SENT)
    nt = want["out_t"].size
    assert np.array_equal(got_t[:nt], want["out_t"]), np.nonzero(got_t[:nt] != want["out_t"])[0][:8]
    assert np.all(got_t[nt:] == SENT)
    np.testing.assert_array_equal(got_amax.view(np.uint32), want["amax"].view(np.uint32))


@pytest.mark.parametrize("sizes,H", [
    ([5], 256),
    ([0, 1, 15, 16, 17, 63, 64, 65, 200, 0], 512),
    ([130, 3, 0, 64, 127, 128, 129], 7168),
    (list(np.random.default_rng(3).integers(0, 300, 40)), 1024),
])
def test_cast_transpose_matches_oracle(sizes, H):
    rng = np.random.default_rng(len(sizes) * 7 + H)
    n = np.array(sizes, np.int64)
    off = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    R = int(off[-1])
    y = make_bf16(rng, (max(R, 1), H), scale=4.0)[:R] if R else np.zeros((0, H), np.uint16)
    if R:
        y[rng.random(y.shape) < 0.01] = 0x8000                  # -0
    E = n.size
    scale = (2.0 ** rng.uniform(-6, 9, size=E)).astype(np.float32)   # some products saturate
    amax0 = np.where(rng.random(E) < 0.5, 0.0, rng.random(E) * 8).astype(np.float32)
    _check(y if R else np.zeros((1, H), np.uint16)[:0], off, scale, amax0)


def test_cast_transpose_8192_experts():
    """The largest expert count the call takes: 8192 per-expert prefixes in
    shared memory, most experts empty, a few with ragged row counts."""
    rng = np.random.default_rng(8192)
    E, H = 8192, 256
    n = np.zeros(E, np.int64)
    hot = rng.choice(E, 40, replace=False)
    n[hot] = rng.integers(1, 150, hot.size)
    n[E - 1] = 65                                                     # the last expert too
    off = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    R = int(off[-1])
    y = make_bf16(rng, (R, H), scale=2.0)
    scale = (2.0 ** rng.uniform(-3, 6, size=E)).astype(np.float32)
    _check(y, off, scale, np.zeros(E, np.float32))


def test_cast_transpose_expert_major_dsv3_step():
    """Dispatch the DeepSeek-V3 batch into the expert-major layout, then cast
    and transpose the received rows with per-expert scales."""
    inp = make_inputs("dsv3", seed=31)
    cfg = inp["cfg"]
    lay = oracle.layout_experts(inp["topk_idx"], cfg.E)
    R = int(lay["expert_offset"][-1])
    recv = run_dispatch(inp["x"], inp["topk_idx"], inp["topk_w"], lay["slot"], R,
                        ep.EP_QUANT_BF16, with_meta=False)["recv_x"]
    rng = np.random.default_rng(32)
    scale = (448.0 / rng.uniform(2.0, 6.0, size=cfg.E)).astype(np.float32)
    _check(recv, lay["expert_offset"], scale, np.zeros(cfg.E, np.float32))


def test_cast_transpose_rows_beyond_capacity_are_skipped():
    rng = np.random.default_rng(33)
    H = 256
    n = np.array([40, 70, 30], np.int64)
    off = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    y = make_bf16(rng, (140, H))
    scale = np.ones(3, np.float32)
    cap = 100                                   # expert 2 (rows 110..139) and expert 1's end are out
    got_c, got_t, got_amax, st = _run(y, off, scale, np.zeros(3, np.float32), cap=cap)
    assert st & ep.EP_STATUS_CAPACITY
    want = oracle.cast_transpose(y[:40], off[:2], scale[:1])    # expert 0 alone is fully inside
    assert_rows_equal(got_c[:40], want["out_c"], "out_c")
    assert np.all(got_c[40:] == SENT)
    assert np.array_equal(got_t[:want["out_t"].size], want["out_t"])
    assert got_amax[0] == want["amax"][0] and got_amax[1] == 0 and got_amax[2] == 0
