"""The Python binding checks every tensor's shape against the sizes it passes
to the library (T, k, E, W, H, capacity) before anything is launched: the
kernels trust those sizes, so a wrong-sized tensor must be refused on the host.

CPU: the shape checks come before the device checks, so CPU tensors exercise
them (a correctly shaped CPU tensor is refused only for not being on the GPU).
GPU: the same refusals leave sentinel-filled outputs untouched."""
import pytest
import torch

import combine_ep_dispatch_gb300 as ep

T, H, E, k, W = 64, 256, 16, 4, 4
CAP = T * W


def _i32(*s):
    return torch.zeros(*s, dtype=torch.int32)


def _layout_args(**over):
    a = dict(topk_idx=_i32(T, k), E=E, W=W, num_tokens_per_expert=_i32(E),
             num_tokens_per_rank=_i32(W), rank_offset=_i32(W + 1), slot=_i32(T, W),
             workspace=torch.zeros(4096, dtype=torch.uint8), status=_i32(1))
    a.update(over)
    return a


def _dispatch_args(quant=ep.EP_QUANT_BF16, **over):
    fp8 = quant == ep.EP_QUANT_FP8_E4M3_B128
    a = dict(x=torch.zeros(T, H, dtype=torch.bfloat16), topk_idx=_i32(T, k),
             topk_w=torch.zeros(T, k), W=W, slot=_i32(T, W),
             recv_x=torch.zeros(CAP, H, dtype=torch.uint8 if fp8 else torch.bfloat16),
             recv_topk_idx=_i32(CAP, k), recv_topk_w=torch.zeros(CAP, k), recv_src=_i32(CAP),
             recv_scale=torch.zeros(CAP, H // 128) if fp8 else None, quant=quant, status=_i32(1))
    a.update(over)
    return a


def _with_layout_args(**over):
    a = _dispatch_args()
    a.update(E=E, num_tokens_per_expert=_i32(E), num_tokens_per_rank=_i32(W),
             rank_offset=_i32(W + 1), workspace=torch.zeros(4096, dtype=torch.uint8))
    a.update(over)
    return a


def _refused_for_shape(fn, **kw):
    with pytest.raises(ValueError, match="shape|2-D|at least one"):
        fn(**kw)


def _refused_for_device(fn, **kw):
    with pytest.raises(ValueError, match="CUDA tensor"):
        fn(**kw)


@pytest.mark.parametrize("fn", [ep.ep_dispatch_layout, ep.ep_dispatch_layout_noalloc])
@pytest.mark.parametrize("bad", [dict(num_tokens_per_expert=_i32(E - 1)),
                                 dict(num_tokens_per_rank=_i32(W + 1)),
                                 dict(rank_offset=_i32(W)),
                                 dict(slot=_i32(T, W - 1)), dict(slot=_i32(T - 1, W)),
                                 dict(topk_idx=_i32(T * k)), dict(status=_i32(0))])
def test_layout_refuses_wrong_shapes(fn, bad):
    args = _layout_args(**bad)
    if fn is ep.ep_dispatch_layout_noalloc:
        args.pop("workspace")
    _refused_for_shape(fn, **args)


@pytest.mark.parametrize("quant", [ep.EP_QUANT_BF16, ep.EP_QUANT_FP8_E4M3_B128])
@pytest.mark.parametrize("bad", [dict(topk_idx=_i32(T - 1, k)), dict(topk_w=torch.zeros(T, k + 1)),
                                 dict(slot=_i32(T, W + 1)), dict(slot=_i32(T + 1, W)),
                                 dict(recv_topk_idx=_i32(CAP, k - 1)),
                                 dict(recv_topk_idx=_i32(CAP - 1, k)),
                                 dict(recv_topk_w=torch.zeros(CAP + 1, k)),
                                 dict(recv_src=_i32(CAP - 1)), dict(recv_src=_i32(CAP, 1)),
                                 dict(status=_i32(0))])
def test_dispatch_refuses_wrong_shapes(quant, bad):
    _refused_for_shape(ep.ep_dispatch, **_dispatch_args(quant, **bad))
    _refused_for_shape(ep.ep_dispatch_with_layout, **_with_layout_args(quant=quant, **bad,
                       recv_x=_dispatch_args(quant)["recv_x"],
                       recv_scale=_dispatch_args(quant)["recv_scale"]))


def test_dispatch_refuses_wrong_payload_shapes():
    _refused_for_shape(ep.ep_dispatch, **_dispatch_args(recv_x=torch.zeros(CAP, H + 8,
                                                                          dtype=torch.bfloat16)))
    fp8 = ep.EP_QUANT_FP8_E4M3_B128
    _refused_for_shape(ep.ep_dispatch, **_dispatch_args(fp8, recv_scale=torch.zeros(CAP, 1)))
    _refused_for_shape(ep.ep_dispatch, **_dispatch_args(fp8, recv_scale=torch.zeros(CAP - 1,
                                                                                   H // 128)))
    _refused_for_shape(ep.ep_dispatch_with_layout, **_with_layout_args(rank_offset=_i32(W + 2)))
    _refused_for_shape(ep.ep_dispatch_with_layout,
                       **_with_layout_args(num_tokens_per_expert=_i32(2 * E)))


def test_fused_and_expert_calls_refuse_wrong_shapes():
    a = _with_layout_args()
    del a["workspace"], a["recv_scale"], a["quant"]
    _refused_for_shape(ep.ep_dispatch_fused, **{**a, "slot": _i32(T, W + 1)})
    _refused_for_shape(ep.ep_dispatch_fused, **{**a, "recv_src": _i32(CAP + 3)})
    x = dict(x=torch.zeros(T, H, dtype=torch.bfloat16), topk_idx=_i32(T, k),
             topk_w=torch.zeros(T, k), E=E, num_tokens_per_expert=_i32(E),
             expert_offset=_i32(E + 1), slot=_i32(T, k),
             workspace=torch.zeros(4096, dtype=torch.uint8),
             recv_x=torch.zeros(T * k, H, dtype=torch.bfloat16))
    _refused_for_shape(ep.ep_dispatch_experts_with_layout, **{**x, "slot": _i32(T, W + 1)})
    _refused_for_shape(ep.ep_dispatch_experts_with_layout, **{**x, "expert_offset": _i32(E)})
    _refused_for_shape(ep.ep_dispatch_layout_experts,
                       topk_idx=_i32(T, k), E=E, num_tokens_per_expert=_i32(E),
                       expert_offset=_i32(E + 1), slot=_i32(T, k + 1),
                       workspace=torch.zeros(16, dtype=torch.uint8))
    _refused_for_device(ep.ep_dispatch_experts_with_layout, **x)


def test_combine_refuses_wrong_shapes():
    y = torch.zeros(CAP, H, dtype=torch.bfloat16)
    out = torch.zeros(T, H, dtype=torch.bfloat16)
    _refused_for_shape(ep.ep_combine, y=y, slot=_i32(T, W), out=torch.zeros(T - 1, H,
                                                                            dtype=torch.bfloat16))
    _refused_for_shape(ep.ep_combine, y=torch.zeros(CAP, H - 8, dtype=torch.bfloat16),
                       slot=_i32(T, W), out=out)
    _refused_for_shape(ep.ep_combine, y=y, slot=_i32(T * W), out=out)
    _refused_for_shape(ep.ep_combine_weighted, y=y, slot=_i32(T, W), w=torch.zeros(T, W + 1),
                       out=out)
    _refused_for_device(ep.ep_combine, y=y, slot=_i32(T, W), out=out)


def test_other_calls_refuse_wrong_shapes():
    _refused_for_shape(ep.ep_localize_expert_ids, recv_topk_idx=_i32(CAP, k),
                       rank_offset=_i32(W), E=E, W=W)
    y = torch.zeros(CAP, H, dtype=torch.bfloat16)
    ct = dict(y=y, expert_offset=_i32(E + 1), scale=torch.zeros(E),
              out_c=torch.zeros(CAP, H, dtype=torch.uint8), out_t=torch.zeros(16, dtype=torch.uint8),
              amax=torch.zeros(E))
    _refused_for_shape(ep.ep_cast_transpose_experts, **{**ct, "scale": torch.zeros(E - 1)})
    _refused_for_shape(ep.ep_cast_transpose_experts, **{**ct, "amax": torch.zeros(E + 1)})
    _refused_for_shape(ep.ep_cast_transpose_experts,
                       **{**ct, "out_c": torch.zeros(CAP, H // 2, dtype=torch.uint8)})


def test_correct_shapes_pass_to_the_device_check():
    _refused_for_device(ep.ep_dispatch_layout, **_layout_args())
    _refused_for_device(ep.ep_dispatch, **_dispatch_args())
    _refused_for_device(ep.ep_dispatch, **_dispatch_args(ep.EP_QUANT_FP8_E4M3_B128))
    _refused_for_device(ep.ep_dispatch_with_layout, **_with_layout_args())


# ----------------------------------------------------------------- on the GPU

SENT = -424242


@pytest.mark.gpu
def test_wrong_shapes_launch_nothing_on_the_gpu():
    import __graft_entry__

    __graft_entry__.build()
    dev = torch.device("cuda", torch.cuda.current_device())

    def cuda(a):
        return {n: (v.to(dev) if isinstance(v, torch.Tensor) else v) for n, v in a.items()}

    # layout: a slot table one column short must not be written
    lay = cuda(_layout_args(slot=torch.full((T, W - 1), SENT, dtype=torch.int32),
                            rank_offset=torch.full((W + 1,), SENT, dtype=torch.int32)))
    with pytest.raises(ValueError):
        ep.ep_dispatch_layout(**lay)
    # dispatch: metadata one row short of the receive rows
    dis = cuda(_dispatch_args(recv_src=torch.full((CAP - 1,), SENT, dtype=torch.int32)))
    dis["recv_topk_idx"].fill_(SENT)
    with pytest.raises(ValueError):
        ep.ep_dispatch(**dis)
    # combine: out one token short
    out = torch.full((T - 1, H), 7.0, dtype=torch.bfloat16, device=dev)
    with pytest.raises(ValueError):
        ep.ep_combine(torch.zeros(CAP, H, dtype=torch.bfloat16, device=dev),
                      torch.zeros(T, W, dtype=torch.int32, device=dev), out)
    torch.cuda.synchronize()
    assert bool((lay["slot"] == SENT).all()) and bool((lay["rank_offset"] == SENT).all())
    assert bool((dis["recv_src"] == SENT).all()) and bool((dis["recv_topk_idx"] == SENT).all())
    assert bool((out == 7.0).all())
