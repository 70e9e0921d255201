"""The block at the limits of the C ABI: E = 1024 experts with k = 32 per
token (forward and backward, BF16 and MXFP8, each checked against the
oracle), bounded in-kernel waits forced to expire in the backward and MXFP8
paths (the call reports MOE_ERR_TIMEOUT and the context stays usable), and
out-of-range expert ids in the MXFP8 forward."""
import numpy as np
import pytest
import torch

import oracle as orc
from gpu_util import assert_bf16_close, assert_rel_to_max, dev, to_np

pytestmark = pytest.mark.gpu
m = pytest.importorskip("moe_expert_dispatch_gb300")


def _case(T, H, F, E, k, seed, wstd=0.05, mx=False):
    g = torch.Generator().manual_seed(seed)
    ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    p = torch.rand((T, k), generator=g) + 0.05
    probs = (p / p.sum(1, keepdim=True)).float()
    bf = lambda *s, sd=1.0: (torch.randn(s, generator=g) * sd).to(torch.bfloat16)  # noqa: E731
    if mx:   # K-contiguous weights
        w = (bf(E, F, H, sd=wstd), bf(E, F, H, sd=wstd), bf(E, H, F, sd=wstd))
    else:
        w = (bf(E, H, F, sd=wstd), bf(E, H, F, sd=wstd), bf(E, F, H, sd=wstd))
    return bf(T, H), bf(T, H), w, ids, probs


def test_bf16_forward_backward_1024_experts_top32():
    T, H, F, E, k = 96, 128, 128, 1024, 32
    dy, x, (wg, wu, wd), ids, probs = _case(T, H, F, E, k, seed=1, wstd=0.02)
    cfg = m.config(save_for_backward=True)
    y, ws = m.moe_expert_forward(dev(x), dev(wg), dev(wu), dev(wd), dev(ids), dev(probs), cfg=cfg)
    g = m.moe_expert_backward(dev(dy), dev(x), dev(wg), dev(wu), dev(wd), dev(ids), dev(probs), ws)
    assert m.moe_get_error() == 0
    args = (to_np(x), to_np(wg), to_np(wu), to_np(wd), ids.numpy(), probs.numpy().astype(np.float64))
    assert_bf16_close(to_np(y), orc.expert_forward(*args), "y")
    ref = orc.expert_backward(to_np(dy), *args)
    assert_bf16_close(to_np(g["dx"]), ref["dx"], "dx")
    for key in ("dw_gate", "dw_up", "dw_down", "dprobs"):
        assert_bf16_close(g[key].cpu().numpy(), ref[key], key)


def test_mxfp8_forward_backward_1024_experts_top32():
    T, H, F, E, k = 96, 128, 128, 1024, 32
    dy, x, (wg, wu, wd), ids, probs = _case(T, H, F, E, k, seed=2, mx=True)
    fq = [t for w in (wg, wu, wd) for t in m.moe_quantize_mxfp8(dev(w))]
    bq = [t for w in (wg, wu, wd) for t in m.moe_quantize_mxfp8_t(dev(w))]
    cfg = m.config(save_for_backward=True)
    y, ws = m.moe_expert_forward_mxfp8(dev(x), *fq, dev(ids), dev(probs), cfg=cfg)
    g = m.moe_expert_backward_mxfp8(dev(dy), dev(x), *bq, dev(ids), dev(probs), ws, cfg=cfg)
    assert m.moe_get_error() == 0
    ref = orc.expert_backward_mxfp8(to_np(dy), to_np(x), to_np(wg), to_np(wu), to_np(wd),
                                    ids.numpy(), probs.numpy().astype(np.float64))
    assert_rel_to_max(to_np(y), ref["y"], 3e-2, "y")
    for key in ("dx", "dw_gate_t", "dw_up_t", "dw_down_t", "dprobs"):
        assert_rel_to_max(to_np(g[key]), ref[key], 3e-2, key)


def test_backward_wait_timeout_reports_and_recovers():
    T, H, F, E, k = 200, 256, 256, 4, 2
    dy, x, (wg, wu, wd), ids, probs = _case(T, H, F, E, k, seed=3, wstd=0.02)
    a = [dev(t) for t in (x, wg, wu, wd, ids, probs)]
    y, ws = m.moe_expert_forward(*a, cfg=m.config(save_for_backward=True))
    m.moe_expert_backward(dev(dy), *a, ws, cfg=m.config(save_for_backward=True, wait_limit_ns=1))
    assert m.moe_get_error() == 5
    g = m.moe_expert_backward(dev(dy), *a, ws)          # the context is still usable
    assert m.moe_get_error() == 0
    ref = orc.expert_backward(to_np(dy), to_np(x), to_np(wg), to_np(wu), to_np(wd), ids.numpy(),
                              probs.numpy().astype(np.float64))
    assert_bf16_close(to_np(g["dx"]), ref["dx"], "dx")


def test_mxfp8_wait_timeout_reports_and_recovers():
    T, H, F, E, k = 200, 256, 256, 4, 2
    dy, x, (wg, wu, wd), ids, probs = _case(T, H, F, E, k, seed=4, mx=True)
    fq = [t for w in (wg, wu, wd) for t in m.moe_quantize_mxfp8(dev(w))]
    bq = [t for w in (wg, wu, wd) for t in m.moe_quantize_mxfp8_t(dev(w))]
    a_ids, a_p, a_x = dev(ids), dev(probs), dev(x)
    m.moe_expert_forward_mxfp8(a_x, *fq, a_ids, a_p, cfg=m.config(wait_limit_ns=1))
    assert m.moe_get_error() == 5
    save = m.config(save_for_backward=True)
    y, ws = m.moe_expert_forward_mxfp8(a_x, *fq, a_ids, a_p, cfg=save)
    assert m.moe_get_error() == 0
    m.moe_expert_backward_mxfp8(dev(dy), a_x, *bq, a_ids, a_p, ws,
                                cfg=m.config(save_for_backward=True, wait_limit_ns=1))
    assert m.moe_get_error() == 5
    g = m.moe_expert_backward_mxfp8(dev(dy), a_x, *bq, a_ids, a_p, ws, cfg=save)
    assert m.moe_get_error() == 0
    ref = orc.expert_backward_mxfp8(to_np(dy), to_np(x), to_np(wg), to_np(wu), to_np(wd),
                                    ids.numpy(), probs.numpy().astype(np.float64))
    assert_rel_to_max(to_np(y), ref["y"], 3e-2, "y")
    assert_rel_to_max(to_np(g["dx"]), ref["dx"], 3e-2, "dx")


def test_mxfp8_forward_bad_ids_reported():
    T, H, F, E, k = 64, 128, 128, 4, 2
    _, x, (wg, wu, wd), ids, probs = _case(T, H, F, E, k, seed=5, mx=True)
    ids = ids.clone()
    ids[5, 1] = 4
    ids[9, 0] = -1
    fq = [t for w in (wg, wu, wd) for t in m.moe_quantize_mxfp8(dev(w))]
    y, _ = m.moe_expert_forward_mxfp8(dev(x), *fq, dev(ids), dev(probs))
    assert m.moe_get_error() == 3
    ok = [t for t in range(T) if t not in (5, 9)]
    xq, xs = orc.quantize_mxfp8(to_np(x[ok]))
    wq = [[orc.quantize_mxfp8(to_np(w[e])) for e in range(E)] for w in (wg, wu, wd)]
    ref = orc.expert_forward_mxfp8(xq, xs, *wq, ids[ok].numpy(),
                                   probs[ok].numpy().astype(np.float64), E)
    assert_rel_to_max(to_np(y)[ok], ref, 3e-2, "y")
