"""GPU parity of the backward (dX, dW1gate, dW1up, dW2, dprobs) against the
CPU oracle under |g - g_ref| <= 1e-2 + 1e-2 |g_ref|: small ragged shapes in
full, the Mixtral-shaped training workload on sampled tokens and sampled
weight-gradient columns, empty experts, accumulation and the micro-batch
split (dX, dprobs bit-identical; dW summed over chunks)."""
import numpy as np
import pytest
import torch

import oracle as orc
import synth
from gpu_util import assert_bf16_close, dev, f32_slices, to_np
from test_gpu_forward import _case

pytestmark = pytest.mark.gpu
m = pytest.importorskip("moe_expert_dispatch_gb300")


def _gpu_fwd_bwd(x, wg, wu, wd, ids, probs, dy, accumulate=False, grads=None, **cfg):
    c = m.config(save_for_backward=True, **cfg)
    y, ws = m.moe_expert_forward(dev(x), dev(wg), dev(wu), dev(wd), dev(ids), dev(probs), cfg=c)
    kw = {} if grads is None else {k: grads[k] for k in ("dw_gate", "dw_up", "dw_down")}
    g = m.moe_expert_backward(dev(dy), dev(x), dev(wg), dev(wu), dev(wd), dev(ids), dev(probs), ws,
                              accumulate_dw=accumulate, cfg=c, **kw)
    assert m.moe_get_error() == 0
    g["y"] = y
    return g


def _oracle_bwd(x, wg, wu, wd, ids, probs, dy):
    return orc.expert_backward(to_np(dy), to_np(x), to_np(wg), to_np(wu), to_np(wd), ids.numpy(),
                               probs.numpy().astype(np.float64))


# Weight scale of the elementwise checks: the workloads' (N(0, 0.01..0.02)).
WSTD = 0.02


def _compare_all(g, ref):
    assert_bf16_close(to_np(g["dx"]), ref["dx"], "dx")
    assert_bf16_close(to_np(g["dprobs"]), ref["dprobs"], "dprobs")
    for key in ("dw_gate", "dw_up", "dw_down"):
        assert_bf16_close(to_np(g[key]), ref[key], key)


@pytest.mark.parametrize("T,H,F,E,k,empty", [
    (300, 256, 384, 5, 2, (3,)),       # ragged tails, an empty expert
    (129, 128, 256, 1, 1, ()),         # one expert
    (517, 384, 640, 9, 3, (0, 8)),     # H, F not multiples of 256
    (64, 256, 512, 4, 4, ()),          # k = E
])
def test_backward_small(T, H, F, E, k, empty):
    case = _case(T, H, F, E, k, seed=T + 1, empty=empty, wstd=WSTD)
    dy = synth.normal_bf16(7, 5, (T, H))
    g = _gpu_fwd_bwd(*case, dy)
    ref = _oracle_bwd(*case, dy)
    _compare_all(g, ref)
    for e in empty:
        assert torch.all(g["dw_gate"][e] == 0) and torch.all(g["dw_down"][e] == 0)


def test_backward_large_weights_stress():
    """Weights five times the workloads' scale make dA large, so a one-ulp
    difference in where GPU (float) and oracle (float64) round an element of
    dA to bf16 moves whole dW columns by ulp(dA) * |Xp|. dX and dprobs stay
    within the elementwise bound; dW is held to a relative norm bound and
    to a small count of elements outside the elementwise one."""
    case = _case(300, 256, 384, 5, 2, seed=301, empty=(3,), wstd=0.1)
    dy = synth.normal_bf16(7, 5, (300, 256))
    g = _gpu_fwd_bwd(*case, dy)
    ref = _oracle_bwd(*case, dy)
    assert_bf16_close(to_np(g["dx"]), ref["dx"], "dx")
    assert_bf16_close(to_np(g["dprobs"]), ref["dprobs"], "dprobs")
    for key in ("dw_gate", "dw_up", "dw_down"):
        got, want = to_np(g[key]), ref[key]
        assert np.linalg.norm(got - want) <= 2e-3 * np.linalg.norm(want), key
        outside = np.abs(got - want) > 1e-2 + 1e-2 * np.abs(want)
        assert outside.mean() < 1e-4, (key, int(outside.sum()))


def test_backward_all_tokens_one_expert():
    case = _case(700, 256, 256, 16, 2, seed=5, hot=3, wstd=WSTD)
    dy = synth.normal_bf16(7, 6, (700, 256))
    _compare_all(_gpu_fwd_bwd(*case, dy), _oracle_bwd(*case, dy))


def test_backward_accumulate_and_ring_depth():
    case = _case(300, 256, 384, 5, 2, seed=8, wstd=WSTD)
    dy = synth.normal_bf16(7, 7, (300, 256))
    g1 = _gpu_fwd_bwd(*case, dy)
    g2 = _gpu_fwd_bwd(*case, dy, accumulate=True, grads={k: g1[k].clone() for k in
                                                         ("dw_gate", "dw_up", "dw_down")})
    for key in ("dw_gate", "dw_up", "dw_down"):
        assert torch.equal(g2[key], 2 * g1[key])        # x + x is exact in float
    g3 = _gpu_fwd_bwd(*case, dy, ring_stages=1, num_sms=7)
    for key in ("dx", "dprobs", "dw_gate", "dw_up", "dw_down"):
        assert torch.equal(g3[key], g1[key]), key


@pytest.mark.parametrize("splits", [4, 8])
def test_backward_microbatch_split(splits):
    T = 512
    case = _case(T, 256, 384, 8, 2, seed=13, wstd=WSTD)
    x, wg, wu, wd, ids, probs = case
    dy = synth.normal_bf16(7, 8, (T, 256))
    full = _gpu_fwd_bwd(*case, dy)
    n = T // splits
    acc = None
    dxs, dps = [], []
    for i in range(splits):
        sl = slice(i * n, (i + 1) * n)
        g = _gpu_fwd_bwd(x[sl], wg, wu, wd, ids[sl], probs[sl], dy[sl],
                         accumulate=acc is not None, grads=acc)
        acc = {k: g[k] for k in ("dw_gate", "dw_up", "dw_down")}
        dxs.append(g["dx"])
        dps.append(g["dprobs"])
    assert torch.equal(torch.cat(dxs), full["dx"])
    assert torch.equal(torch.cat(dps), full["dprobs"])
    for key in ("dw_gate", "dw_up", "dw_down"):
        assert_bf16_close(to_np(acc[key]), to_np(full[key]), key)


def test_backward_train_workload_sampled():
    w = synth.WORKLOADS["train_bf16"]
    inp = synth.make_inputs(w, 0)
    case = (inp["x"], inp["w_gate"], inp["w_up"], inp["w_down"], inp["expert_ids"], inp["probs"])
    dy = inp["dy"]
    g = _gpu_fwd_bwd(*case, dy)
    ws = [f32_slices(t) for t in case[1:4]]
    toks = np.random.default_rng(1).choice(w.T, 12, replace=False).tolist() + [0, w.T - 1]
    dx_ref, dp_ref = orc.backward_rows(to_np(dy), to_np(case[0]), *ws, case[4].numpy(),
                                       case[5].numpy(), toks)
    assert_bf16_close(to_np(g["dx"])[toks], dx_ref, "dx sampled")
    assert_bf16_close(to_np(g["dprobs"])[toks], dp_ref, "dprobs sampled")
    cols = [0, 77, 8191, w.F - 1]
    for e in (0, 5):
        ref = orc.weight_grad_columns(to_np(dy), to_np(case[0]), *ws, case[4].numpy(),
                                      case[5].numpy(), e, cols)
        for key, got in (("dw_gate", g["dw_gate"][e][:, cols]), ("dw_up", g["dw_up"][e][:, cols]),
                         ("dw_down", g["dw_down"][e][cols, :])):
            _check_reduction_over_rows(to_np(got), ref[key], f"{key}[{e}]")


def _check_reduction_over_rows(got, ref, what):
    """Weight gradients sum thousands of rows whose bf16 operands (h, dA)
    come from float32 accumulations on the GPU: a few tenths of a percent of
    them round one way on the GPU and the other way in the float64 oracle
    (measured: 0.45 % of h on this workload). Where a sum cancels heavily
    that can move it past the elementwise bound, so at full size the bound
    must hold for at least 99.9 % of the sampled elements, and every element
    must lie within the bound widened by 1e-3 * max|ref| (the scale of those
    rounding flips summed over the rows)."""
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got)), what
    inside = err <= 1e-2 + 1e-2 * np.abs(ref)
    assert inside.mean() >= 0.999, (what, int((~inside).sum()), inside.size)
    widened = err <= 1e-2 + 1e-2 * np.abs(ref) + 1e-3 * np.max(np.abs(ref))
    assert widened.all(), (what, float(err.max()))
