"""GPU parity of the MXFP8 backward (every GEMM block-scaled, operands
quantised along each GEMM's reduction) against the oracle's
expert_backward_mxfp8, under max|g - g_ref| <= 3e-2 max|g_ref| per output
(the MXFP8 forward's bound: the GPU's bf16 intermediates round from float
accumulations, and a one-step bf16 flip can move an E4M3 code by a step).
The transposed quantiser is checked bit-exact against the oracle's rule."""
import numpy as np
import pytest
import torch

import oracle as orc
import synth
from gpu_util import assert_rel_to_max, dev, to_np

pytestmark = pytest.mark.gpu
m = pytest.importorskip("moe_expert_dispatch_gb300")

TOL = 3e-2


def _case(T, H, F, E, k, seed=0, empty=(), wstd=0.05):
    g = torch.Generator().manual_seed(seed)
    live = [e for e in range(E) if e not in empty]
    ids = torch.stack([torch.tensor(live)[torch.randperm(len(live), generator=g)[:k]]
                       for _ in range(T)]).to(torch.int32)
    p = torch.rand((T, k), generator=g) + 0.05
    bf = lambda *s, sd=1.0: (torch.randn(s, generator=g) * sd).to(torch.bfloat16)  # noqa: E731
    return dict(dy=bf(T, H), x=bf(T, H), wg=bf(E, F, H, sd=wstd), wu=bf(E, F, H, sd=wstd),
                wd=bf(E, H, F, sd=wstd), ids=ids, probs=(p / p.sum(1, keepdim=True)).float())


def _gpu(c, accumulate_dw=False, init=None, **cfg):
    fq = [t for w in ("wg", "wu", "wd") for t in m.moe_quantize_mxfp8(dev(c[w]))]
    bq = [t for w in ("wg", "wu", "wd") for t in m.moe_quantize_mxfp8_t(dev(c[w]))]
    ids, probs, x = dev(c["ids"]), dev(c["probs"]), dev(c["x"])
    y, ws = m.moe_expert_forward_mxfp8(x, *fq, ids, probs,
                                       cfg=m.config(save_for_backward=True, **cfg))
    kw = {} if init is None else {key: dev(v.clone()) for key, v in init.items()}
    g = m.moe_expert_backward_mxfp8(dev(c["dy"]), x, *bq, ids, probs, ws,
                                    accumulate_dw=accumulate_dw,
                                    cfg=m.config(save_for_backward=True, **cfg), **kw)
    assert m.moe_get_error() == 0
    g["y"] = y
    return g


def _oracle(c):
    return orc.expert_backward_mxfp8(to_np(c["dy"]), to_np(c["x"]), to_np(c["wg"]),
                                     to_np(c["wu"]), to_np(c["wd"]), c["ids"].numpy(),
                                     c["probs"].numpy().astype(np.float64))


KEYS = ("dx", "dw_gate_t", "dw_up_t", "dw_down_t", "dprobs", "y")


@pytest.mark.parametrize("shape", [(3, 96, 256), (2, 64, 264), (1, 32, 8), (2, 128, 392)])
def test_transposed_quantiser_bit_exact(shape):
    """Column tiles of 256 with ragged last tiles (264, 392: one or a few
    8-column chunks past the last full tile; 8: a single chunk)."""
    g = torch.Generator().manual_seed(1)
    B, R, C = shape
    w = (torch.randn(shape, generator=g) * torch.logspace(-3, 2, C)).to(torch.bfloat16)
    q, s = m.moe_quantize_mxfp8_t(dev(w))
    for z in range(B):
        rq, rs = orc.quantize_mxfp8(to_np(w[z]).T)
        assert np.array_equal(q[z].cpu().numpy(), rq)
        assert np.array_equal(s[z].cpu().numpy(), rs)


@pytest.mark.parametrize("T,H,F,E,k,empty", [
    (300, 256, 256, 5, 2, (3,)),        # ragged tails, an empty expert
    (129, 128, 128, 1, 1, ()),          # one expert, two M tiles
    (517, 256, 384, 9, 3, (0, 8)),      # F not a multiple of 256
    (64, 384, 256, 4, 4, ()),           # k = E; H not a multiple of 256
])
def test_mxfp8_backward_small(T, H, F, E, k, empty):
    c = _case(T, H, F, E, k, seed=T + E, empty=empty)
    g = _gpu(c)
    ref = _oracle(c)
    for key in KEYS:
        assert_rel_to_max(to_np(g[key]), ref[key], TOL, key)
    for e in empty:                     # an expert without rows has zero gradients
        for key in ("dw_gate_t", "dw_up_t", "dw_down_t"):
            assert torch.count_nonzero(g[key][e]) == 0


def test_mxfp8_backward_accumulates():
    c = _case(200, 256, 256, 6, 2, seed=5, empty=(1,))
    g0 = _gpu(c)
    gen = torch.Generator().manual_seed(6)
    init = {key: torch.randn(g0[key].shape, generator=gen) for key in ("dw_gate_t", "dw_up_t",
                                                                         "dw_down_t")}
    g1 = _gpu(c, accumulate_dw=True, init=init)
    for key in init:
        assert torch.allclose(g1[key].cpu(), init[key] + g0[key].cpu(), rtol=1e-6, atol=1e-6)
        assert torch.equal(g1[key][1].cpu(), init[key][1])     # the empty expert is untouched


@pytest.mark.parametrize("kw", [dict(num_sms=7), dict(ring_stages=2), dict(mxfp8_tile_n=128)])
def test_mxfp8_backward_schedule_independent(kw):
    c = _case(300, 256, 256, 5, 2, seed=7)
    g0 = _gpu(c)
    g1 = _gpu(c, **kw)
    for key in KEYS:
        assert torch.equal(g1[key], g0[key]), (key, kw)


def test_mxfp8_backward_zero_tokens():
    E, F, H = 3, 128, 128
    dw = [torch.full((E, F, H), 7.0, device="cuda") for _ in range(2)] + \
        [torch.full((E, H, F), 7.0, device="cuda")]
    st = m._lib.moe_expert_backward_mxfp8(None, None, None, None, None, None, None, None, None,
                                          None, 0, H, F, E, 2, None, 0, None,
                                          m._p(dw[0]), m._p(dw[1]), m._p(dw[2]), None, 0, None, 0,
                                          None, m._stream(None))
    assert st == 0
    torch.cuda.synchronize()
    assert all(torch.count_nonzero(t) == 0 for t in dw)


def test_mxfp8_backward_training_workload_sampled():
    """The MXFP8 training workload at full size (T=16384, E=8, k=2): dX and
    dprobs of sampled tokens that together reach all 8 experts, and whole
    weight-gradient slices of every expert (rows dW1g^T[e][f, :], dW1u^T[e][f, :]
    and columns dW2^T[e][:, f], each entry a sum over all of the expert's
    rows), against the oracle's sampled forms. Each slice set is held to
    3e-2 of its own largest oracle value."""
    from test_gpu_mxfp8 import tokens_covering_experts
    w = synth.WORKLOADS["train_mxfp8"]
    inp = synth.make_inputs(w, 0)
    c = dict(dy=inp["dy"], x=inp["x"], wg=inp["w_gate_t"], wu=inp["w_up_t"], wd=inp["w_down_t"],
             ids=inp["expert_ids"], probs=inp["probs"])
    g = _gpu(c)
    f32 = synth.F32Slices
    args = (to_np(c["dy"]), to_np(c["x"]), f32(c["wg"]), f32(c["wu"]), f32(c["wd"]),
            c["ids"].numpy(), c["probs"].numpy())
    ids = c["ids"].numpy()
    toks = tokens_covering_experts(ids, w.E, extra=(0, w.T - 1))
    assert set(ids[toks].reshape(-1).tolist()) == set(range(w.E))
    dx, dp = orc.backward_rows_mxfp8(*args, toks)
    assert_rel_to_max(to_np(g["dx"])[toks], dx, TOL, "dx sampled")
    assert_rel_to_max(g["dprobs"].cpu().numpy()[toks], dp, TOL, "dprobs sampled")
    cols = [0, 777, 5000, w.F - 1]
    for e in range(w.E):
        ref = orc.weight_grad_slices_mxfp8(*args, e, cols)
        got = {"dw_gate_t": g["dw_gate_t"][e][cols], "dw_up_t": g["dw_up_t"][e][cols],
               "dw_down_t": g["dw_down_t"][e][:, cols].T}
        for key in ref:
            assert_rel_to_max(got[key].cpu().numpy().astype(np.float64), ref[key], TOL,
                              f"{key}[{e}] slices")


@pytest.mark.parametrize("shape", [(2, 160, 384), (1, 32, 128), (3, 64, 512)])
def test_dual_quantiser_equals_both_single_ones(shape):
    g = torch.Generator().manual_seed(2)
    w = (torch.randn(shape, generator=g) * torch.logspace(-2, 2, shape[2])).to(torch.bfloat16)
    q, s, qt, st = m.moe_quantize_mxfp8_dual(dev(w))
    r = m.moe_quantize_mxfp8(dev(w))
    rt = m.moe_quantize_mxfp8_t(dev(w))
    assert torch.equal(q, r[0]) and torch.equal(s, r[1])
    assert torch.equal(qt, rt[0]) and torch.equal(st, rt[1])
    for z in range(shape[0]):           # and both against the oracle's rule
        rq, rs = orc.quantize_mxfp8(to_np(w[z]))
        assert np.array_equal(q[z].cpu().numpy(), rq) and np.array_equal(s[z].cpu().numpy(), rs)
        rq, rs = orc.quantize_mxfp8(to_np(w[z]).T)
        assert np.array_equal(qt[z].cpu().numpy(), rq) and np.array_equal(st[z].cpu().numpy(), rs)


@pytest.mark.parametrize("splits", [2, 4])
def test_mxfp8_microbatch_split(splits):
    """Micro-batches of the MXFP8 block: y, dX and dprobs are per-row
    results (every row-quantised operand and every reduction is the row's
    own), so they are bit-identical to the unsplit call. The weight
    gradients' 32-row quantisation blocks depend on which rows a chunk gives
    each expert: their sum over chunks must match the oracle's sum over the
    same chunks (3e-2 of max), and stays within the quantisation-level
    distance (0.15 of max, as the oracle's own pins) of the unsplit result."""
    T = 512
    c = _case(T, 256, 256, 6, 2, seed=40 + splits)
    g0 = _gpu(c)
    n = T // splits
    acc, ref = None, None
    for i in range(splits):
        part = {key: (v[i * n:(i + 1) * n] if key in ("dy", "x", "ids", "probs") else v)
                for key, v in c.items()}
        gi = _gpu(part)
        ri = _oracle(part)
        for key in ("y", "dx", "dprobs"):
            assert torch.equal(gi[key], g0[key][i * n:(i + 1) * n]), (key, i)
        keys = ("dw_gate_t", "dw_up_t", "dw_down_t")
        if acc is None:
            acc = {key: gi[key].cpu().numpy().astype(np.float64) for key in keys}
            ref = {key: ri[key] for key in keys}
        else:
            for key in keys:
                acc[key] += gi[key].cpu().numpy()
                ref[key] = ref[key] + ri[key]
    for key in acc:
        assert_rel_to_max(acc[key], ref[key], TOL, key + " vs the oracle per chunk")
        assert_rel_to_max(acc[key], g0[key].cpu().numpy().astype(np.float64), 0.15,
                          key + " vs unsplit")
