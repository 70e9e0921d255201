"""GPU parity of the fused gate (top-k + softmax + counts + offsets in one
kernel) against the oracle's route_topk: expert ids, counts and offsets
bit-exact, weights within a relative 1e-5 (float softmax against float64;
the float32 subtraction l_j - l_0 and expf add a few units in the last
place, under 1e-6 relative for logits of magnitude below 16). Also the
forward with the gate fused in front, which must equal the forward on the
ids and weights the gate wrote, bit for bit."""
import numpy as np
import pytest
import torch

import oracle as orc
import synth
from gpu_util import assert_bf16_close, dev, to_np

pytestmark = pytest.mark.gpu
m = pytest.importorskip("moe_expert_dispatch_gb300")

RTOL, ATOL = 1e-5, 1e-7


def _check(logits, k, ids, probs, counts, offsets, finite_rows=None):
    ref_ids, ref_p, ref_c, ref_o = orc.route_topk(logits.numpy(), k)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    assert np.array_equal(counts.cpu().numpy(), ref_c)
    assert np.array_equal(offsets.cpu().numpy(), ref_o)
    p = probs.cpu().numpy().astype(np.float64)
    rows = slice(None) if finite_rows is None else finite_rows
    np.testing.assert_allclose(p[rows], ref_p[rows], rtol=RTOL, atol=ATOL)


@pytest.mark.parametrize("T,E,k", [
    (1, 1, 1), (37, 8, 2), (1000, 128, 8), (513, 64, 6), (300, 1024, 32), (100, 33, 5),
    (2000, 200, 1), (4097, 16, 16), (50, 32, 32), (700, 500, 3),
])
def test_route_topk_random(T, E, k):
    g = torch.Generator().manual_seed(T * 131 + E)
    logits = (torch.randn((T, E), generator=g) * 3.0).float()
    out = m.moe_route_topk(dev(logits), k)
    _check(logits, k, *out)


def test_route_topk_ties_signed_zeros_inf_nan():
    # logits from a small pool: ties everywhere, -0.0 next to +0.0, -inf and NaN
    rng = np.random.default_rng(5)
    pool = np.array([-0.0, 0.0, 1.0, -1.0, 2.5, -np.inf, np.nan, 0.5], dtype=np.float32)
    for E, k in ((7, 3), (40, 8), (130, 16), (5, 5)):
        logits = torch.from_numpy(pool[rng.integers(0, pool.size, (500, E))])
        out = m.moe_route_topk(dev(logits), k)
        ref_ids, ref_p, _, _ = orc.route_topk(logits.numpy(), k)
        finite = np.isfinite(np.take_along_axis(logits.numpy(), ref_ids[:, :1].astype(np.int64), 1)[:, 0])
        _check(logits, k, *out, finite_rows=finite)


def test_route_topk_equal_logits_take_lowest_indices():
    logits = torch.full((64, 24), 0.75)
    ids, probs, counts, offsets = m.moe_route_topk(dev(logits), 6)
    assert ids.cpu().tolist() == [list(range(6))] * 64
    assert torch.all(probs.cpu() == 1.0 / 6.0)


def test_route_topk_zero_tokens_and_reused_workspace():
    E, k = 12, 3
    ids, probs, counts, offsets = m.moe_route_topk(dev(torch.zeros((0, E))), k)
    assert counts.cpu().tolist() == [0] * E and offsets.cpu().tolist() == [0] * (E + 1)
    ws = torch.empty(m._lib.moe_route_topk_workspace_size(5000, k, E), dtype=torch.uint8,
                     device="cuda")
    for T in (5000, 17, 5000, 1):                 # the scratch is cleared by every call
        logits = torch.randn((T, E), generator=torch.Generator().manual_seed(T))
        _check(logits, k, *m.moe_route_topk(dev(logits), k, workspace=ws))


def test_route_topk_rejects_bad_arguments():
    with pytest.raises(m.MoeError) as e:
        m.moe_route_topk(dev(torch.zeros((4, 3))), 4)           # k > E
    assert e.value.status == 1
    with pytest.raises(m.MoeError) as e:
        m.moe_route_topk(dev(torch.zeros((4, 3))), 2,
                         workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 4


@pytest.mark.parametrize("name", ["tiny_bf16", "mixtral_bf16", "train_bf16"])
def test_route_topk_workload_logits(name):
    w = synth.WORKLOADS[name]
    x = synth.make_inputs(w, 0)["x"] if w.routing == "router" else None
    logits = synth.router_logits(w, 0, x)
    _check(logits, w.k, *m.moe_route_topk(dev(logits), w.k))


def _block(T, H, F, E, k, seed, wstd=0.05):
    g = torch.Generator().manual_seed(seed)
    bf = lambda *s, sd=1.0: (torch.randn(s, generator=g) * sd).to(torch.bfloat16)  # noqa: E731
    return (bf(T, H), bf(E, H, F, sd=wstd), bf(E, H, F, sd=wstd), bf(E, F, H, sd=wstd),
            torch.randn((T, E), generator=g).float())


@pytest.mark.parametrize("T,H,F,E,k", [
    (300, 256, 384, 5, 2),
    (1000, 256, 256, 16, 6),          # 6000 ids: slots straddle the 2048-id chunks
    (129, 128, 128, 1, 1),
    (2500, 128, 256, 64, 8),
])
def test_forward_from_logits(T, H, F, E, k):
    x, wg, wu, wd, logits = _block(T, H, F, E, k, seed=T + E)
    y, ids, probs, _ = m.moe_expert_forward_from_logits(dev(x), dev(wg), dev(wu), dev(wd),
                                                        dev(logits), k)
    assert m.moe_get_error() == 0
    ids_r, probs_r, _, _ = m.moe_route_topk(dev(logits), k)
    assert torch.equal(ids, ids_r) and torch.equal(probs, probs_r)
    y2, _ = m.moe_expert_forward(dev(x), dev(wg), dev(wu), dev(wd), ids, probs)
    assert torch.equal(y, y2)
    ref = orc.expert_forward(to_np(x), to_np(wg), to_np(wu), to_np(wd), ids.cpu().numpy(),
                             probs.cpu().numpy().astype(np.float64))
    assert_bf16_close(to_np(y), ref, "y")
    assert np.array_equal(ids.cpu().numpy(), orc.route_topk(logits.numpy(), k)[0])


def test_forward_from_logits_saves_for_backward():
    T, H, F, E, k = 400, 256, 256, 8, 2
    x, wg, wu, wd, logits = _block(T, H, F, E, k, seed=3, wstd=0.02)
    cfg = m.config(save_for_backward=True)
    y, ids, probs, ws = m.moe_expert_forward_from_logits(dev(x), dev(wg), dev(wu), dev(wd),
                                                         dev(logits), k, cfg=cfg)
    y2, ws2 = m.moe_expert_forward(dev(x), dev(wg), dev(wu), dev(wd), ids, probs, cfg=cfg)
    assert torch.equal(y, y2)
    dy = dev(torch.randn((T, H), generator=torch.Generator().manual_seed(4)).to(torch.bfloat16))
    g1 = m.moe_expert_backward(dy, dev(x), dev(wg), dev(wu), dev(wd), ids, probs, ws)
    g2 = m.moe_expert_backward(dy, dev(x), dev(wg), dev(wu), dev(wd), ids, probs, ws2)
    assert m.moe_get_error() == 0
    for key in g1:
        assert torch.equal(g1[key], g2[key]), key
