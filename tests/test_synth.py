"""The seeded generators give the workloads' structure (checked on CPU with
reduced token counts where the full size is not needed)."""
import numpy as np
import pytest
import torch

import oracle as orc
import synth


def test_deterministic():
    a = synth.normal_bf16(0, 7, (3, 5))
    b = synth.normal_bf16(0, 7, (3, 5))
    assert torch.equal(a, b)
    assert not torch.equal(a, synth.normal_bf16(1, 7, (3, 5)))


def test_chunked_draws_match_shape_and_moments():
    a = synth.normal_f32(3, 9, (1 << 24) + 12345, 0.02)
    assert abs(a.std() - 0.02) < 1e-4 and abs(a.mean()) < 1e-4


def _check_routing(w, ids, probs):
    ids = ids.numpy()
    probs = probs.numpy()
    assert ids.shape == (w.T, w.k) and probs.shape == (w.T, w.k)
    assert ids.min() >= 0 and ids.max() < w.E
    assert all(len(set(r)) == w.k for r in ids.tolist())       # no expert twice per token
    np.testing.assert_allclose(probs.sum(1), 1.0, rtol=1e-5)
    counts = np.bincount(ids.reshape(-1), minlength=w.E)
    assert counts.sum() == w.T * w.k
    return counts


def test_tiny_router_routing():
    w = synth.WORKLOADS["tiny_bf16"]
    inp = synth.make_inputs(w, 0)
    assert inp["x"].shape == (256, 512) and inp["w_gate"].shape == (8, 512, 1024)
    assert inp["w_down"].shape == (8, 1024, 512)
    _check_routing(w, inp["expert_ids"], inp["probs"])


def test_mixtral_routing_near_uniform():
    w = synth.WORKLOADS["mixtral_bf16"]
    ids, probs = synth.routing(w, 0)
    c = _check_routing(w, ids, probs)
    assert c.min() > 900 and c.max() < 1150


def test_skewed_routing_has_empty_experts():
    w = synth.WORKLOADS["skewed_bf16"]
    ids, probs = synth.routing(w, 0)
    c = _check_routing(w, ids, probs)
    assert np.count_nonzero(c == 0) >= synth.ZIPF_ZERO_EXPERTS
    assert c.max() > 4000            # the hot experts take most tokens


def test_uniform_dirichlet_routing():
    w = synth.WORKLOADS["mxfp8"]
    ids, probs = synth.routing(w, 0)
    c = _check_routing(w, ids, probs)
    assert c.min() > 0.8 * c.mean()


@pytest.mark.parametrize("name", ["tiny_bf16", "mixtral_bf16"])
def test_router_logits_reproduce_workload_routing(name):
    # the workloads' routing ranks float64 draws with its own top-k; the
    # oracle's gate on the same draws rounded to float32 picks the same
    # experts with the same weights (to float32 rounding)
    w = synth.WORKLOADS[name]
    inp = synth.make_inputs(w, 0)
    logits = synth.router_logits(w, 0, inp["x"])
    ids, probs, _, _ = orc.route_topk(logits.numpy(), w.k)
    assert np.array_equal(ids, inp["expert_ids"].numpy())
    np.testing.assert_allclose(probs, inp["probs"].numpy(), rtol=1e-6, atol=1e-7)
    assert synth.router_logits(synth.WORKLOADS["skewed_bf16"], 0) is None


def test_exact_inputs_quantise_exactly_to_mxfp8():
    # the MXFP8 layout of the exact-arithmetic inputs: K-contiguous weights
    # holding the BF16 layout's values, and every 32-element block of x and
    # of each weight row an exact E4M3 x E8M0 encoding (the oracle's
    # quantiser round-trips it unchanged)
    w = synth.WORKLOADS["mxfp8"].resized(T=96, H=256, F=384, E=3, k=2)
    mx = synth.exact_inputs(w, 0)
    bf = synth.exact_inputs(w.resized(mxfp8=False), 0)
    assert torch.equal(mx["x"], bf["x"]) and torch.equal(mx["expert_ids"], bf["expert_ids"])
    assert torch.equal(mx["w_gate_t"], bf["w_gate"].transpose(1, 2))
    assert torch.equal(mx["w_up_t"], bf["w_up"].transpose(1, 2))
    assert torch.equal(mx["w_down_t"], bf["w_down"].transpose(1, 2))
    assert mx["w_gate_t"].shape == (3, 384, 256) and mx["w_down_t"].shape == (3, 256, 384)
    mats = [mx["x"]] + [mx[n][e] for n in ("w_gate_t", "w_up_t", "w_down_t") for e in range(3)]
    for a in mats:
        a = a.float().numpy()
        np.testing.assert_array_equal(orc.dequantize_mxfp8(*orc.quantize_mxfp8(a)), a)
    assert mx["w_gate_t"][:, :, 0].eq(synth.EXACT_GATE_BIAS).all()
