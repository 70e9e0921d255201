"""The seeded generators give the workloads' structure (checked on CPU with
reduced token counts where the full size is not needed)."""
import numpy as np
import torch

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
