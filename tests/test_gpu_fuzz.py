"""Seeded fuzz over small shapes: T not a multiple of the tile, E from 1 to
128, k from 1 to 8, H and F not multiples of 256, and three routings (k
distinct random experts per token; one hot expert in every token; k = 1
with every token on one expert, so that all other experts are empty). The
inputs are exact-arithmetic ones (synth.exact_inputs), on which the GPU and
the oracle round the same real numbers at the same points, so every output
must be bit-equal: the BF16 forward and backward on one CTA per tile and on
CTA pairs, and the MXFP8 forward."""
import numpy as np
import pytest
import torch

import oracle as orc
import synth
from gpu_util import dev, to_np

pytestmark = pytest.mark.gpu
m = pytest.importorskip("moe_expert_dispatch_gb300")


def _draw(i):
    """Case i: shape, routing pattern and its expert ids, from a seeded draw."""
    rng = np.random.default_rng(7000 + i)
    E = int(rng.choice([1, 2, 3, 5, 8, 16, 128]))
    k = int(rng.integers(1, min(8, E) + 1))
    T = int(rng.integers(1, 700))
    H = int(rng.choice([128, 256, 384, 512]))
    F = int(rng.choice([128, 256, 384, 640]))
    pattern = ["random", "hot", "single"][i % 3]
    if pattern == "single" and k != 1:
        k = 1
    if pattern == "hot" and E == 1:
        pattern = "random"
    if pattern == "random":
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
    elif pattern == "hot":
        hot = int(rng.integers(E))
        others = [e for e in range(E) if e != hot]
        ids = np.stack([[hot] + list(rng.choice(others, k - 1, replace=False)) for _ in range(T)])
    else:
        ids = np.full((T, 1), int(rng.integers(E)))
    return T, H, F, E, k, pattern, torch.from_numpy(ids.astype(np.int32))


def _inputs(i, mxfp8=False):
    T, H, F, E, k, pattern, ids = _draw(i)
    w = synth.WORKLOADS["tiny_bf16"].resized(T=T, H=H, F=F, E=E, k=k, routing="gaussian",
                                             mxfp8=mxfp8)
    inp = synth.exact_inputs(w, i)
    inp["expert_ids"] = ids
    return (T, H, F, E, k, pattern), inp


def _equal(got, ref, what):
    got = to_np(got) if isinstance(got, torch.Tensor) else np.asarray(got)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    bad = int((got != ref).sum())
    assert bad == 0, f"{what}: {bad} of {got.size} not bit-equal"


@pytest.mark.parametrize("i", range(18))
def test_fuzz_bf16_forward_backward_exact(i):
    shape, inp = _inputs(i)
    x, wg, wu, wd = inp["x"], inp["w_gate"], inp["w_up"], inp["w_down"]
    ids, probs, dy = inp["expert_ids"], inp["probs"], inp["dy"]
    ref = orc.expert_backward(to_np(dy), to_np(x), to_np(wg), to_np(wu), to_np(wd), ids.numpy(),
                              probs.numpy().astype(np.float64))
    for pairs in (1, 2):
        c = m.config(save_for_backward=True, cta_pairs=pairs)
        y, ws = m.moe_expert_forward(dev(x), dev(wg), dev(wu), dev(wd), dev(ids), dev(probs),
                                     cfg=c)
        g = m.moe_expert_backward(dev(dy), dev(x), dev(wg), dev(wu), dev(wd), dev(ids),
                                  dev(probs), ws, cfg=c)
        assert m.moe_get_error() == 0
        what = f"case {i} {shape} pairs={pairs}"
        _equal(y, ref["y"], what + " y")
        for key in ("dx", "dprobs", "dw_gate", "dw_up", "dw_down"):
            _equal(g[key], ref[key], f"{what} {key}")


@pytest.mark.parametrize("i", range(9))
def test_fuzz_mxfp8_forward_exact(i):
    shape, inp = _inputs(100 + i, mxfp8=True)
    x, ids, probs = inp["x"], inp["expert_ids"], inp["probs"]
    E = shape[3]
    wq = []
    for name in ("w_gate_t", "w_up_t", "w_down_t"):
        wq += list(m.moe_quantize_mxfp8(dev(inp[name])))
    y, _ = m.moe_expert_forward_mxfp8(dev(x), *wq, dev(ids), dev(probs))
    assert m.moe_get_error() == 0
    xq, xs = orc.quantize_mxfp8(to_np(x))
    q = {n: [orc.quantize_mxfp8(to_np(inp[n][e])) for e in range(E)]
         for n in ("w_gate_t", "w_up_t", "w_down_t")}
    ref = orc.expert_forward_mxfp8(xq, xs, q["w_gate_t"], q["w_up_t"], q["w_down_t"], ids.numpy(),
                                   probs.numpy().astype(np.float64), E)
    _equal(y, ref, f"case {100 + i} {shape} mxfp8 y")
