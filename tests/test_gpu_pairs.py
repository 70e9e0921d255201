"""CTA pairs in the BF16 grouped GEMMs over routed rows: two CTAs on two SMs
share one M = 256 tensor-core tile (tcgen05 cta_group::2), each loading its
own 128 rows of A and half of the tile's B. Every output element keeps its K
order, so results are bit-identical to one CTA per 128-row tile: at every
ring depth and grid size, with experts whose last tile is half filled, empty
experts and 128-column N tiles, in the forward (fc1, fc2) and the backward
(dH, dXp). Also: exact-arithmetic parity with the oracle, and the bounded
waits of a pair reporting a timeout without losing the context."""
import numpy as np
import pytest
import torch

import synth
from gpu_util import assert_bf16_close, dev, to_np
from test_gpu_backward import _exact_case, _gpu_fwd_bwd, _oracle_bwd
from test_gpu_forward import _case, _gpu, _oracle

pytestmark = pytest.mark.gpu
m = pytest.importorskip("moe_expert_dispatch_gb300")

SHAPES = [
    (300, 256, 384, 5, 2, (3,)),       # odd and even block counts, an empty expert
    (129, 128, 256, 1, 1, ()),         # one expert of 2 blocks: one full pair tile
    (65, 128, 128, 1, 1, ()),          # one expert of 1 block: a half-filled tile only
    (517, 384, 640, 9, 3, (0, 8)),     # H % 256 != 0: fc2 N = 128, 64 columns per CTA
    (1000, 256, 256, 16, 2, ()),
]


@pytest.mark.parametrize("T,H,F,E,k,empty", SHAPES)
def test_forward_pairs_bit_identical(T, H, F, E, k, empty):
    case = _case(T, H, F, E, k, seed=T + 11, empty=empty)
    y1 = _gpu(*case, cta_pairs=1)
    y2 = _gpu(*case, cta_pairs=2)
    assert torch.equal(y2, y1)
    assert_bf16_close(to_np(y2), _oracle(*case), "y")


def test_forward_pairs_ring_depth_and_grid():
    case = _case(700, 256, 384, 6, 2, seed=21)
    y0 = _gpu(*case, cta_pairs=1)
    for kw in (dict(ring_stages=1), dict(ring_stages=3), dict(ring_stages=6), dict(num_sms=2),
               dict(num_sms=7), dict(num_sms=33), dict(ring_stages=2, num_sms=5)):
        assert torch.equal(_gpu(*case, cta_pairs=2, **kw), y0), kw


@pytest.mark.parametrize("T,H,F,E,k,empty", SHAPES[:4])
def test_backward_pairs_bit_identical(T, H, F, E, k, empty):
    case = _case(T, H, F, E, k, seed=T + 13, empty=empty, wstd=0.02)
    dy = synth.normal_bf16(9, 1, (T, H))
    g1 = _gpu_fwd_bwd(*case, dy, cta_pairs=1)
    g2 = _gpu_fwd_bwd(*case, dy, cta_pairs=2)
    for key in ("y", "dx", "dprobs", "dw_gate", "dw_up", "dw_down"):
        assert torch.equal(g2[key], g1[key]), key


def test_backward_pairs_exact_vs_oracle():
    case, dy = _exact_case(517, 384, 640, 9, 3, seed=5, empty=(0, 8))
    g = _gpu_fwd_bwd(*case, dy, cta_pairs=2, ring_stages=5, num_sms=9)
    ref = _oracle_bwd(*case, dy)
    for key in ("y", "dx", "dprobs", "dw_gate", "dw_up", "dw_down"):
        got = to_np(g[key])
        assert np.array_equal(got, ref[key]), (key, int((got != ref[key]).sum()))


def test_pairs_wait_timeout_reports_and_recovers():
    case = _case(300, 256, 384, 5, 2, seed=3)
    y, _ = m.moe_expert_forward(*(dev(t) for t in case),
                                cfg=m.config(wait_limit_ns=1, cta_pairs=2))
    assert m.moe_get_error() == 5
    y = _gpu(*case, cta_pairs=2)   # the context is still usable and results are right
    assert_bf16_close(to_np(y), _oracle(*case), "y")


# ---------------------------------------------------------------- MXFP8

MX_SHAPES = [
    (300, 256, 512, 5, 2, (3,)),       # odd and even block counts, an empty expert
    (65, 256, 256, 1, 1, ()),          # a half-filled tile only
    (517, 512, 768, 9, 3, (0, 8)),
    (1000, 256, 256, 16, 2, ()),
]


@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("T,H,F,E,k,empty", MX_SHAPES)
def test_mxfp8_forward_pairs_bit_identical(T, H, F, E, k, empty, tile_n):
    from test_gpu_mxfp8 import TOL, _gpu as _mx_gpu, _mx_case, _oracle as _mx_oracle
    from gpu_util import assert_rel_to_max
    case = _mx_case(T, H, F, E, k, seed=T + 17, empty=empty)
    y1, _ = _mx_gpu(*case, mxfp8_tile_n=tile_n, cta_pairs=1)
    y2, _ = _mx_gpu(*case, mxfp8_tile_n=tile_n, cta_pairs=2)
    assert torch.equal(y2, y1)
    ref, _ = _mx_oracle(*case)
    assert_rel_to_max(to_np(y2), ref, TOL, "y")


@pytest.mark.parametrize("tile_n", [128, 256])
def test_mxfp8_forward_pairs_ring_depth_and_grid(tile_n):
    from test_gpu_mxfp8 import _gpu as _mx_gpu, _mx_case
    case = _mx_case(700, 256, 512, 6, 2, seed=23)
    y0, _ = _mx_gpu(*case, mxfp8_tile_n=tile_n, cta_pairs=1)
    for kw in (dict(ring_stages=1), dict(ring_stages=4), dict(ring_stages=8), dict(num_sms=2),
               dict(num_sms=9)):
        y1, _ = _mx_gpu(*case, mxfp8_tile_n=tile_n, cta_pairs=2, **kw)
        assert torch.equal(y1, y0), kw


@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("T,H,F,E,k,empty", MX_SHAPES[:3])
def test_mxfp8_backward_pairs_bit_identical(T, H, F, E, k, empty, tile_n):
    from test_gpu_mxfp8_backward import _case as _mxb_case, _gpu as _mxb_gpu
    c = _mxb_case(T, H, F, E, k, seed=T + 19, empty=empty)
    g1 = _mxb_gpu(c, mxfp8_tile_n=tile_n, cta_pairs=1)
    g2 = _mxb_gpu(c, mxfp8_tile_n=tile_n, cta_pairs=2)
    for key in ("y", "dx", "dprobs", "dw_gate_t", "dw_up_t", "dw_down_t"):
        assert torch.equal(g2[key], g1[key]), key


def test_weight_gradients_on_pairs_accumulate():
    # dW1 (M = H) and dW2 (M = F) on CTA pairs, stored then added: x + x is
    # exact in float, and both match one CTA per tile
    case = _case(300, 256, 512, 5, 2, seed=31, wstd=0.02)
    dy = synth.normal_bf16(9, 2, (300, 256))
    g1 = _gpu_fwd_bwd(*case, dy, cta_pairs=2)
    g2 = _gpu_fwd_bwd(*case, dy, accumulate=True, cta_pairs=2,
                      grads={k: g1[k].clone() for k in ("dw_gate", "dw_up", "dw_down")})
    g0 = _gpu_fwd_bwd(*case, dy, cta_pairs=1)
    for key in ("dw_gate", "dw_up", "dw_down"):
        assert torch.equal(g1[key], g0[key]), key
        assert torch.equal(g2[key], 2 * g1[key]), key
