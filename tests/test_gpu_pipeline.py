"""The micro-batch pipeline (routing of chunk c+1 and combine of chunk c on a
second stream while the GEMMs of chunk c run) gives the unsplit forward's y
bit for bit: each chunk is an independent forward and no row's arithmetic
depends on the split."""
import numpy as np
import pytest
import torch

import oracle as orc
import synth
from gpu_util import assert_bf16_close, dev, to_np

pytestmark = pytest.mark.gpu
m = pytest.importorskip("moe_expert_dispatch_gb300")


def _case(T, H, F, E, k, seed, wstd=0.05):
    g = torch.Generator().manual_seed(seed)
    bf = lambda *s, sd=1.0: (torch.randn(s, generator=g) * sd).to(torch.bfloat16)  # noqa: E731
    ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    p = torch.rand((T, k), generator=g) + 0.1
    return (bf(T, H), bf(E, H, F, sd=wstd), bf(E, H, F, sd=wstd), bf(E, F, H, sd=wstd), ids,
            (p / p.sum(1, keepdim=True)).float())


@pytest.mark.parametrize("n_chunks", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("T,H,F,E,k", [(517, 256, 384, 9, 3), (1000, 128, 256, 16, 2)])
def test_pipelined_equals_unsplit(T, H, F, E, k, n_chunks):
    case = [dev(t) for t in _case(T, H, F, E, k, seed=T + n_chunks)]
    y0, _ = m.moe_expert_forward(*case)
    y1, _ = m.moe_expert_forward_pipelined(*case, n_chunks)
    assert m.moe_get_error() == 0
    assert torch.equal(y1, y0)


def test_pipelined_matches_oracle():
    case = _case(300, 256, 384, 5, 2, seed=1)
    y, _ = m.moe_expert_forward_pipelined(*(dev(t) for t in case), 3)
    ref = orc.expert_forward(*(to_np(t) for t in case[:4]), case[4].numpy(),
                             case[5].numpy().astype(np.float64))
    assert_bf16_close(to_np(y), ref, "y")


@pytest.mark.parametrize("kw", [dict(fuse_gather=True), dict(num_sms=7), dict(ring_stages=2)])
def test_pipelined_options(kw):
    case = [dev(t) for t in _case(700, 256, 256, 6, 2, seed=2)]
    y0, _ = m.moe_expert_forward(*case)
    y1, _ = m.moe_expert_forward_pipelined(*case, 4, cfg=m.config(**kw))
    assert torch.equal(y1, y0)


def test_pipelined_more_chunks_than_tokens():
    case = [dev(t) for t in _case(5, 128, 128, 4, 2, seed=3)]
    y0, _ = m.moe_expert_forward(*case)
    y1, _ = m.moe_expert_forward_pipelined(*case, 16)   # 5 chunks of one token
    assert torch.equal(y1, y0)


def test_pipelined_in_cuda_graph():
    case = [dev(t) for t in _case(600, 256, 256, 8, 2, seed=4)]
    y0, _ = m.moe_expert_forward(*case)
    y = torch.empty_like(y0)
    ws = torch.empty(m._lib.moe_workspace_size_pipelined(600, 256, 256, 8, 2, 3),
                     dtype=torch.uint8, device="cuda")
    m.moe_expert_forward_pipelined(*case, 3, y=y, workspace=ws)    # creates the events
    torch.cuda.synchronize()
    y.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        m.moe_expert_forward_pipelined(*case, 3, y=y, workspace=ws, stream=s)
    torch.cuda.synchronize()
    assert not torch.equal(y, y0)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, y0)


def test_pipelined_mixtral_workload():
    inp = synth.make_inputs(synth.WORKLOADS["mixtral_bf16"], 0)
    case = [dev(inp[key]) for key in ("x", "w_gate", "w_up", "w_down", "expert_ids", "probs")]
    y0, _ = m.moe_expert_forward(*case)
    for n in (2, 4):
        y1, _ = m.moe_expert_forward_pipelined(*case, n)
        assert torch.equal(y1, y0), n


def test_pipelined_refusals():
    case = [dev(t) for t in _case(64, 128, 128, 4, 2, seed=5)]
    with pytest.raises(m.MoeError) as e:
        m.moe_expert_forward_pipelined(*case, 2, cfg=m.config(save_for_backward=True))
    assert e.value.status == 2
    s = torch.cuda.current_stream()
    with pytest.raises(m.MoeError) as e:
        m.moe_expert_forward_pipelined(*case, 2, stream=s, aux_stream=s)
    assert e.value.status == 1
    with pytest.raises(m.MoeError) as e:
        m.moe_expert_forward_pipelined(*case, 0)
    assert e.value.status == 1
