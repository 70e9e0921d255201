"""GPU parity of the MXFP8 forward (x quantised while permuted, block-scaled
fc1 with h quantised in its epilogue, block-scaled fc2, bf16 combine)
against the CPU oracle under max|y - y_ref| <= 3e-2 max|y_ref|. The oracle
quantises its own inputs; the GPU's weight quantisation is first checked
bit-exact against it."""
import numpy as np
import pytest
import torch

import oracle as orc
import synth
from gpu_util import assert_rel_to_max, dev, to_np

pytestmark = pytest.mark.gpu
m = pytest.importorskip("moe_expert_dispatch_gb300")

TOL = 3e-2


def _mx_case(T, H, F, E, k, seed=0, empty=(), wstd=0.05):
    rng = np.random.default_rng(seed)
    live = [e for e in range(E) if e not in empty]
    ids = torch.from_numpy(np.stack([rng.choice(live, k, replace=False) for _ in range(T)]).astype(np.int32))
    ex = rng.exponential(1.0, (T, k))
    probs = torch.from_numpy((ex / ex.sum(1, keepdims=True)).astype(np.float32))
    bf = lambda shape, s: torch.from_numpy((rng.standard_normal(shape) * s).astype(np.float32)).to(torch.bfloat16)  # noqa: E731
    return bf((T, H), 1.0), bf((E, F, H), wstd), bf((E, F, H), wstd), bf((E, H, F), wstd), ids, probs


def _gpu_weights(wg, wu, wd):
    out = []
    for w in (wg, wu, wd):
        q, s = m.moe_quantize_mxfp8(dev(w))
        out += [q, s]
    return out


def _gpu(x, wg, wu, wd, ids, probs, **cfg):
    wq = _gpu_weights(wg, wu, wd)
    y, _ = m.moe_expert_forward_mxfp8(dev(x), *wq, dev(ids), dev(probs), cfg=m.config(**cfg))
    assert m.moe_get_error() == 0
    return y, wq


def _oracle(x, wg, wu, wd, ids, probs):
    E = wg.shape[0]
    xq, xs = orc.quantize_mxfp8(to_np(x))
    qg = [orc.quantize_mxfp8(to_np(wg[e])) for e in range(E)]
    qu = [orc.quantize_mxfp8(to_np(wu[e])) for e in range(E)]
    qd = [orc.quantize_mxfp8(to_np(wd[e])) for e in range(E)]
    return orc.expert_forward_mxfp8(xq, xs, qg, qu, qd, ids.numpy(), probs.numpy().astype(np.float64), E), (qg, qu, qd)


@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("T,H,F,E,k,empty", [
    (300, 256, 384, 5, 2, (3,)),       # ragged tails, an empty expert
    (129, 256, 128, 1, 1, ()),         # one expert
    (517, 512, 640, 9, 3, (0, 8)),     # F not a multiple of 256
    (64, 512, 256, 4, 4, ()),          # k = E
])
def test_mxfp8_forward_small(T, H, F, E, k, empty, tile_n):
    case = _mx_case(T, H, F, E, k, seed=T, empty=empty)
    y, wq = _gpu(*case, mxfp8_tile_n=tile_n)
    ref, (qg, qu, qd) = _oracle(*case)
    for e in range(E):       # the GPU's weight codes and scales are the oracle's
        assert np.array_equal(wq[0][e].cpu().numpy(), qg[e][0])
        assert np.array_equal(wq[1][e].cpu().numpy(), qg[e][1])
        assert np.array_equal(wq[4][e].cpu().numpy(), qd[e][0])
    assert_rel_to_max(to_np(y), ref, TOL, "y")


def test_mxfp8_h_not_multiple_of_256_uses_128_tiles():
    case = _mx_case(300, 384, 256, 4, 2, seed=8)
    y, _ = _gpu(*case)
    ref, _ = _oracle(*case)
    assert_rel_to_max(to_np(y), ref, TOL, "y")


@pytest.mark.parametrize("tile_n", [128, 256])
def test_mxfp8_schedule_independent(tile_n):
    case = _mx_case(400, 256, 384, 6, 2, seed=4)
    y0, _ = _gpu(*case, mxfp8_tile_n=tile_n)
    for kw in (dict(ring_stages=1), dict(num_sms=5), dict(ring_stages=2, num_sms=17)):
        y1, _ = _gpu(*case, mxfp8_tile_n=tile_n, **kw)
        assert torch.equal(y1, y0), kw


def test_mxfp8_tile_widths_agree():
    # both tile widths run the same per-row reduction order over K
    case = _mx_case(300, 512, 384, 5, 2, seed=11)
    y128, _ = _gpu(*case, mxfp8_tile_n=128)
    y256, _ = _gpu(*case, mxfp8_tile_n=256)
    assert torch.equal(y128, y256)


def tokens_covering_experts(ids, E, extra=(), seed=0):
    """Tokens, in a seeded random order, taken while they route to an expert
    that no earlier pick reaches, until every expert with a token is reached;
    then `extra`."""
    order = np.random.default_rng(seed).permutation(ids.shape[0])
    seen, toks = set(), []
    for t in order:
        new = set(int(e) for e in ids[t]) - seen
        if new:
            toks.append(int(t))
            seen |= new
        if len(seen) == E:
            break
    return sorted(set(toks) | set(extra))


def test_mxfp8_workload_sampled():
    """The MXFP8 workload at full size (T=16384, H=7168, F=2048, E=64, k=6)
    on sampled tokens that together reach all 64 experts, so that every
    expert's fc1 and fc2 tiles are compared with the oracle."""
    w = synth.WORKLOADS["mxfp8"]
    inp = synth.make_inputs(w, 0)
    x, wg, wu, wd = inp["x"], inp["w_gate_t"], inp["w_up_t"], inp["w_down_t"]
    ids, probs = inp["expert_ids"], inp["probs"]
    y, _ = _gpu(x, wg, wu, wd, ids, probs)
    y = to_np(y)
    toks = tokens_covering_experts(ids.numpy(), w.E, extra=(0, 7777, w.T - 1))
    assert set(ids.numpy()[toks].reshape(-1).tolist()) == set(range(w.E))
    f32 = lambda t: synth.F32Slices(t)  # noqa: E731
    ref = orc.sampled_forward_mxfp8(to_np(x), f32(wg), f32(wu), f32(wd), ids.numpy(), probs.numpy(), toks)
    print(f"{len(toks)} tokens reach all {w.E} experts; max err / max|ref| = "
          f"{np.abs(y[toks] - ref).max() / np.abs(ref).max():.3e}")
    assert_rel_to_max(y[toks], ref, TOL, "y sampled")
    assert np.all(np.isfinite(y))


def test_mxfp8_workload_exact_arithmetic_bit_equal():
    """The MXFP8 workload at full size on exact-arithmetic inputs
    (synth.exact_inputs: small integers that quantise to E4M3 x E8M0 exactly,
    a gate pre-activation of at least 40 so that silu is the identity in
    float32 and float64, dyadic routing weights). Every product and partial
    sum is then exact on both sides, which round the same real numbers at
    the same points: h to bf16, h to its E4M3 codes and E8M0 scales, O and y
    to bf16. Sampled tokens that reach all 64 experts must be bit-equal."""
    w = synth.WORKLOADS["mxfp8"]
    inp = synth.exact_inputs(w, 0)
    x, wg, wu, wd = inp["x"], inp["w_gate_t"], inp["w_up_t"], inp["w_down_t"]
    ids, probs = inp["expert_ids"], inp["probs"]
    y, _ = _gpu(x, wg, wu, wd, ids, probs)
    y = to_np(y)
    rng = np.random.default_rng(1)
    toks = tokens_covering_experts(ids.numpy(), w.E,
                                   extra=tuple(rng.choice(w.T, 40, replace=False).tolist()))
    assert set(ids.numpy()[toks].reshape(-1).tolist()) == set(range(w.E))
    f32 = lambda t: synth.F32Slices(t)  # noqa: E731
    ref = orc.sampled_forward_mxfp8(to_np(x), f32(wg), f32(wu), f32(wd), ids.numpy(), probs.numpy(), toks)
    assert np.abs(ref).max() > 256          # past bf16's exact integers: rounding is exercised
    diff = int((y[toks] != ref).sum())
    print(f"{len(toks)} tokens reach all {w.E} experts; {diff} of {ref.size} outputs differ")
    assert diff == 0


def test_mxfp8_workload_microbatch_splits_full_size():
    """The MXFP8 workload at full size split into 2, 4 and 8 contiguous token
    chunks, each chunk a call of its own: the concatenated y equals the
    unsplit call's y bit for bit (x is quantised per token, so a chunk's
    codes and scales are the unsplit call's rows)."""
    w = synth.WORKLOADS["mxfp8"]
    inp = synth.make_inputs(w, 0)
    wq = _gpu_weights(inp["w_gate_t"], inp["w_up_t"], inp["w_down_t"])
    x, ids, probs = dev(inp["x"]), dev(inp["expert_ids"]), dev(inp["probs"])
    y, _ = m.moe_expert_forward_mxfp8(x, *wq, ids, probs)
    for splits in (2, 4, 8):
        n = w.T // splits
        parts = [m.moe_expert_forward_mxfp8(x[i * n:(i + 1) * n], *wq, ids[i * n:(i + 1) * n],
                                            probs[i * n:(i + 1) * n])[0] for i in range(splits)]
        assert torch.equal(torch.cat(parts), y), splits
    assert m.moe_get_error() == 0


def _with_nonfinite(shape, seed):
    """N(0,1) bf16 values with about one element in 400 replaced by +inf,
    -inf or NaN."""
    g = torch.Generator().manual_seed(seed)
    a = torch.randn(shape, generator=g)
    flat = a.view(-1)
    idx = torch.randperm(flat.numel(), generator=g)[:max(3, flat.numel() // 400)]
    special = torch.tensor([float("inf"), float("-inf"), float("nan")])
    flat[idx] = special[torch.arange(idx.numel()) % 3]
    return a.to(torch.bfloat16)


def test_quantisers_nonfinite_blocks_bit_exact():
    """Blocks holding an infinity or a NaN: every quantiser (along the rows,
    along the columns, both at once, and fused with the permute) writes the
    E8M0 NaN scale and E4M3 NaN codes for them, and the oracle's codes and
    scales elsewhere, bit for bit."""
    a = _with_nonfinite((3, 96, 256), 3)
    ref_rows = [orc.quantize_mxfp8(to_np(a[z])) for z in range(3)]
    ref_cols = [orc.quantize_mxfp8(to_np(a[z]).T) for z in range(3)]
    assert any((s == 255).any() for _, s in ref_rows)
    q, s = m.moe_quantize_mxfp8(dev(a))
    qt, st = m.moe_quantize_mxfp8_t(dev(a))
    dq, ds, dqt, dst = m.moe_quantize_mxfp8_dual(dev(a))
    for z in range(3):
        for got, want in ((q[z], ref_rows[z][0]), (s[z], ref_rows[z][1]), (dq[z], ref_rows[z][0]),
                          (ds[z], ref_rows[z][1]), (qt[z], ref_cols[z][0]),
                          (st[z], ref_cols[z][1]), (dqt[z], ref_cols[z][0]),
                          (dst[z], ref_cols[z][1])):
            assert np.array_equal(got.cpu().numpy(), want)
    x = a[0]                                     # [96, 256] as tokens
    T, k = x.shape[0], 2
    row_of = torch.arange(T * k, dtype=torch.int32).reshape(T, k).flip(0).contiguous()
    pq, ps = m.moe_permute_quantize_mxfp8(dev(x), dev(row_of))
    rq, rs = ref_rows[0]
    assert np.array_equal(ps.cpu().numpy(), rs)
    pq = pq.cpu().numpy()
    for t in range(T):
        for j in range(k):
            assert np.array_equal(pq[row_of[t, j]], rq[t]), (t, j)


@pytest.mark.parametrize("tile_n,pairs", [(128, 1), (256, 1), (256, 2), (128, 2)])
def test_mxfp8_forward_pretiled_scales_bit_identical(tile_n, pairs):
    """The weights' scales tiled once (moe_tile_weight_scales_mxfp8) and handed
    to the forward with mx_scales_pretiled give its output bit for bit."""
    case = _mx_case(300, 256, 384, 5, 2, seed=21, empty=(3,))
    y0, wq = _gpu(*case, mxfp8_tile_n=tile_n, cta_pairs=pairs)
    x, _, _, _, ids, probs = case
    wgu_t, wd_t = m.moe_tile_weight_scales_mxfp8(wq[1], wq[3], wq[5],
                                                  cfg=m.config(mxfp8_tile_n=tile_n))
    cfg = m.config(mxfp8_tile_n=tile_n, cta_pairs=pairs, mx_scales_pretiled=True)
    y1, _ = m.moe_expert_forward_mxfp8(dev(x), wq[0], wgu_t, wq[2], None, wq[4], wd_t, dev(ids),
                                       dev(probs), cfg=cfg)
    assert m.moe_get_error() == 0
    assert torch.equal(y0, y1)


def test_mxfp8_pretiled_scales_rejects_unaligned_buffers():
    case = _mx_case(64, 256, 256, 2, 1, seed=5)
    _, wq = _gpu(*case)
    wgu_t, wd_t = m.moe_tile_weight_scales_mxfp8(wq[1], wq[3], wq[5])
    x, _, _, _, ids, probs = case
    cfg = m.config(mx_scales_pretiled=True)
    shifted = torch.empty(wgu_t.numel() + 16, dtype=torch.uint8, device=wgu_t.device)[4:4 + wgu_t.numel()]
    shifted.copy_(wgu_t)
    with pytest.raises(m.MoeError):
        m.moe_expert_forward_mxfp8(dev(x), wq[0], shifted, wq[2], None, wq[4], wd_t, dev(ids),
                                   dev(probs), cfg=cfg)
