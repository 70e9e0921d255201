"""GPU parity of counts, offsets, permute, unpermute and the MXFP8 quantiser
against the CPU oracle: bit-exact for counts, offsets, row maps, permuted
rows and quantised codes; the BF16 tolerance for the unpermute sums."""
import numpy as np
import pytest
import torch

import oracle as orc
import synth
from gpu_util import assert_bf16_close, dev, to_np

pytestmark = pytest.mark.gpu
m = pytest.importorskip("moe_expert_dispatch_gb300")

WL = list(synth.WORKLOADS)


def _routing(name, seed=0):
    w = synth.WORKLOADS[name]
    x = synth.normal_bf16(seed, 1, (w.T, w.H)) if w.routing == "router" else None
    ids, probs = synth.routing(w, seed, x)
    return w, ids, probs


@pytest.mark.parametrize("name", WL)
def test_counts_offsets_bitexact(name):
    w, ids, _ = _routing(name)
    counts, offsets = m.moe_counts(dev(ids), w.E)
    c_ref = orc.expert_counts(ids.numpy(), w.E)
    np.testing.assert_array_equal(counts.cpu().numpy(), c_ref)
    np.testing.assert_array_equal(offsets.cpu().numpy(), orc.expert_offsets(c_ref))
    assert int(counts.sum()) == w.T * w.k


@pytest.mark.parametrize("n,E", [(1, 1), (2047, 3), (2048, 7), (2049, 7), (10000, 1024), (65, 128)])
def test_counts_shapes(n, E):
    rng = np.random.default_rng(n + E)
    ids = rng.integers(0, E, n).astype(np.int32)
    counts, offsets = m.moe_counts(dev(torch.from_numpy(ids)), E)
    c_ref = orc.expert_counts(ids, E)
    np.testing.assert_array_equal(counts.cpu().numpy(), c_ref)
    np.testing.assert_array_equal(offsets.cpu().numpy(), orc.expert_offsets(c_ref))


def test_counts_all_on_one_expert_and_reuse_workspace():
    ids = torch.full((5000,), 6, dtype=torch.int32, device="cuda")
    ws = torch.empty(m._lib.moe_counts_workspace_size(5000, 9), dtype=torch.uint8, device="cuda")
    for _ in range(2):
        counts, offsets = m.moe_counts(ids, 9, workspace=ws)
        assert counts.cpu().tolist() == [0] * 6 + [5000, 0, 0]
        assert offsets.cpu().tolist() == [0] * 7 + [5000] * 3


def test_bad_ids_reported_without_fault():
    assert m.moe_get_error() == 0
    ids = torch.tensor([0, 1, 9, -2, 1], dtype=torch.int32, device="cuda")
    counts, _ = m.moe_counts(ids, 4)
    assert m.moe_get_error() == 3
    assert counts.cpu().tolist() == [1, 2, 0, 0]
    assert m.moe_get_error() == 0      # the word is cleared by reading it


def _check_permute(w, x, ids, probs, out, align):
    row_ref, tok_ref, slot_ref = orc.permute_map(ids.numpy(), w.E)
    counts = orc.expert_counts(ids.numpy(), w.E)
    off = orc.expert_offsets(counts)
    np.testing.assert_array_equal(out["counts"].cpu().numpy(), counts)
    row_of = out["row_of"].cpu().numpy().astype(np.int64)
    if align == 1:
        np.testing.assert_array_equal(out["offsets"].cpu().numpy(), off)
        np.testing.assert_array_equal(row_of, row_ref)
        rows = np.arange(w.R)
    else:
        off_al = out["offsets"].cpu().numpy().astype(np.int64)
        assert off_al[0] == 0 and np.all(off_al % align == 0)
        assert np.all(np.diff(off_al) == (counts + align - 1) // align * align)
        # padded row -> (expert, rank) equals the dense row -> (expert, rank)
        e_of = np.searchsorted(off[1:], row_ref, side="right")
        np.testing.assert_array_equal(row_of, off_al[e_of] + (row_ref - off[e_of]))
        rows = row_of.reshape(-1)[np.argsort(row_ref.reshape(-1))]
    np.testing.assert_array_equal(out["token_of"].cpu().numpy()[rows], tok_ref)
    np.testing.assert_array_equal(out["prob_of"].cpu().numpy()[rows],
                                  probs.numpy()[tok_ref, slot_ref])
    xp = out["x_perm"].cpu()[torch.from_numpy(rows)]
    assert torch.equal(xp, x[torch.from_numpy(tok_ref)])


@pytest.mark.parametrize("name", WL)
@pytest.mark.parametrize("align", [1, 128])
def test_permute_bitexact(name, align):
    w, ids, probs = _routing(name)
    x = synth.normal_bf16(0, 1, (w.T, w.H))
    out = m.moe_permute(dev(x), dev(ids), dev(probs), w.E, row_align=align)
    _check_permute(w, x, ids, probs, out, align)


@pytest.mark.parametrize("T,k,E,H", [(1, 1, 1, 8), (37, 3, 5, 24), (300, 8, 8, 64), (5000, 2, 3, 8)])
def test_permute_edge_shapes(T, k, E, H):
    rng = np.random.default_rng(T)
    ids = torch.from_numpy(np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32))
    probs = torch.from_numpy(rng.random((T, k)).astype(np.float32))
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16)
    w = synth.Workload("edge", T, H, 128, E, k, "uniform", 0.1)
    for align in (1, 128):
        out = m.moe_permute(dev(x), dev(ids), dev(probs), E, row_align=align)
        _check_permute(w, x, ids, probs, out, align)


@pytest.mark.parametrize("k", [1, 2, 6, 8])
def test_permute_then_unpermute_unit_probs(k):
    T, E, H = 700, 16, 256
    rng = np.random.default_rng(k)
    ids = torch.from_numpy(np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32))
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16)
    out = m.moe_permute(dev(x), dev(ids), None, E)
    y = m.moe_unpermute(out["x_perm"], out["row_of"], None)
    np.testing.assert_array_equal(to_np(y), orc.bf16(k * to_np(x)))


@pytest.mark.parametrize("name", ["tiny_bf16", "mixtral_bf16", "skewed_bf16"])
def test_unpermute_vs_oracle(name):
    w, ids, probs = _routing(name)
    o = synth.normal_bf16(3, 9, (w.R, w.H))
    row_of, _, _ = orc.permute_map(ids.numpy(), w.E)
    y = m.moe_unpermute(dev(o), dev(torch.from_numpy(row_of.astype(np.int32))), dev(probs))
    ref = orc.unpermute(to_np(o), row_of, probs.numpy().astype(np.float64))
    assert_bf16_close(to_np(y), ref, "unpermute")


def test_quantize_mxfp8_bitexact():
    rng = np.random.default_rng(21)
    a = rng.standard_normal((64, 256)) * np.exp(rng.uniform(-30, 30, (64, 1)))
    a[3, :32] = 0.0                     # an all-zero block
    a[5, 32:64] = 1e-38                 # subnormal-range values
    a[7, :] = -a[7, :]
    at = torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16)
    q, s = m.moe_quantize_mxfp8(dev(at))
    q_ref, s_ref = orc.quantize_mxfp8(to_np(at))
    np.testing.assert_array_equal(s.cpu().numpy(), s_ref)
    np.testing.assert_array_equal(q.cpu().numpy(), q_ref)


@pytest.mark.parametrize("T,H,k", [(1, 32, 1), (37, 96, 3), (300, 1056, 8), (64, 4128, 32),
                                   (513, 7168, 6)])
def test_permute_quantize_mxfp8_bitexact(T, H, k):
    # the MXFP8 dispatch: every slot's row holds its token's codes, the
    # scales are per token; H spans whole and ragged passes of 32 blocks
    rng = np.random.default_rng(T + H + k)
    a = rng.standard_normal((T, H)) * np.exp(rng.uniform(-30, 30, (T, 1)))
    a[0, :32] = 0.0                     # an all-zero block
    if T > 2:
        a[2, H - 32:] = 1e-38           # subnormal-range values in the last block
    x = torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16)
    n_rows = T * k + 5
    row_of = rng.permutation(n_rows)[:T * k].reshape(T, k).astype(np.int32)
    row_of[rng.random((T, k)) < 0.1] = -1                  # dropped slots write nothing
    q, s = m.moe_permute_quantize_mxfp8(dev(x), dev(torch.from_numpy(row_of)), n_rows=n_rows)
    q_ref, s_ref = orc.quantize_mxfp8(to_np(x))
    np.testing.assert_array_equal(s.cpu().numpy(), s_ref)
    want = np.zeros((n_rows, H), np.uint8)
    for t in range(T):
        for j in range(k):
            if row_of[t, j] >= 0:
                want[row_of[t, j]] = q_ref[t]
    np.testing.assert_array_equal(q.cpu().numpy(), want)


def test_permute_quantize_mxfp8_workload_sampled():
    # the MXFP8 forward's full workload (T=16384, H=7168, k=6) with the padded
    # row map the forward uses; 64 sampled tokens checked bit for bit
    w, ids, probs = _routing("mxfp8")
    x = synth.normal_bf16(0, 1, (w.T, w.H))
    out = m.moe_permute(dev(x), dev(ids), dev(probs), w.E, row_align=128)
    cap = out["x_perm"].shape[0]
    q, s = m.moe_permute_quantize_mxfp8(dev(x), out["row_of"], n_rows=cap)
    row_of = out["row_of"].cpu().numpy()
    toks = np.random.default_rng(5).choice(w.T, 64, replace=False)
    q_ref, s_ref = orc.quantize_mxfp8(to_np(x[torch.from_numpy(toks)]))
    np.testing.assert_array_equal(s.cpu().numpy()[toks], s_ref)
    qn = q.cpu().numpy()
    for i, t in enumerate(toks):
        for j in range(w.k):
            np.testing.assert_array_equal(qn[row_of[t, j]], q_ref[i])


def test_quantize_mxfp8_weights_bitexact():
    w = synth.normal_bf16(0, 2, (4, 256, 7168), 0.02)
    q, s = m.moe_quantize_mxfp8(dev(w))
    q_ref, s_ref = orc.quantize_mxfp8(to_np(w))
    np.testing.assert_array_equal(s.cpu().numpy(), s_ref)
    np.testing.assert_array_equal(q.cpu().numpy(), q_ref)
