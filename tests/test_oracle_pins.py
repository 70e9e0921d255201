"""Pins of the CPU oracle against things other than itself: library
rounding routines, closed forms, a hand-worked example, pure-Python brute
force, torch float64 references and finite differences.

Each test is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign, index or transposition, a wrong rounding point) fails one of them.
"""
import collections
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_case(T=37, H=64, F=96, E=5, k=2, seed=1, empty=(3,), wstd=0.15):
    rng = np.random.default_rng(seed)
    x = orc.bf16(rng.standard_normal((T, H)))
    live = [e for e in range(E) if e not in empty]
    ids = np.stack([rng.choice(live, size=k, replace=False) for _ in range(T)]).astype(np.int64)
    logits = rng.standard_normal((T, k))
    probs = (np.exp(logits) / np.exp(logits).sum(1, keepdims=True)).astype(np.float32).astype(np.float64)
    wg = orc.bf16(rng.standard_normal((E, H, F)) * wstd)
    wu = orc.bf16(rng.standard_normal((E, H, F)) * wstd)
    wd = orc.bf16(rng.standard_normal((E, F, H)) * wstd)
    return x, wg, wu, wd, ids, probs


# ---------------------------------------------------------------- rounding

def test_bf16_matches_torch_rne():
    rng = np.random.default_rng(0)
    # float32 values over a wide exponent range, plus exact ties and subnormals
    mant = rng.integers(0, 1 << 23, 20000)
    expo = rng.integers(1, 254, 20000)
    sign = rng.integers(0, 2, 20000)
    bits = (sign << 31) | (expo << 23) | mant
    vals = bits.astype(np.uint32).view(np.float32)
    ties = (np.arange(1, 4000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    subn = (rng.integers(1, 1 << 23, 2000).astype(np.uint32)).view(np.float32)
    for v in (vals, ties, subn, -ties):
        want = torch.from_numpy(v.copy()).to(torch.bfloat16).float().numpy().astype(np.float64)
        got = orc.bf16(v.astype(np.float64))
        np.testing.assert_array_equal(got, want)


def test_bf16_overflow_and_zero():
    assert orc.bf16(0.0) == 0.0
    assert np.isinf(orc.bf16(3.5e38))
    assert orc.bf16(float.fromhex("0x1.fep127")) == float.fromhex("0x1.fep127")


def test_e4m3_decode_all_codes_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    got = orc.e4m3_decode(codes)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], want[~nan])
    assert got[0x7E] == 448.0 and got[0x08] == 2.0 ** -6 and got[0x01] == 2.0 ** -9


def test_e4m3_encode_vs_torch():
    rng = np.random.default_rng(3)
    vals = np.concatenate([
        rng.uniform(-448, 448, 20000),
        rng.standard_normal(20000) * 0.01,
        rng.standard_normal(5000) * 2.0 ** -8,
    ]).astype(np.float32)
    # exact midpoints between neighbouring codes (ties to even)
    pos = orc.e4m3_decode(np.arange(0, 0x7F))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    vals = np.concatenate([vals, mids, -mids])
    want = torch.from_numpy(vals.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = orc.e4m3_encode(vals.astype(np.float64))
    np.testing.assert_array_equal(got, want)


def test_e4m3_satfinite():
    got = orc.e4m3_encode(np.array([448.0, 463.9, 464.0, 480.0, 1e6, -1e6]))
    np.testing.assert_array_equal(got, [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE])


def test_e8m0_scale_closed_forms():
    # X = 2^(floor(log2 amax) - 8), code = exponent + 127
    cases = {1.0: 119, 1.5: 119, 2.0: 120, 448.0: 127, 511.0: 127, 2.0 ** -10: 109, 0.0: 0,
             2.0 ** 140: 254, 2.0 ** -140: 0}
    for amax, code in cases.items():
        assert int(orc.e8m0_scale_code(amax)) == code, amax


def test_mxfp8_nonfinite_blocks():
    # a block holding an infinity or a NaN has no finite shared exponent:
    # scale code 255 (the E8M0 NaN) and E4M3 NaN elements, so that IEEE
    # arithmetic with the scale makes every element of the block NaN; the
    # other blocks of the row are quantised as if alone
    rng = np.random.default_rng(5)
    a = orc.bf16(rng.standard_normal((3, 96)))
    a[0, 5], a[1, 40], a[2, 70], a[2, 71] = np.inf, np.nan, -np.inf, np.nan
    q, s = orc.quantize_mxfp8(a)
    bad = {(0, 0), (1, 1), (2, 2)}
    for r in range(3):
        for b in range(3):
            blk = slice(32 * b, 32 * b + 32)
            if (r, b) in bad:
                assert s[r, b] == 255 and np.all(q[r, blk] == 0x7F)
            else:
                q1, s1 = orc.quantize_mxfp8(a[r:r + 1, blk])
                assert s[r, b] == s1[0, 0] and np.array_equal(q[r, blk], q1[0])
    # 0x7F is a NaN of E4M3 (torch's float8_e4m3fn agrees) and 255 of E8M0
    assert torch.tensor([0x7F], dtype=torch.uint8).view(torch.float8_e4m3fn).float().isnan().all()
    d = orc.dequantize_mxfp8(q, s)
    for r in range(3):
        for b in range(3):
            blk = d[r, 32 * b:32 * b + 32]
            assert np.all(np.isnan(blk)) if (r, b) in bad else np.all(np.isfinite(blk))
    assert list(orc.e8m0_scale_code(np.array([np.inf, np.nan, 448.0]))) == [255, 255, 127]


def test_mxfp8_power_of_two_blocks_are_exact():
    rng = np.random.default_rng(5)
    ex = rng.integers(-20, 20, (4, 64))
    sgn = rng.choice([-1.0, 1.0], (4, 64))
    a = sgn * np.ldexp(1.0, ex)
    # within a block every value must lie within 2^-9..2^8 of the block max
    a = np.clip(a, None, None)
    blocks = a.reshape(4, 2, 32)
    m = np.abs(blocks).max(-1, keepdims=True)
    blocks = np.where(np.abs(blocks) < m * 2.0 ** -14, np.sign(blocks) * m * 2.0 ** -14, blocks)
    a = blocks.reshape(4, 64)
    q, s = orc.quantize_mxfp8(a)
    np.testing.assert_array_equal(orc.dequantize_mxfp8(q, s), a)


def test_mxfp8_block_max_lands_in_top_binade():
    rng = np.random.default_rng(6)
    a = orc.bf16(rng.standard_normal((8, 128)) * 3.0)
    q, s = orc.quantize_mxfp8(a)
    vals = orc.e4m3_decode(q).reshape(8, 4, 32)
    top = np.abs(vals).max(-1)
    assert np.all((top >= 256) & (top <= 448))
    err = np.abs(orc.dequantize_mxfp8(q, s) - a).reshape(8, 4, 32)
    scale = np.ldexp(1.0, s.astype(int) - 127)[..., None]
    scaled = np.abs(a).reshape(8, 4, 32) / scale
    # round to nearest: at most half an E4M3 ulp (2^5 at the top binade) in
    # scaled units; beyond 448 the floor-based scale makes satfinite clamp
    bound = np.maximum(16.0, scaled - 448.0) * scale
    assert np.all(err <= bound)


# ---------------------------------------------------------------- counts / permute

def test_counts_bruteforce():
    rng = np.random.default_rng(7)
    ids = rng.integers(0, 13, (211, 3))
    c = collections.Counter(ids.reshape(-1).tolist())
    got = orc.expert_counts(ids, 13)
    assert got.tolist() == [c.get(e, 0) for e in range(13)]
    assert got.sum() == ids.size
    off = orc.expert_offsets(got)
    assert off[0] == 0 and off[-1] == ids.size and np.all(np.diff(off) == got)


def test_counts_rejects_out_of_range():
    with pytest.raises(ValueError):
        orc.expert_counts(np.array([[0, 5]]), 5)
    with pytest.raises(ValueError):
        orc.expert_counts(np.array([[-1, 0]]), 5)


def test_permute_matches_stable_sort():
    rng = np.random.default_rng(8)
    T, k, E = 173, 4, 9
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
    row_of, token_of, slot_of = orc.permute_map(ids, E)
    order = sorted(range(T * k), key=lambda i: (ids.reshape(-1)[i], i))   # Python's sort is stable
    for r, i in enumerate(order):
        assert token_of[r] == i // k and slot_of[r] == i % k
        assert row_of.reshape(-1)[i] == r


def test_permute_rows_carry_token_and_prob():
    x, wg, wu, wd, ids, probs = _rand_case()
    xp, row_of, token_of, prob_of = orc.permute(x, ids, probs, 5)
    for t in range(x.shape[0]):
        for j in range(ids.shape[1]):
            r = row_of[t, j]
            assert np.array_equal(xp[r], x[t]) and prob_of[r] == probs[t, j]


def test_unpermute_unit_probs_gives_k_times_x():
    rng = np.random.default_rng(9)
    for k in (1, 2, 4, 6, 8):
        T, E = 50, 8
        x = orc.bf16(rng.standard_normal((T, 24)))
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
        xp, row_of, _, _ = orc.permute(x, ids, None, E)
        y = orc.unpermute(xp, row_of, None)
        np.testing.assert_array_equal(y, orc.bf16(k * x))
        if k in (1, 2, 4, 8):
            np.testing.assert_array_equal(y, k * x)


# ---------------------------------------------------------------- forward

def test_worked_example_golden():
    g = json.load(open(os.path.join(GOLDEN, "tiny_worked_example.json")))
    y, st = orc.expert_forward(np.array(g["x"]), np.array(g["w_gate"]), np.array(g["w_up"]),
                               np.array(g["w_down"]), np.array(g["expert_ids"]),
                               np.array(g["probs"]), keep=True)
    np.testing.assert_array_equal(y, np.array(g["y"]))
    np.testing.assert_array_equal(st["h"][st["row_of"][0, 0]], g["h_expert0"])


def test_mxfp8_worked_example_golden():
    g = json.load(open(os.path.join(GOLDEN, "mxfp8_worked_example.json")))
    inp = g["inputs"]
    H, F, E = inp["H"], inp["F"], inp["E"]
    ids, probs = np.array(inp["ids"]), np.array(inp["probs"])
    x = np.zeros((len(ids), H))
    for t, c, v in inp["x_nonzero"]:
        x[t, c] = v

    def ones(shape, where):
        a = np.zeros(shape)
        for e, r, c in where:
            a[e, r, c] = 1.0
        return a
    wg = ones((E, F, H), inp["w_gate_t_ones"])
    wu = ones((E, F, H), inp["w_up_t_ones"])
    wd = ones((E, H, F), inp["w_down_t_ones"])
    want = np.zeros_like(x)
    for t, c, v in g["expected"]["y_nonzero"]:
        want[t, c] = v
    np.testing.assert_array_equal(_mx_fwd(x, wg, wu, wd, ids, probs), want)
    xq, xs = orc.quantize_mxfp8(x)
    q = [[orc.quantize_mxfp8(w[e]) for e in range(E)] for w in (wg, wu, wd)]
    np.testing.assert_array_equal(orc.token_forward_mxfp8(xq[0], xs[0], *q, ids[0], probs[0]),
                                  want[0])
    hq, hs = orc.quantize_mxfp8(np.array([[g["expected"]["h_bf16_0"]] + [0.0] * (F - 1)]))
    assert orc.dequantize_mxfp8(hq, hs)[0, 0] == g["expected"]["h_dequantised_0"]


def test_grouped_equals_per_token_dense():
    x, wg, wu, wd, ids, probs = _rand_case()
    y1 = orc.expert_forward(x, wg, wu, wd, ids, probs)
    y2 = orc.dense_forward(x, wg, wu, wd, ids, probs)
    # same dot products in float64; only BLAS summation order can differ, which
    # can move a bf16 rounding by one step in rare elements
    np.testing.assert_allclose(y1, y2, rtol=2 ** -7, atol=1e-6)
    assert np.mean(y1 == y2) > 0.999


def test_forward_pure_python_bruteforce():
    rng = np.random.default_rng(11)
    T, H, F, E, k = 4, 6, 5, 3, 2
    x = rng.standard_normal((T, H))
    wg, wu = rng.standard_normal((E, H, F)), rng.standard_normal((E, H, F))
    wd = rng.standard_normal((E, F, H))
    ids = np.array([[0, 2], [1, 0], [2, 1], [0, 1]])
    probs = rng.uniform(0.1, 1.0, (T, k))
    want = [[0.0] * H for _ in range(T)]
    for t in range(T):
        for j in range(k):
            e = ids[t][j]
            h = []
            for f in range(F):
                g = sum(x[t][i] * wg[e][i][f] for i in range(H))
                u = sum(x[t][i] * wu[e][i][f] for i in range(H))
                h.append(g / (1.0 + math.exp(-g)) * u)
            for c in range(H):
                want[t][c] += probs[t][j] * sum(h[f] * wd[e][f][c] for f in range(F))
    got = orc.expert_forward(x, wg, wu, wd, ids, probs, rounding=False)
    np.testing.assert_allclose(got, np.array(want), rtol=1e-12, atol=1e-12)


def test_single_expert_is_dense_swiglu_mlp_torch():
    rng = np.random.default_rng(12)
    T, H, F = 9, 16, 24
    x = rng.standard_normal((T, H))
    wg, wu, wd = (rng.standard_normal((1, H, F)), rng.standard_normal((1, H, F)),
                  rng.standard_normal((1, F, H)))
    ids = np.zeros((T, 1), np.int64)
    probs = np.ones((T, 1))
    tx = torch.from_numpy(x)
    want = (torch.nn.functional.silu(tx @ torch.from_numpy(wg[0])) * (tx @ torch.from_numpy(wu[0]))
            ) @ torch.from_numpy(wd[0])
    got = orc.expert_forward(x, wg, wu, wd, ids, probs, rounding=False)
    np.testing.assert_allclose(got, want.numpy(), rtol=1e-12, atol=1e-12)
    # with rounding the only change is bf16 at h, O and y
    got_r = orc.expert_forward(x, wg, wu, wd, ids, probs)
    h = orc.bf16((torch.nn.functional.silu(tx @ torch.from_numpy(wg[0])) * (tx @ torch.from_numpy(wu[0]))).numpy())
    np.testing.assert_allclose(got_r, orc.bf16(orc.bf16(h @ wd[0])), rtol=2 ** -7, atol=1e-9)


def test_zero_weights_give_zero():
    x, wg, wu, wd, ids, probs = _rand_case()
    assert np.all(orc.expert_forward(x, wg, np.zeros_like(wu), wd, ids, probs) == 0)
    assert np.all(orc.expert_forward(np.zeros_like(x), wg, wu, wd, ids, probs) == 0)
    assert np.all(orc.expert_forward(x, np.zeros_like(wg), wu, wd, ids, probs) == 0)


def test_probs_weight_linearly():
    x, wg, wu, wd, ids, probs = _rand_case(k=1)
    y1 = orc.expert_forward(x, wg, wu, wd, ids, np.ones_like(probs), rounding=False)
    y2 = orc.expert_forward(x, wg, wu, wd, ids, probs, rounding=False)
    np.testing.assert_allclose(y2, probs * y1, rtol=1e-12, atol=1e-14)


def test_expert_relabelling_changes_nothing():
    # renaming the experts (ids and weights together) gives the same y, bit
    # for bit; a weight of the wrong expert anywhere would show
    x, wg, wu, wd, ids, probs = _rand_case(E=5, empty=(3,))
    perm = np.array([2, 4, 0, 1, 3])            # expert e is called perm[e]
    inv = np.argsort(perm)
    y1 = orc.expert_forward(x, wg, wu, wd, ids, probs)
    y2 = orc.expert_forward(x, wg[inv], wu[inv], wd[inv], perm[ids], probs)
    np.testing.assert_array_equal(y2, y1)


def test_slot_order_within_a_token_changes_only_rounding():
    # swapping a token's slots (ids and probs together) reorders one float
    # sum before its single bf16 rounding
    x, wg, wu, wd, ids, probs = _rand_case(k=2)
    y1 = orc.expert_forward(x, wg, wu, wd, ids, probs)
    y2 = orc.expert_forward(x, wg, wu, wd, ids[:, ::-1].copy(), probs[:, ::-1].copy())
    np.testing.assert_allclose(y2, y1, rtol=2 ** -7, atol=1e-12)
    assert np.mean(y2 == y1) > 0.95


def test_microbatch_split_forward_equal():
    x, wg, wu, wd, ids, probs = _rand_case(T=64, k=2)
    y = orc.expert_forward(x, wg, wu, wd, ids, probs)
    for s in (1, 2, 4, 8):
        ys = orc.microbatched_forward(x, wg, wu, wd, ids, probs, s)
        np.testing.assert_allclose(ys, y, rtol=2 ** -7, atol=1e-6)


# ---------------------------------------------------------------- backward

def _loss(dy, *a):
    return float(np.sum(dy * orc.expert_forward(*a, rounding=False)))


def test_backward_finite_differences():
    x, wg, wu, wd, ids, probs = _rand_case(T=6, H=5, F=7, E=3, k=2, empty=(), wstd=0.7)
    rng = np.random.default_rng(13)
    dy = rng.standard_normal(x.shape)
    g = orc.expert_backward(dy, x, wg, wu, wd, ids, probs, rounding=False)
    eps = 1e-6

    def fd(arr, idx, build):
        a1 = arr.copy(); a1[idx] += eps
        a2 = arr.copy(); a2[idx] -= eps
        return (_loss(dy, *build(a1)) - _loss(dy, *build(a2))) / (2 * eps)

    checks = [
        ("dx", x, lambda a: (a, wg, wu, wd, ids, probs)),
        ("dw_gate", wg, lambda a: (x, a, wu, wd, ids, probs)),
        ("dw_up", wu, lambda a: (x, wg, a, wd, ids, probs)),
        ("dw_down", wd, lambda a: (x, wg, wu, a, ids, probs)),
        ("dprobs", probs, lambda a: (x, wg, wu, wd, ids, a)),
    ]
    for name, arr, build in checks:
        for idx in np.ndindex(arr.shape):
            want = fd(arr, idx, build)
            assert abs(g[name][idx] - want) <= 1e-6 * (1 + abs(want)), (name, idx, g[name][idx], want)


def test_backward_matches_torch_autograd():
    x, wg, wu, wd, ids, probs = _rand_case(T=11, H=8, F=12, E=4, k=2, empty=(2,), wstd=0.5)
    dy = np.random.default_rng(14).standard_normal(x.shape)
    g = orc.expert_backward(dy, x, wg, wu, wd, ids, probs, rounding=False)
    tx, tg, tu, td, tp = (torch.tensor(a, requires_grad=True) for a in (x, wg, wu, wd, probs))
    y = torch.zeros_like(tx)
    for t in range(x.shape[0]):
        for j in range(ids.shape[1]):
            e = int(ids[t, j])
            hh = torch.nn.functional.silu(tx[t] @ tg[e]) * (tx[t] @ tu[e])
            y = y.index_add(0, torch.tensor([t]), (tp[t, j] * (hh @ td[e]))[None])
    (y * torch.from_numpy(dy)).sum().backward()
    for name, tt in (("dx", tx), ("dw_gate", tg), ("dw_up", tu), ("dw_down", td), ("dprobs", tp)):
        np.testing.assert_allclose(g[name], tt.grad.numpy(), rtol=1e-10, atol=1e-12, err_msg=name)


def test_backward_worked_example_golden():
    # a hand-worked token whose two dXp rows each round (ties to even) and then
    # nearly cancel: it fixes that dXp is rounded to bf16 before the k-way sum
    g = json.load(open(os.path.join(GOLDEN, "backward_worked_example.json")))
    args = [np.array(g[key]) for key in ("dy", "x", "w_gate", "w_up", "w_down", "expert_ids",
                                          "probs")]
    out = orc.expert_backward(*args)
    for key in ("y", "dprobs", "dx", "dw_gate", "dw_up", "dw_down"):
        np.testing.assert_array_equal(out[key], np.array(g[key]), err_msg=key)
    dx, dp = orc.backward_rows(*args, [0])
    np.testing.assert_array_equal(dx, np.array(g["dx"]))
    np.testing.assert_array_equal(dp, np.array(g["dprobs"]))
    # the MXFP8 backward with quantisation off shares the rounding points
    t = lambda a: a.transpose(0, 2, 1)  # noqa: E731
    mx = orc.expert_backward_mxfp8(args[0], args[1], t(args[2]), t(args[3]), t(args[4]),
                                   args[5], args[6], quantize=False, keep=True)
    np.testing.assert_array_equal(mx["dx"], np.array(g["dx"]))
    np.testing.assert_array_equal(mx["state"]["dxp"], np.array(g["dxp_rows"]))


def test_backward_sampled_helpers_agree():
    x, wg, wu, wd, ids, probs = _rand_case(T=20, H=16, F=24, E=4, k=2, empty=(1,), wstd=0.3)
    dy = orc.bf16(np.random.default_rng(15).standard_normal(x.shape))
    g = orc.expert_backward(dy, x, wg, wu, wd, ids, probs)
    toks = [0, 3, 7, 19]
    dx, dp, rows = orc.backward_rows(dy, x, wg, wu, wd, ids, probs, toks, with_rows=True)
    np.testing.assert_allclose(dx, g["dx"][toks], rtol=2 ** -7, atol=1e-9)
    np.testing.assert_allclose(rows, g["dxp"][g["row_of"][toks]], rtol=2 ** -7, atol=1e-9)
    np.testing.assert_allclose(dp, g["dprobs"][toks], rtol=1e-9, atol=1e-12)
    for e in (0, 2):
        c = orc.weight_grad_columns(dy, x, wg, wu, wd, ids, probs, e, [1, 5, 23])
        np.testing.assert_allclose(c["dw_gate"], g["dw_gate"][e][:, [1, 5, 23]], rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(c["dw_up"], g["dw_up"][e][:, [1, 5, 23]], rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(c["dw_down"], g["dw_down"][e][[1, 5, 23], :], rtol=1e-9, atol=1e-12)
    assert np.all(g["dw_gate"][1] == 0) and np.all(g["dw_down"][1] == 0)


def test_microbatch_split_backward():
    x, wg, wu, wd, ids, probs = _rand_case(T=32, H=16, F=24, E=4, k=2, empty=(), wstd=0.3)
    dy = orc.bf16(np.random.default_rng(16).standard_normal(x.shape))
    g = orc.expert_backward(dy, x, wg, wu, wd, ids, probs)
    for s in (1, 4, 8):
        gs = orc.microbatched_backward(dy, x, wg, wu, wd, ids, probs, s)
        np.testing.assert_allclose(gs["dx"], g["dx"], rtol=2 ** -7, atol=1e-9)
        np.testing.assert_allclose(gs["dprobs"], g["dprobs"], rtol=1e-9, atol=1e-12)
        for key in ("dw_gate", "dw_up", "dw_down"):
            np.testing.assert_allclose(gs[key], g[key], rtol=1e-9, atol=1e-12)


# ---------------------------------------------------------------- MXFP8 forward

def test_mxfp8_grouped_equals_per_token():
    rng = np.random.default_rng(17)
    T, H, F, E, k = 24, 64, 96, 5, 3
    x = orc.bf16(rng.standard_normal((T, H)))
    wg = orc.bf16(rng.standard_normal((E, F, H)) * 0.1)
    wu = orc.bf16(rng.standard_normal((E, F, H)) * 0.1)
    wd = orc.bf16(rng.standard_normal((E, H, F)) * 0.1)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
    probs = rng.dirichlet(np.ones(k), T)
    xq, xs = orc.quantize_mxfp8(x)
    qg = [orc.quantize_mxfp8(wg[e]) for e in range(E)]
    qu = [orc.quantize_mxfp8(wu[e]) for e in range(E)]
    qd = [orc.quantize_mxfp8(wd[e]) for e in range(E)]
    y1 = orc.expert_forward_mxfp8(xq, xs, qg, qu, qd, ids, probs, E)
    y2 = np.stack([orc.token_forward_mxfp8(xq[t], xs[t], qg, qu, qd, ids[t], probs[t]) for t in range(T)])
    np.testing.assert_allclose(y1, y2, rtol=2 ** -6, atol=1e-6)
    # against the unquantised block: MXFP8 is an approximation of it
    wgt = np.transpose(wg, (0, 2, 1)); wut = np.transpose(wu, (0, 2, 1)); wdt = np.transpose(wd, (0, 2, 1))
    yb = orc.expert_forward(x, wgt, wut, wdt, ids, probs)
    assert np.max(np.abs(y1 - yb)) <= 0.1 * np.max(np.abs(yb))


def test_sampled_forward_equals_dense():
    x, wg, wu, wd, ids, probs = _rand_case(T=23)
    toks = [0, 5, 22, 7]
    np.testing.assert_array_equal(orc.sampled_forward(x, wg, wu, wd, ids, probs, toks),
                                  orc.dense_forward(x, wg, wu, wd, ids, probs, toks))


def test_quantizer_rounding_step_equals_definition():
    # quantize_mxfp8 rounds with torch's float8 conversion; e4m3_encode is the
    # rule written out: they must agree bit for bit on every block
    rng = np.random.default_rng(30)
    a = orc.bf16(rng.standard_normal((40, 256)) * np.exp(rng.uniform(-20, 20, (40, 1))))
    a[0, :32] = 0.0
    q, sc = orc.quantize_mxfp8(a)
    x_scale = np.ldexp(1.0, sc.astype(np.int64) - 127)
    want = orc.e4m3_encode(a.reshape(40, 8, 32) / x_scale[..., None]).reshape(40, 256)
    np.testing.assert_array_equal(q, want)


def test_sampled_mxfp8_equals_token_forward():
    rng = np.random.default_rng(31)
    T, H, F, E, k = 6, 64, 96, 4, 2
    x = orc.bf16(rng.standard_normal((T, H)))
    wg, wu = orc.bf16(rng.standard_normal((E, F, H)) * 0.1), orc.bf16(rng.standard_normal((E, F, H)) * 0.1)
    wd = orc.bf16(rng.standard_normal((E, H, F)) * 0.1)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
    probs = rng.dirichlet(np.ones(k), T)
    xq, xs = orc.quantize_mxfp8(x)
    qg = [orc.quantize_mxfp8(wg[e]) for e in range(E)]
    qu = [orc.quantize_mxfp8(wu[e]) for e in range(E)]
    qd = [orc.quantize_mxfp8(wd[e]) for e in range(E)]
    toks = [0, 3, 5]
    want = np.stack([orc.token_forward_mxfp8(xq[t], xs[t], qg, qu, qd, ids[t], probs[t]) for t in toks])
    np.testing.assert_array_equal(orc.sampled_forward_mxfp8(x, wg, wu, wd, ids, probs, toks), want)


# ---------------------------------------------------------------- router (gate ahead of the block)

def test_route_topk_worked_example_golden():
    g = json.load(open(os.path.join(GOLDEN, "router_worked_example.json")))
    logits = np.array([[float(v) for v in row] for row in g["logits"]], dtype=np.float32)  # "-inf", "nan", "-0.0"
    assert np.signbit(logits[3, 0]) and not np.signbit(logits[3, 1])
    ids, probs, counts, offsets = orc.route_topk(logits, g["k"])
    assert ids.tolist() == g["expert_ids"]
    np.testing.assert_allclose(probs, np.array(g["probs"]), rtol=1e-15, atol=0)
    assert counts.tolist() == g["counts"] and offsets.tolist() == g["offsets"]


def _beats(a, b, ea, eb):
    """a (expert ea) ranks before b (expert eb); NaN as -inf."""
    a = -math.inf if math.isnan(a) else a
    b = -math.inf if math.isnan(b) else b
    return a > b or (a == b and ea < eb)


def test_route_topk_order_bruteforce():
    # values from a small set so that ties, signed zeros, -inf and NaN all occur
    rng = np.random.default_rng(21)
    pool = np.array([-0.0, 0.0, 1.0, -1.0, 2.5, -np.inf, np.nan, 0.5], dtype=np.float32)
    for E, k in ((7, 3), (5, 5), (9, 1), (12, 4)):
        logits = pool[rng.integers(0, pool.size, (60, E))]
        ids, _, counts, offsets = orc.route_topk(logits, k)
        for t in range(60):
            row = [float(v) for v in logits[t]]
            chosen = ids[t].tolist()
            assert len(set(chosen)) == k
            for a, b in zip(chosen, chosen[1:]):              # in rank order
                assert _beats(row[a], row[b], a, b)
            for a in chosen:                                   # beats every expert left out
                for b in set(range(E)) - set(chosen):
                    assert _beats(row[a], row[b], a, b)
        assert counts.tolist() == np.bincount(ids.reshape(-1), minlength=E).tolist()
        assert offsets.tolist() == [0] + np.cumsum(counts).tolist()


def test_route_topk_softmax_closed_forms():
    rng = np.random.default_rng(22)
    logits = rng.standard_normal((200, 16)).astype(np.float32)
    l64 = logits.astype(np.float64)
    # k = 2: the first weight is the logistic function of the logit gap
    ids, p, _, _ = orc.route_topk(logits, 2)
    gap = np.take_along_axis(l64, ids[:, :1], 1) - np.take_along_axis(l64, ids[:, 1:], 1)
    np.testing.assert_allclose(p[:, :1], 1.0 / (1.0 + np.exp(-gap)), rtol=1e-14)
    # k = 1: weight one
    _, p1, _, _ = orc.route_topk(logits, 1)
    assert np.all(p1 == 1.0)
    # k = E: a full softmax over the row (scipy's), in rank order
    from scipy.special import softmax
    ids, p, _, _ = orc.route_topk(logits, 16)
    np.testing.assert_allclose(p, np.take_along_axis(softmax(l64, axis=1), ids, 1), rtol=1e-13)
    # any k: the softmax over all E restricted to the top k and renormalised
    for k in (3, 6):
        ids, p, _, _ = orc.route_topk(logits, k)
        full = np.take_along_axis(softmax(l64, axis=1), ids, 1)
        np.testing.assert_allclose(p, full / full.sum(1, keepdims=True), rtol=1e-13)


def test_route_topk_shift_and_ties():
    # integer logits shifted by an integer: exact in float32 and float64, so
    # neither the order nor the weights may change
    rng = np.random.default_rng(23)
    logits = rng.integers(-4, 5, (100, 10)).astype(np.float32)
    ids0, p0, _, _ = orc.route_topk(logits, 4)
    ids1, p1, _, _ = orc.route_topk(logits + 37.0, 4)
    assert np.array_equal(ids0, ids1)
    np.testing.assert_allclose(p0, p1, rtol=1e-15)
    # a row of equal logits: experts 0..k-1, weight 1/k each
    ids, p, _, _ = orc.route_topk(np.full((3, 8), 1.25, np.float32), 4)
    assert ids.tolist() == [[0, 1, 2, 3]] * 3 and np.all(p == 0.25)


def test_route_topk_rejects_bad_k():
    with pytest.raises(ValueError):
        orc.route_topk(np.zeros((2, 4), np.float32), 5)
    with pytest.raises(ValueError):
        orc.route_topk(np.zeros((2, 4), np.float32), 0)


# ---------------------------------------------------------------- MXFP8 backward

def _mx_bwd_case(T=60, H=64, F=96, E=4, k=2, seed=31, wstd=0.1):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
    ex = rng.exponential(1.0, (T, k))
    probs = ex / ex.sum(1, keepdims=True)
    b = lambda *s_, sd=1.0: orc.bf16(rng.standard_normal(s_) * sd)  # noqa: E731
    return (b(T, H), b(T, H), b(E, F, H, sd=wstd), b(E, F, H, sd=wstd), b(E, H, F, sd=wstd),
            ids, probs)


def test_quantized_along_columns_blocks_by_hand():
    # blocks of 32 rows per column, the last one zero-completed; each block
    # worked with the pinned element rules (e8m0_scale_code, e4m3 codes)
    rng = np.random.default_rng(32)
    a = orc.bf16(rng.standard_normal((70, 3)) * np.array([1e-3, 1.0, 300.0]))
    a[40:64, 1] *= 1e-4                         # a block far below its neighbours
    got = orc.quantized_along_columns(a)
    for c in range(3):
        col = np.concatenate([a[:, c], np.zeros(26)])
        for b in range(3):
            blk = col[32 * b:32 * b + 32]
            code = int(orc.e8m0_scale_code(np.abs(blk).max()))
            scale = 2.0 ** (code - 127)
            want = orc.e4m3_decode(orc.e4m3_encode(blk / scale)) * scale
            rows = slice(32 * b, min(32 * b + 32, 70))
            np.testing.assert_array_equal(got[rows, c], want[:rows.stop - rows.start])
    np.testing.assert_array_equal(orc.quantized_along_columns(a, quantize=False), a)


def test_mxfp8_backward_unquantized_is_bf16_backward():
    dy, x, wgt, wut, wdt, ids, probs = _mx_bwd_case()
    mx = orc.expert_backward_mxfp8(dy, x, wgt, wut, wdt, ids, probs, quantize=False)
    ref = orc.expert_backward(dy, x, wgt.transpose(0, 2, 1), wut.transpose(0, 2, 1),
                              wdt.transpose(0, 2, 1), ids, probs)
    pairs = [("dx", "dx", None), ("dprobs", "dprobs", None), ("y", "y", None),
             ("dw_gate_t", "dw_gate", (0, 2, 1)), ("dw_up_t", "dw_up", (0, 2, 1)),
             ("dw_down_t", "dw_down", (0, 2, 1))]
    for a, b, perm in pairs:
        want = ref[b] if perm is None else ref[b].transpose(perm)
        # the same products in float64; only BLAS summation order differs,
        # which can move a bf16 rounding of h, dA or y by one step
        scale = np.abs(want).max()
        np.testing.assert_allclose(mx[a], want, rtol=2 ** -6, atol=2 ** -6 * scale, err_msg=a)
        assert np.mean(np.isclose(mx[a], want, rtol=1e-9, atol=1e-12 * scale)) > 0.97, a


def test_mxfp8_backward_elements_by_definition():
    # single elements of every quantised GEMM rebuilt from the kept
    # intermediates with explicit per-block quantisation
    dy, x, wgt, wut, wdt, ids, probs = _mx_bwd_case(T=40, E=2, k=1, seed=33)
    out = orc.expert_backward_mxfp8(dy, x, wgt, wut, wdt, ids, probs, keep=True)
    st = out["state"]

    def q_vec(v):                     # one vector, blocks of 32 from its start
        v = np.concatenate([v, np.zeros((-len(v)) % 32)])
        res = np.zeros_like(v)
        for b in range(0, len(v), 32):
            blk = v[b:b + 32]
            sc = 2.0 ** (int(orc.e8m0_scale_code(np.abs(blk).max())) - 127)
            res[b:b + 32] = orc.e4m3_decode(orc.e4m3_encode(blk / sc)) * sc
        return res

    off = st["off"]
    for e in range(2):
        lo, hi = int(off[e]), int(off[e + 1])
        n = hi - lo
        r, f, hh = lo + n // 2, 17, 9
        # dH[r, f] = sum_h q(dO[r, :])[h] q(W2[f, :])[h]  (W2 = w_down_t^T, along H)
        dh = np.dot(q_vec(st["d_o"][r]), q_vec(wdt[e][:, f]))
        np.testing.assert_allclose(st["dh"][r, f], dh, rtol=1e-12)
        # dXp[r, hh] = q(dA_g[r])·q(W1g[hh, :]) + q(dA_u[r])·q(W1u[hh, :])  (along F)
        # then rounded to bf16 (another summation order may move that rounding a step)
        dxp = (np.dot(q_vec(st["da_g"][r]), q_vec(wgt[e][:, hh])) +
               np.dot(q_vec(st["da_u"][r]), q_vec(wut[e][:, hh])))
        assert orc.bf16(st["dxp"][r, hh]) == st["dxp"][r, hh]
        np.testing.assert_allclose(st["dxp"][r, hh], orc.bf16(dxp), rtol=2 ** -8)
        # dW1g^T[f, hh] = sum_r q(dA_g[:, f])[r] q(Xp[:, hh])[r]  (along the expert's rows)
        xp_col = x[st["token_of"][lo:hi], hh]
        want = np.dot(q_vec(st["da_g"][lo:hi, f]), q_vec(xp_col))[()]
        np.testing.assert_allclose(out["dw_gate_t"][e][f, hh], want, rtol=1e-12, atol=1e-300)
        # dW2^T[hh, f] = sum_r q(dO[:, hh])[r] q(h[:, f])[r]
        want = np.dot(q_vec(st["d_o"][lo:hi, hh]), q_vec(st["h"][lo:hi, f]))
        np.testing.assert_allclose(out["dw_down_t"][e][hh, f], want, rtol=1e-12, atol=1e-300)


def test_mxfp8_backward_close_to_unquantized():
    # each operand carries at most 2^-4 relative E4M3 rounding: the
    # quantised gradients stay within a few percent of the unquantised ones
    dy, x, wgt, wut, wdt, ids, probs = _mx_bwd_case(seed=34)
    mx = orc.expert_backward_mxfp8(dy, x, wgt, wut, wdt, ids, probs)
    ex = orc.expert_backward_mxfp8(dy, x, wgt, wut, wdt, ids, probs, quantize=False)
    for key in ("dx", "dw_gate_t", "dw_up_t", "dw_down_t", "dprobs"):
        err = np.abs(mx[key] - ex[key]).max() / np.abs(ex[key]).max()
        assert err < 0.15, (key, err)


def test_mxfp8_backward_sampled_helpers_agree():
    dy, x, wgt, wut, wdt, ids, probs = _mx_bwd_case(T=50, E=3, k=2, seed=35)
    full = orc.expert_backward_mxfp8(dy, x, wgt, wut, wdt, ids, probs)
    toks = [0, 17, 49]
    dx, dp = orc.backward_rows_mxfp8(dy, x, wgt, wut, wdt, ids, probs, toks)
    np.testing.assert_allclose(dx, full["dx"][toks], rtol=2 ** -7, atol=1e-12)
    np.testing.assert_allclose(dp, full["dprobs"][toks], rtol=1e-9, atol=1e-12)
    pairs = [(0, 0), (5, 63), (95, 17)]
    for e in range(3):
        got = orc.weight_grad_entries_mxfp8(dy, x, wgt, wut, wdt, ids, probs, e, pairs)
        for i, (f, h) in enumerate(pairs):
            want = (full["dw_gate_t"][e][f, h], full["dw_up_t"][e][f, h],
                    full["dw_down_t"][e][h, f])
            np.testing.assert_allclose(got[i], want, rtol=1e-9, atol=1e-12)
        sl = orc.weight_grad_slices_mxfp8(dy, x, wgt, wut, wdt, ids, probs, e, [0, 5, 95])
        np.testing.assert_allclose(sl["dw_gate_t"], full["dw_gate_t"][e][[0, 5, 95]], rtol=1e-9,
                                   atol=1e-12)
        np.testing.assert_allclose(sl["dw_up_t"], full["dw_up_t"][e][[0, 5, 95]], rtol=1e-9,
                                   atol=1e-12)
        np.testing.assert_allclose(sl["dw_down_t"], full["dw_down_t"][e][:, [0, 5, 95]].T,
                                   rtol=1e-9, atol=1e-12)


# ---------------------------------------------------------------- MXFP8 symmetries

def _mx_fwd(x, wgt, wut, wdt, ids, probs):
    E = len(wgt)
    xq, xs = orc.quantize_mxfp8(x)
    q = [[orc.quantize_mxfp8(w[e]) for e in range(E)] for w in (wgt, wut, wdt)]
    return orc.expert_forward_mxfp8(xq, xs, *q, ids, probs, E)


def test_mxfp8_forward_linear_in_probs():
    # the weights enter only the combine, after every quantisation: doubling
    # them doubles y exactly (a power of two moves no rounding)
    _, x, wgt, wut, wdt, ids, probs = _mx_bwd_case(T=30, seed=40)
    y1 = _mx_fwd(x, wgt, wut, wdt, ids, probs)
    y2 = _mx_fwd(x, wgt, wut, wdt, ids, 2.0 * probs)
    np.testing.assert_array_equal(y2, 2.0 * y1)
    assert np.abs(y1).max() > 0


def test_mxfp8_forward_expert_relabelling():
    # renaming the experts (ids and weights together) changes nothing:
    # every routed row meets its own expert's weights
    _, x, wgt, wut, wdt, ids, probs = _mx_bwd_case(T=30, E=5, k=3, seed=41)
    perm = np.array([3, 0, 4, 1, 2])            # expert e is called perm[e]
    inv = np.argsort(perm)
    y1 = _mx_fwd(x, wgt, wut, wdt, ids, probs)
    y2 = _mx_fwd(x, wgt[inv], wut[inv], wdt[inv], perm[ids], probs)
    np.testing.assert_array_equal(y2, y1)


def test_mxfp8_forward_token_order():
    # tokens are independent: permuting them permutes y's rows
    _, x, wgt, wut, wdt, ids, probs = _mx_bwd_case(T=30, seed=42)
    order = np.random.default_rng(43).permutation(30)
    y1 = _mx_fwd(x, wgt, wut, wdt, ids, probs)
    y2 = _mx_fwd(x[order], wgt, wut, wdt, ids[order], probs[order])
    # a different row order can change BLAS's blocking, so a bf16 rounding
    # may move by one step
    np.testing.assert_allclose(y2, y1[order], rtol=2 ** -7, atol=1e-12)
    assert np.mean(y2 == y1[order]) > 0.99


def test_mxfp8_dprobs_is_dy_dot_slot_output():
    # dprobs[t, j] = <dY_t, O of slot (t, j)>, O from the forward of that
    # slot alone with weight 1
    dy, x, wgt, wut, wdt, ids, probs = _mx_bwd_case(T=12, E=3, k=2, seed=44)
    g = orc.expert_backward_mxfp8(dy, x, wgt, wut, wdt, ids, probs)
    xq, xs = orc.quantize_mxfp8(x)
    q = [[orc.quantize_mxfp8(w[e]) for e in range(3)] for w in (wgt, wut, wdt)]
    for t in (0, 5, 11):
        for j in range(2):
            o = orc.token_forward_mxfp8(xq[t], xs[t], *q, ids[t, j:j + 1], [1.0])
            np.testing.assert_allclose(g["dprobs"][t, j], np.dot(dy[t], o),
                                       rtol=2 ** -7, atol=1e-9 * np.abs(o).max())
