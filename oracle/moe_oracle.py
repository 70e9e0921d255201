"""Plain CPU oracle of the MoE expert block.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports, calls or runs
this module: only the tests, the package smoke check and the benchmark's CPU
baseline / reference arm use it. It shares no code with the CUDA library.

What it computes is the expert block that the pages describe, written out
from its definition with NumPy in float64 (matmuls through NumPy's BLAS,
everything else elementwise), with no blocking, fusion or reordering beyond
the definition:

  * counts      per-expert token counts, the histc step of ep_mc2_forward
                ("NPU Training Operators - MC2", section "execution path",
                step 2). For integer ids in [0, E) a histogram with E bins over
                [0, E] equals a bincount (the same page's PR table notes the
                swap from bincount to histc).
  * offsets     the exclusive scan of the counts; on one device the send and
                receive counts of steps 4-5 are both the local counts.
  * route_topk  the gate ahead of the block: top-k experts of the router
                logits with a softmax over the chosen k, and their counts.
  * permute     step 6: routed rows gathered into expert-contiguous order,
                stable by flat index t*k+j within an expert.
  * fc1+SwiGLU  steps 7-8: A_g = Xp_e W1g_e, A_u = Xp_e W1u_e,
                h = bf16(silu(A_g) * A_u), silu(z) = z / (1 + exp(-z)).
                The separate gate / up weights follow the mc2_fused_expert
                call in the MC2 for MoE All-to-All article (section "usage").
  * fc2         step 9: O = bf16(h_e W2_e).
  * unpermute   step 10: y_t = bf16(sum_j p_tj O[row_of[t, j]]), j in order.
  * backward    the gradients the autograd Functions of the same page wrap
                (section "PR changes"), and the fc1/fc2 gradient comparison of
                its section "validation items".
  * MXFP8       the quantised AllToAll+Matmul of "MC2 通算融合架构总览"
                (section 1, and the scale buffers of section 5): E4M3 values
                with one E8M0 scale per 32 K-contiguous elements, following the
                OCP Microscaling Formats (MX) v1.0 specification; its backward
                quantises every GEMM operand along that GEMM's reduction.
  * micro-batch the split of the MC2 for MoE All-to-All article (section
                "pipeline design"): chunks processed independently and
                reassembled in token order.

Readings where the pages are silent (listed with the rest in the design
notes): h rounded to bf16 (A_g, A_u not rounded in the forward); O rounded to
bf16 before the combine; the combine sums j in order, then rounds once;
backward uses A_g, A_u as saved in bf16 and rounds dXp to bf16, because, like
O in the forward, it is a tensor of its own between two ops (the grouped
matmul's backward and the permute's backward); dX = bf16 of the float sum of
a token's k rows of dXp, rounded once; dW is float (here float64, on the GPU
float32); in MXFP8 mode h is first rounded to bf16 then quantised per 32
along F.

Every function here is pinned by tests against something other than itself
(library routines, closed forms, brute force, finite differences).
"""
from __future__ import annotations

import numpy as np

BF16_MAX = float.fromhex("0x1.fep127")
E4M3_MAX = 448.0
E4M3_EMAX = 8          # exponent of the largest E4M3 normal (448 = 1.75 * 2^8)
MX_BLOCK = 32          # elements per shared scale


# --------------------------------------------------------------------------
# rounding
# --------------------------------------------------------------------------

def bf16(a) -> np.ndarray:
    """Round to the nearest bfloat16, ties to even, returned as float64.

    bfloat16 keeps 8 significant bits, exponents down to 2^-126 for normals
    and a fixed quantum of 2^-133 below that; values whose rounding exceeds
    the largest finite bf16 become infinities.
    """
    a = np.asarray(a, dtype=np.float64)
    _, e = np.frexp(a)                       # a = m 2^e, 0.5 <= |m| < 1
    q = np.ldexp(1.0, np.maximum(e, -125) - 8)
    r = np.rint(a / q) * q                   # np.rint: half to even
    return np.where(np.abs(r) > BF16_MAX, np.copysign(np.inf, a), r)


def silu(z):
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def sigmoid(z):
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


# --------------------------------------------------------------------------
# counts, offsets, permute, unpermute
# --------------------------------------------------------------------------

def expert_counts(expert_ids, num_experts: int) -> np.ndarray:
    """c_e = number of routed slots (t, j) with expert_ids[t, j] == e.

    An id outside [0, E) is a caller error (the migration checks of "NPU
    Training Operators - MC2" require ids in [0, num_experts)); it raises.
    """
    ids = np.asarray(expert_ids).reshape(-1)
    if ids.size and (ids.min() < 0 or ids.max() >= num_experts):
        raise ValueError("expert id outside [0, num_experts)")
    return np.array([np.count_nonzero(ids == e) for e in range(num_experts)], dtype=np.int64)


def expert_offsets(counts) -> np.ndarray:
    """off[0] = 0, off[e+1] = off[e] + c_e."""
    counts = np.asarray(counts, dtype=np.int64)
    off = np.zeros(counts.size + 1, dtype=np.int64)
    for e in range(counts.size):
        off[e + 1] = off[e] + counts[e]
    return off


def route_topk(logits, k: int):
    """Top-k routing from router logits: the gate step just ahead of the block.

    The block takes the routing weights and selected experts that the
    dispatcher call of "NPU Training Operators - MC2" (section "suggested
    configuration") passes in; they come from the gate computation that the
    MC2 for MoE All-to-All article counts as the first part of a step
    (section on why communication is the bottleneck). The pages do not spell
    the gate out. Reading used here:

      * ids[t] are the k experts with the largest logits, in descending order
        of logit; equal logits rank the lower expert index first (so -0.0 and
        +0.0 tie); a NaN logit ranks as -inf.
      * probs[t, j] = exp(l_j - l_0) / sum_i exp(l_i - l_0) over the chosen k,
        l_0 the largest: a softmax over all E restricted to the top k and
        renormalised.
      * counts and offsets are those of the chosen ids (expert_counts,
        expert_offsets).

    logits: float32 [T, E]. The order is decided on those float32 values
    (exact in float64); the weights are computed in float64.
    Returns ids int32 [T, k], probs float64 [T, k], counts [E], offsets [E+1].
    """
    lg = np.asarray(logits, dtype=np.float32).astype(np.float64)
    T, E = lg.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    lg = np.where(np.isnan(lg), -np.inf, lg)
    index = np.broadcast_to(np.arange(E), lg.shape)
    order = np.lexsort((index, -lg), axis=1)[:, :k]      # primary -logit, then index
    chosen = np.take_along_axis(lg, order, axis=1)
    with np.errstate(invalid="ignore"):
        ex = np.exp(chosen - chosen[:, :1])
        probs = ex / ex.sum(axis=1, keepdims=True)
    ids = order.astype(np.int32)
    counts = expert_counts(ids, E)
    return ids, probs, counts, expert_offsets(counts)


def permute_map(expert_ids, num_experts: int):
    """Row map of the stable permute.

    Flat slot i = t*k + j goes to row off[e] + (number of earlier slots with
    the same expert), e = expert_ids[t, j]. Returns (row_of [T,k],
    token_of [R], slot_of [R]) where slot_of[r] = j.
    """
    ids = np.asarray(expert_ids)
    T, k = ids.shape
    flat = ids.reshape(-1)
    off = expert_offsets(expert_counts(ids, num_experts))
    nxt = [int(v) for v in off[:-1]]
    row_of = np.empty(flat.size, dtype=np.int64)
    for i, e in enumerate(flat.tolist()):
        row_of[i] = nxt[e]
        nxt[e] += 1
    token_of = np.empty(flat.size, dtype=np.int64)
    slot_of = np.empty(flat.size, dtype=np.int64)
    token_of[row_of] = np.arange(flat.size) // k
    slot_of[row_of] = np.arange(flat.size) % k
    return row_of.reshape(T, k), token_of, slot_of


def permute(x, expert_ids, probs, num_experts: int):
    """Xp[row_of[t,j]] = x[t]; prob_of[row_of[t,j]] = probs[t,j]."""
    x = _f64(x)
    row_of, token_of, slot_of = permute_map(expert_ids, num_experts)
    xp = x[token_of]
    prob_of = None if probs is None else _f64(probs)[token_of, slot_of]
    return xp, row_of, token_of, prob_of


def unpermute(o, row_of, probs=None, rounding: bool = True):
    """y_t = bf16(sum_j p_tj O[row_of[t, j]]) with j summed in order; p = 1
    when probs is None."""
    o = _f64(o)
    row_of = np.asarray(row_of)
    T, k = row_of.shape
    acc = np.zeros((T, o.shape[1]))
    for j in range(k):
        p = 1.0 if probs is None else _f64(probs)[:, j:j + 1]
        acc = acc + p * o[row_of[:, j]]
    return bf16(acc) if rounding else acc


# --------------------------------------------------------------------------
# grouped expert matmuls (O1: the permuted grouped path)
# --------------------------------------------------------------------------

def grouped_fc1_swiglu(xp, counts, w_gate, w_up, rounding: bool = True):
    """Per expert e over its rows: A_g = Xp_e W1g_e, A_u = Xp_e W1u_e,
    h = bf16(silu(A_g) A_u). Weights [E, H, F]. Returns (h, A_g, A_u)."""
    xp = _f64(xp)
    off = expert_offsets(counts)
    F = np.asarray(w_gate[0]).shape[1]
    h = np.zeros((xp.shape[0], F))
    a_g = np.zeros_like(h)
    a_u = np.zeros_like(h)
    for e in range(len(counts)):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        a_g[lo:hi] = xp[lo:hi] @ _f64(w_gate[e])
        a_u[lo:hi] = xp[lo:hi] @ _f64(w_up[e])
    hv = silu(a_g) * a_u
    h = bf16(hv) if rounding else hv
    return h, a_g, a_u


def grouped_fc2(h, counts, w_down, rounding: bool = True):
    """O_e = bf16(h_e W2_e), W2 [E, F, H]."""
    h = _f64(h)
    off = expert_offsets(counts)
    H = np.asarray(w_down[0]).shape[1]
    o = np.zeros((h.shape[0], H))
    for e in range(len(counts)):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi > lo:
            o[lo:hi] = h[lo:hi] @ _f64(w_down[e])
    return bf16(o) if rounding else o


def expert_forward(x, w_gate, w_up, w_down, expert_ids, probs, num_experts=None,
                   rounding: bool = True, keep: bool = False):
    """The whole block, step by step: counts, offsets, permute, fc1+SwiGLU,
    fc2, unpermute. Returns y [T, H] (and the intermediates when keep)."""
    E = len(w_gate) if num_experts is None else num_experts
    counts = expert_counts(expert_ids, E)
    xp, row_of, token_of, prob_of = permute(x, expert_ids, probs, E)
    h, a_g, a_u = grouped_fc1_swiglu(xp, counts, w_gate, w_up, rounding)
    o = grouped_fc2(h, counts, w_down, rounding)
    y = unpermute(o, row_of, probs, rounding)
    if not keep:
        return y
    return y, dict(counts=counts, xp=xp, row_of=row_of, token_of=token_of, prob_of=prob_of,
                   h=h, a_g=a_g, a_u=a_u, o=o)


# --------------------------------------------------------------------------
# O2: per-token dense loop, no permutation at all
# --------------------------------------------------------------------------

def token_forward(x_t, w_gate, w_up, w_down, ids_t, probs_t, rounding: bool = True):
    """y_t = bf16(sum_j p_tj bf16(W2_e^T bf16(silu(W1g_e^T x_t) * (W1u_e^T x_t))))."""
    x_t = _f64(x_t)
    acc = None
    for j, e in enumerate(np.asarray(ids_t).tolist()):
        g = x_t @ _f64(w_gate[e])
        u = x_t @ _f64(w_up[e])
        hv = silu(g) * u
        hv = bf16(hv) if rounding else hv
        ov = hv @ _f64(w_down[e])
        ov = bf16(ov) if rounding else ov
        term = float(np.asarray(probs_t)[j]) * ov
        acc = term if acc is None else acc + term
    return bf16(acc) if rounding else acc


def dense_forward(x, w_gate, w_up, w_down, expert_ids, probs, tokens=None, rounding: bool = True):
    """token_forward for every token in `tokens` (all tokens by default)."""
    x = np.asarray(x)
    ids = np.asarray(expert_ids)
    pr = np.asarray(probs)
    tokens = range(x.shape[0]) if tokens is None else tokens
    return np.stack([token_forward(x[t], w_gate, w_up, w_down, ids[t], pr[t], rounding)
                     for t in tokens])


def sampled_forward(x, w_gate, w_up, w_down, expert_ids, probs, tokens):
    """token_forward for the listed tokens, visiting one expert at a time so
    that each expert's weights are converted to float64 once. Every (t, j)
    slot's O row is the same per-token expression; the combine then sums j
    in order per token."""
    x = np.asarray(x)
    ids = np.asarray(expert_ids)
    pr = np.asarray(probs)
    tokens = list(tokens)
    o_rows = {}
    for e in sorted(set(int(v) for t in tokens for v in ids[t])):
        wg, wu, wd = _f64(w_gate[e]), _f64(w_up[e]), _f64(w_down[e])
        for t in tokens:
            for j, ee in enumerate(ids[t].tolist()):
                if ee == e:
                    xt = _f64(x[t])
                    hv = bf16(silu(xt @ wg) * (xt @ wu))
                    o_rows[(t, j)] = bf16(hv @ wd)
    out = []
    for t in tokens:
        acc = None
        for j in range(ids.shape[1]):
            term = float(pr[t, j]) * o_rows[(t, j)]
            acc = term if acc is None else acc + term
        out.append(bf16(acc))
    return np.stack(out)


# --------------------------------------------------------------------------
# backward
# --------------------------------------------------------------------------

def expert_backward(dy, x, w_gate, w_up, w_down, expert_ids, probs, rounding: bool = True):
    """Gradients of y = expert_forward(...) with respect to x, the three
    weight tensors and probs.

      dO_r   = bf16(p_r dY_t(r))
      dp_tj  = <dY_t, O_row(t,j)>
      dH     = dO_e W2_e^T
      dA_g   = bf16(dH * A_u * sigma(A_g) (1 + A_g (1 - sigma(A_g))))
      dA_u   = bf16(dH * silu(A_g))
      dXp    = bf16(dA_g W1g_e^T + dA_u W1u_e^T)
      dW2_e  = h_e^T dO_e,  dW1g_e = Xp_e^T dA_g,e,  dW1u_e = Xp_e^T dA_u,e
      dX_t   = bf16(sum_j dXp[row_of[t, j]])

    With rounding, A_g and A_u enter as bf16 (as saved by the forward).
    With rounding=False every bf16() is the identity: the exact gradient of
    the unrounded forward, which the finite-difference test checks.
    Returns dict(dx, dw_gate, dw_up, dw_down, dprobs, y), plus the rows of
    dXp (dxp, in permuted order) and row_of.
    """
    E = len(w_gate)
    rnd = bf16 if rounding else (lambda v: _f64(v))
    y, st = expert_forward(x, w_gate, w_up, w_down, expert_ids, probs, E, rounding, keep=True)
    dy = _f64(dy)
    counts, off = st["counts"], expert_offsets(st["counts"])
    token_of, prob_of, row_of = st["token_of"], st["prob_of"], st["row_of"]
    a_g, a_u = rnd(st["a_g"]), rnd(st["a_u"])
    xp, h, o = st["xp"], st["h"], st["o"]
    T, k = np.asarray(expert_ids).shape
    d_o = rnd(prob_of[:, None] * dy[token_of])
    dprobs = np.zeros((T, k))
    for j in range(k):
        dprobs[:, j] = np.sum(dy * o[row_of[:, j]], axis=1)
    H = xp.shape[1]
    F = h.shape[1]
    dxp = np.zeros_like(xp)
    dw_gate = np.zeros((E, H, F))
    dw_up = np.zeros((E, H, F))
    dw_down = np.zeros((E, F, H))
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        dh = d_o[lo:hi] @ _f64(w_down[e]).T
        sg = sigmoid(a_g[lo:hi])
        da_g = rnd(dh * a_u[lo:hi] * sg * (1.0 + a_g[lo:hi] * (1.0 - sg)))
        da_u = rnd(dh * a_g[lo:hi] * sg)
        dxp[lo:hi] = rnd(da_g @ _f64(w_gate[e]).T + da_u @ _f64(w_up[e]).T)
        dw_down[e] = h[lo:hi].T @ d_o[lo:hi]
        dw_gate[e] = xp[lo:hi].T @ da_g
        dw_up[e] = xp[lo:hi].T @ da_u
    dx = unpermute(dxp, row_of, None, rounding)
    return dict(dx=dx, dw_gate=dw_gate, dw_up=dw_up, dw_down=dw_down, dprobs=dprobs, y=y,
                dxp=dxp, row_of=row_of)


def backward_rows(dy, x, w_gate, w_up, w_down, expert_ids, probs, tokens, with_rows=False):
    """dX and dprobs of the listed tokens only (rounding as expert_backward);
    with_rows adds their dXp rows, [len(tokens), k, H], slot by slot.

    Each token's gradient depends only on its own rows, so this is the same
    arithmetic as expert_backward restricted to those rows; it lets the
    full-size workloads be checked on a sample of tokens. Experts are
    visited one at a time so that each expert's weights are converted once.
    """
    dy = _f64(dy)
    x = np.asarray(x)
    ids = np.asarray(expert_ids)
    pr = np.asarray(probs)
    tokens = list(tokens)
    dxr, dpt = {}, {}
    for e in sorted(set(int(v) for t in tokens for v in ids[t])):
        wg, wu, wd = _f64(w_gate[e]), _f64(w_up[e]), _f64(w_down[e])
        for t in tokens:
            for j, ee in enumerate(ids[t].tolist()):
                if ee != e:
                    continue
                xt = _f64(x[t])
                g = xt @ wg
                u = xt @ wu
                hv = bf16(silu(g) * u)
                ov = bf16(hv @ wd)
                dpt[(t, j)] = float(np.dot(dy[t], ov))
                d_o = bf16(float(pr[t, j]) * dy[t])
                dh = wd @ d_o
                ga, ua = bf16(g), bf16(u)
                sg = sigmoid(ga)
                da_g = bf16(dh * ua * sg * (1.0 + ga * (1.0 - sg)))
                da_u = bf16(dh * ga * sg)
                dxr[(t, j)] = bf16(wg @ da_g + wu @ da_u)
    k = ids.shape[1]
    dx, dp = [], []
    for t in tokens:
        acc = dxr[(t, 0)]
        for j in range(1, k):
            acc = acc + dxr[(t, j)]
        dx.append(bf16(acc))
        dp.append([dpt[(t, j)] for j in range(k)])
    if with_rows:
        rows = np.stack([np.stack([dxr[(t, j)] for j in range(k)]) for t in tokens])
        return np.stack(dx), np.array(dp), rows
    return np.stack(dx), np.array(dp)


def weight_grad_columns(dy, x, w_gate, w_up, w_down, expert_ids, probs, e, f_cols):
    """Exact slices of the weight gradients of expert e for each f in f_cols:
    the columns dW1g_e[:, f] and dW1u_e[:, f] (over all H) and the row
    dW2_e[f, :] (over all H). Each needs only column f of A_g, A_u and dH
    over the rows routed to e, so this is expert_backward's arithmetic
    restricted to those columns."""
    ids = np.asarray(expert_ids)
    pr = np.asarray(probs)
    dy = _f64(dy)
    flat = ids.reshape(-1)
    slots = np.nonzero(flat == e)[0]
    k = ids.shape[1]
    toks, js = slots // k, slots % k
    cols = list(f_cols)
    xe = _f64(np.asarray(x)[toks])                        # rows of expert e
    p = pr[toks, js].astype(np.float64)
    d_o = bf16(p[:, None] * dy[toks])
    wg, wu, wd = _f64(np.asarray(w_gate[e])[:, cols]), _f64(np.asarray(w_up[e])[:, cols]), \
        _f64(np.asarray(w_down[e])[cols])
    a_g = xe @ wg                                         # [c_e, len(cols)]
    a_u = xe @ wu
    dh = d_o @ wd.T
    ga, ua = bf16(a_g), bf16(a_u)
    sg = sigmoid(ga)
    da_g = bf16(dh * ua * sg * (1.0 + ga * (1.0 - sg)))
    da_u = bf16(dh * ga * sg)
    h = bf16(silu(a_g) * a_u)
    return {"dw_gate": xe.T @ da_g,                       # [H, len(cols)]
            "dw_up": xe.T @ da_u,
            "dw_down": h.T @ d_o}                         # [len(cols), H]


# --------------------------------------------------------------------------
# MXFP8 (OCP MX v1.0: E4M3 elements, E8M0 shared scale per 32)
# --------------------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    """Value of each E4M3 (fn) code: sign, 4 exponent bits (bias 7), 3
    mantissa bits; exponent 0 is subnormal (m 2^-9); S.1111.111 is NaN; there
    is no infinity."""
    c = np.asarray(codes, dtype=np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    ex = (c >> 3) & 0xF
    man = (c & 0x7).astype(np.float64)
    val = np.where(ex == 0, man * 2.0 ** -9, (1.0 + man / 8.0) * np.ldexp(1.0, ex - 7))
    val = np.where((ex == 15) & ((c & 7) == 7), np.nan, val)
    return s * val


def e4m3_encode(v) -> np.ndarray:
    """Round to the nearest E4M3 value, ties to even, saturating at +-448
    (satfinite); returns the uint8 codes. Zero keeps its sign bit."""
    v = _f64(v)
    a = np.abs(v)
    _, e = np.frexp(a)
    q = np.ldexp(1.0, np.maximum(e, -5) - 4)      # 4 significant bits, min normal 2^-6
    r = np.minimum(np.rint(a / q) * q, E4M3_MAX)
    normal = r >= 2.0 ** -6
    with np.errstate(divide="ignore"):
        ex = np.where(normal, np.floor(np.log2(np.where(normal, r, 1.0))), 0).astype(np.int64)
    man_n = np.rint(np.where(normal, r / np.ldexp(1.0, ex), 0.0) * 8.0 - 8.0).astype(np.int64)
    man_s = np.rint(r / 2.0 ** -9).astype(np.int64)
    code = np.where(normal, ((ex + 7) << 3) | man_n, man_s)
    code = code | np.where(np.signbit(v), 0x80, 0)
    return code.astype(np.uint8)


def e8m0_scale_code(amax) -> np.ndarray:
    """Shared scale of one block: X = 2^(floor(log2(amax)) - 8), the
    exponent clamped to E8M0's [-127, 127]; code = exponent + 127. A block of
    zeros gets the smallest scale, 2^-127 (code 0). A block holding an
    infinity or a NaN (amax not finite) has no such exponent: it gets 255,
    the E8M0 NaN, so that the whole block decodes to NaN."""
    amax = _f64(amax)
    live = np.isfinite(amax) & (amax > 0)
    with np.errstate(divide="ignore", invalid="ignore"):
        ex = np.where(live, np.floor(np.log2(np.where(live, amax, 1.0))), -np.inf)
    ex = np.clip(ex - E4M3_EMAX, -127, 127)
    return np.where(np.isfinite(amax), ex + 127, 255).astype(np.uint8)


E8M0_NAN = 255
E4M3_NAN = 0x7F


_E4M3_TABLE = None


def _e4m3_table() -> np.ndarray:
    global _E4M3_TABLE
    if _E4M3_TABLE is None:
        _E4M3_TABLE = e4m3_decode(np.arange(256))
    return _E4M3_TABLE


def quantize_mxfp8(a):
    """Quantise the last axis in blocks of 32: per block the E8M0 scale code
    from its amax, then each element E4M3(v / X). Returns (codes uint8 of a's
    shape, scale codes uint8 of shape [..., K/32]). A block holding an
    infinity or a NaN gets the NaN scale code and E4M3 NaN (0x7F) elements.

    v / X is a power-of-two scaling, exact for bf16-valued inputs, so the
    only rounding is the E4M3 one. That rounding step uses torch's
    float8_e4m3fn conversion (round to nearest even) after clamping to
    +-448, which together are E4M3 satfinite; e4m3_encode is the same rule
    written out, and the tests hold the two bit-identical."""
    import torch
    a = _f64(a)
    K = a.shape[-1]
    assert K % MX_BLOCK == 0
    blocks = a.reshape(a.shape[:-1] + (K // MX_BLOCK, MX_BLOCK))
    sc = e8m0_scale_code(np.abs(blocks).max(axis=-1))
    bad = sc == E8M0_NAN
    x_scale = np.ldexp(1.0, np.where(bad, 127, sc.astype(np.int64)) - 127)
    with np.errstate(invalid="ignore"):
        scaled = np.clip(blocks / x_scale[..., None], -E4M3_MAX, E4M3_MAX).astype(np.float32)
    codes = torch.from_numpy(scaled).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    codes = np.where(bad[..., None], np.uint8(E4M3_NAN), codes)
    return codes.reshape(a.shape), sc


def dequantize_mxfp8(codes, scales):
    codes = np.asarray(codes)
    K = codes.shape[-1]
    vals = _e4m3_table()[codes].reshape(codes.shape[:-1] + (K // MX_BLOCK, MX_BLOCK))
    sc = np.asarray(scales).astype(np.int64)
    x_scale = np.where(sc == E8M0_NAN, np.nan, np.ldexp(1.0, np.minimum(sc, 254) - 127))
    return (vals * x_scale[..., None]).reshape(codes.shape)


def token_forward_mxfp8(xq_t, xs_t, wg, wu, wd, ids_t, probs_t):
    """One token of the MXFP8 block. wg/wu/wd are indexable by expert and
    give (codes, scales) of the K-contiguous weights: W1g_e, W1u_e as [F, H]
    with scales [F, H/32], W2_e as [H, F] with scales [H, F/32].

      A_g = deq(x_t) . deq(W1g_e)^T,  A_u likewise
      h   = bf16(silu(A_g) A_u), then quantised per 32 along F
      O   = bf16(deq(h) . deq(W2_e)^T)
      y_t = bf16(sum_j p_tj O_j)
    """
    xd = dequantize_mxfp8(xq_t, xs_t)
    acc = None
    for j, e in enumerate(np.asarray(ids_t).tolist()):
        g = dequantize_mxfp8(*wg[e]) @ xd
        u = dequantize_mxfp8(*wu[e]) @ xd
        h = bf16(silu(g) * u)
        hq, hs = quantize_mxfp8(h)
        o = bf16(dequantize_mxfp8(*wd[e]) @ dequantize_mxfp8(hq, hs))
        term = float(np.asarray(probs_t)[j]) * o
        acc = term if acc is None else acc + term
    return bf16(acc)


def expert_forward_mxfp8(xq, xs, wg, wu, wd, expert_ids, probs, num_experts):
    """Grouped MXFP8 path: permute the quantised rows (with their scales),
    per expert fc1 on dequantised operands, h rounded to bf16 then quantised
    per 32 along F, fc2, combine."""
    counts = expert_counts(expert_ids, num_experts)
    off = expert_offsets(counts)
    row_of, token_of, _ = permute_map(expert_ids, num_experts)
    xd = dequantize_mxfp8(np.asarray(xq)[token_of], np.asarray(xs)[token_of])
    H = np.asarray(wd[0][0]).shape[0]
    o = np.zeros((xd.shape[0], H))
    for e in range(num_experts):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        a_g = xd[lo:hi] @ dequantize_mxfp8(*wg[e]).T
        a_u = xd[lo:hi] @ dequantize_mxfp8(*wu[e]).T
        h = bf16(silu(a_g) * a_u)
        hq, hs = quantize_mxfp8(h)
        o[lo:hi] = bf16(dequantize_mxfp8(hq, hs) @ dequantize_mxfp8(*wd[e]).T)
    return unpermute(o, row_of, probs)


def sampled_forward_mxfp8(x, w_gate_t, w_up_t, w_down_t, expert_ids, probs, tokens):
    """token_forward_mxfp8 for the listed tokens from bf16-valued inputs:
    x [T, H] and the K-contiguous weights W1g, W1u [E, F, H], W2 [E, H, F]
    (indexable by expert) are quantised here, one expert at a time, so that
    only the experts the sampled tokens use are quantised."""
    x = np.asarray(x)
    ids = np.asarray(expert_ids)
    pr = np.asarray(probs)
    tokens = list(tokens)
    xq, xs = quantize_mxfp8(x[tokens])
    xd = {t: dequantize_mxfp8(xq[i], xs[i]) for i, t in enumerate(tokens)}
    o_rows = {}
    for e in sorted(set(int(v) for t in tokens for v in ids[t])):
        wg = dequantize_mxfp8(*quantize_mxfp8(w_gate_t[e]))
        wu = dequantize_mxfp8(*quantize_mxfp8(w_up_t[e]))
        wd = dequantize_mxfp8(*quantize_mxfp8(w_down_t[e]))
        for t in tokens:
            for j, ee in enumerate(ids[t].tolist()):
                if ee == e:
                    h = bf16(silu(wg @ xd[t]) * (wu @ xd[t]))
                    hq, hs = quantize_mxfp8(h)
                    o_rows[(t, j)] = bf16(wd @ dequantize_mxfp8(hq, hs))
    out = []
    for t in tokens:
        acc = None
        for j in range(ids.shape[1]):
            term = float(pr[t, j]) * o_rows[(t, j)]
            acc = term if acc is None else acc + term
        out.append(bf16(acc))
    return np.stack(out)


def quantized_along_rows(a, quantize: bool = True) -> np.ndarray:
    """deq(quant(a)) with blocks of 32 along the last axis (the rule of
    quantize_mxfp8), or a itself when quantize is False."""
    a = _f64(a)
    if not quantize:
        return a
    return dequantize_mxfp8(*quantize_mxfp8(a))


def quantized_along_columns(a, quantize: bool = True) -> np.ndarray:
    """deq(quant(a)) of a [n, C] with blocks of 32 along axis 0: rows
    32 i .. 32 i + 31 of each column share a scale, the blocks start at row 0
    and the last one is completed with zero rows. Returned as [n, C]."""
    a = _f64(a)
    if not quantize:
        return a
    n = a.shape[0]
    pad = (-n) % MX_BLOCK
    if pad:
        a = np.concatenate([a, np.zeros((pad,) + a.shape[1:])])
    return dequantize_mxfp8(*quantize_mxfp8(a.T)).T[:n]


def expert_backward_mxfp8(dy, x, w_gate_t, w_up_t, w_down_t, expert_ids, probs,
                          quantize: bool = True, keep: bool = False):
    """Gradients of the MXFP8 block (FP8 training of the expert block, the
    quantised AllToAll+Matmul of "MC2 通算融合架构总览" section 1 carried to
    the backward). The pages fix no rule for the backward. Reading used
    here: every GEMM runs on MXFP8 operands, each quantised by the
    forward's rule per 32 elements along that GEMM's reduction dimension,
    with the rounding points of expert_backward:

      forward   x quantised along H; W1g_e, W1u_e [F, H] along H;
                A_g = deq(x) deq(W1g_e)^T, A_u likewise; h = bf16(silu(A_g) A_u);
                O = bf16(deq(h quantised along F) deq(W2_e [H, F] along F)^T)
      dO        bf16(p dY_t), one row per routed slot; dp_tj = <dY_t, O_row>
      dH        deq(dO along H) deq(W2_e as [F, H], along H)^T
      dA_g, dA_u  the SwiGLU backward of dH on A_g, A_u as saved (bf16)
      dXp       bf16(deq(dA_g along F) deq(W1g_e as [H, F], along F)^T + the same for up)
      dX        bf16(sum_j dXp[row_of[t, j]])
      dW1g_e^T  deq(dA_g,e along rows)^T deq(Xp_e along rows)   [F, H]
      dW1u_e^T  the same with dA_u,e
      dW2_e^T   deq(dO_e along rows)^T deq(h_e along rows)       [H, F]

    "Along rows" quantises the expert's routed rows (in permuted order) in
    blocks of 32 starting at its first row (quantized_along_columns). Xp_e
    are the bf16 rows of x, h_e the bf16 h. Weights come in the MXFP8
    forward's K-contiguous layout, w_gate_t / w_up_t [E, F, H] and
    w_down_t [E, H, F], and the weight gradients are returned in that
    layout: dw_gate_t, dw_up_t [E, F, H], dw_down_t [E, H, F].

    With quantize=False every deq(quant(.)) is the identity and the result
    is expert_backward's on the same bf16 values. keep=True adds the
    intermediates (row maps, offsets, A_g, A_u, h, O, dO, dH, dA_g, dA_u, dXp)
    under "state".
    """
    q_rows = lambda a: quantized_along_rows(a, quantize)      # noqa: E731
    q_cols = lambda a: quantized_along_columns(a, quantize)   # noqa: E731
    E = len(w_gate_t)
    x, dy = _f64(x), _f64(dy)
    ids = np.asarray(expert_ids)
    pr = _f64(probs)
    T, k = ids.shape
    counts = expert_counts(ids, E)
    off = expert_offsets(counts)
    row_of, token_of, slot_of = permute_map(ids, E)
    prob_of = pr[token_of, slot_of]
    H = x.shape[1]
    F = np.asarray(w_gate_t[0]).shape[0]
    R = T * k
    xd = q_rows(x)[token_of]
    xp = x[token_of]
    a_g, a_u, h = np.zeros((R, F)), np.zeros((R, F)), np.zeros((R, F))
    o = np.zeros((R, H))
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        a_g[lo:hi] = xd[lo:hi] @ q_rows(w_gate_t[e]).T
        a_u[lo:hi] = xd[lo:hi] @ q_rows(w_up_t[e]).T
        h[lo:hi] = bf16(silu(a_g[lo:hi]) * a_u[lo:hi])
        o[lo:hi] = bf16(q_rows(h[lo:hi]) @ q_rows(w_down_t[e]).T)
    y = unpermute(o, row_of, pr)
    d_o = bf16(prob_of[:, None] * dy[token_of])
    dprobs = np.zeros((T, k))
    for j in range(k):
        dprobs[:, j] = np.sum(dy * o[row_of[:, j]], axis=1)
    ag_s, au_s = bf16(a_g), bf16(a_u)
    dxp = np.zeros((R, H))
    dw_gate_t, dw_up_t = np.zeros((E, F, H)), np.zeros((E, F, H))
    dw_down_t = np.zeros((E, H, F))
    dh_all, dag_all, dau_all = np.zeros((R, F)), np.zeros((R, F)), np.zeros((R, F))
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        dh = q_rows(d_o[lo:hi]) @ q_rows(_f64(w_down_t[e]).T).T
        sg = sigmoid(ag_s[lo:hi])
        da_g = bf16(dh * au_s[lo:hi] * sg * (1.0 + ag_s[lo:hi] * (1.0 - sg)))
        da_u = bf16(dh * ag_s[lo:hi] * sg)
        dxp[lo:hi] = bf16(q_rows(da_g) @ q_rows(_f64(w_gate_t[e]).T).T +
                          q_rows(da_u) @ q_rows(_f64(w_up_t[e]).T).T)
        xq_e = q_cols(xp[lo:hi])
        dw_gate_t[e] = q_cols(da_g).T @ xq_e
        dw_up_t[e] = q_cols(da_u).T @ xq_e
        dw_down_t[e] = q_cols(d_o[lo:hi]).T @ q_cols(h[lo:hi])
        dh_all[lo:hi], dag_all[lo:hi], dau_all[lo:hi] = dh, da_g, da_u
    dx = unpermute(dxp, row_of, None)
    out = dict(dx=dx, dw_gate_t=dw_gate_t, dw_up_t=dw_up_t, dw_down_t=dw_down_t,
               dprobs=dprobs, y=y)
    if keep:
        out["state"] = dict(row_of=row_of, token_of=token_of, off=off, a_g=a_g, a_u=a_u, h=h,
                            o=o, d_o=d_o, dh=dh_all, da_g=dag_all, da_u=dau_all, dxp=dxp)
    return out


def backward_rows_mxfp8(dy, x, w_gate_t, w_up_t, w_down_t, expert_ids, probs, tokens):
    """dX and dprobs of the listed tokens of expert_backward_mxfp8.

    A token's data gradients depend only on its own rows, and every
    row-quantised operand (x, h, dO, dA, and the weights) is quantised per
    row, so this is the same arithmetic restricted to those rows. Experts
    are visited one at a time and their weights quantised once."""
    dy, x = np.asarray(dy), np.asarray(x)
    ids = np.asarray(expert_ids)
    pr = np.asarray(probs)
    tokens = list(tokens)
    dxr, dpt = {}, {}
    for e in sorted(set(int(v) for t in tokens for v in ids[t])):
        wg = quantized_along_rows(w_gate_t[e])           # [F, H] along H
        wu = quantized_along_rows(w_up_t[e])
        wd = quantized_along_rows(w_down_t[e])           # [H, F] along F
        w2b = quantized_along_rows(_f64(w_down_t[e]).T)  # [F, H] along H
        w1gb = quantized_along_rows(_f64(w_gate_t[e]).T)  # [H, F] along F
        w1ub = quantized_along_rows(_f64(w_up_t[e]).T)
        for t in tokens:
            for j, ee in enumerate(ids[t].tolist()):
                if ee != e:
                    continue
                xd = quantized_along_rows(x[t])
                a_g, a_u = wg @ xd, wu @ xd
                hv = bf16(silu(a_g) * a_u)
                ov = bf16(wd @ quantized_along_rows(hv))
                dpt[(t, j)] = float(np.dot(_f64(dy[t]), ov))
                d_o = bf16(float(pr[t, j]) * _f64(dy[t]))
                dh = w2b @ quantized_along_rows(d_o)
                ga, ua = bf16(a_g), bf16(a_u)
                sg = sigmoid(ga)
                da_g = bf16(dh * ua * sg * (1.0 + ga * (1.0 - sg)))
                da_u = bf16(dh * ga * sg)
                dxr[(t, j)] = bf16(w1gb @ quantized_along_rows(da_g) +
                                   w1ub @ quantized_along_rows(da_u))
    k = ids.shape[1]
    dx, dp = [], []
    for t in tokens:
        acc = dxr[(t, 0)]
        for j in range(1, k):
            acc = acc + dxr[(t, j)]
        dx.append(bf16(acc))
        dp.append([dpt[(t, j)] for j in range(k)])
    return np.stack(dx), np.array(dp)


def weight_grad_entries_mxfp8(dy, x, w_gate_t, w_up_t, w_down_t, expert_ids, probs, e, pairs):
    """For each (f, h) in pairs, the entries dw_gate_t[e][f, h],
    dw_up_t[e][f, h] and dw_down_t[e][h, f] of expert_backward_mxfp8.

    Each is a sum over the expert's routed rows of two column-quantised
    vectors: column f of dA_g (or dA_u, or h) and column h of Xp (or dO).
    Column f of A_g, A_u and dH over those rows needs only row f of the
    quantised weights, so the full [rows, F] tensors are never formed."""
    dy, x = np.asarray(dy), np.asarray(x)
    ids = np.asarray(expert_ids)
    pr = np.asarray(probs)
    E = len(w_gate_t)
    counts = expert_counts(ids, E)
    off = expert_offsets(counts)
    _, token_of, slot_of = permute_map(ids, E)
    lo, hi = int(off[e]), int(off[e + 1])
    toks = token_of[lo:hi]
    q_col = lambda v: quantized_along_columns(np.asarray(v)[:, None])[:, 0]  # noqa: E731
    xe = _f64(x[toks])
    xd = quantized_along_rows(xe)
    d_o = bf16(_f64(pr[toks, slot_of[lo:hi]])[:, None] * _f64(dy[toks]))
    d_oq = quantized_along_rows(d_o)
    out = []
    for f, h in pairs:
        a_g = xd @ quantized_along_rows(w_gate_t[e][f])
        a_u = xd @ quantized_along_rows(w_up_t[e][f])
        hv = bf16(silu(a_g) * a_u)
        dh = d_oq @ quantized_along_rows(_f64(w_down_t[e])[:, f])
        ga, ua = bf16(a_g), bf16(a_u)
        sg = sigmoid(ga)
        da_g = bf16(dh * ua * sg * (1.0 + ga * (1.0 - sg)))
        da_u = bf16(dh * ga * sg)
        xh = q_col(xe[:, h])
        out.append((float(np.dot(q_col(da_g), xh)), float(np.dot(q_col(da_u), xh)),
                    float(np.dot(q_col(d_o[:, h]), q_col(hv)))))
    return np.array(out).reshape(len(pairs), 3)


def weight_grad_slices_mxfp8(dy, x, w_gate_t, w_up_t, w_down_t, expert_ids, probs, e, f_cols):
    """Whole slices of expert e's weight gradients in expert_backward_mxfp8,
    for each f in f_cols: the rows dw_gate_t[e][f, :] and dw_up_t[e][f, :]
    and the column dw_down_t[e][:, f], each over all H.

    They need column f of A_g, A_u, h and dH over the expert's routed rows
    (row f of the quantised weights) and the column-quantised Xp_e and dO_e
    [rows, H], so the [rows, F] tensors are never formed. Returns a dict of
    [len(f_cols), H] arrays."""
    dy, x = np.asarray(dy), np.asarray(x)
    ids = np.asarray(expert_ids)
    pr = np.asarray(probs)
    E = len(w_gate_t)
    counts = expert_counts(ids, E)
    off = expert_offsets(counts)
    _, token_of, slot_of = permute_map(ids, E)
    lo, hi = int(off[e]), int(off[e + 1])
    toks = token_of[lo:hi]
    xe = _f64(x[toks])
    xd = quantized_along_rows(xe)                        # fc1's A: along H
    xq_cols = quantized_along_columns(xe)                # dW1's B: along the rows
    d_o = bf16(_f64(pr[toks, slot_of[lo:hi]])[:, None] * _f64(dy[toks]))
    d_oq = quantized_along_rows(d_o)                     # dH's A: along H
    do_cols = quantized_along_columns(d_o)               # dW2's A: along the rows
    q_col = lambda v: quantized_along_columns(np.asarray(v)[:, None])[:, 0]  # noqa: E731
    out = {"dw_gate_t": [], "dw_up_t": [], "dw_down_t": []}
    for f in f_cols:
        a_g = xd @ quantized_along_rows(w_gate_t[e][f])
        a_u = xd @ quantized_along_rows(w_up_t[e][f])
        hv = bf16(silu(a_g) * a_u)
        dh = d_oq @ quantized_along_rows(_f64(w_down_t[e])[:, f])
        ga, ua = bf16(a_g), bf16(a_u)
        sg = sigmoid(ga)
        da_g = bf16(dh * ua * sg * (1.0 + ga * (1.0 - sg)))
        da_u = bf16(dh * ga * sg)
        out["dw_gate_t"].append(q_col(da_g) @ xq_cols)
        out["dw_up_t"].append(q_col(da_u) @ xq_cols)
        out["dw_down_t"].append(q_col(hv) @ do_cols)
    return {key: np.array(v) for key, v in out.items()}


# --------------------------------------------------------------------------
# micro-batch split
# --------------------------------------------------------------------------

def microbatched_forward(x, w_gate, w_up, w_down, expert_ids, probs, splits: int):
    """Split the tokens into `splits` contiguous equal chunks, run the block
    on each, and reassemble in token order."""
    x = np.asarray(x)
    T = x.shape[0]
    assert T % splits == 0
    n = T // splits
    ids, pr = np.asarray(expert_ids), np.asarray(probs)
    return np.concatenate([expert_forward(x[i * n:(i + 1) * n], w_gate, w_up, w_down,
                                          ids[i * n:(i + 1) * n], pr[i * n:(i + 1) * n],
                                          len(w_gate))
                           for i in range(splits)])


def microbatched_backward(dy, x, w_gate, w_up, w_down, expert_ids, probs, splits: int):
    """Backward on `splits` contiguous chunks: dX and dprobs concatenated,
    weight gradients summed over chunks in chunk order."""
    x, dy = np.asarray(x), np.asarray(dy)
    T = x.shape[0]
    assert T % splits == 0
    n = T // splits
    ids, pr = np.asarray(expert_ids), np.asarray(probs)
    parts = [expert_backward(dy[i * n:(i + 1) * n], x[i * n:(i + 1) * n], w_gate, w_up, w_down,
                             ids[i * n:(i + 1) * n], pr[i * n:(i + 1) * n])
             for i in range(splits)]
    out = dict(dx=np.concatenate([p["dx"] for p in parts]),
               dprobs=np.concatenate([p["dprobs"] for p in parts]))
    for key in ("dw_gate", "dw_up", "dw_down"):
        acc = parts[0][key]
        for p in parts[1:]:
            acc = acc + p[key]
        out[key] = acc
    return out
