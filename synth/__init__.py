"""Seeded synthetic inputs for the MoE expert block.

This module draws random tensors and routing decisions. It holds none of the
expert block's own arithmetic (no counting, permuting, matmul, activation,
combine or quantisation): both the CPU oracle and the CUDA path receive what
it returns, as plain host tensors, and compute from there.

Random numbers come from NumPy's Philox4x32-10 counter-based generator
(Salmon et al., "Parallel random numbers: as easy as 1, 2, 3", SC'11), one
independent stream per (seed, tensor id, chunk) so that large tensors are
drawn in parallel threads yet stay identical run to run.

Workloads (shapes and distributions) follow the five expert-block
configurations: a tiny BF16 block, a Mixtral-8x7B-shaped layer, a
fine-grained skewed layer, an MXFP8 layer and a Mixtral-shaped training step.
The pages measured Mixtral 8x7B / LLaMA models with trained weights and real
data; those are not available here and these seeded inputs stand in for them.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os

import numpy as np
import torch

_CHUNK = 1 << 24  # elements per independent stream


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int          # tokens
    H: int          # hidden size
    F: int          # ffn size
    E: int          # experts
    k: int          # experts per token (top-k)
    routing: str    # "router" | "gaussian" | "zipf" | "uniform"
    w_std: float    # std of the expert weights
    mxfp8: bool = False
    backward: bool = False

    @property
    def R(self) -> int:
        return self.T * self.k

    def resized(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny_bf16": Workload("tiny_bf16", 256, 512, 1024, 8, 2, "router", 0.02),
    "mixtral_bf16": Workload("mixtral_bf16", 4096, 4096, 14336, 8, 2, "gaussian", 0.01),
    "skewed_bf16": Workload("skewed_bf16", 8192, 2048, 768, 128, 8, "zipf", 0.01),
    "mxfp8": Workload("mxfp8", 16384, 7168, 2048, 64, 6, "uniform", 0.02, mxfp8=True),
    "train_bf16": Workload("train_bf16", 16384, 4096, 14336, 8, 2, "gaussian", 0.01, backward=True),
    # a smaller Mixtral-shaped case (2 experts, every token on both) for
    # profiler captures that must hold only about 1 GB on the device
    "mixtral_2experts": Workload("mixtral_2experts", 2048, 4096, 14336, 2, 2, "gaussian", 0.01),
    "mxfp8_16experts": Workload("mxfp8_16experts", 4096, 7168, 2048, 16, 6, "uniform", 0.02,
                                mxfp8=True),
    "train_2experts": Workload("train_2experts", 2048, 4096, 14336, 2, 2, "gaussian", 0.01,
                               backward=True),
    # the training workload in MXFP8 (FP8 training of the expert block), and
    # its 2-expert profiling case
    "train_mxfp8": Workload("train_mxfp8", 16384, 4096, 14336, 8, 2, "gaussian", 0.01,
                            mxfp8=True, backward=True),
    "train_mxfp8_2experts": Workload("train_mxfp8_2experts", 2048, 4096, 14336, 2, 2, "gaussian",
                                     0.01, mxfp8=True, backward=True),
}

# Zipf exponent and the number of experts given zero popularity in the
# skewed workload (so that at least that many experts receive no token).
ZIPF_ALPHA = 1.2
ZIPF_ZERO_EXPERTS = 5


def _gen(seed: int, tensor_id: int, chunk: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, tensor_id, chunk])))


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def normal_f32(seed: int, tensor_id: int, n: int, std: float = 1.0) -> np.ndarray:
    """n draws of N(0, std^2) as float32, filled chunk by chunk in threads."""
    out = np.empty(n, dtype=np.float32)
    nchunks = (n + _CHUNK - 1) // _CHUNK

    def fill(c):
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        g = _gen(seed, tensor_id, c)
        g.standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])
        if std != 1.0:
            out[lo:hi] *= np.float32(std)

    if nchunks <= 1:
        for c in range(nchunks):
            fill(c)
    else:
        with _cf.ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(nchunks)))
    return out


def normal_bf16(seed: int, tensor_id: int, shape, std: float = 1.0) -> torch.Tensor:
    """A bf16 host tensor of N(0, std^2) draws (float32 draw, then cast)."""
    n = int(np.prod(shape))
    a = normal_f32(seed, tensor_id, n, std)
    return torch.from_numpy(a).to(torch.bfloat16).reshape(shape)


def _softmax_rows(logits: np.ndarray) -> np.ndarray:
    z = logits - logits.max(axis=1, keepdims=True)
    p = np.exp(z)
    return p / p.sum(axis=1, keepdims=True)


def _topk_desc(scores: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest scores per row, largest first; ties go to the
    lower expert index (a stable sort on the negated score)."""
    order = np.argsort(-scores, axis=1, kind="stable")
    return order[:, :k]


def routing(w: Workload, seed: int, x: torch.Tensor | None = None):
    """(expert_ids int32 [T,k], probs float32 [T,k]) for a workload.

    router   : logits = x @ Wr, Wr ~ N(0, 0.02) [H, E]; top-k; softmax over the k.
    gaussian : logits ~ N(0,1) [T, E]; top-k; softmax over the k.
    zipf     : k experts drawn without replacement with Zipf(1.2) popularity
               over a seeded permutation of the experts, the last five of
               which get popularity 0 (Gumbel-top-k sampling); probs are a
               softmax of N(0,1) logits over the chosen k.
    uniform  : k of E uniformly without replacement; probs ~ Dirichlet(1)
               (k iid Exp(1) draws, normalised).
    """
    T, E, k = w.T, w.E, w.k
    g = _gen(seed, 100, 0)
    if w.routing == "router":
        assert x is not None
        wr = normal_f32(seed, 101, w.H * E, 0.02).astype(np.float64).reshape(w.H, E)
        logits = x.float().numpy().astype(np.float64) @ wr
        ids = _topk_desc(logits, k)
        chosen = np.take_along_axis(logits, ids, axis=1)
        probs = _softmax_rows(chosen)
    elif w.routing == "gaussian":
        logits = g.standard_normal((T, E))
        ids = _topk_desc(logits, k)
        probs = _softmax_rows(np.take_along_axis(logits, ids, axis=1))
    elif w.routing == "zipf":
        perm = g.permutation(E)
        pop = np.zeros(E)
        live = E - ZIPF_ZERO_EXPERTS
        pop[perm[:live]] = np.arange(1, live + 1, dtype=np.float64) ** (-ZIPF_ALPHA)
        with np.errstate(divide="ignore"):
            logpop = np.log(pop)
        gumbel = -np.log(-np.log(g.random((T, E))))
        keys = logpop[None, :] + gumbel
        ids = _topk_desc(keys, k)
        probs = _softmax_rows(g.standard_normal((T, k)))
    elif w.routing == "uniform":
        keys = g.random((T, E))
        ids = _topk_desc(keys, k)
        ex = g.exponential(1.0, (T, k))
        probs = ex / ex.sum(axis=1, keepdims=True)
    else:
        raise ValueError(w.routing)
    return (torch.from_numpy(np.ascontiguousarray(ids.astype(np.int32))),
            torch.from_numpy(np.ascontiguousarray(probs.astype(np.float32))))


def router_logits(w: Workload, seed: int, x: torch.Tensor | None = None) -> torch.Tensor | None:
    """float32 router logits [T, E] of the 'router' and 'gaussian' routings
    (the same draws routing() ranks, rounded to float32); None for the
    routings that sample experts directly ('zipf', 'uniform')."""
    g = _gen(seed, 100, 0)
    if w.routing == "router":
        assert x is not None
        wr = normal_f32(seed, 101, w.H * w.E, 0.02).astype(np.float64).reshape(w.H, w.E)
        logits = x.float().numpy().astype(np.float64) @ wr
    elif w.routing == "gaussian":
        logits = g.standard_normal((w.T, w.E))
    else:
        return None
    return torch.from_numpy(np.ascontiguousarray(logits.astype(np.float32)))


def make_inputs(w: Workload, seed: int = 0, with_dy: bool | None = None) -> dict:
    """All host inputs of one workload.

    BF16 workloads: x [T,H], w_gate/w_up [E,H,F], w_down [E,F,H] (N
    contiguous, as the pages' mc2_fused_expert weights).
    MXFP8 workload: the same draws but the weights are laid out K-contiguous,
    w_gate_t/w_up_t [E,F,H] and w_down_t [E,H,F], still in bf16; quantising
    them is the block's own work and happens downstream.
    """
    T, H, F, E = w.T, w.H, w.F, w.E
    out = {"workload": w}
    out["x"] = normal_bf16(seed, 1, (T, H), 1.0)
    if w.mxfp8:
        out["w_gate_t"] = normal_bf16(seed, 2, (E, F, H), w.w_std)
        out["w_up_t"] = normal_bf16(seed, 3, (E, F, H), w.w_std)
        out["w_down_t"] = normal_bf16(seed, 4, (E, H, F), w.w_std)
    else:
        out["w_gate"] = normal_bf16(seed, 2, (E, H, F), w.w_std)
        out["w_up"] = normal_bf16(seed, 3, (E, H, F), w.w_std)
        out["w_down"] = normal_bf16(seed, 4, (E, F, H), w.w_std)
    ids, probs = routing(w, seed, out["x"])
    out["expert_ids"], out["probs"] = ids, probs
    if with_dy if with_dy is not None else w.backward:
        out["dy"] = normal_bf16(seed, 5, (T, H), 1.0)
    return out


# Small-integer inputs of the BF16 block whose arithmetic is exact (see
# exact_inputs): the gate bias, and the nonzero entries per weight column.
EXACT_GATE_BIAS = 44
EXACT_GATE_NNZ = 4
EXACT_UP_NNZ = 6
EXACT_DOWN_NNZ = 8


def _sparse_columns(g: np.random.Generator, E: int, K: int, N: int, nnz: int,
                    row0: int) -> np.ndarray:
    """int8 [E, K, N]: in every column (e, :, n), nnz draws of +-1 added at
    rows drawn uniformly from [row0, K) (two draws may land on one row)."""
    w = np.zeros((E, K, N), dtype=np.int8)
    rows = g.integers(row0, K, size=(E, nnz, N))
    signs = (2 * g.integers(0, 2, size=(E, nnz, N)) - 1).astype(np.int8)
    e_idx = np.broadcast_to(np.arange(E)[:, None, None], rows.shape)
    n_idx = np.broadcast_to(np.arange(N)[None, None, :], rows.shape)
    np.add.at(w, (e_idx, rows, n_idx), signs)
    return w


def exact_inputs(w: Workload, seed: int = 0) -> dict:
    """Inputs of the block (with dY) whose arithmetic is exact in float32.

    Shapes and routing are the workload's (routing() draws ids as usual), but
    every value is a small integer or a dyadic fraction:
      x     in {-1, 0, 1}, with column 0 fixed at 1 (a bias input);
      W1g   row 0 = EXACT_GATE_BIAS, plus EXACT_GATE_NNZ draws of +-1 per
            column in rows 1..H-1, so every gate pre-activation lies in
            [bias - nnz, bias + nnz] = [40, 48];
      W1u   row 0 in {-2..2}, plus EXACT_UP_NNZ draws of +-1 per column;
      W2    EXACT_DOWN_NNZ draws of +-1 per output column, over all F rows;
      probs dyadic: k positive multiples of 2^-m summing to 1;
      dY    in {-1, 0, 1}.
    A gate input of 40 or more puts exp(-z) below half an ulp of 1 in float64
    (and in float32), so silu(z) = z and the sigmoid is exactly 1 on both the
    GPU and the oracle, and every product and partial sum of the block and its
    backward is an integer or a multiple of 2^-m far below 2^24 units. Both
    sides then round the same real numbers at the same points, and any
    remaining difference is a mistake, not rounding.
    MXFP8 workloads get the same values with the weights laid out
    K-contiguous, as make_inputs lays them out (w_gate_t, w_up_t [E,F,H],
    w_down_t [E,H,F]). A 32-element block of x or of a weight row then holds
    integers of magnitude at most 44; under the E8M0 scale that its largest
    sets, each of them is an E4M3 value, so quantising them is exact.
    """
    T, H, F, E, k = w.T, w.H, w.F, w.E, w.k
    g = _gen(seed, 200, 0)
    x = g.integers(-1, 2, size=(T, H)).astype(np.int8)
    x[:, 0] = 1
    wg = _sparse_columns(_gen(seed, 201, 0), E, H, F, EXACT_GATE_NNZ, 1)
    wg[:, 0, :] = EXACT_GATE_BIAS
    wu = _sparse_columns(_gen(seed, 202, 0), E, H, F, EXACT_UP_NNZ, 1)
    wu[:, 0, :] = _gen(seed, 203, 0).integers(-2, 3, size=(E, F))
    wd = _sparse_columns(_gen(seed, 204, 0), E, F, H, EXACT_DOWN_NNZ, 0)
    dy = _gen(seed, 205, 0).integers(-1, 2, size=(T, H)).astype(np.int8)
    # dyadic routing weights: a random composition of 2^m into k positive parts
    m = max(2, int(np.ceil(np.log2(k))) + 1)
    gp = _gen(seed, 206, 0)
    cuts = np.sort(np.stack([gp.choice(np.arange(1, 2 ** m), k - 1, replace=False)
                             for _ in range(T)]), axis=1) if k > 1 else np.zeros((T, 0), int)
    edges = np.concatenate([np.zeros((T, 1), int), cuts, np.full((T, 1), 2 ** m)], axis=1)
    probs = (np.diff(edges, axis=1) / 2.0 ** m).astype(np.float32)
    ids, _ = routing(w, seed, torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
                     if w.routing == "router" else None)
    bf = lambda a: torch.from_numpy(a).to(torch.bfloat16)  # noqa: E731
    out = {"workload": w, "x": bf(x), "expert_ids": ids, "probs": torch.from_numpy(probs),
           "dy": bf(dy)}
    if w.mxfp8:
        kc = lambda a: bf(np.ascontiguousarray(a.transpose(0, 2, 1)))  # noqa: E731
        out.update(w_gate_t=kc(wg), w_up_t=kc(wu), w_down_t=kc(wd))
    else:
        out.update(w_gate=bf(wg), w_up=bf(wu), w_down=bf(wd))
    return out


class F32Slices:
    """Indexable view that hands out one expert's weights at a time as a
    float32 NumPy array (bf16 -> f32 is exact), so that callers never hold a
    float copy of every expert at once."""

    def __init__(self, t: torch.Tensor):
        self.t = t

    def __len__(self):
        return self.t.shape[0]

    def __getitem__(self, e):
        return self.t[e].float().numpy()


def bf16_to_f32(t: torch.Tensor) -> np.ndarray:
    return t.float().numpy()
