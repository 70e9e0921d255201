"""Helpers shared by the GPU tests: device transfer and the tolerance of the
BF16 path, |got - ref| <= 1e-2 + 1e-2 |ref| elementwise."""
import numpy as np
import torch

ATOL = 1e-2
RTOL = 1e-2


def dev(t):
    return t.cuda() if t is not None else None


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_bf16_close(got, ref, what="", atol=ATOL, rtol=RTOL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first at "
                             f"{tuple(i)} got {got[tuple(i)]} ref {ref[tuple(i)]}")


def bf16_step(v):
    """The spacing of bfloat16 values at |v| (8 significant bits); 0 at 0."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.ldexp(1.0, (np.maximum(e, -126) - 7).astype(np.int64)), 0.0)


def check_dx(got, ref, dxp_rows, what="dx"):
    """dX = bf16(sum_j dXp_j) where every dXp_j is itself rounded to bf16.
    Where the GPU's float32 value of a dXp_j and the oracle's float64 one lie
    on two sides of a bf16 rounding boundary, the two roundings differ by one
    bf16 step of dXp_j, and that step survives the k-way sum even when the
    rows nearly cancel. So every element must lie within the BF16 bound
    widened by one step of each of its rows (sum_j bf16_step(dXp_j)); the
    elements outside the unwidened bound are counted and returned, for the
    caller to hold against the count it expects."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    widened = bound + bf16_step(dxp_rows).sum(axis=1)
    bad = err > widened
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside the widened bound; "
                             f"first at {i} got {got[i]} ref {ref[i]}")
    return int((err > bound).sum())


def assert_rel_to_max(got, ref, tol, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    m = np.max(np.abs(ref))
    e = np.max(np.abs(got - ref))
    assert e <= tol * m, f"{what}: max err {e} > {tol} * max|ref| {m}"


def f32_slices(t):
    class S:
        def __getitem__(self, e):
            return t[e].float().numpy()

        def __len__(self):
            return t.shape[0]
    return S()
