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
