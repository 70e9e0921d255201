"""moe_counts_static, the counting entry point for callers that cannot
allocate device memory at call time (its scratch is a fixed array inside the
library), against the CPU oracle and against moe_counts with a caller
workspace: identical counts and offsets on two calls in a row, no device
memory taken by a call, and a clear error past its size limit.

Kept in a file that pytest collects last, so that a run stopping at the
first failure has run every other test before this one."""
import ctypes

import numpy as np
import pytest
import torch

import oracle as orc

pytestmark = pytest.mark.gpu
m = pytest.importorskip("moe_expert_dispatch_gb300")


def _via_c_abi(ids: torch.Tensor, E: int):
    counts = torch.full((E,), -7, dtype=torch.int32, device="cuda")
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    st = m._lib.moe_counts_static(ctypes.c_void_p(ids.data_ptr()), ids.numel(), E,
                                  ctypes.c_void_p(counts.data_ptr()),
                                  ctypes.c_void_p(offsets.data_ptr()),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, st
    return counts, offsets


def test_counts_static_matches_workspace_counts_twice():
    rng = np.random.default_rng(2024)
    cases = [(rng.integers(0, 128, (8192, 8)), 128),      # first call: many chunks, many experts
             (rng.integers(0, 8, (4096, 2)), 8)]           # second call: fewer chunks, reuses the array
    for ids_np, E in cases:
        ids = torch.from_numpy(ids_np.astype(np.int32)).cuda()
        want_c, want_o = m.moe_counts(ids, E)
        got_c, got_o = _via_c_abi(ids, E)
        assert m.moe_get_error() == 0
        assert torch.equal(got_c, want_c)
        assert torch.equal(got_o, want_o)
        ref_c = orc.expert_counts(ids_np, E)
        assert np.array_equal(got_c.cpu().numpy(), ref_c)
        assert np.array_equal(got_o.cpu().numpy(), orc.expert_offsets(ref_c))


def test_counts_static_takes_no_device_memory():
    """After one call on the device (which loads its kernels and looks up
    the scratch address), a call with preallocated outputs changes neither
    the device's free memory nor what torch has allocated."""
    ids = torch.from_numpy(np.random.default_rng(7).integers(0, 64, (4096, 6))
                           .astype(np.int32)).cuda()
    _via_c_abi(ids, 64)
    counts = torch.empty(64, dtype=torch.int32, device="cuda")
    offsets = torch.empty(65, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    st = m._lib.moe_counts_static(ctypes.c_void_p(ids.data_ptr()), ids.numel(), 64,
                                  ctypes.c_void_p(counts.data_ptr()),
                                  ctypes.c_void_p(offsets.data_ptr()),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert st == 0
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_allocated() == alloc0
    assert int(counts.sum()) == ids.numel()


def test_counts_static_rejects_sizes_past_its_scratch():
    E = 1024
    n = 2048 * 64 + 1                      # 65 chunks x 1024 experts > 65536 entries
    ids = torch.zeros(n, dtype=torch.int32, device="cuda")
    out = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    st = m._lib.moe_counts_static(ctypes.c_void_p(ids.data_ptr()), n, E,
                                  ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                  None)
    assert st == 4
