"""moe_build_permutation_static, the entry point for callers that cannot
allocate device memory on the call path (for example a host runtime that owns
every device buffer, or a hot loop that must not call cudaMalloc because it
synchronises the device). It keeps its chunk histogram in the library's fixed
device array instead of a caller workspace.

Called through the C ABI and compared bit-exactly (integer outputs) with the
workspace entry point moe_build_permutation, on two calls in a row so that the
second runs over the array the first left behind. This file sorts last so a
run that stops at the first failure has run every other test first; it also
passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from grouped_gemm_moe_gb300 import binding as B

from _parity import ensure_built

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _static_call(lib, idx, E):
    T, K = idx.shape
    dev = idx.device
    counts = torch.full((E,), -7, dtype=torch.int32, device=dev)
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device=dev)
    perm = torch.full((T * K,), -7, dtype=torch.int32, device=dev)
    inv = torch.full((T * K,), -7, dtype=torch.int32, device=dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    rc = lib.moe_build_permutation_static(_ptr(idx), T, E, K, _ptr(counts), _ptr(offsets),
                                          _ptr(perm), _ptr(inv), stream)
    assert rc == B.MOE_OK, lib.moe_status_string(rc)
    return counts, offsets, perm, inv


def test_static_scratch_matches_workspace_entry_point_twice():
    ensure_built()
    lib = B.load()
    dev = torch.device("cuda:0")
    cases = [(8192, 128, 8, 0), (20000, 64, 6, 1)]     # second call: different shape and data
    for T, E, K, seed in cases:
        rng = np.random.default_rng(seed)
        idx = torch.from_numpy(np.stack([rng.permutation(E)[:K] for _ in range(T)])
                               .astype(np.int32)).to(dev)
        got = _static_call(lib, idx, E)
        want = B.moe_build_permutation(idx, E)
        torch.cuda.synchronize()
        for g, w, name in zip(got, want, ("counts", "offsets", "perm", "inv_perm")):
            assert torch.equal(g, w), name


def test_static_scratch_rejects_problems_beyond_its_size():
    ensure_built()
    lib = B.load()
    fake = ctypes.c_void_p(0x10000)   # never dereferenced: the size check comes first
    E, K = 1024, 8
    T = ((1 << 18) // E + 1) * 1024 // K      # one chunk row more than the array holds
    rc = lib.moe_build_permutation_static(fake, T, E, K, fake, fake, fake, fake, None)
    assert rc == B.MOE_ERR_WORKSPACE
