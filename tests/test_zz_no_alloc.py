"""The allocation-free batched Newton-Schulz entry point.

Callers that may not allocate device memory (a framework whose caching
allocator must own every allocation, a process with a pre-planned memory
budget) use muon_ns_batched_noalloc, whose workspace is a fixed array inside
the library.  This file checks, through the C ABI, that two calls in a row
give the same result as the allocating muon_ns_batched on the same input.
It is named so that pytest collects it after every other test file.
"""
import ctypes

import numpy as np
import pytest
import torch

from newton_schulz_gb300 import binding

pytestmark = pytest.mark.gpu

NS_TOL = 3e-2   # the NS tolerance the other parity tests use
ABC = (3.4445, -4.7750, 2.0315)


def _lib():
    lib = binding.load()
    f = lib.muon_ns_batched_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                  ctypes.c_float, ctypes.c_float, ctypes.c_float, ctypes.c_void_p]
    f.restype = ctypes.c_int32
    return lib


def _rel(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return max(np.linalg.norm(a[i] - b[i]) / np.linalg.norm(b[i]) for i in range(a.shape[0]))


@pytest.mark.parametrize("shape", [(3, 96, 200), (2, 333, 130), (4, 24, 2048)])
def test_noalloc_matches_allocating_entry_point(lib, cuda_ok, shape):
    lib = _lib()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):      # two calls in a row share (and reuse) the fixed array
        g = torch.Generator().manual_seed(100 * call + sum(shape))
        x = torch.randn(shape, generator=g).to(torch.bfloat16).cuda()
        ref = x.clone()
        got = x.clone()
        B, M, N = shape
        assert lib.muon_ns_batched(ref.data_ptr(), B, M, N, 5, *ABC, stream) == 0
        assert lib.muon_ns_batched_noalloc(got.data_ptr(), B, M, N, 5, *ABC, stream) == 0
        torch.cuda.synchronize()
        assert torch.isfinite(got.float()).all()
        assert _rel(got, ref) <= NS_TOL


def test_noalloc_rejects_oversize_and_bad_args(lib, cuda_ok):
    lib = _lib()
    stream = torch.cuda.current_stream().cuda_stream
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    # a [64, 1024, 1024] problem needs far more than the fixed array; nothing runs
    assert lib.muon_ns_batched_noalloc(x.data_ptr(), 64, 1024, 1024, 5, *ABC, stream) == 2
    assert lib.muon_ns_batched_noalloc(None, 1, 4, 4, 5, *ABC, stream) == 1
    assert lib.muon_ns_batched_noalloc(x.data_ptr(), 1, 4, 4, -1, *ABC, stream) == 1
    assert lib.muon_ns_batched_noalloc(x.data_ptr(), 0, 4, 4, 5, *ABC, stream) == 0
