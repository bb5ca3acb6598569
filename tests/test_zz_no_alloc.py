"""The allocation-free batched Newton-Schulz entry point.

Callers that may not allocate device memory -- a framework whose caching
allocator must own every allocation, a process whose memory budget is planned
before it starts -- use muon_ns_batched_noalloc, whose workspace is a fixed
array inside the library.  Through the C ABI this file checks that two calls
in a row agree with the allocating muon_ns_batched on the same input within
the NS tolerance, that the result matches the float64 oracle, that steps = 0
returns X / ||X||_F, that a non-finite input is reported by muon_query_status,
and that oversize or bad arguments are refused.  It is named so that pytest
collects it after every other test file.
"""
import ctypes

import numpy as np
import pytest
import torch

from newton_schulz_gb300 import binding
from oracle import muon_ref as R

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


def _np(t):
    return t.double().cpu().numpy()


def _rel(a, b):
    a, b = _np(a), np.asarray(b, np.float64)
    return max(np.linalg.norm(a[i] - b[i]) / np.linalg.norm(b[i]) for i in range(a.shape[0]))


def _input(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.bfloat16).cuda()


@pytest.mark.parametrize("shape", [(3, 96, 200), (2, 333, 130), (4, 24, 2048)])
def test_noalloc_matches_allocating_entry_point(lib, cuda_ok, shape):
    lib = _lib()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):      # two calls in a row share (and reuse) the fixed array
        x = _input(shape, 100 * call + sum(shape))
        ref = x.clone()
        got = x.clone()
        B, M, N = shape
        assert lib.muon_ns_batched(ref.data_ptr(), B, M, N, 5, *ABC, stream) == 0
        assert lib.muon_ns_batched_noalloc(got.data_ptr(), B, M, N, 5, *ABC, stream) == 0
        torch.cuda.synchronize()
        assert binding.muon_query_status() == 0
        assert torch.isfinite(got.float()).all()
        assert _rel(got, _np(ref)) <= NS_TOL


@pytest.mark.parametrize("shape", [(3, 96, 200), (2, 333, 130)])   # wide, tall (transposed)
def test_noalloc_matches_oracle(lib, cuda_ok, shape):
    lib = _lib()
    stream = torch.cuda.current_stream().cuda_stream
    x = _input(shape, 7 + sum(shape))
    want = R.ns_batched_ref(_np(x))
    B, M, N = shape
    assert lib.muon_ns_batched_noalloc(x.data_ptr(), B, M, N, 5, *ABC, stream) == 0
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 0
    assert _rel(x, want) <= NS_TOL


def test_noalloc_zero_steps_is_normalised_input(lib, cuda_ok):
    """steps = 0: X0 = X / (||X||_F + eps) per matrix (the copy-back applies
    the norm's reciprocal; bf16 output, so one bf16 rounding apart)."""
    lib = _lib()
    stream = torch.cuda.current_stream().cuda_stream
    x = _input((3, 40, 90), 11)
    want = R.ns_batched_ref(_np(x), steps=0)
    assert lib.muon_ns_batched_noalloc(x.data_ptr(), 3, 40, 90, 0, *ABC, stream) == 0
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 0
    assert _rel(x, want) <= 5e-3


def test_noalloc_reports_nonfinite_input(lib, cuda_ok):
    lib = _lib()
    stream = torch.cuda.current_stream().cuda_stream
    x = _input((2, 64, 96), 12)
    x[1, 5, 7] = float("nan")
    assert lib.muon_ns_batched_noalloc(x.data_ptr(), 2, 64, 96, 5, *ABC, stream) == 0
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 7            # MUON_ERR_NONFINITE
    assert binding.muon_query_status() == 0            # the read cleared it
    y = _input((2, 64, 96), 13)
    assert lib.muon_ns_batched_noalloc(y.data_ptr(), 2, 64, 96, 5, *ABC, stream) == 0
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 0


def test_noalloc_rejects_oversize_and_bad_args(lib, cuda_ok):
    lib = _lib()
    stream = torch.cuda.current_stream().cuda_stream
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    # a [64, 1024, 1024] problem needs far more than the fixed array; nothing runs
    assert lib.muon_ns_batched_noalloc(x.data_ptr(), 64, 1024, 1024, 5, *ABC, stream) == 2
    assert lib.muon_ns_batched_noalloc(None, 1, 4, 4, 5, *ABC, stream) == 1
    assert lib.muon_ns_batched_noalloc(x.data_ptr(), 1, 4, 4, -1, *ABC, stream) == 1
    assert lib.muon_ns_batched_noalloc(x.data_ptr(), 0, 4, 4, 5, *ABC, stream) == 0
