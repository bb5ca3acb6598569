"""The failure path of the bounded device-side waits, without a GPU fault.

Every wait in the library's kernels gives up after MUON_WAIT_TIMEOUT_MS: the
kernel then sets MUON_ERR_TIMEOUT in the status word, waits (bounded) for its
own copies and MMAs in flight, frees its tensor memory and returns.  The
testing hook muon_debug_inject_stall makes the next launch of one kind wait on
something nothing provides (a pipeline stage never armed, a matrix never
published), so the bound runs out; nothing traps and nothing is left running.
Each test checks that the call returns, that the status word reports the
timeout (once: reading clears it), and that the next clean call gives the
same bits as a clean call made before the stall (the workspace counters and
the small-m path's launch tags recover).  The wait bound is set to 50 ms for
the stalled launch.
"""
import pytest
import torch

from newton_schulz_gb300 import binding, synth

pytestmark = pytest.mark.gpu
HP = dict(mu=0.95, nesterov=True, lr=0.02, wd=0.01, scale_rule=0)
TIMEOUT = 6


@pytest.fixture(autouse=True)
def _dev(lib, cuda_ok):
    yield
    binding.muon_debug_inject_stall(binding.INJECT_NONE)
    torch.cuda.synchronize()
    assert binding.muon_query_status() in (0, TIMEOUT)


def _copies(shape, n=3):
    g = synth.random_group(shape, torch.bfloat16, torch.float32, "cuda", sum(shape), 1e-3, 1e-3)
    return [{k: g[k].clone() for k in ("W", "G", "Mom")} for _ in range(n)]


@pytest.mark.parametrize("kind,shape", [
    (binding.INJECT_GEMM, (3, 200, 333)),     # grouped GEMM path (Gram launch of step 1)
    (binding.INJECT_SMALL, (12, 24, 4096)),   # small-m path (its last matrix withheld)
])
def test_step_stall_times_out_and_recovers(kind, shape, monkeypatch):
    ref, stalled, again = _copies(shape)
    binding.muon_step_grouped([ref], **HP)
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 0
    monkeypatch.setenv("MUON_WAIT_TIMEOUT_MS", "50")
    binding.muon_debug_inject_stall(kind)
    binding.muon_step_grouped([stalled], **HP)
    torch.cuda.synchronize()
    assert binding.muon_query_status() == TIMEOUT
    assert binding.muon_query_status() == 0            # the read cleared it
    monkeypatch.delenv("MUON_WAIT_TIMEOUT_MS")
    binding.muon_step_grouped([again], **HP)
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 0
    assert torch.equal(again["W"], ref["W"]) and torch.equal(again["Mom"], ref["Mom"])


def test_ns_stall_in_gemm_path_times_out_and_recovers(monkeypatch):
    x = torch.randn((2, 300, 300), generator=torch.Generator().manual_seed(4)).cuda()
    ref, out = torch.empty_like(x), torch.empty_like(x)
    binding.muon_ns_batched_ex(x, binding.make_config(), ref)
    monkeypatch.setenv("MUON_WAIT_TIMEOUT_MS", "50")
    binding.muon_debug_inject_stall(binding.INJECT_GEMM)
    binding.muon_ns_batched_ex(x, binding.make_config(), out)
    torch.cuda.synchronize()
    assert binding.muon_query_status() == TIMEOUT
    monkeypatch.delenv("MUON_WAIT_TIMEOUT_MS")
    binding.muon_ns_batched_ex(x, binding.make_config(), out)
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 0
    assert torch.equal(out, ref)


def test_pending_request_is_one_shot_and_cancellable():
    shape = (2, 200, 333)
    a, b = _copies(shape, 2)
    binding.muon_debug_inject_stall(binding.INJECT_GEMM)
    binding.muon_debug_inject_stall(binding.INJECT_NONE)   # cancelled before any launch
    binding.muon_step_grouped([a], **HP)
    binding.muon_step_grouped([b], **HP)
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 0
    assert torch.equal(a["W"], b["W"])
