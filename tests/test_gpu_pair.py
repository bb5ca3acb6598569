"""The grouped GEMM path run by CTA pairs that share the B tile.

Large launches run their tiles two at a time on a cluster of two CTAs: each
CTA loads its own 128-row A tile and half of the common 256-row B tile, which
TMA multicasts into both.  Each CTA still issues the same MMAs over the same
K blocks in the same order into its own accumulator, so the results must be
bit-identical to the unpaired kernel's.  MUON_GEMM_PAIR=1 forces pairs on the
small shapes below (0 forbids them): ragged edges, transposed layouts, an odd
number of 128-row tiles (the pair's second tile then lies past the matrix and
stores nothing), square and tall-wide mixes, all against the float64 oracle
too.
"""
import numpy as np
import pytest
import torch

from newton_schulz_gb300 import binding, synth
from oracle import muon_ref as R

pytestmark = pytest.mark.gpu
NS_TOL, DW_TOL = 3e-2, 1e-2
HP = dict(mu=0.95, nesterov=True, lr=0.02, wd=0.01, scale_rule=0)


@pytest.fixture(autouse=True)
def _dev(lib, cuda_ok, monkeypatch):
    monkeypatch.setenv("MUON_GEMM_WIDE", "0")   # pairs, not WIDE blocks
    yield
    torch.cuda.synchronize()


def _ns(x, pair, monkeypatch):
    monkeypatch.setenv("MUON_GEMM_PAIR", "1" if pair else "0")
    out = torch.empty_like(x)
    binding.muon_ns_batched_ex(x, binding.make_config(), out)
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 0
    return out


@pytest.mark.parametrize("shape", [
    (3, 200, 333),     # two row tiles, ragged columns
    (2, 333, 200),     # transposed
    (1, 640, 1000),    # five 128-row tiles: the last pair's second tile is empty
    (2, 300, 300),     # square, three row tiles
    (2, 1024, 1536),   # several full pairs per column tile
])
@pytest.mark.parametrize("ksplit", ["64", "1"])   # few Gram tiles: split-K (unpaired) or not
def test_pair_equals_unpaired_and_oracle(shape, ksplit, monkeypatch):
    monkeypatch.setenv("MUON_MAX_KSPLIT", ksplit)
    x = torch.randn(shape, generator=torch.Generator().manual_seed(sum(shape))).cuda()
    a = _ns(x, False, monkeypatch)
    b = _ns(x, True, monkeypatch)
    assert torch.equal(a, b)
    ref = R.ns_batched_ref(x.double().cpu().numpy())
    got = b.double().cpu().numpy()
    for i in range(shape[0]):
        e = np.linalg.norm(got[i] - ref[i]) / np.linalg.norm(ref[i])
        assert e <= NS_TOL, (shape, i, e)


def test_pair_step_mixed_groups(monkeypatch):
    """A step over several core shapes in one launch, paired and unpaired."""
    def groups():
        return [synth.random_group((3, 200, 333), torch.bfloat16, torch.float32, "cuda", 1, 1e-3),
                synth.random_group((2, 640, 256), torch.bfloat16, torch.float32, "cuda", 2, 1e-3),
                synth.random_group((1, 1000, 300), torch.float32, torch.float32, "cuda", 3, 1.0)]
    out = []
    for pair in (False, True):
        monkeypatch.setenv("MUON_GEMM_PAIR", "1" if pair else "0")
        g = groups()
        binding.muon_step_grouped(g, **HP)
        torch.cuda.synchronize()
        assert binding.muon_query_status() == 0
        out.append(g)
    for ga, gb in zip(*out):
        assert torch.equal(ga["W"], gb["W"]) and torch.equal(ga["Mom"], gb["Mom"])


def test_pair_stall_times_out_and_recovers(monkeypatch):
    """The testing hook's stalled stage in a paired launch: the stalled CTA's
    MMA issuer gives up, and so does its partner, which never receives that
    CTA's half of B; both drain, pass the pair's exit barrier and return."""
    monkeypatch.setenv("MUON_GEMM_PAIR", "1")
    monkeypatch.setenv("MUON_MAX_KSPLIT", "1")   # the first launch (the Gram) is paired
    x = torch.randn((2, 512, 768), generator=torch.Generator().manual_seed(9)).cuda()
    ref, out = torch.empty_like(x), torch.empty_like(x)
    binding.muon_ns_batched_ex(x, binding.make_config(), ref)
    monkeypatch.setenv("MUON_WAIT_TIMEOUT_MS", "50")
    binding.muon_debug_inject_stall(binding.INJECT_GEMM)
    binding.muon_ns_batched_ex(x, binding.make_config(), out)
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 6
    monkeypatch.delenv("MUON_WAIT_TIMEOUT_MS")
    binding.muon_ns_batched_ex(x, binding.make_config(), out)
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 0
    assert torch.equal(out, ref)
