"""The grouped GEMM path in WIDE blocks: one CTA computes both 128-row halves
of a 256 x 256 output block from one stage holding the two A tiles and the
common B tile, half h into TMEM accumulator h.  Each half's MMAs run over the
same K blocks in the same order as a single 128 x 256 tile's, so the results
must be bit-identical to the single-tile kernel's.  MUON_GEMM_WIDE=1 forces
WIDE blocks (0 forbids them; MUON_GEMM_PAIR=0 keeps CTA pairs out): ragged
edges, transposed layouts, an odd number of 128-row tiles (the block's second
half then lies past the matrix and stores nothing), square and mixed groups,
one Muon step, all against the float64 oracle too.
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
    monkeypatch.setenv("MUON_GEMM_PAIR", "0")
    monkeypatch.setenv("MUON_MAX_KSPLIT", "1")   # WIDE launches are unsplit
    yield
    torch.cuda.synchronize()


def _ns(x, wide, monkeypatch):
    monkeypatch.setenv("MUON_GEMM_WIDE", "1" if wide else "0")
    out = torch.empty_like(x)
    binding.muon_ns_batched_ex(x, binding.make_config(), out)
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 0
    return out


@pytest.mark.parametrize("shape", [
    (3, 200, 333),     # two row tiles, ragged columns
    (2, 333, 200),     # transposed
    (1, 640, 1000),    # five 128-row tiles: the last block's second half is empty
    (2, 300, 300),     # square, three row tiles
    (2, 1024, 1536),   # several full blocks per column tile
    (1, 130, 2000),    # two row tiles, the second nearly empty
])
def test_wide_equals_single_and_oracle(shape, monkeypatch):
    x = torch.randn(shape, generator=torch.Generator().manual_seed(sum(shape))).cuda()
    a = _ns(x, False, monkeypatch)
    b = _ns(x, True, monkeypatch)
    assert torch.equal(a, b)
    ref = R.ns_batched_ref(x.double().cpu().numpy())
    got = b.double().cpu().numpy()
    for i in range(shape[0]):
        e = np.linalg.norm(got[i] - ref[i]) / np.linalg.norm(ref[i])
        assert e <= NS_TOL, (shape, i, e)


def test_wide_step_mixed_groups(monkeypatch):
    """One Muon step over three core shapes in one chunk, WIDE against single."""
    def groups():
        return [synth.random_group((3, 256, 1024), torch.bfloat16, torch.float32, "cuda", 1, 1e-3),
                synth.random_group((2, 700, 384), torch.float32, torch.float32, "cuda", 2, 1.0, 0.5),
                synth.random_group((1, 520, 520), torch.bfloat16, torch.float32, "cuda", 3, 1e-3)]
    outs = []
    for wide in ("0", "1"):
        monkeypatch.setenv("MUON_GEMM_WIDE", wide)
        gs = groups()
        host = [{k: g[k].double().cpu().numpy() for k in ("W", "G", "Mom")} for g in gs]
        binding.muon_step_grouped(gs, **HP)
        torch.cuda.synchronize()
        assert binding.muon_query_status() == 0
        outs.append([g["W"].clone() for g in gs])
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    for g, h in zip(gs, host):
        w2, _, _ = R.muon_step_ref(h["W"], h["G"], h["Mom"], **HP)
        w = g["W"].double().cpu().numpy()
        for i in range(w.shape[0]):
            assert np.linalg.norm(w[i] - w2[i]) / np.linalg.norm(w2[i] - h["W"][i]) <= DW_TOL
