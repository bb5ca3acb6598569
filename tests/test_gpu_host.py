"""The host-resident step (muon_step_grouped_host): W, G and Mom in pinned
host memory, staged through device slots in chunks, against the float64
oracle, with the tolerances of the device entry points."""
import numpy as np
import pytest
import torch

from newton_schulz_gb300 import binding, synth
from oracle import muon_ref as R

pytestmark = pytest.mark.gpu
MOM_TOL, DW_TOL = 1e-6, 1e-2


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


@pytest.fixture(autouse=True)
def _dev(lib, cuda_ok):
    yield


def _host_groups(specs):
    out = []
    for shape, gdt, wdt, seed in specs:
        g = synth.random_group(shape, gdt, wdt, "cpu", seed, 1e-3, 1e-3)
        out.append({k: g[k].pin_memory() for k in ("W", "G", "Mom")})
    return out


def _check(groups, host0, sample):
    for g, h in zip(groups, host0):
        B = g["W"].shape[0]
        idx = list(range(0, B, max(1, B // sample)))[:sample]
        w2, m2, _ = R.muon_step_ref(h["W"][idx], h["G"][idx], h["Mom"][idx])
        assert _rel(_np(g["Mom"])[idx], m2) <= MOM_TOL
        w = _np(g["W"])[idx]
        for k in range(len(idx)):
            err = np.linalg.norm(w[k] - w2[k]) / np.linalg.norm(w2[k] - h["W"][idx][k])
            assert err <= DW_TOL, (g["W"].shape, idx[k], err)


def test_host_step_many_chunks_mixed_paths():
    """About 250 MB of state: five or more chunks (48 MB each at least)
    through the three device slots, so the slots are reused, with small-m and
    GEMM-path shapes in the same call."""
    groups = _host_groups([((100, 24, 10240), torch.bfloat16, torch.float32, 61),
                           ((3, 300, 700), torch.bfloat16, torch.float32, 62),
                           ((2, 1000, 48), torch.float32, torch.float32, 63)])
    host0 = [{k: _np(g[k]) for k in ("W", "G", "Mom")} for g in groups]
    stream = torch.cuda.current_stream()
    binding.muon_step_grouped_host(groups, mu=0.95, nesterov=True, lr=0.02, wd=0.01)
    stream.synchronize()
    assert binding.muon_query_status() == 0
    assert binding.muon_last_launch_count() >= 5
    _check(groups, host0, sample=4)


def test_host_step_matches_device_step_single_chunk():
    """A call small enough for one chunk runs the same launches as the device
    entry point on the same values: identical bits."""
    specs = [((4, 64, 256), torch.float32, torch.float32, 71), ((1, 256, 64), torch.float32, torch.float32, 72)]
    groups = _host_groups(specs)
    dev = [{k: v.cuda() for k, v in g.items()} for g in groups]
    binding.muon_step_grouped_host(groups)
    binding.muon_step_grouped(dev)
    torch.cuda.synchronize()
    for g, d in zip(groups, dev):
        assert torch.equal(g["W"], d["W"].cpu()) and torch.equal(g["Mom"], d["Mom"].cpu())


def test_host_step_repeat_and_two_steps():
    groups = _host_groups([((12, 24, 4096), torch.bfloat16, torch.float32, 81)])
    h = {k: _np(groups[0][k]) for k in ("W", "G", "Mom")}
    for _ in range(2):
        binding.muon_step_grouped_host(groups)
        torch.cuda.current_stream().synchronize()
        w2, m2, _ = R.muon_step_ref(h["W"], h["G"], h["Mom"])
        assert _rel(_np(groups[0]["Mom"]), m2) <= MOM_TOL
        w = _np(groups[0]["W"])
        for i in range(w.shape[0]):
            assert np.linalg.norm(w[i] - w2[i]) <= DW_TOL * np.linalg.norm(w2[i] - h["W"][i])
        h["W"], h["Mom"] = w, _np(groups[0]["Mom"])
