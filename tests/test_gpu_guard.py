"""Workspace guard bands: a check for out-of-bounds writes into the
library's workspace that needs no memory sanitizer.

With MUON_WS_GUARD=1 every buffer of the library's workspace is followed by a
4 KB band filled with a fixed byte before the kernels that use that layout;
a small kernel counts the band bytes that changed right after them, and
muon_debug_guard_check returns the count.  Every path below must leave the
bands intact and give the same bits as without guard mode.
"""
import pytest
import torch

from newton_schulz_gb300 import binding, synth

pytestmark = pytest.mark.gpu
HP = dict(mu=0.95, nesterov=True, lr=0.02, wd=0.01, scale_rule=0)


@pytest.fixture(autouse=True)
def _dev(lib, cuda_ok):
    yield
    torch.cuda.synchronize()


def _groups(kind):
    if kind == "small":          # Gram-space kernel, both layouts, ragged n
        return [synth.random_group((5, 24, 3000), torch.bfloat16, torch.float32, "cuda", 1, 1e-3),
                synth.random_group((3, 1000, 40), torch.float32, torch.bfloat16, "cuda", 2, 1.0)]
    if kind == "long":           # split-K Gram on the grouped GEMM path
        return [synth.random_group((2, 96, 8192), torch.bfloat16, torch.float32, "cuda", 3, 1e-3)]
    return [synth.random_group((3, 200, 333), torch.bfloat16, torch.float32, "cuda", 4, 1e-3),
            synth.random_group((2, 640, 256), torch.float32, torch.bfloat16, "cuda", 5, 1.0),
            synth.random_group((1, 1000, 300), torch.bfloat16, torch.float32, "cuda", 6, 1e-3)]


@pytest.mark.parametrize("kind,env", [
    ("small", {}),
    ("gemm", {}),
    ("gemm", {"MUON_GEMM_PAIR": "1", "MUON_GEMM_WIDE": "0", "MUON_MAX_KSPLIT": "1"}),
    ("gemm", {"MUON_GEMM_WIDE": "1", "MUON_MAX_KSPLIT": "1"}),
    ("long", {}),
    ("gemm", {"PRECISE": "1"}),
    ("small", {"PRECISE": "1"}),
])
def test_guard_bands_intact_and_results_unchanged(kind, env, monkeypatch):
    precise = env.pop("PRECISE", None) is not None
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    cfg = binding.make_config(precision=binding.NS_TF32) if precise else None
    out = []
    for guard in ("0", "1"):
        monkeypatch.setenv("MUON_WS_GUARD", guard)
        g = _groups(kind)
        binding.muon_step_grouped(g, ns_cfg=cfg, **HP)
        torch.cuda.synchronize()
        assert binding.muon_query_status() == 0
        assert binding.muon_debug_guard_check() == 0
        out.append(g)
    for a, b in zip(*out):
        assert torch.equal(a["W"], b["W"]) and torch.equal(a["Mom"], b["Mom"])


def test_guard_bands_host_resident_step(monkeypatch):
    monkeypatch.setenv("MUON_WS_GUARD", "1")
    host = [{k: v.cpu().pin_memory() for k, v in g.items() if k != "name"} for g in _groups("gemm")]
    binding.muon_step_grouped_host(host, **HP)
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 0
    assert binding.muon_debug_guard_check() == 0
