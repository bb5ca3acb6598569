"""The update kernel in two row passes (tiles twice as tall, 16 elements a
thread), which the library runs when every weight of a launch is bf16,
against the one-pass kernel (MUON_FIN_PASSES=1).  Each element goes through
the same arithmetic, W' = RNE(decay W - lr s O), so W' and the momentum must
be bit-identical: ragged rows and columns in both layouts (O read through the
transposed tile, or in place), the high-precision mode (O's lo half added to
its hi half), and the NS-only copy-back into bf16 with steps = 5 and steps = 0
(the 1 / ||X|| factor).  The bf16-weight update itself is checked against the
float64 oracle by the parity tests, which run the two-pass kernel by default.
"""
import pytest
import torch

from newton_schulz_gb300 import binding, synth

pytestmark = pytest.mark.gpu
HP = dict(mu=0.95, nesterov=True, lr=0.02, wd=0.01, scale_rule=0)
BF, F32 = torch.bfloat16, torch.float32


@pytest.fixture(autouse=True)
def _dev(lib, cuda_ok):
    yield
    torch.cuda.synchronize()


def _groups(specs):
    return [synth.random_group(shape, gd, BF, "cuda", seed, gs, 0.1)
            for shape, gd, seed, gs in specs]


def _step(specs, passes, monkeypatch, ns_cfg=None):
    if passes:
        monkeypatch.setenv("MUON_FIN_PASSES", str(passes))
    else:
        monkeypatch.delenv("MUON_FIN_PASSES", raising=False)
    groups = _groups(specs)
    binding.muon_step_grouped(groups, ns_cfg=ns_cfg, **HP)
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 0
    return groups


@pytest.mark.parametrize("specs", [
    [((2, 130, 1001), BF, 1, 1e-3)],                          # transposed O, ragged rows and columns
    [((1, 1001, 130), F32, 2, 1.0)],                          # O in place, ragged rows and columns
    [((2, 200, 1536), BF, 3, 1e-3), ((1, 1544, 264), BF, 4, 1e-3)],   # full vectors, both layouts
    [((1, 96, 4096), BF, 5, 1e-3), ((3, 520, 300), BF, 6, 1e-3)],     # last tile half filled, both layouts
])
@pytest.mark.parametrize("precise", [False, True])
def test_two_passes_equal_one_pass(specs, precise, monkeypatch):
    cfg = binding.make_config(precision=binding.NS_TF32) if precise else None
    a = _step(specs, 1, monkeypatch, cfg)
    b = _step(specs, None, monkeypatch, cfg)
    for ga, gb in zip(a, b):
        assert ga["W"].dtype == BF
        assert torch.equal(ga["W"], gb["W"])
        assert torch.equal(ga["Mom"], gb["Mom"])


@pytest.mark.parametrize("shape", [(1, 130, 1001), (2, 1001, 130), (2, 256, 1024), (1, 1024, 256)])
@pytest.mark.parametrize("steps", [0, 5])
def test_two_passes_copy_back(shape, steps, monkeypatch):
    # the output has X's dtype: a bf16 X makes the copy-back a bf16-only launch
    x = torch.randn(shape, generator=torch.Generator().manual_seed(sum(shape) + steps)).to("cuda", BF)
    outs = []
    for passes in ("1", None):
        if passes:
            monkeypatch.setenv("MUON_FIN_PASSES", passes)
        else:
            monkeypatch.delenv("MUON_FIN_PASSES", raising=False)
        o = torch.empty(shape, dtype=BF, device="cuda")
        binding.muon_ns_batched_ex(x, binding.make_config(steps=steps), o)
        torch.cuda.synchronize()
        assert binding.muon_query_status() == 0
        outs.append(o)
    assert torch.equal(outs[0], outs[1])
