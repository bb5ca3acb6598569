"""GPU parity of the AdamW update (non-matrix parameters) against the
float64 oracle, through the C ABI.  fp32 arithmetic on the device: relative
error per tensor within 1e-5 for p' (fp32), the moments within 1e-6; bf16
parameters within one bf16 ulp of the oracle."""
import numpy as np
import pytest
import torch

from newton_schulz_gb300 import binding
from oracle.adamw_ref import adamw_step_ref

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _dev(lib, cuda_ok):
    yield


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def _tensors(sizes, pdt, gdt, seed):
    g = torch.Generator().manual_seed(seed)
    out = []
    for n in sizes:
        out.append({"param": (torch.randn(n, generator=g) * 0.02).to(pdt).cuda(),
                    "grad": (torch.randn(n, generator=g) * 1e-3).to(gdt).cuda(),
                    "exp_avg": (torch.randn(n, generator=g) * 1e-4).cuda(),
                    "exp_avg_sq": (torch.rand(n, generator=g) * 1e-6).cuda()})
    return out


HP = dict(lr=3e-4, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1)


@pytest.mark.parametrize("pdt,gdt", [(torch.float32, torch.float32),
                                     (torch.float32, torch.bfloat16),
                                     (torch.bfloat16, torch.bfloat16)])
def test_adamw_parity_ragged_sizes(pdt, gdt):
    sizes = [1, 7, 8, 9, 4096, 4097, 123457, 1 << 20]
    ts = _tensors(sizes, pdt, gdt, 1)
    host = [{k: _np(v) for k, v in t.items()} for t in ts]
    for step in (1, 2, 10):
        binding.muon_adamw_grouped(ts, step=step, **HP)
        torch.cuda.synchronize()
        assert binding.muon_last_launch_count() == 1
        for t, h in zip(ts, host):
            p2, m2, v2 = adamw_step_ref(h["param"], h["grad"], h["exp_avg"], h["exp_avg_sq"], step,
                                        lr=HP["lr"], beta1=HP["betas"][0], beta2=HP["betas"][1],
                                        eps=HP["eps"], wd=HP["weight_decay"])
            assert _rel(_np(t["exp_avg"]), m2) <= 1e-6
            assert _rel(_np(t["exp_avg_sq"]), v2) <= 1e-6
            if pdt == torch.float32:
                assert _rel(_np(t["param"]), p2) <= 1e-5
            else:
                # within one bf16 ulp (at most 2^-7 relative) of the oracle's
                # value: the fp32 result may round to the other neighbour
                assert np.all(np.abs(_np(t["param"]) - p2) <= 2.0 ** -7 * np.abs(p2) + 1e-30)
            h["param"], h["exp_avg"], h["exp_avg_sq"] = _np(t["param"]), _np(t["exp_avg"]), _np(t["exp_avg_sq"])


def test_adamw_many_tensors_and_unaligned_views():
    # more tensors than one launch carries, and views at odd element offsets
    base = _tensors([70 * 33 + 5], torch.float32, torch.float32, 2)[0]
    views = []
    for i in range(70):
        sl = slice(i * 33 + 1, i * 33 + 34)
        views.append({k: v[sl] for k, v in base.items()})
    host = [{k: _np(v) for k, v in t.items()} for t in views]
    binding.muon_adamw_grouped(views, step=3, **HP)
    torch.cuda.synchronize()
    assert binding.muon_last_launch_count() == 2
    for t, h in zip(views, host):
        p2, m2, v2 = adamw_step_ref(h["param"], h["grad"], h["exp_avg"], h["exp_avg_sq"], 3,
                                    lr=HP["lr"], beta1=0.9, beta2=0.95, eps=1e-8, wd=0.1)
        assert _rel(_np(t["param"]), p2) <= 1e-5 and _rel(_np(t["exp_avg"]), m2) <= 1e-6


def test_adamw_first_step_closed_form():
    # from zero state the first step is lr * g / (|g| + eps) plus the decay
    n = 100000
    g = torch.randn(n, generator=torch.Generator().manual_seed(3)).cuda()
    p = torch.randn(n, generator=torch.Generator().manual_seed(4)).cuda()
    t = {"param": p.clone(), "grad": g, "exp_avg": torch.zeros(n, device="cuda"),
         "exp_avg_sq": torch.zeros(n, device="cuda")}
    binding.muon_adamw_grouped([t], step=1, lr=1e-2, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.0)
    torch.cuda.synchronize()
    want = _np(p) - 1e-2 * _np(g) / (np.abs(_np(g)) + 1e-8)
    assert _rel(_np(t["param"]), want) <= 1e-6
