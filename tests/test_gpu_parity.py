"""GPU parity of the CUDA path against the float64 oracle (through the C ABI).

Tolerances (per matrix): NS output relative Frobenius error <= 3e-2 for the
bf16 NS path; fp32 momentum <= 1e-6 relative; updated weights within
1e-2 * ||dW_oracle||_F of the oracle's W'.
"""
import numpy as np
import pytest
import torch

from newton_schulz_gb300 import binding, synth
from oracle import muon_ref as R

pytestmark = pytest.mark.gpu

NS_TOL = 3e-2
MOM_TOL = 1e-6
DW_TOL = 1e-2


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


@pytest.fixture(scope="module", autouse=True)
def _dev(lib, cuda_ok):
    torch.cuda.init()
    yield
    torch.cuda.synchronize()


def _ns_gpu_f32(x_cpu, steps=5, **cfgkw):
    X = x_cpu.cuda().contiguous()
    out = torch.empty_like(X)
    cfg = binding.make_config(steps=steps, **cfgkw)
    binding.muon_ns_batched_ex(X, cfg, out)
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 0
    return out


NS_SHAPES = [
    (5, 64, 256),      # the small reference shape
    (1, 256, 64),      # transposed path
    (3, 200, 333),     # two row tiles, ragged n
    (2, 333, 200),     # transposed, ragged
    (2, 300, 300),     # square, 3 tiles per side
    (4, 24, 10240),    # tall-skinny: split-K Gram
    (1, 1, 17),        # a row vector
    (2, 9, 1),         # column vectors
    (1, 130, 1000),    # ragged M tile
]


@pytest.mark.parametrize("shape", NS_SHAPES)
def test_ns_parity_f32_input(shape):
    g = torch.Generator().manual_seed(hash(shape) % 2**31)
    x = torch.randn(shape, generator=g)
    out = _ns_gpu_f32(x)
    ref = R.ns_batched_ref(_np(x))
    got = _np(out)
    for i in range(shape[0]):
        assert _rel(got[i], ref[i]) <= NS_TOL, (shape, i, _rel(got[i], ref[i]))


@pytest.mark.parametrize("shape", [(3, 200, 333), (74, 24, 10240)])
def test_ns_batched_bf16_inplace(shape):
    g = torch.Generator().manual_seed(7)
    x = (torch.randn(shape, generator=g) * 1e-3).to(torch.bfloat16)
    ref = R.ns_batched_ref(_np(x))
    X = x.cuda()
    binding.muon_ns_batched(X)
    torch.cuda.synchronize()
    got = _np(X)
    for i in range(shape[0]):
        assert _rel(got[i], ref[i]) <= NS_TOL


def test_steps_zero_and_coefficient_table():
    x = torch.randn((2, 40, 90), generator=torch.Generator().manual_seed(3))
    out = _ns_gpu_f32(x, steps=0)
    ref = R.ns_batched_ref(_np(x), steps=0)
    for i in range(2):
        assert _rel(_np(out)[i], ref[i]) <= 5e-3
    table = [(3.0, -3.2, 1.2), (2.5, -2.0, 0.6), (1.9, -1.2, 0.3)]
    out = _ns_gpu_f32(x, steps=3, coeffs=table)
    ref = R.ns_batched_ref(_np(x), steps=3, coeffs=table)
    for i in range(2):
        assert _rel(_np(out)[i], ref[i]) <= NS_TOL


def _step_and_check(groups_dev, hp, steps_of_training=1):
    """Run the step on device copies; compare W', Mom' with the oracle."""
    host = [{k: _np(g[k]) for k in ("W", "G", "Mom")} for g in groups_dev]
    for _ in range(steps_of_training):
        binding.muon_step_grouped(groups_dev, **hp)
        torch.cuda.synchronize()
        assert binding.muon_query_status() == 0
        outs = [R.muon_step_ref(h["W"], h["G"], h["Mom"], mu=hp["mu"], nesterov=hp["nesterov"],
                                lr=hp["lr"], wd=hp["wd"], scale_rule=hp["scale_rule"])
                for h in host]
        for g, h, (w2, m2, o) in zip(groups_dev, host, outs):
            mom = _np(g["Mom"])
            assert _rel(mom, m2) <= MOM_TOL
            dw_ref = w2 - h["W"]
            w_gpu = _np(g["W"])
            for i in range(w2.shape[0]):
                err = np.linalg.norm(w_gpu[i] - w2[i]) / np.linalg.norm(dw_ref[i])
                assert err <= DW_TOL, (g.get("name"), i, err)
            h["W"], h["Mom"] = w_gpu, mom   # next step starts from the GPU state


def test_c1_reference_step():
    groups = synth.config_c1("cuda")
    _step_and_check(groups, dict(mu=0.95, nesterov=True, lr=0.02, wd=0.01, scale_rule=0),
                    steps_of_training=2)
    # both core shapes fold to (64, 256): one fused cluster launch for the step
    assert binding.muon_last_launch_count() == 1


@pytest.mark.parametrize("rule", [0, 1, 2])
@pytest.mark.parametrize("nesterov", [True, False])
def test_mixed_groups_step(rule, nesterov):
    groups = [
        synth.random_group((3, 200, 333), torch.bfloat16, torch.float32, "cuda", 1, 1e-3, 1e-3),
        synth.random_group((2, 333, 200), torch.float32, torch.bfloat16, "cuda", 2, 1.0, 0.5),
        synth.random_group((1, 130, 1000), torch.float32, torch.float32, "cuda", 3, 1.0, 0.0),
        synth.random_group((2, 1000, 130), torch.bfloat16, torch.float32, "cuda", 4, 1e-2, 0.0),
    ]
    hp = dict(mu=0.9, nesterov=nesterov, lr=0.05, wd=0.1, scale_rule=rule)
    # bf16 weights: the update is a few ulps of W; compare an fp32 rerun instead
    groups[1]["W"] = groups[1]["W"].float()
    _step_and_check(groups, hp)


def test_batched_equals_singleton_bitwise():
    x = torch.randn((4, 150, 260), generator=torch.Generator().manual_seed(5)).cuda()
    out_b = torch.empty_like(x)
    binding.muon_ns_batched_ex(x, binding.make_config(), out_b)
    out_1 = torch.empty_like(x[2:3])
    binding.muon_ns_batched_ex(x[2:3].contiguous(), binding.make_config(), out_1)
    torch.cuda.synchronize()
    assert torch.equal(out_b[2:3], out_1)


def test_transpose_bitwise_and_repeatable():
    x = torch.randn((2, 150, 260), generator=torch.Generator().manual_seed(6)).cuda()
    xt = x.transpose(1, 2).contiguous()
    o1 = torch.empty_like(x)
    o2 = torch.empty_like(xt)
    o3 = torch.empty_like(x)
    binding.muon_ns_batched_ex(x, binding.make_config(), o1)
    binding.muon_ns_batched_ex(xt, binding.make_config(), o2)
    binding.muon_ns_batched_ex(x, binding.make_config(), o3)
    torch.cuda.synchronize()
    assert torch.equal(o1.transpose(1, 2), o2)
    assert torch.equal(o1, o3)


def test_zero_matrix_and_nonfinite_flag():
    x = torch.zeros((2, 32, 64), device="cuda")
    out = torch.full_like(x, 7.0)
    binding.muon_ns_batched_ex(x, binding.make_config(), out)
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 0
    assert torch.count_nonzero(out).item() == 0
    x[1, 3, 5] = float("nan")
    binding.muon_ns_batched_ex(x, binding.make_config(), out)
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 7          # MUON_ERR_NONFINITE
    assert binding.muon_query_status() == 0          # read clears it


def test_checkpoint_resume_bitwise():
    """Two steps == one step, save/restore Mom and W, one step (bitwise)."""
    def fresh():
        return [synth.random_group((3, 96, 200), torch.bfloat16, torch.float32, "cuda", 9, 1e-3)]
    hp = dict(mu=0.95, nesterov=True, lr=0.02, wd=0.01, scale_rule=0)
    a = fresh()
    g_seq = [synth.random_group((3, 96, 200), torch.bfloat16, torch.float32, "cuda", s, 1e-3)["G"]
             for s in (11, 12)]
    for g in g_seq:
        a[0]["G"] = g
        binding.muon_step_grouped(a, **hp)
    b = fresh()
    b[0]["G"] = g_seq[0]
    binding.muon_step_grouped(b, **hp)
    torch.cuda.synchronize()
    saved = {k: b[0][k].cpu().clone() for k in ("W", "Mom")}
    c = fresh()
    c[0]["W"].copy_(saved["W"])
    c[0]["Mom"].copy_(saved["Mom"])
    c[0]["G"] = g_seq[1]
    binding.muon_step_grouped(c, **hp)
    torch.cuda.synchronize()
    assert torch.equal(a[0]["W"], c[0]["W"]) and torch.equal(a[0]["Mom"], c[0]["Mom"])


@pytest.mark.parametrize("shape", [(160, 256, 2048), (2, 2048, 2304)])
def test_long_k_launches(shape):
    """Long-K launches: 160 x [256, 2048] (Gram over K = 2048 without
    split-K), 2 x [2048, 2304] (the polynomial's tiles have 32 K blocks, so
    it takes the 4-stage ring with one staging box per epilogue set)."""
    g = torch.Generator().manual_seed(shape[0] + shape[1])
    x = torch.randn(shape, generator=g)
    out = _ns_gpu_f32(x)
    idx = list(range(0, shape[0], max(1, shape[0] // 6)))
    ref = R.ns_batched_ref(_np(x[idx]))
    got = _np(out)
    for k, i in enumerate(idx):
        assert _rel(got[i], ref[k]) <= NS_TOL, (shape, i, _rel(got[i], ref[k]))
