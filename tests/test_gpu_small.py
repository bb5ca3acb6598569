"""GPU parity of the fused small-m kernel (m <= 64, Gram-space Newton-Schulz),
and of the grouped GEMM path on the same shapes (MUON_SMALL_PATH=0), against
the float64 oracle."""
import os

import numpy as np
import pytest
import torch

from newton_schulz_gb300 import binding, synth
from oracle import muon_ref as R

pytestmark = pytest.mark.gpu
NS_TOL, MOM_TOL, DW_TOL = 3e-2, 1e-6, 1e-2


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


@pytest.fixture(autouse=True)
def _dev(lib, cuda_ok):
    yield
    os.environ.pop("MUON_SMALL_PATH", None)


SHAPES = [
    (3, 8, 300),        # m = 8
    (2, 33, 1000),      # m = 33: 48-wide MMA N, ragged n
    (2, 1000, 48),      # transposed, m = 48
    (6, 64, 4097),      # m = 64, several items per matrix, ragged tail, element-wise copies
    (20, 24, 2048),     # many matrices
    (1, 24, 10240),     # the tall-skinny shape, one matrix split into many items
    (3, 5000, 17),      # transposed, odd m, element-wise copies (17 fp32 = 68 B rows)
]


@pytest.mark.parametrize("generic", [False, True])
@pytest.mark.parametrize("shape", SHAPES)
def test_small_ns_parity(shape, generic):
    if generic:
        os.environ["MUON_SMALL_PATH"] = "0"
    x = torch.randn(shape, generator=torch.Generator().manual_seed(sum(shape)))
    X = x.cuda()
    out = torch.empty_like(X)
    binding.muon_ns_batched_ex(X, binding.make_config(), out)
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 0
    ref = R.ns_batched_ref(_np(x))
    got = _np(out)
    for i in range(shape[0]):
        assert _rel(got[i], ref[i]) <= NS_TOL, (shape, i, _rel(got[i], ref[i]))
    # one fused launch per core shape on the small path
    assert binding.muon_last_launch_count() == (17 if generic else 1)


@pytest.mark.parametrize("shape", [(4, 24, 3000), (3, 3000, 24), (2, 64, 256)])
def test_small_step_parity_bf16_grad(shape):
    g = synth.random_group(shape, torch.bfloat16, torch.float32, "cuda", 31, 1e-3, 1e-3)
    host = {k: _np(g[k]) for k in ("W", "G", "Mom")}
    binding.muon_step_grouped([g], mu=0.95, nesterov=True, lr=0.02, wd=0.01, scale_rule=0)
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 0
    w2, m2, _ = R.muon_step_ref(host["W"], host["G"], host["Mom"])
    assert _rel(_np(g["Mom"]), m2) <= MOM_TOL
    w = _np(g["W"])
    for i in range(shape[0]):
        assert np.linalg.norm(w[i] - w2[i]) <= DW_TOL * np.linalg.norm(w2[i] - host["W"][i])


def test_small_transpose_bitwise():
    x = torch.randn((3, 40, 700), generator=torch.Generator().manual_seed(4)).cuda()
    o1 = torch.empty_like(x)
    o2 = torch.empty((3, 700, 40), device="cuda")
    binding.muon_ns_batched_ex(x, binding.make_config(), o1)
    binding.muon_ns_batched_ex(x.transpose(1, 2).contiguous(), binding.make_config(), o2)
    torch.cuda.synchronize()
    assert torch.equal(o1.transpose(1, 2), o2)


def test_small_steps_zero_and_table():
    x = torch.randn((2, 20, 500), generator=torch.Generator().manual_seed(8))
    X = x.cuda()
    for steps, table in ((0, None), (3, [(3.0, -3.2, 1.2), (2.5, -2.0, 0.6), (1.9, -1.2, 0.3)])):
        out = torch.empty_like(X)
        binding.muon_ns_batched_ex(X, binding.make_config(steps=steps, coeffs=table), out)
        torch.cuda.synchronize()
        ref = R.ns_batched_ref(_np(x), steps=steps, coeffs=table)
        tol = 5e-3 if steps == 0 else NS_TOL
        for i in range(2):
            assert _rel(_np(out)[i], ref[i]) <= tol


def test_small_and_large_groups_in_one_call():
    groups = [
        synth.random_group((3, 24, 2048), torch.bfloat16, torch.float32, "cuda", 41, 1e-3),
        synth.random_group((2, 300, 700), torch.bfloat16, torch.float32, "cuda", 42, 1e-3),
        synth.random_group((2, 2048, 24), torch.float32, torch.float32, "cuda", 43, 1.0),
    ]
    host = [{k: _np(g[k]) for k in ("W", "G", "Mom")} for g in groups]
    binding.muon_step_grouped(groups)
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 0
    for g, h in zip(groups, host):
        w2, m2, _ = R.muon_step_ref(h["W"], h["G"], h["Mom"])
        w = _np(g["W"])
        for i in range(w.shape[0]):
            assert np.linalg.norm(w[i] - w2[i]) <= DW_TOL * np.linalg.norm(w2[i] - h["W"][i])


@pytest.mark.parametrize("trans", [False, True])
def test_small_step_multistage_items(trans):
    """Enough matrices that a work item spans many ring stages (2048 columns),
    so the ring wraps several times within an item and across the phases."""
    shape = (160, 4096, 16) if trans else (160, 16, 4096)
    g = synth.random_group(shape, torch.bfloat16, torch.float32, "cuda", 51, 1e-3, 1e-3)
    host = {k: _np(g[k]) for k in ("W", "G", "Mom")}
    binding.muon_step_grouped([g], mu=0.95, nesterov=True, lr=0.02, wd=0.01, scale_rule=0)
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 0
    w2, m2, _ = R.muon_step_ref(host["W"][:8], host["G"][:8], host["Mom"][:8])
    assert _rel(_np(g["Mom"])[:8], m2) <= MOM_TOL
    w = _np(g["W"])
    for i in range(8):
        assert np.linalg.norm(w[i] - w2[i]) <= DW_TOL * np.linalg.norm(w2[i] - host["W"][i])
    assert binding.muon_last_launch_count() == 1


def test_small_repeat_bitwise_across_counter_ring():
    """70 launches in a row (more than the 64 per-launch counter slots) give
    the same bits: no launch depends on counters an earlier one left."""
    x = torch.randn((5, 24, 3000), generator=torch.Generator().manual_seed(12)).cuda()
    outs = [torch.empty_like(x) for _ in range(70)]
    for o in outs:
        binding.muon_ns_batched_ex(x, binding.make_config(), o)
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 0
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    ref = R.ns_batched_ref(_np(x.cpu()))
    for i in range(5):
        assert _rel(_np(outs[0])[i], ref[i]) <= NS_TOL


HP_TOL = 1e-3   # NS tolerance of the high-precision mode


@pytest.mark.parametrize("shape", SHAPES + [(2, 64, 256), (4, 40, 3000)])
def test_precise_ns_parity(shape):
    """MUON_NS_TF32: X0 as bf16 hi + lo, fp32 Gram space; relative error per
    matrix within 1e-3 of the float64 oracle."""
    x = torch.randn(shape, generator=torch.Generator().manual_seed(sum(shape) + 1))
    X = x.cuda()
    out = torch.empty_like(X)
    binding.muon_ns_batched_ex(X, binding.make_config(precision=binding.NS_TF32), out)
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 0
    ref = R.ns_batched_ref(_np(x))
    got = _np(out)
    errs = [_rel(got[i], ref[i]) for i in range(shape[0])]
    print(shape, "max rel err", max(errs))
    assert max(errs) <= HP_TOL, (shape, errs)
    assert binding.muon_last_launch_count() == 1


@pytest.mark.parametrize("shape", [(4, 24, 3000), (3, 3000, 24), (2, 64, 1000), (74, 24, 10240)])
def test_precise_step_parity(shape):
    g = synth.random_group(shape, torch.bfloat16, torch.float32, "cuda", 33, 1e-3, 1e-3)
    host = {k: _np(g[k]) for k in ("W", "G", "Mom")}
    binding.muon_step_grouped([g], mu=0.95, nesterov=True, lr=0.02, wd=0.01, scale_rule=0,
                              ns_cfg=binding.make_config(precision=binding.NS_TF32))
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 0
    k = min(shape[0], 6)
    w2, m2, _ = R.muon_step_ref(host["W"][:k], host["G"][:k], host["Mom"][:k])
    assert _rel(_np(g["Mom"])[:k], m2) <= MOM_TOL
    w = _np(g["W"])
    for i in range(k):
        err = np.linalg.norm(w[i] - w2[i]) / np.linalg.norm(w2[i] - host["W"][i])
        assert err <= HP_TOL, (shape, i, err)


@pytest.mark.parametrize("shape,generic", [((2, 128, 300), False), ((1, 300, 200), False),
                                           ((2, 200, 333), False), ((3, 24, 2000), True),
                                           ((1, 520, 700), False)])
def test_precise_gemm_path_parity(shape, generic):
    """The high-precision mode on the grouped GEMM path (hi + lo operands,
    three K segments per product), including a small shape forced there."""
    if generic:
        os.environ["MUON_SMALL_PATH"] = "0"
    x = torch.randn(shape, generator=torch.Generator().manual_seed(sum(shape) + 5))
    X = x.cuda()
    out = torch.empty_like(X)
    binding.muon_ns_batched_ex(X, binding.make_config(precision=binding.NS_TF32), out)
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 0
    ref = R.ns_batched_ref(_np(x))
    errs = [_rel(_np(out)[i], ref[i]) for i in range(shape[0])]
    print(shape, "GEMM path max rel err", max(errs))
    assert max(errs) <= HP_TOL, (shape, errs)


def test_precise_gemm_step_parity():
    g = synth.random_group((2, 300, 520), torch.bfloat16, torch.float32, "cuda", 35, 1e-3, 1e-3)
    host = {k: _np(g[k]) for k in ("W", "G", "Mom")}
    binding.muon_step_grouped([g], ns_cfg=binding.make_config(precision=binding.NS_TF32))
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 0
    w2, m2, _ = R.muon_step_ref(host["W"], host["G"], host["Mom"])
    assert _rel(_np(g["Mom"]), m2) <= MOM_TOL
    w = _np(g["W"])
    for i in range(2):
        err = np.linalg.norm(w[i] - w2[i]) / np.linalg.norm(w2[i] - host["W"][i])
        assert err <= HP_TOL, (i, err)


@pytest.mark.parametrize("generic", [False, True])
def test_precise_steps_zero_and_table(generic):
    """The high-precision mode with steps = 0 (O = X0 / ||X0||) and with a
    per-step coefficient table, on both paths."""
    if generic:
        os.environ["MUON_SMALL_PATH"] = "0"
    x = torch.randn((2, 40, 700), generator=torch.Generator().manual_seed(17))
    X = x.cuda()
    for steps, table, tol in ((0, None, 1e-5), (3, [(3.0, -3.2, 1.2), (2.5, -2.0, 0.6), (1.9, -1.2, 0.3)], HP_TOL)):
        out = torch.empty_like(X)
        binding.muon_ns_batched_ex(X, binding.make_config(steps=steps, coeffs=table,
                                                          precision=binding.NS_TF32), out)
        torch.cuda.synchronize()
        assert binding.muon_query_status() == 0
        ref = R.ns_batched_ref(_np(x), steps=steps, coeffs=table)
        for i in range(2):
            assert _rel(_np(out)[i], ref[i]) <= tol, (generic, steps, _rel(_np(out)[i], ref[i]))


def test_precise_host_step():
    g = synth.random_group((6, 24, 4096), torch.bfloat16, torch.float32, "cpu", 37, 1e-3, 1e-3)
    host = {k: g[k].pin_memory() for k in ("W", "G", "Mom")}
    h0 = {k: _np(v) for k, v in host.items()}
    binding.muon_step_grouped_host([host], ns_cfg=binding.make_config(precision=binding.NS_TF32))
    torch.cuda.current_stream().synchronize()
    w2, m2, _ = R.muon_step_ref(h0["W"], h0["G"], h0["Mom"])
    w = _np(host["W"])
    for i in range(6):
        err = np.linalg.norm(w[i] - w2[i]) / np.linalg.norm(w2[i] - h0["W"][i])
        assert err <= HP_TOL, (i, err)
