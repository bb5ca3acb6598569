"""Gram-space Newton-Schulz on the grouped GEMM path (DMuon-2 Appendix C.3).

For n >= 2 m the library iterates on the m x m Gram matrix in phases of P
steps (the restart period: 3 for m >= 1024, else 2): R = X X^T of the phase's input, per
step B' = b R + c R^2 + alpha I, Q <- (a - alpha) Q + Q B',
T = (a - alpha) R + R B', R <- (a - alpha) T + T B', and X <- Q X at the
phase's end.  In exact arithmetic this is the X-space iteration; in bf16 it
rounds R, B', T and Q instead of the iterate, so the test holds it to the same
tolerances against the float64 oracle: NS error <= 3e-2 per matrix and W'
within 1e-2 * ||dW||.  On ill-conditioned inputs, where bf16 NS in either
form is farther from the float64 result, Gram space is held to 2.5x the
X-space error of the same input.  Gram space is the default for m >= 1024
and n >= 2 m (MUON_GRAM_SPACE unset or 1), =force applies it to every shape
(used here), 0 turns it off; MUON_GRAM_RESTART sets P (0: no restart).
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
def _dev(lib, cuda_ok):
    yield
    torch.cuda.synchronize()


def _ns(x, gs, monkeypatch, **cfgkw):
    monkeypatch.setenv("MUON_GRAM_SPACE", "force" if gs else "0")
    out = torch.empty_like(x)
    binding.muon_ns_batched_ex(x, binding.make_config(**cfgkw), out)
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 0
    return out


def _errs(got, x, **kw):
    ref = R.ns_batched_ref(x.double().cpu().numpy(), **kw)
    g = got.double().cpu().numpy()
    return [float(np.linalg.norm(g[i] - ref[i]) / np.linalg.norm(ref[i])) for i in range(g.shape[0])]


def test_path_choice(monkeypatch):
    assert binding.muon_ns_gram_restart(768) == 2
    assert binding.muon_ns_gram_restart(1024) == 3
    monkeypatch.setenv("MUON_GRAM_RESTART", "0")
    assert binding.muon_ns_gram_restart(4096) == 0
    monkeypatch.delenv("MUON_GRAM_RESTART")
    monkeypatch.delenv("MUON_GRAM_SPACE", raising=False)
    assert binding.muon_ns_path(1024, 4096) == binding.PATH_GRAM_SPACE    # the default
    monkeypatch.setenv("MUON_GRAM_SPACE", "0")
    assert binding.muon_ns_path(1024, 4096) == binding.PATH_XSPACE
    monkeypatch.setenv("MUON_GRAM_SPACE", "1")
    assert binding.muon_ns_path(1024, 4096) == binding.PATH_GRAM_SPACE
    assert binding.muon_ns_path(14336, 4096) == binding.PATH_GRAM_SPACE
    assert binding.muon_ns_path(4096, 4096) == binding.PATH_XSPACE
    assert binding.muon_ns_path(24, 10240) == binding.PATH_SMALL
    assert binding.muon_ns_path(100, 1000) == binding.PATH_XSPACE    # m < 1024
    assert binding.muon_ns_path(768, 2048) == binding.PATH_XSPACE
    assert binding.muon_ns_path(1024, 4096, binding.make_config(precision=binding.NS_TF32)) == \
        binding.PATH_XSPACE
    monkeypatch.setenv("MUON_GRAM_SPACE", "force")
    assert binding.muon_ns_path(4096, 4096) == binding.PATH_GRAM_SPACE
    assert binding.muon_ns_path(24, 10240) == binding.PATH_SMALL


@pytest.mark.parametrize("shape", [
    (2, 130, 1000),    # ragged m and n, r = 7.7
    (2, 1000, 300),    # transposed, r = 3.3
    (1, 256, 1024),    # whole tiles, r = 4
    (3, 200, 520),     # ragged, r = 2.6
    (1, 640, 2048),    # five 128-row tiles, long K for the Gram
    (2, 300, 300),     # square: Gram space forced where it would not be chosen
])
def test_gram_space_matches_oracle(shape, monkeypatch):
    x = torch.randn(shape, generator=torch.Generator().manual_seed(sum(shape))).cuda()
    eg = _errs(_ns(x, True, monkeypatch), x)
    ex = _errs(_ns(x, False, monkeypatch), x)
    print(f"{shape}: Gram space {max(eg):.4f}, X space {max(ex):.4f}")
    assert max(eg) <= NS_TOL and max(ex) <= NS_TOL


@pytest.mark.parametrize("period", ["0", "1", "3", "5"])
def test_gram_space_restart_periods(period, monkeypatch):
    """Every restart period gives the X-space result on well-conditioned
    inputs; period 1 is one Gram, one Q = P(R) and one apply per step."""
    monkeypatch.setenv("MUON_GRAM_RESTART", period)
    x = torch.randn((2, 256, 1024), generator=torch.Generator().manual_seed(7)).cuda()
    assert max(_errs(_ns(x, True, monkeypatch), x)) <= NS_TOL


def _ill_conditioned(kind, m, n, seed):
    """Rectangular inputs with a wide spectrum: U diag(s) V^T with
    log-spaced s over `kind` decades, or a rank-8 signal x 10 plus noise."""
    rng = np.random.default_rng(seed)
    if kind == "lowrank":
        x = rng.standard_normal((m, 8)) @ rng.standard_normal((8, n)) * 10 + rng.standard_normal((m, n))
    else:
        u = np.linalg.qr(rng.standard_normal((m, m)))[0]
        v = np.linalg.qr(rng.standard_normal((n, m)))[0]
        x = (u * np.logspace(0, -kind, m)) @ v.T
    return torch.from_numpy(x[None]).float().cuda()


@pytest.mark.parametrize("m,n", [(256, 1024), (1024, 4096)])   # restart period 2, 3
@pytest.mark.parametrize("kind", [1, 2, 3, 5, "lowrank"])
def test_gram_space_ill_conditioned(kind, m, n, monkeypatch):
    x = _ill_conditioned(kind, m, n, 11)
    eg = max(_errs(_ns(x, True, monkeypatch), x))
    ex = max(_errs(_ns(x, False, monkeypatch), x))
    print(f"{kind}: Gram space {eg:.4f}, X space {ex:.4f}")
    assert eg <= 2.5 * ex + 1e-3


@pytest.mark.parametrize("steps", [1, 2, 3])
def test_gram_space_steps_and_tables(steps, monkeypatch):
    x = torch.randn((2, 192, 800), generator=torch.Generator().manual_seed(steps)).cuda()
    table = [(3.0, -3.2, 1.2), (2.5, -2.0, 0.6), (1.9, -1.2, 0.3)][:steps]
    got = _ns(x, True, monkeypatch, steps=steps, coeffs=table)
    assert max(_errs(got, x, steps=steps, coeffs=table)) <= NS_TOL


def test_gram_space_step_weights(monkeypatch):
    """One Muon step over mixed groups in Gram space, W' against the oracle."""
    monkeypatch.setenv("MUON_GRAM_SPACE", "force")
    groups = [synth.random_group((3, 256, 1024), torch.bfloat16, torch.float32, "cuda", 1, 1e-3),
              synth.random_group((2, 1536, 384), torch.float32, torch.float32, "cuda", 2, 1.0, 0.5)]
    host = [{k: g[k].double().cpu().numpy() for k in ("W", "G", "Mom")} for g in groups]
    binding.muon_step_grouped(groups, **HP)
    torch.cuda.synchronize()
    assert binding.muon_query_status() == 0
    for g, h in zip(groups, host):
        w2, m2, _ = R.muon_step_ref(h["W"], h["G"], h["Mom"], **HP)
        w = g["W"].double().cpu().numpy()
        assert np.linalg.norm(g["Mom"].double().cpu().numpy() - m2) <= 1e-6 * np.linalg.norm(m2)
        for i in range(w.shape[0]):
            assert np.linalg.norm(w[i] - w2[i]) / np.linalg.norm(w2[i] - h["W"][i]) <= DW_TOL


def test_gram_space_pairs_bitwise(monkeypatch):
    """CTA pairs on every Gram-space product (forced) give the same bits."""
    monkeypatch.setenv("MUON_MAX_KSPLIT", "1")
    x = torch.randn((2, 640, 2048), generator=torch.Generator().manual_seed(3)).cuda()
    outs = []
    for pair in ("0", "1"):
        monkeypatch.setenv("MUON_GEMM_PAIR", pair)
        outs.append(_ns(x, True, monkeypatch))
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("shape", [(1, 4096, 14336), (1, 14336, 4096), (2, 1024, 4096)])
def test_gram_space_full_size_llama_shapes(shape, monkeypatch):
    """The Llama-3-8B shapes Gram space would take with MUON_GRAM_SPACE=1
    (gate/up/down and k/v), at full size: NS error against the float64 oracle
    within 3e-2; the X-space error of the same input printed beside it."""
    x = torch.randn(shape, generator=torch.Generator().manual_seed(shape[1] + shape[2])).cuda()
    monkeypatch.setenv("MUON_GRAM_SPACE", "1")
    assert binding.muon_ns_path(shape[1], shape[2]) == binding.PATH_GRAM_SPACE
    eg = _errs(_ns(x, True, monkeypatch), x)
    ex = _errs(_ns(x, False, monkeypatch), x)
    print(f"{shape}: Gram space {max(eg):.4f}, X space {max(ex):.4f}")
    assert max(eg) <= NS_TOL


def test_gram_space_wide_bitwise(monkeypatch):
    """WIDE blocks on the Gram-space launches (forced) give the same bits."""
    monkeypatch.setenv("MUON_MAX_KSPLIT", "1")
    monkeypatch.setenv("MUON_GEMM_PAIR", "0")
    x = torch.randn((2, 640, 2048), generator=torch.Generator().manual_seed(4)).cuda()
    outs = []
    for wide in ("0", "1"):
        monkeypatch.setenv("MUON_GEMM_WIDE", wide)
        outs.append(_ns(x, True, monkeypatch))
    assert torch.equal(outs[0], outs[1])
