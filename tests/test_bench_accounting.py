"""Host-side pieces of the measurement: the algorithmic flop count bench.py
reports per GEMM kind, and the library's path choice and Gram-space restart
period it is built on (decided on the host, no GPU needed).

The Gram-space count is checked against an independent walk through the
phase structure the library issues (per phase: the Gram; per step B' unless
it is a one-step phase, Q, and T and R unless it is the phase's last step;
the apply), and against the closed form (3 r + 4 P - 2) m^3 per phase of
P >= 2 steps that include/muon.h states (m(m+1) ~ m^2).
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _walk(steps, period):
    """(Grams, m x m products, applies) of one matrix in Gram space."""
    grams = prods = applies = 0
    k0 = 0
    while k0 < steps:
        k1 = min(steps, k0 + period)
        grams += 1
        for it in range(k0, k1):
            more = it + 1 < k1
            if it > k0 or more:
                prods += 1          # B'
            prods += 1              # Q (P_k at the phase's first step, else the update)
            if more:
                prods += 2          # T, R
        applies += 1
        k0 = k1
    return grams, prods, applies


@pytest.mark.parametrize("steps,period", [(5, 3), (5, 2), (5, 1), (5, 5), (3, 2), (1, 3), (4, 3)])
def test_gram_space_count_matches_phase_walk(steps, period):
    m, n = 1024, 4096
    f = bench.matrix_flops(m, n, 2, steps=steps, restart=period)
    g, p, a = _walk(steps, period)
    assert f["gram"] == g * m * (m + 1) * n
    assert f["poly"] == p * m * m * (m + 1)
    assert f["apply"] == a * 2 * m * m * n


def test_gram_space_closed_form_and_x_space():
    m, n = 2048, 7168          # r = 3.5
    r = n / m
    f = bench.matrix_flops(m, n, 2, steps=5, restart=3)       # phases of 3 and 2 steps
    closed = ((3 * r + 4 * 3 - 2) + (3 * r + 4 * 2 - 2)) * m ** 3
    assert abs(sum(f.values()) - closed) / closed < 1e-3       # m(m+1) against m^2
    x = bench.matrix_flops(m, n, 1, steps=5)
    assert x == {"gram": 5 * m * (m + 1) * n, "poly": 5 * m * m * (m + 1),
                 "apply": 5 * 2 * m * m * n}
    assert abs(sum(x.values()) - (15 * r + 5) * m ** 3) / ((15 * r + 5) * m ** 3) < 1e-3
    # no restart: one phase of five steps
    f0 = bench.matrix_flops(m, n, 2, steps=5, restart=0)
    assert f0["gram"] == m * (m + 1) * n and f0["apply"] == 2 * m * m * n
    assert f0["poly"] == 18 * m * m * (m + 1)


def test_nominal_flops():
    assert bench.ns_flops(24, 10240) == 5 * (4 * 24 * 24 * 10240 + 2 * 24 ** 3)
    assert bench.ns_flops(10240, 24) == bench.ns_flops(24, 10240)


def test_path_choice_and_restart(lib, monkeypatch):
    from newton_schulz_gb300 import binding
    for k in ("MUON_GRAM_SPACE", "MUON_GRAM_SPACE_RATIO", "MUON_GRAM_RESTART", "MUON_SMALL_PATH"):
        monkeypatch.delenv(k, raising=False)
    P = binding
    assert P.muon_ns_path(24, 10240) == P.PATH_SMALL
    assert P.muon_ns_path(10240, 64) == P.PATH_SMALL
    assert P.muon_ns_path(4096, 4096) == P.PATH_XSPACE          # n < 2m
    assert P.muon_ns_path(768, 2048) == P.PATH_XSPACE           # m < 1024
    assert P.muon_ns_path(1024, 2048) == P.PATH_GRAM_SPACE      # n = 2m
    assert P.muon_ns_path(14336, 4096) == P.PATH_GRAM_SPACE     # transposed
    assert P.muon_ns_path(1024, 2047) == P.PATH_XSPACE
    assert P.muon_ns_path(1024, 4096, P.make_config(precision=P.NS_TF32)) == P.PATH_XSPACE
    assert P.muon_ns_path(1024, 4096, P.make_config(steps=0)) == P.PATH_XSPACE
    assert P.muon_ns_path(0, 4096) == -1
    monkeypatch.setenv("MUON_GRAM_SPACE", "0")
    assert P.muon_ns_path(1024, 4096) == P.PATH_XSPACE
    monkeypatch.setenv("MUON_GRAM_SPACE", "force")
    assert P.muon_ns_path(300, 300) == P.PATH_GRAM_SPACE
    assert P.muon_ns_path(24, 10240) == P.PATH_SMALL
    monkeypatch.setenv("MUON_SMALL_PATH", "0")
    assert P.muon_ns_path(24, 10240) == P.PATH_GRAM_SPACE
    monkeypatch.delenv("MUON_GRAM_SPACE")
    assert P.muon_ns_path(24, 10240) == P.PATH_XSPACE
    assert P.muon_ns_gram_restart(768) == 2
    assert P.muon_ns_gram_restart(1024) == 3
    assert P.muon_ns_gram_restart(0) == -1
    monkeypatch.setenv("MUON_GRAM_RESTART", "4")
    assert P.muon_ns_gram_restart(8192) == 4
    monkeypatch.setenv("MUON_GRAM_RESTART", "0")
    assert P.muon_ns_gram_restart(8192) == 0
