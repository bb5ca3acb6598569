"""Host-only checks of the C ABI: the library loads without a GPU, exports
every entry point declared in include/muon.h, and rejects bad arguments before
touching CUDA (nothing is enqueued, so no device is needed)."""
import ctypes
import os
import re

import pytest

from newton_schulz_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "muon.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(muon_[a-z_]+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    names = _declared_functions()
    for n in ("muon_ns_batched", "muon_step_grouped", "muon_ns_batched_ex",
              "muon_step_grouped_ex", "muon_query_status", "muon_status_string",
              "muon_release_workspace"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
    for name in binding.EXPORTED:
        assert name in _declared_functions()


def test_status_strings(lib):
    for code, name in binding.STATUS_NAMES.items():
        assert lib.muon_status_string(code).decode() == name
    assert lib.muon_status_string(99).decode() == "MUON_ERR_UNKNOWN"


def test_default_config(lib):
    cfg = binding.NsConfig()
    assert lib.muon_ns_default_config(ctypes.byref(cfg)) == 0
    assert cfg.steps == 5 and cfg.precision == 0
    assert abs(cfg.a - 3.4445) < 1e-6 and abs(cfg.b + 4.775) < 1e-6 and abs(cfg.c - 2.0315) < 1e-6
    assert abs(cfg.eps - 1e-7) < 1e-12
    assert lib.muon_ns_default_config(None) == 1


E_INV, E_UNS, E_ALIAS = 1, 2, 3


def _grp(W=0x1000, G=0x100000, M_=0x200000, B=1, M=4, N=8, wdt=0, gdt=0):
    return binding.Group(W, wdt, G, gdt, M_, B, M, N)


def _step(lib, groups, n=None, mu=0.95, lr=0.02, wd=0.01, rule=0, cfg=None):
    arr = (binding.Group * max(1, len(groups)))(*groups)
    n = len(groups) if n is None else n
    if cfg is None:
        return lib.muon_step_grouped(arr, n, mu, 1, lr, wd, rule, None)
    return lib.muon_step_grouped_ex(arr, n, mu, 1, lr, wd, rule, ctypes.byref(cfg), None)


def test_step_argument_errors(lib):
    assert lib.muon_step_grouped(None, 1, 0.95, 1, 0.02, 0.01, 0, None) == E_INV
    assert lib.muon_step_grouped(None, -1, 0.95, 1, 0.02, 0.01, 0, None) == E_INV
    assert _step(lib, [_grp(B=-1)]) == E_INV
    assert _step(lib, [_grp(M=-2)]) == E_INV
    assert _step(lib, [_grp(W=0)]) == E_INV
    assert _step(lib, [_grp(G=0)]) == E_INV
    assert _step(lib, [_grp(M_=0)]) == E_INV
    assert _step(lib, [_grp(wdt=7)]) == E_INV
    assert _step(lib, [_grp(gdt=-1)]) == E_INV
    assert _step(lib, [_grp(W=0x1001)]) == E_INV          # misaligned f32
    assert _step(lib, [_grp()], rule=9) == E_INV
    assert _step(lib, [_grp()], mu=float("nan")) == E_INV
    assert _step(lib, [_grp()], lr=float("inf")) == E_INV


def test_step_alias_errors(lib):
    # W overlaps Mom
    assert _step(lib, [_grp(W=0x1000, M_=0x1040)]) == E_ALIAS
    # G overlaps W
    assert _step(lib, [_grp(W=0x1000, G=0x1010)]) == E_ALIAS
    # W of one group overlaps Mom of another
    assert _step(lib, [_grp(W=0x1000, G=0x100000, M_=0x200000),
                       _grp(W=0x300000, G=0x400000, M_=0x1000)]) == E_ALIAS


def test_ns_config_errors(lib):
    assert _step(lib, [_grp()], cfg=binding.make_config(steps=-1)) == E_INV
    assert _step(lib, [_grp()], cfg=binding.make_config(steps=65)) == E_INV
    assert _step(lib, [_grp()], cfg=binding.make_config(eps=-1.0)) == E_INV
    assert _step(lib, [_grp()], cfg=binding.make_config(precision=5)) == E_INV
    bad = binding.make_config(steps=2, coeffs=[[1, 2, 3], [float("nan"), 0, 0]])
    assert _step(lib, [_grp()], cfg=bad) == E_INV


def test_empty_inputs_are_noops(lib):
    assert lib.muon_step_grouped(None, 0, 0.95, 1, 0.02, 0.01, 0, None) == 0
    assert _step(lib, [_grp(B=0, W=0, G=0, M_=0)]) == 0
    assert lib.muon_ns_batched(None, 0, 3, 4, 5, 1.0, 0.0, 0.0, None) == 0
    assert lib.muon_ns_batched(0x1000, 2, 0, 4, 5, 1.0, 0.0, 0.0, None) == 0


def test_ns_argument_errors(lib):
    assert lib.muon_ns_batched(None, 1, 3, 4, 5, 1.0, 0.0, 0.0, None) == E_INV
    assert lib.muon_ns_batched(0x1001, 1, 3, 4, 5, 1.0, 0.0, 0.0, None) == E_INV
    assert lib.muon_ns_batched(0x1000, -1, 3, 4, 5, 1.0, 0.0, 0.0, None) == E_INV
    assert lib.muon_ns_batched(0x1000, 1, 3, 4, -1, 1.0, 0.0, 0.0, None) == E_INV
    assert lib.muon_ns_batched(0x1000, 1, 3, 4, 5, float("nan"), 0.0, 0.0, None) == E_INV
    assert lib.muon_ns_batched_ex(0x1000, 3, 1, 3, 4, None, None, None) == E_INV
    # out overlapping X
    assert lib.muon_ns_batched_ex(0x1000, 0, 1, 3, 4, None, 0x1008, None) == E_ALIAS


def test_host_step_argument_errors(lib):
    def host(groups, **kw):
        arr = (binding.Group * max(1, len(groups)))(*groups)
        cfg = kw.get("cfg")
        return lib.muon_step_grouped_host(arr, len(groups), 0.95, 1, kw.get("lr", 0.02), 0.01,
                                          kw.get("rule", 0),
                                          ctypes.byref(cfg) if cfg is not None else None, None)
    assert lib.muon_step_grouped_host(None, 1, 0.95, 1, 0.02, 0.01, 0, None, None) == E_INV
    assert host([_grp(W=0)]) == E_INV
    assert host([_grp(wdt=3)]) == E_INV
    assert host([_grp()], rule=7) == E_INV
    assert host([_grp()], lr=float("nan")) == E_INV
    assert host([_grp(W=0x1000, M_=0x1040)]) == E_ALIAS
    assert host([_grp(B=0, W=0, G=0, M_=0)]) == 0


def test_adamw_argument_errors(lib):
    def grp(p=0x1000, g=0x100000, m=0x200000, v=0x300000, n=16, pdt=0, gdt=0):
        return binding.AdamwGroup(p, pdt, g, gdt, m, v, n)

    def call(groups, **kw):
        cfg = binding.AdamwConfig(kw.get("lr", 1e-3), kw.get("b1", 0.9), kw.get("b2", 0.999),
                                  kw.get("eps", 1e-8), kw.get("wd", 0.01), kw.get("step", 1))
        arr = (binding.AdamwGroup * max(1, len(groups)))(*groups)
        return lib.muon_adamw_grouped(arr, len(groups), ctypes.byref(cfg), None)
    assert lib.muon_adamw_grouped(None, 1, None, None) == E_INV
    assert call([grp()], step=0) == E_INV
    assert call([grp()], b1=1.0) == E_INV
    assert call([grp()], b2=-0.1) == E_INV
    assert call([grp()], eps=-1.0) == E_INV
    assert call([grp()], lr=float("nan")) == E_INV
    assert call([grp(p=0)]) == E_INV
    assert call([grp(pdt=4)]) == E_INV
    assert call([grp(n=-1)]) == E_INV
    assert call([grp(p=0x1002)]) == E_INV            # misaligned f32
    assert call([grp(m=0x1020)]) == E_ALIAS          # exp_avg inside param
    assert call([grp(g=0x1010)]) == E_ALIAS          # grad inside param
    assert call([grp(p=0, g=0, m=0, v=0, n=0)]) == 0  # empty tensors are skipped


def test_debug_inject_stall_arguments(lib):
    """The failure-path testing hook takes 0 (cancel), 1 (GEMM) or 2 (small-m)
    and only records the request (nothing is launched by it)."""
    assert lib.muon_debug_inject_stall(3) == 1
    assert lib.muon_debug_inject_stall(-1) == 1
    assert lib.muon_debug_inject_stall(1) == 0
    assert lib.muon_debug_inject_stall(2) == 0
    assert lib.muon_debug_inject_stall(0) == 0


def test_debug_guard_check_needs_an_output(lib):
    assert lib.muon_debug_guard_check(None, None) == 1


def test_binding_rejects_out_of_another_dtype_or_shape():
    """muon_ns_batched_ex writes `out` in X's dtype and shape; the C entry point
    sees only a pointer, so the binding refuses a mismatched `out` (fp32 data
    into a bf16 buffer would write past its end) before the library is
    reached (CPU tensors: nothing runs)."""
    import torch
    x = torch.zeros((2, 8, 16), dtype=torch.float32)
    for out in (torch.zeros((2, 8, 16), dtype=torch.bfloat16),
                torch.zeros((2, 16, 8), dtype=torch.float32),
                torch.zeros((1, 8, 16), dtype=torch.float32)):
        with pytest.raises(ValueError, match="out must match X"):
            binding.muon_ns_batched_ex(x, binding.make_config(), out)
