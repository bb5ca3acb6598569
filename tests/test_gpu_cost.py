"""The per-shape NS cost table measured on the GPU (DMuon-2 Appendix B: NS
time is measured per shape, not estimated from element counts)."""
import pytest

from newton_schulz_gb300 import binding

pytestmark = pytest.mark.gpu


def test_cost_table_sane(lib, cuda_ok):
    shapes = [(1024, 4096), (4096, 4096), (4096, 14336), (24, 10240), (4096, 1024)]
    ms = binding.muon_ns_cost_table(shapes, reps=3)
    assert all(x > 0 for x in ms)
    # more work costs more; a transposed shape costs what its core shape does
    assert ms[0] < ms[1] < ms[2]
    assert ms[3] < ms[0]
    assert 0.7 < ms[4] / ms[0] < 1.4
