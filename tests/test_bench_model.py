"""The benchmark's FLOP model (bench.py `model_flops`) against the per-configuration
figures it is meant to reproduce: the coupling matrix's nonzeros, the weight term
per output component, backward = 3 x forward.

The plan stand-in is built from the oracle's path list (the library's plan needs a
GPU); the nonzero counts come from the library's host CG blocks, as in bench.py.
Expected values: NequIP-like forward 14.7 GFLOP, high-L batched 34 GFLOP, radial uvw
295 GFLOP on the edges plus 459 GFLOP of node GEMM.
"""

import importlib.util
import os

import pytest

from clebsch_gordan_tensor_racah_gb300 import workloads as wl
from oracle import irreps as oirr

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


class _Plan:
    """The attributes model_flops reads, from the oracle's plan."""

    def __init__(self, name, radial_k=0):
        s = wl.SPECS[name]
        self.mode = s["mode"]
        self.radial_k = radial_k
        self._p = oirr.make_plan(s["in1"], s["in2"], s["out"], s["mode"])
        self.n_paths = len(self._p.paths)
        self.d_out = self._p.d_out

    def path(self, i):
        q = self._p.paths[i]
        return (q.l1, q.l2, q.l3, q.mul1, q.mul_out), None


@pytest.fixture(scope="module")
def bench():
    return _bench()


def test_flop_model_nequip(bench):
    p = _Plan("nequip")
    fwd, tensor = bench.model_flops(p, 10_000, 320_000, graph=True)
    assert tensor == 0.0
    assert abs(fwd / 1e9 - 14.7) < 0.05, fwd / 1e9


def test_flop_model_high_l_batched(bench):
    p = _Plan("highl")
    fwd, _ = bench.model_flops(p, 50_000, 50_000, graph=False)
    assert abs(fwd / 1e9 - 34.0) < 0.1, fwd / 1e9


def test_flop_model_radial_uvw(bench):
    p = _Plan("uvw", radial_k=8)
    edge, node = bench.model_flops(p, 200_000, 6_400_000, graph=True)
    assert abs(edge / 1e9 - 295.0) < 1.0, edge / 1e9
    assert abs(node / 1e9 - 459.0) < 1.0, node / 1e9


def test_cg_counts_small_blocks(bench):
    # (0,0,0): one nonzero; (1,1,0): the dot product (3 nonzeros, m1 = m3 pattern of 3);
    # (1,1,1): the cross product (6 nonzeros, every (m1, m3) with m1 != m3)
    assert bench._cg_counts(0, 0, 0) == (1, 1)
    assert bench._cg_counts(1, 1, 0) == (3, 3)
    assert bench._cg_counts(1, 1, 1) == (6, 6)
