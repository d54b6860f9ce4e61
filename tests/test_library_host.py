"""Host-side checks of the C-ABI library (no GPU needed).

* libcgtp.so loads and exports every function declared in include/*.h;
* the planner's real CG blocks (an independent C++ Racah implementation) agree
  with the oracle's to 1e-14 for every (l1, l2, l3) with l <= 7;
* argument checks that fail before any device work.
"""

import ctypes
import os
import re

import numpy as np
import pytest

import clebsch_gordan_tensor_racah_gb300 as cg
from oracle import cg as ocg

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include")


def declared_functions():
    names = set()
    for h in sorted(os.listdir(INCLUDE)):
        if h.endswith(".h"):
            text = re.sub(r"/\*.*?\*/", "", open(os.path.join(INCLUDE, h)).read(), flags=re.S)
            names |= set(re.findall(r"\b(cgtp_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_binding_exports():
    assert set(declared_functions()) == set(cg.EXPORTS)


def test_library_loads_and_exports_every_symbol():
    L = cg.lib()
    for name in declared_functions():
        assert hasattr(L, name), name


def test_planner_cg_blocks_match_oracle():
    worst = 0.0
    for l1 in range(8):
        for l2 in range(8):
            for l3 in range(0, 8):
                a = cg.cgtp_real_cg_block(l1, l2, l3)
                b = ocg.real_cg_block(l1, l2, l3)
                worst = max(worst, float(np.abs(a - b).max()))
    assert worst < 1e-14


def test_real_cg_block_rejects_bad_l():
    with pytest.raises(cg.CgtpError) as e:
        cg.cgtp_real_cg_block(8, 0, 8)
    assert e.value.status == cg.CGTP_EINVAL


def test_plan_create_rejects_bad_arguments_before_device_work():
    L = cg.lib()
    h = ctypes.c_void_p()
    cases = [
        (b"8x0e+", b"0e", b"0e", 0, 0, 0, cg.CGTP_EINVAL),      # empty term
        (b"8x0q", b"0e", b"0e", 0, 0, 0, cg.CGTP_EINVAL),       # bad parity letter
        (b"8x9e", b"0e", b"9e", 0, 0, 0, cg.CGTP_EINVAL),       # l > 7
        (b"8x0e", b"2x0e", b"0e", 0, 0, 0, cg.CGTP_EUNSUPPORTED),  # in2 multiplicity
        (b"8x0e", b"0e", b"0e", 0, 0, 3, cg.CGTP_EINVAL),       # radial_k in uvu
        (b"8x0e", b"0e", b"0e", 1, 1, 8, cg.CGTP_EUNSUPPORTED),  # uvw FP64 with a radial basis
        (b"8x0e", b"0e", b"0e", 1, 0, 9, cg.CGTP_EUNSUPPORTED),  # more than 8 radial functions
        (b"8x0e", b"0e", b"0e", 1, 0, -1, cg.CGTP_EUNSUPPORTED),  # negative radial_k
        (b"8x0e", b"0e", b"0e", 1, 2, 8, cg.CGTP_EUNSUPPORTED),  # radial uvw in bfloat16
        (b"8x0e", b"0e", b"0e", 7, 0, 0, cg.CGTP_EINVAL),       # bad mode
        (b"8x1o", b"1o", b"1o", 0, 0, 0, cg.CGTP_EINVAL),       # no parity-allowed path
    ]
    for in1, in2, out, mode, dt, k, want in cases:
        st = L.cgtp_plan_create(ctypes.byref(h), in1, in2, out, None, 0, mode, dt, k)
        assert st == want, (in1, in2, out, st, L.cgtp_last_error())
        assert not h.value


def test_forbidden_instruction_rejected():
    L = cg.lib()
    h = ctypes.c_void_p()
    ins = (ctypes.c_int * 3)(0, 0, 0)          # 1o x 1o -> 1o violates parity
    st = L.cgtp_plan_create(ctypes.byref(h), b"4x1o", b"1o", b"1o+1e", ctypes.cast(ins, ctypes.c_void_p),
                            1, 0, 0, 0)
    assert st == cg.CGTP_EINVAL
    assert b"parity" in L.cgtp_last_error()


def test_null_handles_rejected():
    L = cg.lib()
    assert L.cgtp_conv_forward(None, None, None, None, None, None, None, None) == cg.CGTP_EINVAL
    assert L.cgtp_forward(None, None, None, None, None, 0, None) == cg.CGTP_EINVAL
    assert L.cgtp_plan_info(None, None, None, None, None, None) == cg.CGTP_EINVAL


def test_library_sh_matches_oracle():
    # the harmonics the kernels evaluate from edge vectors (host build of the same
    # code) against the oracle's scipy-based ones, values and Jacobian, l <= 7
    rng = np.random.default_rng(41)
    r = rng.normal(size=(60, 3)) * rng.uniform(0.1, 5.0, size=(60, 1))
    Y, dY = cg.cgtp_real_sh(7, r, jacobian=True)
    u = r / np.linalg.norm(r, axis=1, keepdims=True)
    assert np.abs(Y - ocg.sh_real_concat(7, u)).max() < 1e-12
    assert np.abs(dY - ocg.sh_real_concat_jacobian(7, r)).max() < 1e-11


def test_mixed_plan_create_rejects_bad_arguments_before_device_work():
    L = cg.lib()
    h = ctypes.c_void_p()
    ins = (ctypes.c_int * 6)(0, 0, 0, 1, 1, 0)
    good = (ctypes.c_int * 2)(cg.CGTP_UVU, cg.CGTP_UVW)
    bad_mode = (ctypes.c_int * 2)(cg.CGTP_UVU, 5)
    cases = [
        (b"2x0e+2x1o", b"0e+1o", b"2x0e", good, 2, 7, cg.CGTP_EINVAL),    # unknown dtype
        (b"2x0e+2x1o", b"0e+1o", b"3x0e", good, 2, cg.CGTP_F32, cg.CGTP_EINVAL),   # uvu changes multiplicity
        (b"2x0e+2x1o", b"0e+1o", b"2x0e", bad_mode, 2, cg.CGTP_F32, cg.CGTP_EINVAL),
        (b"2x0e+2x1o", b"0e+1o", b"2x0e", good, 0, cg.CGTP_F32, cg.CGTP_EINVAL),   # empty list
        (b"2x0e+2x1o+", b"0e+1o", b"2x0e", good, 2, cg.CGTP_F32, cg.CGTP_EINVAL),  # bad irreps
    ]
    for in1, in2, out, modes, n, dt, want in cases:
        st = L.cgtp_mixed_plan_create(ctypes.byref(h), in1, in2, out, ctypes.cast(ins, ctypes.c_void_p),
                                      ctypes.cast(modes, ctypes.c_void_p), n, dt)
        assert st == want, (in1, out, n, dt, st, L.cgtp_last_error())
        assert not h.value
    oob = (ctypes.c_int * 3)(0, 0, 4)
    st = L.cgtp_mixed_plan_create(ctypes.byref(h), b"2x0e", b"0e", b"2x0e", ctypes.cast(oob, ctypes.c_void_p),
                                  ctypes.cast(good, ctypes.c_void_p), 1, cg.CGTP_F32)
    assert st == cg.CGTP_EINVAL and b"out of range" in L.cgtp_last_error()
