"""Build libcgtp.so in-tree for sm_103a (nvcc + g++, translation units in parallel).

The library is the product: every step of the fused CG tensor-product
convolution runs in its kernels.  Objects go to ``_build/`` at the repository
root; the shared object is written next to this file.
"""

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INC = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libcgtp.so")

CU_SOURCES = ["api.cu", "graph.cu", "uvu.cu", "uvu_f32.cu", "uvu_f32_l7.cu", "uvu_f64.cu",
              "uvu_f64_l7.cu", "uvu2.cu", "uvu3.cu", "uvu3_f32_2.cu", "uvu3_f32_8.cu", "uvu3_f32_32.cu",
              "uvu3_f64_2.cu", "uvu3_f64_8.cu", "uvu3_f64_32.cu", "uvw.cu", "bt.cu", "dbl.cu",
              "uvu3_bf16_2.cu", "uvu3_bf16_8.cu", "uvu3_bf16_32.cu", "sh.cu",
              "uvu3_sh_f32_2.cu", "uvu3_sh_f32_8.cu", "uvu3_sh_f32_32.cu", "uvu3_sh_f64_2.cu",
              "uvu3_sh_f64_8.cu", "uvu3_sh_f64_32.cu", "uvwe.cu", "mixed.cu", "measure.cu"]
CPP_SOURCES = ["planner.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    for cand in (os.environ.get("CUDACXX"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


_INC_RE = None


def _deps_mtime(path, seen=None):
    """Newest mtime of a source and the quoted headers it includes, transitively
    (looked up next to it, in include/ and in the generated-code folder)."""
    global _INC_RE
    import re
    if _INC_RE is None:
        _INC_RE = re.compile(r'^\s*#\s*include\s+"([^"]+)"', re.M)
    seen = set() if seen is None else seen
    if path in seen or not os.path.exists(path):
        return 0.0
    seen.add(path)
    m = os.path.getmtime(path)
    for name in _INC_RE.findall(open(path, errors="replace").read()):
        for d in (os.path.dirname(path), CSRC, INC, GEN):
            cand = os.path.join(d, name)
            if os.path.exists(cand):
                m = max(m, _deps_mtime(cand, seen))
                break
    return m


def _stale(src, obj):
    return not os.path.exists(obj) or os.path.getmtime(obj) < _deps_mtime(src)


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("build failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


GEN = os.path.join(BUILD, "gen")


def _bake():
    """Build and run gen_baked: the planner's CG blocks (l <= 3) as compile-time code."""
    os.makedirs(GEN, exist_ok=True)
    exe = os.path.join(GEN, "gen_baked")
    out = os.path.join(GEN, "cg_baked.cuh")
    srcs = [os.path.join(CSRC, "gen_baked.cpp"), os.path.join(CSRC, "planner.cpp")]
    deps = srcs + [os.path.join(CSRC, "internal.h"), os.path.join(INC, "cgtp.h")]
    if not os.path.exists(out) or os.path.getmtime(out) < max(os.path.getmtime(d) for d in deps):
        _run(["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-I", INC, "-I", CSRC, *srcs, "-o", exe])
        _run([exe, out + ".tmp"])
        os.replace(out + ".tmp", out)
    return os.path.getmtime(out)


def build(verbose=False, jobs=None):
    """Compile (incrementally) and link libcgtp.so; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    _bake()
    cmds = []
    objs = []
    for f in CU_SOURCES:
        src, obj = os.path.join(CSRC, f), os.path.join(BUILD, f + ".o")
        objs.append(obj)
        if _stale(src, obj):
            cmds.append([nvcc, "-std=c++17", "-O3", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC",
                         "-Xcompiler", "-ffp-contract=off", "-I", INC, "-I", GEN, "-c", src, "-o", obj])
    for f in CPP_SOURCES:
        src, obj = os.path.join(CSRC, f), os.path.join(BUILD, f + ".o")
        objs.append(obj)
        if _stale(src, obj):
            cmds.append(["g++", "-std=c++17", "-O2", "-fPIC", "-ffp-contract=off", "-I", INC,
                         "-c", src, "-o", obj])
    jobs = jobs or max(1, min(len(cmds), os.cpu_count() or 4))
    if cmds:
        # longest translation units first
        cmds.sort(key=lambda c: ("_l7" not in c[-3] and "uvu3_" not in c[-3], c[-3]))
        with cf.ThreadPoolExecutor(jobs) as ex:
            for out in ex.map(_run, cmds):
                if verbose and out.strip():
                    print(out)
    if cmds or not os.path.exists(LIB) or os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs):
        tmp = LIB + ".tmp"
        _run([nvcc, "-shared", *ARCH, "-o", tmp, *objs, "-cudart=static"])
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
