"""The HQ_DEBUG build (libhq_debug.so): the same C ABI as libhq.so with device
bounds checks on the kernels' global writes.

CPU: it builds, exports every function include/hq.h declares, reports itself
as the debug build, and the release library refuses the debug self-test.
GPU: in a child process with HQ_DEBUG=1, the self-test's failed check sets
HQ_STATUS_BOUNDS without touching memory; every hot-path kernel on valid
inputs sets no status bit and writes the same bytes as the release library
(debug_build_cases.py computes both)."""

import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest

from fp4_grouped_gemm_gb300 import _abi, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, os.path.join(ROOT, "tests"))
from test_abi_host import declared_functions  # noqa: E402


@pytest.fixture(scope="module")
def libs():
    rel = ctypes.CDLL(build.build())
    dbg = ctypes.CDLL(build.build(debug=True))
    return rel, dbg


def test_debug_library_exports_the_abi(libs):
    rel, dbg = libs
    for name in declared_functions():
        assert hasattr(dbg, name), name


def test_debug_flag_and_release_refusal(libs):
    rel, dbg = libs
    assert rel.hq_debug_build() == 0 and dbg.hq_debug_build() == 1
    # the release library launches nothing for the self-test
    assert rel.hq_debug_selftest(None) == _abi.HQ_ERR_UNSUPPORTED


def test_package_selects_the_debug_library_by_environment():
    code = ("import fp4_grouped_gemm_gb300 as hq, os; "
            "print(os.path.basename(hq._abi.lib_path()), hq.debug_build())")
    env = dict(os.environ, HQ_DEBUG="1")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                         timeout=300)
    assert out.returncode == 0, out.stderr
    assert out.stdout.split() == ["libhq_debug.so", "True"]


@pytest.mark.gpu
def test_debug_kernels_match_release_and_flag_nothing(cuda_dev, tmp_path):
    build.build(debug=True)
    script = os.path.join(ROOT, "tests", "debug_build_cases.py")
    env = dict(os.environ, HQ_DEBUG="1")
    dbg = subprocess.run([sys.executable, script, str(tmp_path / "debug.npz")], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=900)
    assert dbg.returncode == 0, dbg.stdout + dbg.stderr
    lines = dbg.stdout.strip().splitlines()
    assert lines[0] == "selftest status 0x40", lines[0]   # the failed check, recorded
    assert lines[1] == "cases status 0x0", lines[1]       # valid inputs: no check fails
    env = dict(os.environ, HQ_DEBUG="0")
    rel = subprocess.run([sys.executable, script, str(tmp_path / "release.npz")], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=900)
    assert rel.returncode == 0, rel.stdout + rel.stderr
    a = np.load(tmp_path / "debug.npz")
    b = np.load(tmp_path / "release.npz")
    assert sorted(a.files) == sorted(b.files) and len(a.files) >= 10
    for k in a.files:
        if k.startswith("sum_"):
            # float-atomic sums: equal up to the order of the adds, whose
            # rounding scales with the partial sums (the row's largest), not
            # with a result that cancels
            assert np.allclose(a[k], b[k], rtol=1e-4, atol=1e-5 * np.abs(b[k]).max()), k
        else:
            assert np.array_equal(a[k], b[k]), k
