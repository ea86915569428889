"""The checked build (compiled with AQ_DEBUG_CHECKS): every plain output store of the hot-path
kernels checks its index against the extent of the output it addresses, skips an out-of-range
store and records AQ_ERR_BOUNDS in the device status word (no trap, no device assert). The
brute-force sweep of tiny shapes with every path forced, the parity suite and the NVFP4 tests
run again on that library in a child process; each of their tests also asserts that the
device status word reads AQ_OK, so a store the checks skipped fails them."""
import ctypes
import os
import subprocess
import sys

import pytest

from rank_weight_reconstruction_gb300 import binding, build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checked_library_builds_and_exports():
    """Runs without a GPU: the checked library builds and exports every declared symbol."""
    lib = ctypes.CDLL(build_lib.build(debug=True))
    for name in binding.EXPORTED_SYMBOLS:
        assert hasattr(lib, name), name
    lib.aq_checked_build.restype = ctypes.c_int32
    assert lib.aq_checked_build() == 1


@pytest.mark.gpu
def test_suites_on_the_checked_library():
    path = build_lib.build(debug=True)
    env = dict(os.environ, AQ_TEST_CHECKED_LIB=path)
    code = "\n".join([
        "import rank_weight_reconstruction_gb300 as aq",
        "from rank_weight_reconstruction_gb300 import binding",
        f"lib = binding.load({path!r})",
        "assert lib.aq_checked_build() == 1, 'not the checked library'",
        "st = aq.aq_device_status(); assert st == aq.AQ_OK, ('status before', st)",
        "rc = lib.aq_selftest_bounds_check(None); assert rc == aq.AQ_OK, ('launch', rc)",
        "st = aq.aq_device_status(); assert st == binding.AQ_ERR_BOUNDS, ('status after', st)",
        "st = aq.aq_device_status(); assert st == aq.AQ_OK, ('status cleared', st)",
    ])
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_tiny_sweep_gpu.py", "tests/test_parity_gpu.py",
                        "tests/test_nvfp4_gpu.py", "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=3000)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout


@pytest.mark.gpu
def test_normal_build_reports_no_bounds_check():
    """In the normal build the self test checks nothing: the status word stays AQ_OK."""
    import rank_weight_reconstruction_gb300 as aq
    lib = binding.load()
    if os.environ.get("AQ_TEST_CHECKED_LIB"):
        pytest.skip("running on the checked library")
    assert lib.aq_checked_build() == 0
    assert aq.aq_device_status() == aq.AQ_OK
    lib.aq_selftest_bounds_check(None)
    assert aq.aq_device_status() == aq.AQ_OK
