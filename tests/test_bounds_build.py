"""The debug bounds-check build compiles, and the normal build checks nothing.

The GPU side (tests/test_bounds_check_gpu.py) runs parity cases through the
checked library; here, without a GPU, the translation units that carry checks
are compiled with -DGDN_BOUNDS_CHECK for sm_103a, and the normal library's
gdn_bounds_violation reports -1 (no checks compiled in).
"""
import os
import shutil
import subprocess
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

import gated_deltanet_recurrence_gdn_gb300 as gdn
from gated_deltanet_recurrence_gdn_gb300 import _build

CHECKED_UNITS = ["gdn_tc.cu", "gdn_ut.cu", "gdn_prep.cu", "gdn_fused.cu", "gdn_bwd_tc.cu",
                 "gdn_api.cu"]


@pytest.mark.skipif(shutil.which(_build.NVCC) is None, reason="nvcc not available")
def test_checked_units_compile():
    with tempfile.TemporaryDirectory() as tmp:
        def compile_one(name):
            cmd = [_build.NVCC] + _build._flags() + _build.VARIANTS["check"] + [
                "-c", os.path.join(_build.CSRC, name), "-o", os.path.join(tmp, name + ".o")]
            r = subprocess.run(cmd, capture_output=True, text=True)
            return name, r.returncode, r.stdout + r.stderr

        with ThreadPoolExecutor(max_workers=len(CHECKED_UNITS)) as ex:
            results = list(ex.map(compile_one, CHECKED_UNITS))
    failed = [(n, out[-2000:]) for n, rc, out in results if rc != 0]
    assert not failed, failed


def test_normal_build_reports_no_checks():
    assert gdn.load().gdn_bounds_violation(0) == -1
