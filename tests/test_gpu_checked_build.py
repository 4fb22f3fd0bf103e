"""The bounds-checked build (libglance_check.so, -DGLANCE_CHECK): on a fixed
set of in-range calls — a single-request round, a ragged batch (ticket-mode
attention, the LM head's CTA-pair kernel), the fp32 attention path and the
tree-row K/V scatter — it returns exactly what libglance.so returns, and no
check fires (every device status word stays 0). Each library runs in its own
process (the binding loads one library per process)."""
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_DIR = os.path.join(os.path.dirname(HERE), "tree_verified_block_gb300", "_lib")


def run_cases(lib, out):
    r = subprocess.run([sys.executable, os.path.join(HERE, "_checked_cases.py"), lib, out],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    return np.load(out)


def test_checked_build_matches_and_reports_nothing(tmp_path):
    checked = os.path.join(LIB_DIR, "libglance_check.so")
    if not os.path.exists(checked):
        pytest.skip("libglance_check.so not built (run __graft_entry__.build())")
    normal = run_cases(os.path.join(LIB_DIR, "libglance.so"), str(tmp_path / "normal.npz"))
    chk = run_cases(checked, str(tmp_path / "checked.npz"))
    assert sorted(normal.files) == sorted(chk.files)
    assert np.all(chk["status"] == 0), chk["status"]
    assert np.all(normal["status"] == 0), normal["status"]
    for k in normal.files:
        assert np.array_equal(normal[k], chk[k], equal_nan=True), k
