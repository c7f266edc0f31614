"""The bounds-checked build (libqsa_bounds.so, compiled with QSA_DEBUG_BOUNDS):
every kernel checks the indices it derives from data -- page ids and token
offsets of its copies, list / union / selection slots, output rows, workspace
units -- records the first failed check in a device word and skips the access.
Here the small parity cases of the other GPU test files run again in a child
process against that build (QSA_BOUNDS_CHECKED=1); the conftest fixture there
asserts after every test that no check failed, and each test still compares
with the oracle as usual.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu

# Small parity cases: every kernel and path (decode-row attention, verify
# attention, the fused selection, row-tile attention, index and selection,
# token store and rollback) at sizes that span several tiles and ragged tails.
SELECT = ("small_configs or forced_splits or edge_cases or all_pages_invalid or "
          "all_equal_scores or fused_selection or prefill_matches or prefill_all_pages or "
          "prefill_on_verify or store_small or store_edge or rollback")


def test_bounds_checked_build_is_loaded_and_armed():
    code = subprocess.run(
        [sys.executable, "-c",
         "import nvfp4_block_sparse_gb300 as q; q.load(); "
         "print(q.library_path()); print(q.qsa_debug_bounds_status())"],
        cwd=ROOT, env=dict(os.environ, QSA_BOUNDS_CHECKED="1"), capture_output=True, text=True,
        timeout=600)
    assert code.returncode == 0, code.stderr[-2000:]
    path, status = code.stdout.split()[-2:]
    assert path.endswith("libqsa_bounds.so")
    assert status == "0"    # -1 would mean the checks are not compiled in


def test_parity_cases_hold_every_bounds_check():
    r = subprocess.run(
        [sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider",
         "tests/test_gpu_parity.py", "tests/test_gpu_prefill.py", "tests/test_gpu_store.py",
         "-k", SELECT],
        cwd=ROOT, env=dict(os.environ, QSA_BOUNDS_CHECKED="1"), capture_output=True, text=True,
        timeout=1800)
    tail = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and " failed" not in r.stdout, tail
