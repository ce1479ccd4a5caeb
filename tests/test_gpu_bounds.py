"""The bounds-checked build (libbsa_bounds.so, -DBSA_BOUNDS_CHECK=1).

1. On valid inputs it gives the default build's results bit for bit: prefill
   (route, worklist, attention forward and backward on the tensor-core and SIMT
   paths), paged decode and a chunk over a paged cache.
2. Worklist col_idx entries outside [0, r] (below 0, past the diagonal, far past
   the table) and a chunk block-table entry past the cache's pages are reported as
   BSA_ERR_INDEX_RANGE by the forward, the backward and the chunk attention, and
   the calls complete (the checked kernels clamp the index instead of using it).
   These inputs run only on the bounds-checked library: the child refuses them
   otherwise.

Each library runs in a child process (tests/bounds_child.py), since the package
loads one library per process (BSA_BOUNDS_CHECK selects it).
"""
import os
import subprocess
import sys

import numpy as np
import pytest

from dynamic_block_sparse_mean_gb300 import build as bsa_build

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
INDEX_RANGE = 16


def run_child(path, bounds, corrupt):
    env = dict(os.environ, BSA_BOUNDS_CHECK="1" if bounds else "0")
    cmd = [sys.executable, os.path.join(HERE, "bounds_child.py"), str(path)]
    if corrupt:
        cmd.append("--corrupt")
    res = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-3000:]
    return dict(np.load(path))


@pytest.fixture(scope="module")
def outputs(tmp_path_factory):
    bsa_build.build()
    bsa_build.build(bounds_check=True)
    d = tmp_path_factory.mktemp("bounds")
    plain = run_child(d / "plain.npz", bounds=False, corrupt=False)
    checked = run_child(d / "checked.npz", bounds=True, corrupt=True)
    return plain, checked


def test_libraries_report_their_build(outputs):
    plain, checked = outputs
    assert int(plain["bounds_checked"][0]) == 0
    assert int(checked["bounds_checked"][0]) == 1


# The FP32 SIMT backward adds dK / dV contributions with atomics, whose order (and
# so the last bits) varies from call to call in either build; those two outputs are
# compared to a relative 1e-5 of their largest magnitude instead.
ATOMIC_SUMS = {"fp32_d64_dk", "fp32_d64_dv"}


def test_bounds_checked_build_matches_default_bit_for_bit(outputs):
    plain, checked = outputs
    keys = [k for k in plain if k != "bounds_checked"]
    assert len(keys) > 20
    for k in keys:
        if k.endswith("_status"):
            assert int(plain[k][0]) == 0 and int(checked[k][0]) == 0, k
            continue
        assert plain[k].shape == checked[k].shape, k
        if k in ATOMIC_SUMS:
            scale = float(np.abs(plain[k]).max())
            assert float(np.abs(plain[k] - checked[k]).max()) <= 1e-5 * scale, k
        else:
            assert np.array_equal(plain[k], checked[k]), k


@pytest.mark.parametrize("tag", ["bf16_b64", "bf16_b128", "fp32_d64"])
@pytest.mark.parametrize("call", ["fwd", "bwd"])
def test_out_of_range_worklist_entries_are_reported(outputs, tag, call):
    _, checked = outputs
    assert int(checked[f"{tag}_corrupt_{call}_status"][0]) == INDEX_RANGE


def test_out_of_range_block_table_entry_is_reported(outputs):
    _, checked = outputs
    assert int(checked["chunk_corrupt_status"][0]) == INDEX_RANGE
