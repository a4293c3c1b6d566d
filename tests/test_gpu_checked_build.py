"""The bounds-checked build of the library (compiled with CLCG_BOUNDS_CHECK) against the
oracle: every work tile's problem index, row and column block, log entry and k-loop
length, and every worker index written to the first-tile log, is checked before use; a
failed check sets a bit of the device error word (gemm_sync then raises GEMM_ERR_BOUNDS)
and the tile is skipped, so a wrong tile map shows up as an error and as a tile that is
missing from the log.  Nothing traps.

The checked library is built here and a representative part of the parity suite (every
cluster shape and schedule, ragged edges, grouped problems of different shapes, random
shapes, injected cancel failures) runs against it in a child process: each of those tests
ends in gemm_sync, so passing means no check failed.  The full parity suite is run against
the checked build the same way (CLCGEMM_CHECKED=1) when the tile map changes."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUBSET = ("integer_inputs_bit_exact or uniform_ragged_tail or grouped_small or grouped_varied_shapes_small "
          "or randomized_shapes or injected_failure or static_owner_map or deep_products or fetch_ahead")


def test_parity_subset_passes_on_the_checked_build():
    import __graft_entry__
    lib = __graft_entry__._load_build_module().build(checked=True)
    assert os.path.basename(lib) == "libclcgemm_checked.so"
    env = dict(os.environ, CLCGEMM_CHECKED="1")
    probe = subprocess.run([sys.executable, "-c", "import blackwell_clc_dynamic_gb300 as m; print(m.LIB_PATH)"],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert probe.returncode == 0 and probe.stdout.strip().endswith("libclcgemm_checked.so"), probe.stderr
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_gpu_parity.py", "-m", "gpu", "-q", "-x",
                        "-p", "no:cacheprovider", "-k", SUBSET],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    tail = "\n".join(r.stdout.splitlines()[-15:])
    assert r.returncode == 0, tail
    assert " passed" in tail and "failed" not in tail
