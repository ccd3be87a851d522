"""The bounds-checked build (MOE_DEBUG_BOUNDS) on the GPU: parity cases of every kernel family
run with every index checked -- no check fires and the outputs still match the oracle -- and
records planted out of range are rejected (tests/bounds_cases.py).  They run in a child
process because the bounds-checked library is chosen when the binding loads (one library per
process)."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bounds_checked_build_parity_and_rejection():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as g
    g.build()
    env = dict(os.environ, MOE_DEBUG_BOUNDS="1")
    cmd = [sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider", "-m", "gpu",
           "tests/bounds_cases.py",
           "tests/test_gpu_parity.py::test_layer_parity",
           "tests/test_gpu_parity.py::test_drain_plan_matches_single_steps",
           "tests/test_gpu_parity.py::test_duplicate_wave_does_not_overwrite_pool",
           "tests/test_gpu_parity.py::test_cancel_withheld_request_then_reuse",
           "tests/test_gpu_split.py", "tests/test_gpu_wide.py",
           "tests/test_gpu_tick.py::test_tick_equals_separate_calls",
           "tests/test_gpu_tick.py::test_tick_duplicate_of_a_token_it_collects",
           "tests/test_gpu_stream.py::test_stream_small_parity"]
    out = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert out.returncode == 0, out.stdout[-4000:] + out.stderr[-2000:]
    import re
    m = re.search(r"(\d+) passed", out.stdout)
    assert m and int(m.group(1)) >= 20 and "skipped" not in out.stdout, out.stdout[-2000:]
