"""bench.py's host-side parts on the CPU: workload and policy options, the bounded oracle
sample behind `cpu_baseline`, and the reference arm's JSON line (no GPU needed)."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from workloads import get_config  # noqa: E402


def _args(*extra):
    old = sys.argv
    sys.argv = ["bench.py", *extra]
    try:
        return bench.parse()
    finally:
        sys.argv = old


def test_workload_spec_policy_options():
    s = bench.workload_spec(_args())
    assert (s.policy, s.max_groups) == ("mtfs", 0) and bench.policy_name(s) == "mtfs"
    s = bench.workload_spec(_args("--ranks", "16"))
    assert (s.policy, s.max_groups, s.fallback_groups) == ("ranks", 16, 1)
    assert bench.policy_name(s) == "ranks (R = 16, with stealing)"
    s = bench.workload_spec(_args("--ranks", "8", "--no-steal"))
    assert (s.policy, s.max_groups, s.fallback_groups) == ("ranks", 8, 0)
    assert bench.policy_name(s) == "ranks (R = 8, no stealing)"
    s = bench.workload_spec(_args("--max-groups", "4"))
    assert (s.policy, s.max_groups) == ("mtfs", 4) and bench.policy_name(s) == "mtfs (G = 4)"
    s = bench.workload_spec(_args("--workload", "c4"))
    assert s.policy == "threshold" and s.min_batch == 64


@pytest.fixture(scope="module")
def c1_inputs():
    spec = get_config("c1")
    x, logits, ws, waves = bench.build_inputs(spec, 0, "cpu")
    return spec, x, logits, ws, waves


def test_host_weights_cover_first_wave(c1_inputs):
    from oracle import moe_oracle as om
    spec, x, logits, ws, waves = c1_inputs
    idx, _ = om.route(logits.numpy(), spec.layer.top_k)
    first = sorted(waves, key=lambda w: w.tick)[0]
    need = set(idx[np.asarray(first.tokens)].ravel().tolist())
    wh = bench.host_weights_for_sample(ws, waves, logits, spec.layer.top_k)
    assert set(wh["w1"]) == need
    # a byte cap below one expert still keeps the first wave's experts, and nothing more
    wh = bench.host_weights_for_sample(ws, waves, logits, spec.layer.top_k, max_waves=len(waves), max_bytes=1)
    assert set(wh["w1"]) == need
    wh = bench.host_weights_for_sample(ws, waves, logits, spec.layer.top_k, max_waves=len(waves))
    assert set(wh["w1"]) == set(idx.ravel().tolist())


@pytest.mark.parametrize("ranks", [0, 3])
def test_oracle_sample_bounded(c1_inputs, ranks):
    spec, x, logits, ws, waves = c1_inputs
    if ranks:
        spec = bench.workload_spec(_args("--workload", "c1", "--ranks", str(ranks)))
    wh = bench.host_weights_for_sample(ws, waves, logits, spec.layer.top_k, max_waves=len(waves))
    nonempty = [w for w in sorted(waves, key=lambda w: w.tick) if len(w.tokens)]
    p, t, desc = bench.oracle_sample(spec, x, logits, wh, waves)             # no budget: one wave
    assert p == len(nonempty[0].tokens) * spec.layer.top_k and t > 0
    assert desc.startswith("first 1 arriving wave(s)")
    p, t, desc = bench.oracle_sample(spec, x, logits, wh, waves, budget_s=1e9)   # every wave
    assert p == spec.tokens * spec.layer.top_k
    assert desc.startswith(f"first {len(nonempty)} arriving wave(s)")


def test_reference_arm_json_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "c1", "--steps", "2",
                          "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads([ln for ln in out.stdout.splitlines() if ln.startswith("{")][-1])
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 3
    assert line["unit"] == "pairs/s" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "pairs/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"] == "c1_tiny_fp32"
