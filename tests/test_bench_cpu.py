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
    s = bench.workload_spec(_args())                                  # the headline: DeepSeek-wide
    assert s.name == "c4_deepseek_wide_shared" and s.policy == "threshold" and s.min_batch == 64
    s = bench.workload_spec(_args("--workload", "c2"))
    assert (s.policy, s.max_groups) == ("mtfs", 0) and bench.policy_name(s) == "mtfs"
    s = bench.workload_spec(_args("--workload", "c2", "--ranks", "16"))
    assert (s.policy, s.max_groups, s.fallback_groups) == ("ranks", 16, 1)
    assert bench.policy_name(s) == "ranks (R = 16, with stealing)"
    s = bench.workload_spec(_args("--workload", "c2", "--ranks", "8", "--no-steal"))
    assert (s.policy, s.max_groups, s.fallback_groups) == ("ranks", 8, 0)
    assert bench.policy_name(s) == "ranks (R = 8, no stealing)"
    s = bench.workload_spec(_args("--workload", "c2", "--max-groups", "4"))
    assert (s.policy, s.max_groups) == ("mtfs", 4) and bench.policy_name(s) == "mtfs (G = 4)"
    s = bench.workload_spec(_args(), "c5")                            # streaming: options left alone
    assert s.num_layers == 4
    a = _args()
    assert a.subconfigs == "c2,c3,c5" and a.steps >= 50


@pytest.fixture(scope="module")
def c1_inputs():
    spec = get_config("c1")
    x, logits, ws, waves = bench.build_inputs(spec, 0, "cpu")
    return spec, x, logits, ws, waves


def test_oracle_sample_tokens_bounded_by_host_bytes(c1_inputs):
    from oracle import moe_oracle as om
    spec, x, logits, ws, waves = c1_inputs
    idx, _ = om.route(logits.numpy(), spec.layer.top_k)
    order = [int(t) for w in sorted(waves, key=lambda w: w.tick) for t in w.tokens]
    tokens, need = bench.oracle_sample_tokens(spec, logits, waves)          # everything fits
    assert tokens == order and need == set(idx.ravel().tolist())
    per_expert = 3 * spec.layer.hidden * spec.layer.inter * 4
    tokens, need = bench.oracle_sample_tokens(spec, logits, waves, max_bytes=3 * per_expert)
    assert tokens == order[:len(tokens)] and len(need) <= 3 and len(tokens) >= 1
    assert need == set(idx[tokens].ravel().tolist())
    tokens, need = bench.oracle_sample_tokens(spec, logits, waves, max_bytes=1)   # at least one token
    assert tokens == order[:1]


@pytest.mark.parametrize("ranks", [0, 3])
def test_oracle_sample_bounded(c1_inputs, ranks):
    spec, x, logits, ws, waves = c1_inputs
    if ranks:
        spec = bench.workload_spec(_args("--workload", "c1", "--ranks", str(ranks)))
    tokens, need = bench.oracle_sample_tokens(spec, logits, waves, max_bytes=4 * 3 * 64 * 128 * 4)
    wh = bench.host_weights(ws, need, spec.layer.has_shared)
    p, t, desc, threads = bench.oracle_sample(spec, x, logits, wh, tokens)       # no budget: once
    assert p == len(tokens) * spec.layer.top_k and t > 0
    assert desc.startswith(f"the first {len(tokens)} arriving tokens") and "1 time(s)" in desc
    assert "BLAS threads" in desc
    p, t, desc, threads = bench.oracle_sample(spec, x, logits, wh, tokens, budget_s=t * 3)   # repeated
    assert p % (len(tokens) * spec.layer.top_k) == 0 and p >= 2 * len(tokens) * spec.layer.top_k


def test_schedule_independent_bytes(c1_inputs):
    from oracle import moe_oracle as om
    spec, x, logits, ws, waves = c1_inputs
    touched, b = bench.schedule_independent_bytes(spec, logits)
    idx, _ = om.route(logits.numpy(), spec.layer.top_k)
    assert touched == len(set(idx.ravel().tolist()))
    assert b == touched * 3 * spec.layer.hidden * spec.layer.inter * 4


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


def test_drain_is_one_asynchronous_plan_except_for_ranks():
    """After the last wave the pass drains MTFS / threshold buckets with one device plan
    (moe_async_schedule_steps, no host read in the timed pass) and RANKS through
    moe_async_wait, whose status must be 0."""
    from asynchronous_expert_execution_gb300.api import Policy

    class Fake:
        def __init__(self, status=0):
            self.calls, self.status = [], status

        def schedule_steps(self, layer, policy, max_steps):
            self.calls.append(("plan", layer, policy.kind, max_steps))

        def wait(self, layer, policy, max_steps=0, check_every=0):
            self.calls.append(("wait", layer, policy.kind))
            return self.status

    for pol in (Policy("threshold", min_batch=64, fallback_groups=1), Policy("mtfs", max_groups=4)):
        m = Fake()
        bench.drain(m, pol)
        assert m.calls == [("plan", 0, pol.kind, bench.DRAIN_STEPS)]
    assert bench.DRAIN_STEPS >= 1025                 # one bucket a step at least: never cut short
    m = Fake()
    bench.drain(m, Policy("ranks", max_groups=16, fallback_groups=1))
    assert m.calls == [("wait", 0, "ranks")]
    with pytest.raises(AssertionError):
        bench.drain(Fake(status=5), Policy("ranks", max_groups=4))
