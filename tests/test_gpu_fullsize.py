"""Full-size workloads (GPT-OSS decode c2, Zipf prefill c3, DeepSeek-wide + shared c4) in the
launch configuration the benchmark times.  Indexing is compared in full -- routing ids, the
pick trace of every step, each token's emission step, exactly-once collection -- and the
float output on a seeded sample of 64 tokens (for the DeepSeek-wide layer: the shared expert,
four K chunks of GEMM1 and wide token tiles together)."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as om
from workloads import get_config, make_tokens, make_logits, make_waves
from workloads.build import expert_weight_slice, make_layer_weights
from tests.gpu_helpers import TOL, gpu_layer, trace_steps, oracle_steps, oracle_policy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as g
    g.build()
    import asynchronous_expert_execution_gb300 as p
    return p


class _Wl:
    pass


def _device_workload(spec, seed):
    """Inputs generated on the device (as the benchmark does); the oracle copies slices."""
    L = spec.layer
    wl = _Wl()
    wl.spec = spec
    wl.x = make_tokens(spec, seed)
    wl.logits = make_logits(spec, seed)
    wl.waves = make_waves(spec, seed)
    ws = {}
    for kind, shape in (("w1", (L.hidden, L.inter)), ("w3", (L.hidden, L.inter)), ("w2", (L.inter, L.hidden))):
        t = torch.empty((L.num_experts,) + shape, dtype=torch.bfloat16, device="cuda")
        for e in range(L.num_experts):
            t[e] = expert_weight_slice(L, seed, 0, kind, e, device="cuda")
        ws[kind] = t
    if L.has_shared:
        sh = make_layer_weights(L, seed, 0, device="cuda", experts=[])
        ws.update({k: sh[k] for k in ("sw1", "sw3", "sw2")})
    return wl, ws


@pytest.mark.parametrize("name", ["c2", "c3", "c4"])
def test_fullsize_sampled_parity(pkg, name):
    spec = get_config(name)
    L = spec.layer
    wl, ws = _device_workload(spec, seed=0)
    res = gpu_layer(pkg, spec, wl, weights_dev=ws, trace_capacity=1 << 20, drain="wait")   # as bench.py
    assert res["status"] == 0 and res["drained"] >= 0
    T = spec.tokens
    ii, ww = om.route(wl.logits.numpy(), L.top_k)
    assert np.array_equal(res["idx"], ii)
    assert sorted(res["slots"].tolist()) == list(range(T))           # each token exactly once
    # replay of the whole workload on the oracle: picks, counts and emission steps of every
    # token, and the float output of a seeded sample of 64 tokens (the oracle runs each picked
    # bucket's sampled rows through the expert, one expert's weights on the host at a time)
    rng = np.random.default_rng(123)
    sample = sorted(rng.choice(T, size=64, replace=False).tolist())

    def experts(e):
        src = (ws["sw1"], ws["sw3"], ws["sw2"]) if e == L.num_experts else (ws["w1"][e], ws["w3"][e], ws["w2"][e])
        return tuple(m.to("cpu", torch.float64).numpy() for m in src)
    sim = om.replay_layer(L.num_experts, L.top_k, wl.x.double().numpy(), ii, ww, wl.waves, oracle_policy(spec),
                          experts, has_shared=L.has_shared, compute=set(sample))
    assert trace_steps(res["trace"]) == oracle_steps(sim)
    em = np.zeros(T, dtype=np.int64)
    em[res["slots"]] = res["emit"]
    assert all(em[t] == sim.emit_step[t] for t in range(T))
    pos = {int(s): i for i, s in enumerate(res["slots"])}
    got = np.stack([res["y"][pos[t]] for t in sample])
    ref = np.stack([sim.y[t] for t in sample])
    err = float(np.abs(got - ref).max() / np.abs(ref).max())
    assert err <= TOL[L.dtype], err
    del ws
    torch.cuda.empty_cache()
