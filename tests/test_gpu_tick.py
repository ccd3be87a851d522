"""GPU: the serving tick (``moe_async_tick``: collect of what was ready and the wave's
Receptor in one control kernel, then the scheduling step) against the separate calls and the
oracle.

The tick changes when tokens are handed back (a call returns the tokens that earlier steps
made ready) but not what is computed: the pick trace, every token's emission step and its
output must equal those of enqueue / schedule_step / collect, bit for bit, and the outputs
meet the oracle's bound.  A pair delivered for a slot that the same call collects is judged
against the request it completed: a duplicate, dropped.
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as om
from workloads import get_config, make_workload
from tests.gpu_helpers import TOL, rel_err, expert_getter, oracle_policy, gpu_layer, trace_steps, by_token
from tests.test_gpu_fullsize import _device_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as g
    g.build()
    import asynchronous_expert_execution_gb300 as p
    return p


def _same(a, b, T, H):
    assert a["status"] == 0 and b["status"] == 0
    assert sorted(a["slots"].tolist()) == sorted(b["slots"].tolist()) == list(range(T))
    assert trace_steps(a["trace"]) == trace_steps(b["trace"])
    ea, eb = np.zeros(T, dtype=np.int64), np.zeros(T, dtype=np.int64)
    ea[a["slots"]], eb[b["slots"]] = a["emit"], b["emit"]
    assert np.array_equal(ea, eb)
    ya, yb = by_token(a["slots"], a["y"], T, H), by_token(b["slots"], b["y"], T, H)
    assert np.array_equal(ya.view(np.uint64), yb.view(np.uint64))
    for k in ("pairs_executed", "expert_runs", "steps", "tokens_combined", "open_tokens", "duplicates"):
        assert a["stats"][k] == b["stats"][k], k


# single steps after the last arrival (drain="steps"): MTFS, the CUDA-core fp32 path,
# ragged tails, simulated ranks with stealing, the shared expert
@pytest.mark.parametrize("name", ["c1", "m1", "m2", "m4", "r1"])
def test_tick_equals_separate_calls(pkg, name):
    spec = get_config(name)
    wl = make_workload(spec, seed=0)
    a = gpu_layer(pkg, spec, wl)
    b = gpu_layer(pkg, spec, wl, fused=True)
    _same(a, b, spec.tokens, spec.layer.hidden)


@pytest.mark.parametrize("name", ["c2", "c4"])
def test_tick_fullsize_as_benchmarked(pkg, name):
    """The launch sequence the benchmark times (ticks, then moe_async_wait and one collect):
    equal to the separate calls bit for bit, and a seeded sample of 32 tokens against the
    oracle's replay."""
    spec = get_config(name)
    L = spec.layer
    wl, ws = _device_workload(spec, seed=0)
    a = gpu_layer(pkg, spec, wl, weights_dev=ws, trace_capacity=1 << 20, drain="wait")
    b = gpu_layer(pkg, spec, wl, weights_dev=ws, trace_capacity=1 << 20, drain="wait", fused=True)
    _same(a, b, spec.tokens, L.hidden)
    T = spec.tokens
    ii, ww = om.route(wl.logits.numpy(), L.top_k)
    rng = np.random.default_rng(321)
    sample = sorted(rng.choice(T, size=32, replace=False).tolist())

    def experts(e):
        src = (ws["sw1"], ws["sw3"], ws["sw2"]) if e == L.num_experts else (ws["w1"][e], ws["w3"][e], ws["w2"][e])
        return tuple(m.to("cpu", torch.float64).numpy() for m in src)
    sim = om.replay_layer(L.num_experts, L.top_k, wl.x.double().numpy(), ii, ww, wl.waves, oracle_policy(spec),
                          experts, has_shared=L.has_shared, compute=set(sample))
    pos = {int(s): i for i, s in enumerate(b["slots"])}
    got = np.stack([b["y"][pos[t]] for t in sample])
    ref = np.stack([sim.y[t] for t in sample])
    assert rel_err(got, ref) <= TOL["bf16"]


def test_tick_duplicate_of_a_token_it_collects(pkg):
    """Token 5's pairs are delivered again by the tick that collects token 5: they are
    duplicates of the completed request, dropped; token 5 is collected once, correct."""
    from workloads import LayerSpec, WorkloadSpec
    E, K, H, I, T = 8, 2, 64, 64, 16
    spec = WorkloadSpec(name="small", layer=LayerSpec(E, K, H, I, "bf16"), tokens=T, router="normal",
                        waves="even", num_waves=1, arrival="index", policy="mtfs")
    wl = make_workload(spec, seed=9)
    ws = [{k: v.cuda().contiguous() for k, v in wl.weights[0].items()}]
    moe = pkg.MoEAsync(E, K, H, I, torch.bfloat16, T, weights=ws)
    x = wl.x.cuda()
    idx, w = pkg.route(wl.logits.cuda(), K)
    y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    slots = torch.empty(T, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    pol = pkg.Policy("mtfs")
    moe.tick(0, pol, x=x, expert=idx, w=w, y_out=y, slot_out=slots, n_out=n, append=True)   # all run
    assert int(n.item()) == 0
    again = torch.tensor([5], dtype=torch.int32, device="cuda")
    moe.tick(0, pol, x=x, expert=idx, w=w, rows=again, y_out=y, slot_out=slots, n_out=n, append=True)
    assert int(n.item()) == T                                      # every token, collected once
    assert moe.sync() == 3                                         # MOE_ERR_DUPLICATE (sticky)
    s = moe.stats()
    assert s["duplicates"] == K and s["pairs_executed"] == T * K and s["open_tokens"] == 0
    ii, ww = om.route(wl.logits.numpy(), K)
    ref = om.dense_moe(wl.x.double().numpy(), ii, ww, expert_getter(wl.weights[0], E))
    got = by_token(slots.cpu().numpy(), y.float().cpu().numpy().astype(np.float64), T, H)
    assert rel_err(got, ref) <= TOL["bf16"]
    moe.close()


def test_tick_without_outputs_or_wave(pkg):
    """No wave and nothing to collect: the call is one scheduling step (here of a queue filled
    by an enqueue); max_out = 0 needs no output buffers."""
    spec = get_config("m1")
    L = spec.layer
    wl = make_workload(spec, seed=0)
    ws = [{k: v.cuda().contiguous() for k, v in wl.weights[0].items()}]
    moe = pkg.MoEAsync(L.num_experts, L.top_k, L.hidden, L.inter, wl.x.dtype, spec.tokens, weights=ws,
                       has_shared=L.has_shared)
    idx, w = pkg.route(wl.logits.cuda(), L.top_k)
    moe.enqueue(0, wl.x.cuda(), idx, w)
    pol = pkg.Policy("mtfs")
    for _ in range(L.num_experts + 1):
        moe.tick(0, pol)
    assert moe.sync() == 0
    s = moe.stats()
    assert s["open_tokens"] == 0 and s["ready"] == spec.tokens
    T = spec.tokens
    y = torch.empty((T, L.hidden), dtype=wl.x.dtype, device="cuda")
    slots = torch.empty(T, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.collect(0, y, slots, n)
    assert int(n.item()) == T
    ii, ww = om.route(wl.logits.numpy(), L.top_k)
    ex = expert_getter(wl.weights[0], L.num_experts)
    ref = om.dense_moe(wl.x.double().numpy(), ii, ww, ex, shared=ex(L.num_experts) if L.has_shared else None)
    got = by_token(slots.cpu().numpy(), y.float().cpu().numpy().astype(np.float64), T, L.hidden)
    assert rel_err(got, ref) <= TOL[L.dtype]
    moe.close()
