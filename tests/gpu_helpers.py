"""Shared helpers for the GPU tests: run a workload through the library and through
the oracle on the same seeded inputs."""
import numpy as np
import torch

from oracle import moe_oracle as om
from workloads import make_workload

TOL = {"f32": 1e-5, "bf16": 2e-2}


def rel_err(got, ref):
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))


def expert_getter(weights, E, host=True):
    """(W1, W3, W2) float64 for expert e (e == E: the shared expert)."""
    cache = {}

    def get(e):
        if e not in cache:
            if e == E:
                t = (weights["sw1"], weights["sw3"], weights["sw2"])
            else:
                t = (weights["w1"][e], weights["w3"][e], weights["w2"][e])
            cache[e] = tuple(m.detach().to("cpu", torch.float64).numpy() for m in t)
        return cache[e]
    return get


def oracle_policy(spec):
    if spec.policy == "mtfs":
        return lambda d: om.mtfs_pick(d, spec.max_groups)
    if spec.policy == "ranks":
        return lambda d: om.rank_pick(d, spec.max_groups, spec.fallback_groups != 0)
    return lambda d: om.threshold_pick(d, spec.min_batch, spec.max_groups, spec.fallback_groups)


def gpu_layer(pkg, spec, wl, waves=None, dev="cuda", expert_kind="swiglu", x=None, idx=None, w=None,
              trace_capacity=65536, max_drain=20000, weights_dev=None, drain="steps", fused=False):
    """Run one layer of `wl` through the library; returns a dict of host results.

    drain = "steps": after the last arrival, single steps each followed by a collect (the
    emission step of every token is also derived on the host from the per-step counts and
    must equal the device's); "wait": ``moe_async_wait`` then one collect, as the benchmark
    drains (one device plan of the remaining steps under MTFS / THRESHOLD).  fused: one
    ``moe_async_tick`` a tick instead of enqueue, schedule_step and collect."""
    L = spec.layer
    waves = wl.waves if waves is None else waves
    dt = wl.x.dtype
    ws = None
    if expert_kind == "swiglu":
        ws = [weights_dev if weights_dev is not None else {k: v.to(dev).contiguous() for k, v in wl.weights[0].items()}]
    moe = pkg.MoEAsync(L.num_experts, L.top_k, L.hidden, L.inter, dt, spec.tokens, weights=ws,
                       has_shared=L.has_shared, expert_kind=expert_kind, trace_capacity=trace_capacity)
    xd = (wl.x if x is None else x).to(dev).contiguous()
    if idx is None:
        idx, w = pkg.route(wl.logits.to(dev).contiguous(), L.top_k)
    else:
        idx, w = idx.to(dev).contiguous(), w.to(dev).contiguous()
    rep = pkg.LayerReplay(moe, waves, spec.tokens, device=dev, idx_host=idx.cpu().numpy())
    pol = pkg.Policy.from_spec(spec)
    rep.run_ticks(xd, idx, w, pol, fused=fused)
    if drain == "wait":
        drained = 0 if rep.finish(pol, max_steps=max_drain) == 0 else -1
        slots, y, _ = rep.results()
        emit = rep.device_steps()
    else:
        drained = rep.drain(pol, max_steps=max_drain)
        slots, y, emit = rep.results()
        assert np.array_equal(rep.device_steps(), emit), "device emission steps differ from the per-step counts"
    status = moe.sync()
    stats = moe.stats()
    trace = moe.trace()
    moe.close()
    return dict(slots=slots, y=y, emit=emit, idx=idx.cpu().numpy(), w=w.cpu().numpy(), status=status,
                stats=stats, trace=trace, drained=drained)


def trace_steps(trace):
    """Group a (step, layer, expert, count) trace into {step: [(expert, count), ...]}."""
    out = {}
    for s, _, e, c in trace.tolist():
        out.setdefault(s, []).append((e, c))
    return out


def oracle_steps(sim):
    return {r.step: [(e, c) for e, c, _ in r.picks] for r in sim.steps if r.picks}


def by_token(slots, y, T, H):
    got = np.full((T, H), np.nan)
    got[slots] = y
    return got
