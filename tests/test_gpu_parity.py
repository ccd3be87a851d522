"""GPU parity: the CUDA path through the C ABI against the CPU oracle, element by element.

Indexing (routing ids, queue contents, pick traces, emission steps, slot maps) must match
bit-exactly; float outputs within max|gpu - oracle| / max|oracle| <= 1e-5 (fp32) and
<= 2e-2 (bf16 storage, fp32 accumulation).
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as om
from workloads import get_config, make_workload, make_logits, shuffled_waves, repartitioned_waves, Wave
from tests.gpu_helpers import (TOL, rel_err, expert_getter, oracle_policy, gpu_layer, trace_steps,
                               oracle_steps, by_token)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as g
    g.build()
    import asynchronous_expert_execution_gb300 as p
    return p


# ---------------------------------------------------------------- routing

@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4", "m2"])
def test_route_parity(pkg, name):
    spec = get_config(name)
    z = make_logits(spec, seed=1)
    idx, w = pkg.route(z.cuda(), spec.layer.top_k)
    ri, rw = om.route(z.numpy(), spec.layer.top_k)
    assert np.array_equal(idx.cpu().numpy(), ri)                 # bit-exact ids and k order
    assert np.abs(w.cpu().numpy() - rw).max() <= 2e-6


def test_route_ties_and_edges(pkg):
    z = torch.tensor([[1.0, 3.0, 2.0, 3.0], [0.0, 0.0, 0.0, 0.0], [-1.0, 5.0, 5.0, 5.0]])
    idx, w = pkg.route(z.cuda(), 2)
    assert idx.cpu().tolist() == [[1, 3], [0, 1], [1, 2]]
    assert np.allclose(w.cpu().numpy(), 0.5)
    z = torch.randn(37, 1000)                                      # E not a multiple of 32
    idx, w = pkg.route(z.cuda(), 32)
    ri, rw = om.route(z.numpy(), 32)
    assert np.array_equal(idx.cpu().numpy(), ri)
    assert np.abs(w.cpu().numpy() - rw).max() <= 2e-6


# ------------------------------------------------------ identity: exact merge

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shared", [False, True])
def test_identity_experts_bitexact(pkg, dtype, shared):
    """E(x) = x, integer-valued x, power-of-two weights: y = (sum_j w_j) x exactly."""
    from workloads import LayerSpec, WorkloadSpec
    T, E, K, H = 300, 24, 4, 136
    spec = WorkloadSpec(name="ident", layer=LayerSpec(E, K, H, 64, dtype, has_shared=shared, shared_inter=64),
                        tokens=T, router="normal", waves="even", num_waves=6, arrival="exp", policy="mtfs")
    wl = make_workload(spec, seed=3, weights=False)
    rng = np.random.default_rng(5)
    # |y| <= (K/2 + 1) * 8 on a 1/4 grid: exact in bf16 as well as fp32
    xi = rng.integers(-8, 8, size=(T, H)).astype(np.float32)
    x = torch.tensor(xi).to(wl.x.dtype)
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    wv = (rng.integers(1, 3, size=(T, K)) / 4.0).astype(np.float32)
    res = gpu_layer(pkg, spec, wl, expert_kind="identity", x=x, idx=torch.tensor(idx), w=torch.tensor(wv))
    assert res["status"] == 0 and res["drained"] >= 0
    assert sorted(res["slots"].tolist()) == list(range(T))         # each token exactly once
    sim = om.replay_layer(E, K, xi, idx, wv, wl.waves, om.mtfs_pick, None, has_shared=shared)
    want = np.stack([sim.y[t] for t in range(T)])
    got = by_token(res["slots"], res["y"], T, H)
    assert np.array_equal(got, want)
    assert np.array_equal(got, (wv.sum(1, dtype=np.float64) + (1.0 if shared else 0.0))[:, None] * xi)
    assert trace_steps(res["trace"]) == oracle_steps(sim)
    em = np.zeros(T, dtype=np.int64)
    em[res["slots"]] = res["emit"]
    assert all(em[t] == sim.emit_step[t] for t in range(T))


# ------------------------------------------------------------- SwiGLU layers

@pytest.mark.parametrize("name", ["c1", "m1", "m2", "m3", "m4", "r1", "r2", "r3", "r4"])
def test_layer_parity(pkg, name):
    _check_layer(pkg, get_config(name))


# degenerate shapes the method admits: one expert, top-1, every expert picked (K = E), one
# token, top-1 with the shared expert; and the largest the library accepts: 1024 routed
# experts plus the shared one (1025 buckets), top-30
@pytest.mark.parametrize("E,K,H,I,T,dtype,shared", [
    (1024, 8, 64, 64, 256, "bf16", True),
    (32, 30, 64, 64, 20, "bf16", False),
    (1, 1, 64, 64, 40, "bf16", False),
    (32, 1, 256, 128, 100, "bf16", False),
    (6, 6, 128, 64, 50, "f32", False),
    (6, 6, 136, 80, 50, "bf16", False),
    (8, 2, 64, 64, 1, "bf16", False),
    (4, 1, 200, 96, 30, "bf16", True),
])
def test_layer_parity_degenerate(pkg, E, K, H, I, T, dtype, shared):
    from workloads import LayerSpec, WorkloadSpec
    spec = WorkloadSpec(name="degenerate", layer=LayerSpec(E, K, H, I, dtype, has_shared=shared, shared_inter=I),
                        tokens=T, router="normal", waves="even", num_waves=min(3, T), arrival="exp",
                        policy="mtfs")
    _check_layer(pkg, spec)


def _check_layer(pkg, spec):
    L = spec.layer
    wl = make_workload(spec, seed=0)
    res = gpu_layer(pkg, spec, wl)
    assert res["status"] == 0, res["status"]
    assert res["drained"] >= 0
    T = spec.tokens
    ii, ww = om.route(wl.logits.numpy(), L.top_k)
    assert np.array_equal(res["idx"], ii)
    ex = expert_getter(wl.weights[0], L.num_experts)
    sim = om.replay_layer(L.num_experts, L.top_k, wl.x.double().numpy(), ii, ww,
                          wl.waves, oracle_policy(spec), ex, has_shared=L.has_shared)
    assert sorted(res["slots"].tolist()) == list(range(T))
    want = np.stack([sim.y[t] for t in range(T)])
    got = by_token(res["slots"], res["y"], T, L.hidden)
    err = rel_err(got, want)
    assert err <= TOL[L.dtype], err
    assert trace_steps(res["trace"]) == oracle_steps(sim)
    em = np.zeros(T, dtype=np.int64)
    em[res["slots"]] = res["emit"]
    assert all(em[t] == sim.emit_step[t] for t in range(T))
    st = res["stats"]
    assert st["pairs_executed"] == T * (L.top_k + (1 if L.has_shared else 0))
    assert st["tokens_combined"] == T and st["open_tokens"] == 0 and st["pending_pairs"] == 0
    assert st["duplicates"] == 0 and st["error"] == 0


def test_route_weights_into_oracle_tolerance(pkg):
    """The oracle's own float64 weights (not the GPU's fp32 ones) also meet the bound."""
    spec = get_config("m1")
    L = spec.layer
    wl = make_workload(spec, seed=2)
    res = gpu_layer(pkg, spec, wl)
    ii, ww = om.route(wl.logits.numpy(), L.top_k)
    ref = om.dense_moe(wl.x.double().numpy(), ii, ww, expert_getter(wl.weights[0], L.num_experts))
    assert rel_err(by_token(res["slots"], res["y"], spec.tokens, L.hidden), ref) <= TOL[L.dtype]


def test_queue_snapshot_parity(pkg):
    """Queue contents after delivering every wave (no step yet): per-expert multisets and
    depths equal the oracle's, bit for bit."""
    spec = get_config("m2")
    L = spec.layer
    wl = make_workload(spec, seed=0)
    ws = [{k: v.cuda().contiguous() for k, v in wl.weights[0].items()}]
    moe = pkg.MoEAsync(L.num_experts, L.top_k, L.hidden, L.inter, wl.x.dtype, spec.tokens, weights=ws,
                       has_shared=True)
    idx, w = pkg.route(wl.logits.cuda(), L.top_k)
    x = wl.x.cuda()
    for wv in wl.waves:
        rows = torch.tensor(wv.tokens, dtype=torch.int32, device="cuda")
        moe.enqueue(0, x, idx, w, rows=rows)
    depths, recs = moe.snapshot(0)
    sim = om.AsyncMoEOracle(L.num_experts, L.top_k, wl.x.double().numpy(), None, has_shared=True)
    ii, ww = om.route(wl.logits.numpy(), L.top_k)
    for wv in wl.waves:
        sim.deliver(wv.tokens, ii, ww)
    assert depths.tolist() == sim.depths()
    assert recs == [list(b) for b in sim.snapshot()]
    moe.close()


@pytest.mark.parametrize("name", ["m1", "m2"])
def test_arrival_order_and_partition_bitwise_invariance(pkg, name):
    """Shuffled arrival ticks and different wave partitions give bitwise-identical y."""
    spec = get_config(name)
    wl = make_workload(spec, seed=1)
    outs = []
    variants = [wl.waves, shuffled_waves(wl.waves, 1), shuffled_waves(wl.waves, 2),
                repartitioned_waves(spec.tokens, 3, 7), repartitioned_waves(spec.tokens, 9, 8)]
    for wv in variants:
        res = gpu_layer(pkg, spec, wl, waves=wv)
        assert res["status"] == 0 and res["drained"] >= 0
        outs.append(by_token(res["slots"], res["y"], spec.tokens, spec.layer.hidden))
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


# ------------------------------------------------------ protocol / failures

def _small(pkg, dtype="bf16", shared=False, cap=0, T=64, E=8, K=2, H=64, I=64):
    from workloads import LayerSpec, WorkloadSpec
    spec = WorkloadSpec(name="small", layer=LayerSpec(E, K, H, I, dtype, has_shared=shared, shared_inter=I),
                        tokens=T, router="normal", waves="even", num_waves=2, arrival="index", policy="mtfs")
    wl = make_workload(spec, seed=4)
    ws = [{k: v.cuda().contiguous() for k, v in wl.weights[0].items()}]
    moe = pkg.MoEAsync(E, K, H, I, wl.x.dtype, T, weights=ws, has_shared=shared, bucket_capacity=cap)
    idx, w = pkg.route(wl.logits.cuda(), K)
    return spec, wl, moe, wl.x.cuda(), idx, w


def test_withheld_pair_times_out(pkg):
    spec, wl, moe, x, idx, w = _small(pkg)
    T = spec.tokens
    kmask = torch.full((T,), 3, dtype=torch.int32, device="cuda")
    kmask[5] = 1                                                   # token 5 withholds k = 1
    moe.enqueue(0, x, idx, w, kmask=kmask)
    st = moe.wait(0, pkg.Policy(), max_steps=6, check_every=2)
    assert st == 5                                                  # MOE_ERR_TIMEOUT
    y = torch.empty((T, spec.layer.hidden), dtype=x.dtype, device="cuda")
    slots = torch.empty(T, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.collect(0, y, slots, n)
    got = sorted(slots[: int(n.item())].cpu().tolist())
    assert got == [t for t in range(T) if t != 5]                  # never emitted early
    s = moe.stats()
    assert s["open_tokens"] == 1 and s["error"] == 0
    # the missing pair arrives late: the token completes
    one = torch.tensor([5], dtype=torch.int32, device="cuda")
    moe.enqueue(0, x, idx, w, rows=one, kmask=torch.tensor([2], dtype=torch.int32, device="cuda"))
    assert moe.wait(0, pkg.Policy(), max_steps=4) == 0
    moe.collect(0, y, slots, n)
    assert int(n.item()) == 1 and int(slots[0].item()) == 5
    moe.close()


def test_duplicate_pair_rejected_once(pkg):
    spec, wl, moe, x, idx, w = _small(pkg, shared=True)
    T, H = spec.tokens, spec.layer.hidden
    moe.enqueue(0, x, idx, w)
    rows = torch.tensor([3, 7], dtype=torch.int32, device="cuda")
    moe.enqueue(0, x, idx, w, rows=rows)                            # duplicates of tokens 3 and 7
    for _ in range(2):
        moe.schedule_step(0, pkg.Policy())
    assert moe.sync() == 3                                          # MOE_ERR_DUPLICATE (sticky)
    s = moe.stats()
    assert s["duplicates"] == 2 * spec.layer.top_k
    assert s["pairs_executed"] == T * (spec.layer.top_k + 1)       # nothing accumulated twice
    y = torch.empty((T, H), dtype=x.dtype, device="cuda")
    slots = torch.empty(T, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.collect(0, y, slots, n)
    assert int(n.item()) == T
    L = spec.layer
    ii, ww = om.route(wl.logits.numpy(), L.top_k)
    ref = om.dense_moe(wl.x.double().numpy(), ii, ww, expert_getter(wl.weights[0], L.num_experts),
                       shared=expert_getter(wl.weights[0], L.num_experts)(L.num_experts))
    got = by_token(slots.cpu().numpy(), y.float().cpu().numpy().astype(np.float64), T, H)
    assert rel_err(got, ref) <= TOL["bf16"]
    moe.close()


def test_stale_generation_and_slot_reuse(pkg):
    spec, wl, moe, x, idx, w = _small(pkg, dtype="f32")
    T, H = spec.tokens, spec.layer.hidden
    y = torch.empty((T, H), dtype=x.dtype, device="cuda")
    slots = torch.empty(T, dtype=torch.int32, device="cuda")
    gens = torch.empty(T, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    g0 = torch.zeros(T, dtype=torch.int32, device="cuda")
    moe.enqueue(0, x, idx, w, gen=g0)
    assert moe.wait(0, pkg.Policy(), max_steps=4) == 0
    moe.collect(0, y, slots, n, gen_out=gens)
    assert int(n.item()) == T and gens.cpu().tolist() == [0] * T
    first = by_token(slots.cpu().numpy(), y.cpu().numpy().astype(np.float64), T, H)
    # second request generation on the same slots (gen 1): same values again
    g1 = torch.ones(T, dtype=torch.int32, device="cuda")
    moe.enqueue(0, x, idx, w, gen=g1)
    assert moe.wait(0, pkg.Policy(), max_steps=4) == 0
    moe.collect(0, y, slots, n, gen_out=gens)
    assert gens.cpu().tolist() == [1] * T
    assert np.array_equal(by_token(slots.cpu().numpy(), y.cpu().numpy().astype(np.float64), T, H), first)
    # a late pair from generation 0 is stale now
    rows = torch.tensor([2], dtype=torch.int32, device="cuda")
    moe.enqueue(0, x, idx, w, rows=rows, gen=torch.zeros(1, dtype=torch.int32, device="cuda"))
    assert moe.sync() == 4                                          # MOE_ERR_STALE
    assert moe.stats()["stale"] == 1 and moe.stats()["open_tokens"] == 0
    moe.close()


def test_bucket_capacity_overflow_reported(pkg):
    spec, wl, moe, x, idx, w = _small(pkg, cap=2, T=64, E=4, K=2)
    moe.enqueue(0, x, idx, w)
    assert moe.sync() == 2                                          # MOE_ERR_CAPACITY
    moe.close()


def test_empty_inputs(pkg):
    spec, wl, moe, x, idx, w = _small(pkg)
    moe.enqueue(0, x, idx, w, n=0)                                  # empty wave: no-op
    moe.schedule_step(0, pkg.Policy())                              # nothing to pick
    y = torch.empty((4, spec.layer.hidden), dtype=x.dtype, device="cuda")
    slots = torch.empty(4, dtype=torch.int32, device="cuda")
    n = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    moe.collect(0, y, slots, n)
    assert int(n.item()) == 0
    s = moe.stats()
    assert s["steps"] == 1 and s["pairs_executed"] == 0 and s["error"] == 0
    e0 = torch.empty(0, 4, device="cuda")
    i0, w0 = pkg.route(e0, 2)
    assert i0.shape == (0, 2)
    moe.close()


# ------------------------------------------------------------- cancellation

def _ident(pkg, T=64, E=8, K=2, H=64):
    moe = pkg.MoEAsync(E, K, H, 64, torch.float32, T, expert_kind="identity")
    rng = np.random.default_rng(21)
    x = torch.tensor(rng.integers(-8, 8, size=(T, H)).astype(np.float32)).cuda()
    idx = torch.tensor(np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)).cuda()
    w = torch.tensor((rng.integers(1, 3, size=(T, K)) / 4.0).astype(np.float32)).cuda()
    return moe, x, idx, w


def _collect_all(moe, T, H):
    y = torch.empty((T, H), dtype=torch.float32, device="cuda")
    slots = torch.empty(T, dtype=torch.int32, device="cuda")
    gens = torch.empty(T, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.collect(0, y, slots, n, gen_out=gens)
    k = int(n.item())
    return slots[:k].cpu().numpy(), y[:k].cpu().numpy(), gens[:k].cpu().numpy()


def test_cancel_withheld_request_then_reuse(pkg):
    """A request whose second pair never comes is cancelled: the others complete, its slot is
    freed once its queued pair has run, and a new request then uses the slot cleanly."""
    T, H = 64, 64
    moe, x, idx, w = _ident(pkg, T=T, H=H)
    kmask = torch.full((T,), 3, dtype=torch.int32, device="cuda")
    kmask[5] = 1                                                   # pair k = 1 of token 5 withheld
    moe.enqueue(0, x, idx, w, kmask=kmask)
    moe.cancel(0, torch.tensor([5], dtype=torch.int32, device="cuda"))
    assert moe.wait(0, pkg.Policy(), max_steps=8) == 0             # nothing open after the cancel
    slots, y, gens = _collect_all(moe, T, H)
    assert sorted(slots.tolist()) == [t for t in range(T) if t != 5]
    st = moe.stats()
    assert st["cancelled"] == 1 and st["open_tokens"] == 0 and st["error"] == 0
    # the slot was reclaimed after its queued pair ran: generation 1 takes it
    x2 = (x[5:6] * 2 + 1).contiguous()
    moe.enqueue(0, x2, idx[5:6].contiguous(), w[5:6].contiguous(), slots=torch.tensor([5], dtype=torch.int32, device="cuda"),
                gen=torch.ones(1, dtype=torch.int32, device="cuda"))
    assert moe.wait(0, pkg.Policy(), max_steps=8) == 0
    slots, y, gens = _collect_all(moe, T, H)
    assert slots.tolist() == [5] and gens.tolist() == [1]
    want = w[5].sum().item() * x2[0].cpu().numpy()
    assert np.array_equal(y[0], want)                              # no trace of the old request
    # the old request's late pair is stale now
    moe.enqueue(0, x, idx, w, rows=torch.tensor([5], dtype=torch.int32, device="cuda"),
                kmask=torch.tensor([2], dtype=torch.int32, device="cuda"),
                gen=torch.zeros(1, dtype=torch.int32, device="cuda"))
    assert moe.sync() == 4
    moe.close()


def test_cancel_queued_requests_are_not_published(pkg):
    T, H = 64, 64
    moe, x, idx, w = _ident(pkg, T=T, H=H)
    moe.enqueue(0, x, idx, w)
    moe.cancel(0, torch.tensor([3, 7, 7], dtype=torch.int32, device="cuda"))   # duplicate id: once
    assert moe.wait(0, pkg.Policy(), max_steps=8) == 0
    slots, y, _ = _collect_all(moe, T, H)
    assert sorted(slots.tolist()) == [t for t in range(T) if t not in (3, 7)]
    xs, ws = x.cpu().numpy().astype(np.float64), w.cpu().numpy().astype(np.float64)
    for s, row in zip(slots, y):
        assert np.array_equal(row, ws[s].sum() * xs[s])
    st = moe.stats()
    assert st["cancelled"] == 2 and st["error"] == 0
    # both slots are free again (generation 1)
    moe.enqueue(0, x, idx, w, rows=torch.tensor([3, 7], dtype=torch.int32, device="cuda"),
                gen=torch.ones(2, dtype=torch.int32, device="cuda"))
    assert moe.wait(0, pkg.Policy(), max_steps=8) == 0
    slots, y, gens = _collect_all(moe, T, H)
    assert sorted(slots.tolist()) == [3, 7] and gens.tolist() == [1, 1]
    moe.close()


def test_cancel_after_merge_is_too_late(pkg):
    T, H = 64, 64
    moe, x, idx, w = _ident(pkg, T=T, H=H)
    moe.enqueue(0, x, idx, w)
    assert moe.wait(0, pkg.Policy(), max_steps=8) == 0
    moe.cancel(0, torch.tensor([2], dtype=torch.int32, device="cuda"))
    slots, _, _ = _collect_all(moe, T, H)
    assert sorted(slots.tolist()) == list(range(T))
    assert moe.stats()["cancelled"] == 0
    moe.close()


# ------------------------------------ several steps in one plan (the drain)
# StreamEP section 4 / CascadeEP streamFFN: with nothing arriving, consecutive steps pick one
# deepest-first order of the buckets; one device plan of those steps must reproduce them.

@pytest.mark.parametrize("name,over", [
    ("m2", {}),                                                          # threshold + shared
    ("m1", {"max_groups": 3}),                                           # MTFS, 3 buckets a step
    ("c1", {"max_groups": 1}),                                           # fp32 (SIMT path)
    ("m4", {"policy": "threshold", "min_batch": 6, "max_groups": 2, "fallback_groups": 2}),
])
def test_drain_plan_matches_single_steps(pkg, name, over):
    spec = get_config(name, **over)
    L = spec.layer
    wl = make_workload(spec, seed=2)
    one = gpu_layer(pkg, spec, wl, drain="steps")
    many = gpu_layer(pkg, spec, wl, drain="wait")
    assert one["status"] == 0 and many["status"] == 0 and many["drained"] == 0
    T = spec.tokens
    ii, ww = om.route(wl.logits.numpy(), L.top_k)
    sim = om.replay_layer(L.num_experts, L.top_k, wl.x.double().numpy(), ii, ww, wl.waves, oracle_policy(spec),
                          expert_getter(wl.weights[0], L.num_experts), has_shared=L.has_shared)
    for res in (one, many):
        assert trace_steps(res["trace"]) == oracle_steps(sim)          # every step's picks
        em = np.zeros(T, dtype=np.int64)
        em[res["slots"]] = res["emit"]
        assert all(em[t] == sim.emit_step[t] for t in range(T))        # each token's emission step
        assert res["stats"]["steps"] >= max(sim.emit_step.values())
    got1 = by_token(one["slots"], one["y"], T, L.hidden)
    got2 = by_token(many["slots"], many["y"], T, L.hidden)
    assert np.array_equal(got1, got2)                                  # bitwise: same arithmetic
    ref = np.stack([sim.y[t] for t in range(T)])
    assert rel_err(got2, ref) <= TOL[L.dtype]
    # the plan ran the remaining steps in one scheduling launch pair: fewer launches
    assert many["stats"]["kernel_launches"] < one["stats"]["kernel_launches"]


# ------------------------------------------- rejected pairs leave the pool alone
# "asynchronous MoE serving" notes, inferred obligations: accept exactly the selected
# contributions, and return a slot only after its last read; CascadeEP: generation-tagged
# readiness.  A delivery whose pairs are all rejected must not touch the token pool row of
# the slot's current request: the row is what GEMM1 gathers for that request.

def _oracle_y(spec, wl, x_rows, idx, w):
    L = spec.layer
    ii, ww = idx.cpu().numpy().astype(np.int64), w.cpu().numpy().astype(np.float64)
    return om.dense_moe(x_rows, ii, ww, expert_getter(wl.weights[0], L.num_experts))


def test_stale_wave_does_not_overwrite_pool(pkg):
    """Generation 1 of slot 5 is enqueued with a new vector; before any step, a late
    generation-0 wave for slot 5 arrives carrying the old vector.  Its pairs are stale and
    dropped, and the step must still compute generation 1 from the new vector."""
    spec, wl, moe, x, idx, w = _small(pkg, dtype="f32")
    T, H = spec.tokens, spec.layer.hidden
    g0 = torch.zeros(T, dtype=torch.int32, device="cuda")
    moe.enqueue(0, x, idx, w, gen=g0)
    assert moe.wait(0, pkg.Policy(), max_steps=4) == 0
    y = torch.empty((T, H), dtype=x.dtype, device="cuda")
    slots = torch.empty(T, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.collect(0, y, slots, n)                                      # every slot -> generation 1
    assert int(n.item()) == T
    five = torch.tensor([5], dtype=torch.int32, device="cuda")
    x_new = (x[5:6] * -1.5 + 0.25).contiguous()
    moe.enqueue(0, x_new, idx[5:6].contiguous(), w[5:6].contiguous(), slots=five,
                gen=torch.ones(1, dtype=torch.int32, device="cuda"))
    moe.enqueue(0, x, idx, w, rows=five, gen=torch.zeros(1, dtype=torch.int32, device="cuda"))   # stale
    moe.schedule_step(0, pkg.Policy())
    n.zero_()
    moe.collect(0, y, slots, n)
    assert moe.sync() == 4                                          # MOE_ERR_STALE latched
    assert int(n.item()) == 1 and int(slots[0].item()) == 5
    want = _oracle_y(spec, wl, x_new.cpu().double().numpy(), idx[5:6], w[5:6])
    got = y[:1].cpu().double().numpy()
    assert rel_err(got, want) <= TOL["f32"], rel_err(got, want)
    assert moe.stats()["stale"] == 1
    moe.close()


def test_retired_slot_late_pair_is_dropped(pkg):
    """A cancelled request's late pair, carrying another vector, arrives while its slot is
    retired with a record still queued.  The pair is dropped silently; the queued record runs
    and is discarded, the slot is freed, and the next request of that slot is computed from
    its own vector alone (element by element against the oracle).  The retired slot's pool row
    is read only by records whose results are discarded, so this sequence checks the
    bookkeeping around the drop; the pool payload itself is checked by the stale and duplicate
    cases and, over every interleaving, by the protocol model."""
    spec, wl, moe, x, idx, w = _small(pkg, dtype="f32")
    T, H = spec.tokens, spec.layer.hidden
    kmask = torch.full((T,), 3, dtype=torch.int32, device="cuda")
    kmask[5] = 1                                                   # pair k = 1 of token 5 withheld
    moe.enqueue(0, x, idx, w, kmask=kmask)
    five = torch.tensor([5], dtype=torch.int32, device="cuda")
    moe.cancel(0, five)
    x_bad = (x * 3.0 - 1.0).contiguous()
    moe.enqueue(0, x_bad, idx, w, rows=five, kmask=torch.tensor([2], dtype=torch.int32, device="cuda"))
    moe.schedule_step(0, pkg.Policy())
    y = torch.empty((T, H), dtype=x.dtype, device="cuda")
    slots = torch.empty(T, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.collect(0, y, slots, n)
    assert moe.sync() == 0                                          # a retired drop is not an error
    k = int(n.item())
    assert sorted(slots[:k].cpu().tolist()) == [t for t in range(T) if t != 5]
    want = _oracle_y(spec, wl, x.cpu().double().numpy(), idx, w)
    got = by_token(slots[:k].cpu().numpy(), y[:k].cpu().double().numpy(), T, H)
    keep = [t for t in range(T) if t != 5]
    assert rel_err(got[keep], want[keep]) <= TOL["f32"]
    st = moe.stats()
    assert st["cancelled"] == 1 and st["open_tokens"] == 0 and st["duplicates"] == 0
    # generation 1 of slot 5, its own vector
    x_new = (x[5:6] * 0.5 - 2.0).contiguous()
    moe.enqueue(0, x_new, idx[5:6].contiguous(), w[5:6].contiguous(), slots=five,
                gen=torch.ones(1, dtype=torch.int32, device="cuda"))
    moe.schedule_step(0, pkg.Policy())
    n.zero_()
    moe.collect(0, y, slots, n)
    assert moe.sync() == 0 and int(n.item()) == 1
    want = _oracle_y(spec, wl, x_new.cpu().double().numpy(), idx[5:6], w[5:6])
    assert rel_err(y[:1].cpu().double().numpy(), want) <= TOL["f32"]
    moe.close()


def test_duplicate_wave_does_not_overwrite_pool(pkg):
    """Every token is delivered; before any step a duplicate wave for tokens 3 and 7 arrives
    carrying other vectors.  The duplicates are dropped (and reported), and every output must
    still come from the first delivery's vectors."""
    spec, wl, moe, x, idx, w = _small(pkg, dtype="f32", shared=True)
    T, H = spec.tokens, spec.layer.hidden
    moe.enqueue(0, x, idx, w)
    x_bad = (x * -2.0 + 3.0).contiguous()
    moe.enqueue(0, x_bad, idx, w, rows=torch.tensor([3, 7], dtype=torch.int32, device="cuda"))
    moe.schedule_step(0, pkg.Policy())
    y = torch.empty((T, H), dtype=x.dtype, device="cuda")
    slots = torch.empty(T, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.collect(0, y, slots, n)
    assert moe.sync() == 3                                          # MOE_ERR_DUPLICATE latched
    assert int(n.item()) == T
    L = spec.layer
    ii, ww = idx.cpu().numpy().astype(np.int64), w.cpu().numpy().astype(np.float64)
    get = expert_getter(wl.weights[0], L.num_experts)
    want = om.dense_moe(x.cpu().double().numpy(), ii, ww, get, shared=get(L.num_experts))
    got = by_token(slots.cpu().numpy(), y.cpu().double().numpy(), T, H)
    assert rel_err(got, want) <= TOL["f32"], rel_err(got, want)
    assert moe.stats()["duplicates"] == 2 * L.top_k
    moe.close()


def test_collect_into_pinned_host_memory(pkg):
    """Collect outputs written by the kernels straight into pinned host buffers (when
    moe_async_host_writable says the kernels can address them) equal those written to device
    buffers, token by token; pageable host memory is reported as not writable."""
    spec, wl, moe, x, idx, w = _small(pkg, shared=True)
    T, H = spec.tokens, spec.layer.hidden
    yh = torch.empty((T, H), dtype=x.dtype).pin_memory()
    sh = torch.empty(T, dtype=torch.int32).pin_memory()
    assert not pkg.host_writable(torch.empty((T, H), dtype=x.dtype))      # pageable
    if not (pkg.host_writable(yh) and pkg.host_writable(sh)):
        pytest.skip("pinned host memory is not mapped into the device's address space here")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.enqueue(0, x, idx, w, rows=torch.arange(0, T // 2, dtype=torch.int32, device="cuda"))
    moe.schedule_step(0, pkg.Policy())
    moe.collect(0, yh, sh, n, append=True)
    moe.enqueue(0, x, idx, w, rows=torch.arange(T // 2, T, dtype=torch.int32, device="cuda"))
    moe.schedule_step(0, pkg.Policy())
    moe.collect(0, yh, sh, n, append=True)
    assert moe.sync() == 0 and int(n.item()) == T
    L = spec.layer
    ii, ww = om.route(wl.logits.numpy(), L.top_k)
    ref = om.dense_moe(wl.x.double().numpy(), ii, ww, expert_getter(wl.weights[0], L.num_experts),
                       shared=expert_getter(wl.weights[0], L.num_experts)(L.num_experts))
    got = by_token(sh.numpy(), yh.float().numpy().astype(np.float64), T, H)
    assert rel_err(got, ref) <= TOL["bf16"]
    moe.close()
