"""Pins for the CPU oracle: facts that do not come from the oracle itself.

Each ``pin_*`` function checks the oracle against a closed form, a value the
pages print, a brute-force enumeration or an invariant.  The mutation tests at
the bottom plant plausible mistakes in the oracle (on the CPU) and check that
some pin catches each one.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import moe_oracle as om
from workloads import Wave

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng([seed, 7])


def _rand_experts(rng, E, H, I, shared=False):
    ws = [(rng.standard_normal((H, I)) / math.sqrt(H), rng.standard_normal((H, I)) / math.sqrt(H),
           rng.standard_normal((I, H)) / math.sqrt(I)) for _ in range(E + (1 if shared else 0))]
    return ws


# ------------------------------------------------------------------ routing

def pin_route_bruteforce():
    rng = _rng(1)
    for (T, E, K) in [(25, 7, 3), (10, 8, 2), (6, 5, 5), (9, 6, 1)]:
        z = rng.standard_normal((T, E)).astype(np.float32)
        i1, w1 = om.route(z, K)
        i2, w2 = om.route_bruteforce(z, K)
        assert np.array_equal(i1, i2)
        assert np.allclose(w1, w2, rtol=0, atol=1e-14)


def pin_route_hand():
    # equal logits go to the lower expert index; the weights are a softmax over
    # the kept logits: logits (0, ln 3) -> (3/4, 1/4) with expert 1 first.
    idx, w = om.route(np.array([[1.0, 3.0, 2.0, 3.0]]), 2)
    assert idx.tolist() == [[1, 3]]
    assert np.allclose(w, [[0.5, 0.5]], atol=1e-15)
    idx, w = om.route(np.array([[0.0, math.log(3.0), -5.0]]), 2)
    assert idx.tolist() == [[1, 0]]
    assert np.allclose(w, [[0.75, 0.25]], atol=1e-15)
    # K = E: the weights are the plain softmax
    z = np.array([[0.3, -1.2, 2.0, 0.0]])
    idx, w = om.route(z, 4)
    p = np.exp(z[0]) / np.exp(z[0]).sum()
    assert np.allclose(w[0], p[idx[0]], atol=1e-15)
    # K = 1: weight one
    _, w = om.route(np.random.default_rng(3).standard_normal((5, 9)), 1)
    assert np.all(w == 1.0)


def test_route_bruteforce():
    pin_route_bruteforce()


def test_route_hand():
    pin_route_hand()


def test_route_weights_sum_to_one():
    z = _rng(2).standard_normal((64, 128))
    _, w = om.route(z, 4)
    assert np.allclose(w.sum(axis=1), 1.0, atol=4e-16)
    assert np.all(w > 0)


# --------------------------------------------------------------- SwiGLU FFN

def pin_silu():
    assert om.silu(0.0) == 0.0
    assert abs(om.silu(1.0) - 0.7310585786300049) < 1e-15          # sigmoid(1)
    assert abs(om.silu(-1.0) + 0.2689414213699951) < 1e-15          # -sigmoid(-1)
    assert abs(om.silu(40.0) - 40.0) < 1e-12
    assert abs(om.silu(-40.0)) < 1e-15
    a = np.linspace(-6, 6, 101)
    assert np.allclose(om.silu(a) - om.silu(-a), a, atol=1e-14)      # silu(a) - silu(-a) = a


def pin_ffn_closed_form():
    rng = _rng(4)
    # identity projections: E(x) = silu(x) * x, elementwise
    H = 6
    x = rng.standard_normal((3, H))
    eye = np.eye(H)
    assert np.allclose(om.expert_ffn(x, eye, eye, eye), om.silu(x) * x, atol=1e-14)
    # rank-one projections with H != I pin operand order and transposition:
    # W1 = a b^T, W3 = c d^T, W2 = f g^T  =>
    # E(x) = [ (silu((x.a) b) * ((x.c) d)) . f ] g
    H, I = 5, 3
    a, c = rng.standard_normal(H), rng.standard_normal(H)
    b, d, f = rng.standard_normal(I), rng.standard_normal(I), rng.standard_normal(I)
    g = rng.standard_normal(H)
    W1, W3, W2 = np.outer(a, b), np.outer(c, d), np.outer(f, g)
    x = rng.standard_normal((4, H))
    for r in range(4):
        s1, s3 = x[r] @ a, x[r] @ c
        hvec = np.array([s1 * b[i] / (1 + math.exp(-s1 * b[i])) * s3 * d[i] for i in range(I)])
        want = (hvec @ f) * g
        assert np.allclose(om.expert_ffn(x[r:r + 1], W1, W3, W2)[0], want, atol=1e-12)


def test_silu():
    pin_silu()


def test_ffn_closed_form():
    pin_ffn_closed_form()


# ------------------------------------------------------- async layer vs dense

def _tiny_case(seed, E=8, K=2, H=16, I=12, T=32, shared=False):
    rng = _rng(seed)
    x = rng.standard_normal((T, H))
    z = rng.standard_normal((T, E)).astype(np.float32)
    idx, w = om.route(z, K)
    ws = _rand_experts(rng, E, H, I, shared)
    return x, idx, w, ws


def _waves_random(T, n, seed):
    rng = np.random.default_rng([seed, 11])
    perm = rng.permutation(T)
    ticks = rng.permutation(n) + 1
    return [Wave(tick=int(ticks[i]), tokens=np.sort(g)) for i, g in enumerate(np.array_split(perm, n))]


def pin_async_equals_dense(seed=0, shared=False, policy="mtfs"):
    E, K, T = 8, 2, 32
    x, idx, w, ws = _tiny_case(seed, E=E, K=K, T=T, shared=shared)
    waves = _waves_random(T, 4, seed)
    pol = (lambda d: om.mtfs_pick(d)) if policy == "mtfs" else (lambda d: om.threshold_pick(d, 5, 0, 1))
    sim = om.replay_layer(E, K, x, idx, w, waves, pol, lambda e: ws[e], has_shared=shared)
    dense = om.dense_moe(x, idx, w, lambda e: ws[e], shared=ws[E] if shared else None)
    assert sorted(sim.y) == list(range(T))
    got = np.stack([sim.y[t] for t in range(T)])
    assert np.allclose(got, dense, rtol=0, atol=1e-13)


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("shared", [False, True])
@pytest.mark.parametrize("policy", ["mtfs", "threshold"])
def test_async_equals_dense(seed, shared, policy):
    pin_async_equals_dense(seed, shared, policy)


def pin_identity_experts_exact():
    # integer x and power-of-two weights summing to one: y == x exactly
    T, E, K, H = 24, 6, 3, 10
    rng = _rng(5)
    x = rng.integers(-50, 50, size=(T, H)).astype(np.float64)
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)])
    w = np.tile(np.array([0.5, 0.25, 0.25]), (T, 1))
    sim = om.replay_layer(E, K, x, idx, w, _waves_random(T, 3, 5), om.mtfs_pick, None)
    for t in range(T):
        assert np.array_equal(sim.y[t], x[t])
    # general weights: y = (sum_j w_j) x
    w2 = rng.integers(1, 8, size=(T, K)) / 8.0
    sim = om.replay_layer(E, K, x, idx, w2, _waves_random(T, 3, 6), om.mtfs_pick, None)
    for t in range(T):
        assert np.array_equal(sim.y[t], w2[t].sum() * x[t])


def test_identity_experts_exact():
    pin_identity_experts_exact()


# ------------------------------------------------------ readiness/conservation

def test_conservation_and_readiness():
    E, K, T = 8, 2, 32
    x, idx, w, ws = _tiny_case(3, E=E, K=K, T=T, shared=True)
    waves = _waves_random(T, 4, 3)
    sim = om.AsyncMoEOracle(E, K, x, lambda e: ws[e], has_shared=True)
    for wv in sorted(waves, key=lambda v: v.tick):
        sim.deliver(wv.tokens, idx, w)
    assert sum(sim.depths()) == T * K + T                     # every pair + one shared each
    snap = sim.snapshot()
    for e in range(E):
        want = sorted((t, k) for t in range(T) for k in range(K) if idx[t, k] == e)
        assert snap[e] == want
    assert snap[E] == [(t, K) for t in range(T)]
    while sim.pending():
        sim.step(om.mtfs_pick)
    assert all(s.combined == 1 for s in sim.slots)


def test_withheld_pair_never_emitted():
    E, K, T = 8, 2, 16
    x, idx, w, ws = _tiny_case(4, E=E, K=K, T=T)
    sim = om.AsyncMoEOracle(E, K, x, lambda e: ws[e])
    sim.deliver(np.arange(1, T), idx, w)
    sim.deliver([0], idx, w, rank=(int(idx[0, 0]), E))           # only k = 0 of token 0
    for _ in range(5):
        sim.step(om.mtfs_pick)
    assert 0 not in sim.y and sim.slots[0].combined == 0
    assert all(sim.slots[t].combined == 1 for t in range(1, T))


def test_duplicate_delivery_rejected():
    E, K, T = 8, 2, 8
    x, idx, w, ws = _tiny_case(5, E=E, K=K, T=T)
    sim = om.AsyncMoEOracle(E, K, x, lambda e: ws[e])
    sim.deliver(np.arange(T), idx, w)
    sim.deliver([2, 3], idx, w)
    assert sim.duplicates == 2 * K
    while sim.pending():
        sim.step(om.mtfs_pick)
    dense = om.dense_moe(x, idx, w, lambda e: ws[e])
    for t in range(T):
        assert np.allclose(sim.y[t], dense[t], atol=1e-13)


def test_arrival_order_and_partition_invariance():
    E, K, T = 8, 2, 32
    x, idx, w, ws = _tiny_case(6, E=E, K=K, T=T)
    ref = None
    for seed in range(4):
        waves = _waves_random(T, 2 + seed, 100 + seed)
        sim = om.replay_layer(E, K, x, idx, w, waves, om.mtfs_pick, lambda e: ws[e])
        got = np.stack([sim.y[t] for t in range(T)])
        if ref is None:
            ref = got
        assert np.allclose(got, ref, rtol=0, atol=1e-13)


# ------------------------------------------------------------------ policies

def pin_policies_hand():
    d = [3, 0, 5, 5, 1]
    assert om.mtfs_pick(d) == [2, 3, 0, 4]
    assert om.mtfs_pick(d, 2) == [2, 3]
    assert om.mtfs_pick([0, 0]) == []
    assert om.threshold_pick(d, 4) == [2, 3]
    assert om.threshold_pick(d, 4, 1) == [2]
    assert om.threshold_pick(d, 6) == [2]                    # fallback: deepest, G = 1
    assert om.threshold_pick(d, 6, 0, 2) == [2, 3]
    assert om.threshold_pick([0, 0, 0], 1) == []


def pin_rank_pick_hand():
    # worked by hand: expert e belongs to rank e mod R; a rank runs its deepest bucket (tie ->
    # lower id); an idle rank steals the deepest bucket nobody picked; picks in rank order
    d = [5, 0, 3, 0, 2, 7, 0, 1]
    assert om.rank_pick(d, 2) == [0, 5]
    assert om.rank_pick(d, 4) == [0, 5, 2, 7]
    d = [5, 0, 0, 0, 2, 0, 4, 0]
    assert om.rank_pick(d, 4) == [0, 4, 6]                   # rank 1 steals bucket 4
    assert om.rank_pick(d, 4, steal=False) == [0, 6]
    assert om.rank_pick([2, 2, 2, 2], 2) == [0, 1]
    assert om.rank_pick([2, 2, 2, 2], 3) == [0, 1, 2]
    assert om.rank_pick([0, 3, 0, 3, 0, 0], 3) == [3, 1]     # nothing left to steal
    assert om.rank_pick([6, 0, 5, 0], 2) == [0, 2]
    assert om.rank_pick([6, 0, 5, 0], 2, steal=False) == [0]
    assert om.rank_pick([5, 0, 0, 0, 4, 0, 1, 0], 2) == [0, 4]   # the deeper of two candidates
    assert om.rank_pick([5, 0, 0, 0, 4, 0, 1, 0], 4) == [0, 4, 6]
    assert om.rank_pick([0, 0, 0], 2) == []


def test_rank_pick_hand():
    pin_rank_pick_hand()


def test_rank_pick_invariants():
    rng = np.random.default_rng(7)
    for _ in range(300):
        nb = int(rng.integers(1, 12))
        R = int(rng.integers(1, 14))
        d = [int(v) if rng.random() < 0.6 else 0 for v in rng.integers(1, 5, nb)]
        nonempty = [e for e in range(nb) if d[e] > 0]
        owners = {r for r in range(R) if any(d[e] > 0 for e in range(r, nb, R))}
        for steal in (True, False):
            p = om.rank_pick(d, R, steal)
            assert len(set(p)) == len(p) and all(d[e] > 0 for e in p)
            assert len(p) == (min(R, len(nonempty)) if steal else len(owners))
        if R == 1:                                       # one rank: plain MTFS, one bucket
            assert om.rank_pick(d, 1) == om.mtfs_pick(d, 1)
        if R >= nb:                                      # a rank per bucket: every non-empty one
            assert om.rank_pick(d, R) == nonempty


def pin_schedule_trace_hand():
    # t0 -> e0, t1 -> e1, t2 -> e1, t3 -> e2 (K = 1); waves at ticks 1, 1, 3
    idx = np.array([[0], [1], [1], [2]])
    w = np.ones((4, 1))
    x = np.eye(4)
    waves = [Wave(1, np.array([0, 1])), Wave(1, np.array([2])), Wave(3, np.array([3]))]
    sim = om.replay_layer(3, 1, x, idx, w, waves, om.mtfs_pick, None)
    got = [([(e, c) for e, c, _ in s.picks], s.emitted) for s in sim.steps]
    assert got == [([(1, 2), (0, 1)], [0, 1, 2]), ([], []), ([(2, 1)], [3])]
    assert sim.steps[0].picks[0][2] == ((1, 0), (2, 0))
    sim = om.replay_layer(3, 1, x, idx, w, waves, lambda d: om.threshold_pick(d, 2), None)
    got = [([(e, c) for e, c, _ in s.picks], s.emitted) for s in sim.steps]
    assert got == [([(1, 2)], [1, 2]), ([(0, 1)], [0]), ([(2, 1)], [3])]


def test_policies_hand():
    pin_policies_hand()


def test_schedule_trace_hand():
    pin_schedule_trace_hand()


def pin_defrag_golden():
    with open(os.path.join(GOLDEN, "defrag_worked_example.json")) as f:
        g = json.load(f)
    scores = []
    for case in g["cases"]:
        s = om.defrag_score(case["Q"], [(q, 0) for q in case["lookahead_q_plus_h"]], g["delta"])
        assert s == case["expected"]
        scores.append(s)
    assert scores[0] > scores[1]


def test_defrag_golden():
    pin_defrag_golden()


def test_transfer_bytes_golden():
    from workloads import get_config
    with open(os.path.join(GOLDEN, "transfer_bytes_example.json")) as f:
        g = json.load(f)
    layer = get_config("c2").layer
    assert layer.hidden == g["hidden"]
    assert g["tokens"] * layer.hidden * g["bytes_per_element"] == g["expected_bytes"]


def test_rmsnorm_stub_closed_form():
    x = np.array([[3.0, 4.0]])                  # mean square 12.5
    r = om.rmsnorm(x, eps=0.0)
    assert np.allclose(r, x / math.sqrt(12.5), atol=1e-15)
    P = np.array([[1.0, 2.0], [0.0, 1.0]])
    assert np.allclose(om.attention_stub(x, P), (x / math.sqrt(12.5 + 1e-6)) @ P, atol=1e-15)


# ------------------------------------------------- y for sampled tokens

def pin_y_sample_dense():
    """y_sample (the merge formula per token, no queues) against the brute-force dense MoE
    on every token of a tiny case, with and without the shared expert."""
    for shared in (False, True):
        x, idx, w, ws = _tiny_case(5, E=6, K=3, H=10, I=7, T=12, shared=shared)
        ex = lambda e: ws[e]
        sh = ws[6] if shared else None
        dense = om.dense_moe(x, idx, w, ex, shared=sh)
        got = om.y_sample(range(12), x, idx, w, ex, shared=sh)
        for t in range(12):
            assert np.allclose(got[t], dense[t], rtol=0, atol=1e-13), (shared, t)


def pin_y_sample_hand():
    """H = I = 1 worked by hand: expert e is E_e(x) = silu(a_e x) (c_e x) f_e, so a token
    x = 2 routed to (2, 0) with weights (3/4, 1/4) gives
    y = 3/4 silu(0.5) (-4) + 1/4 silu(2) 6 / 2, and the shared expert (a = c = f = 1)
    adds silu(2) 2 with weight one."""
    a, c, f = (1.0, -0.5, 0.25), (3.0, 1.0, -2.0), (0.5, 2.0, 1.0)
    ws = [(np.array([[a[e]]]), np.array([[c[e]]]), np.array([[f[e]]])) for e in range(3)]
    sh = (np.array([[1.0]]), np.array([[1.0]]), np.array([[1.0]]))
    x = np.array([[2.0], [-1.0]])
    idx = np.array([[2, 0], [1, 2]])
    w = np.array([[0.75, 0.25], [0.4, 0.6]])
    sig = lambda v: 1.0 / (1.0 + math.exp(-v))
    s = lambda v: v * sig(v)
    y0 = 0.75 * s(0.5) * (-4.0) * 1.0 + 0.25 * s(2.0) * 6.0 * 0.5
    y1 = 0.4 * s(0.5) * (-1.0) * 2.0 + 0.6 * s(-0.25) * 2.0 * 1.0
    got = om.y_sample([0, 1], x, idx, w, lambda e: ws[e])
    assert abs(got[0][0] - y0) < 1e-15 and abs(got[1][0] - y1) < 1e-15
    got = om.y_sample([1, 0], x, idx, w, lambda e: ws[e], shared=sh)
    assert abs(got[0][0] - (y0 + s(2.0) * 2.0)) < 1e-15
    assert abs(got[1][0] - (y1 + s(-1.0) * (-1.0))) < 1e-15


def test_y_sample_dense():
    pin_y_sample_dense()


def test_y_sample_hand():
    pin_y_sample_hand()


# ------------------------------------------------- planted-mistake detection

def _fails(pin, *args):
    try:
        pin(*args)
    except AssertionError:
        return True
    return False


def test_pins_catch_planted_mistakes(monkeypatch):
    real_silu = om.silu
    # 1. silu without the sigmoid denominator's exponent sign
    monkeypatch.setattr(om, "silu", lambda a: np.asarray(a, float) / (1.0 + np.exp(np.asarray(a, float))))
    assert _fails(pin_silu)
    monkeypatch.setattr(om, "silu", real_silu)
    # 2. W1 and W3 swapped inside the expert
    real_ffn = om.expert_ffn
    monkeypatch.setattr(om, "expert_ffn", lambda X, W1, W3, W2: real_ffn(X, W3, W1, W2))
    assert _fails(pin_ffn_closed_form)
    monkeypatch.setattr(om, "expert_ffn", real_ffn)
    # 3. combine drops its last term
    real_combine = om.combine
    monkeypatch.setattr(om, "combine", lambda c: real_combine(c[:-1]) if len(c) > 1 else real_combine(c))
    assert _fails(pin_identity_experts_exact)
    assert _fails(pin_async_equals_dense, 0, True, "mtfs")
    monkeypatch.setattr(om, "combine", real_combine)
    # 4. weights not renormalised over the top K
    real_route = om.route

    def route_no_renorm(z, K):
        idx, w = real_route(z, K)
        zz = np.asarray(z, float)
        p = np.exp(zz - zz.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        return idx, np.take_along_axis(p, idx, 1)
    monkeypatch.setattr(om, "route", route_no_renorm)
    assert _fails(pin_route_bruteforce)
    monkeypatch.setattr(om, "route", real_route)
    # 5. MTFS breaking depth ties toward the higher expert id
    real_mtfs = om.mtfs_pick
    monkeypatch.setattr(om, "mtfs_pick", lambda d, g=0: [-ne for _, ne in sorted((-x, -e) for e, x in enumerate(d) if x > 0)][:g or None])
    assert _fails(pin_policies_hand)
    monkeypatch.setattr(om, "mtfs_pick", real_mtfs)
    # 6. defrag score without the decay exponent
    monkeypatch.setattr(om, "defrag_score", lambda q, la, dl: q + sum(dl * (a + b) for a, b in la))
    assert _fails(pin_defrag_golden)
    monkeypatch.undo()
    # 7. stealing the shallowest bucket instead of the deepest
    real_rank = om.rank_pick

    def rank_shallow(d, R, steal=True):
        own = real_rank(d, R, steal=False)
        if not steal:
            return own
        picks = {r: e for r in range(R) for e in own if e % R == r}
        left = [e for e in reversed(om.mtfs_pick(d)) if e not in own]
        for r in range(R):
            if r not in picks and left:
                picks[r] = left.pop(0)
        return [picks[r] for r in range(R) if r in picks]
    monkeypatch.setattr(om, "rank_pick", rank_shallow)
    assert _fails(pin_rank_pick_hand)
    monkeypatch.undo()
    # 8. y_sample weighting the shared expert by the first routed weight
    real_ffn = om.expert_ffn

    def y_sample_shared_weighted(tokens, x, idx, w, experts, shared=None):
        out = {}
        for t in tokens:
            t = int(t)
            xt = np.asarray(x[t], float)[None, :]
            cs = [w[t, k] * real_ffn(xt, *experts(int(idx[t, k])))[0] for k in range(idx.shape[1])]
            if shared is not None:
                cs.append(w[t, 0] * real_ffn(xt, *shared)[0])
            out[t] = om.combine(cs)
        return out
    monkeypatch.setattr(om, "y_sample", y_sample_shared_weighted)
    assert _fails(pin_y_sample_dense) and _fails(pin_y_sample_hand)
    monkeypatch.undo()
    # 9. y_sample pairing weight k with the expert of the reversed k order
    def y_sample_reversed_w(tokens, x, idx, w, experts, shared=None):
        out = {}
        K = idx.shape[1]
        for t in tokens:
            t = int(t)
            xt = np.asarray(x[t], float)[None, :]
            cs = [w[t, K - 1 - k] * real_ffn(xt, *experts(int(idx[t, k])))[0] for k in range(K)]
            if shared is not None:
                cs.append(real_ffn(xt, *shared)[0])
            out[t] = om.combine(cs)
        return out
    monkeypatch.setattr(om, "y_sample", y_sample_reversed_w)
    assert _fails(pin_y_sample_dense) and _fails(pin_y_sample_hand)


def test_pins_pass_unmodified():
    pin_rank_pick_hand()
    for p in (pin_route_bruteforce, pin_route_hand, pin_silu, pin_ffn_closed_form,
              pin_identity_experts_exact, pin_policies_hand, pin_schedule_trace_hand, pin_defrag_golden,
              pin_y_sample_dense, pin_y_sample_hand):
        p()


def test_c1_workload_async_equals_dense():
    """The tiny exactness workload end to end on the oracle: waves + MTFS vs dense."""
    from workloads import get_config, make_workload
    wl = make_workload(get_config("c1"), seed=0)
    L = wl.spec.layer
    x = wl.x.double().numpy()
    idx, w = om.route(wl.logits.numpy(), L.top_k)
    ws = wl.weights[0]
    ex = lambda e: (ws["w1"][e].double().numpy(), ws["w3"][e].double().numpy(), ws["w2"][e].double().numpy())
    sim = om.replay_layer(L.num_experts, L.top_k, x, idx, w, wl.waves, om.mtfs_pick, ex)
    dense = om.dense_moe(x, idx, w, ex)
    got = np.stack([sim.y[t] for t in range(wl.spec.tokens)])
    assert np.allclose(got, dense, rtol=0, atol=1e-13)
    assert len(sim.steps) == max(v.tick for v in wl.waves)
