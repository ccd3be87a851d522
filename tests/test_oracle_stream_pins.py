"""Pins for the streaming multi-layer oracle (2L micro-queues, layer-level MTFS,
dispatch delays, stop rule) against hand-derived traces, a scalar closed form and
invariants."""
import math

import numpy as np

from oracle import moe_oracle as om


def _mk(R, L, E, K, H, delays, stop, max_steps, logits=None, experts=None, proj=None, x0=None, values=True,
        admit=None):
    rng = np.random.default_rng(0)
    if logits is None:
        tab = rng.uniform(size=(R, max_steps, E))
        logits = lambda r, n: tab[r, n]
    if x0 is None:
        x0 = rng.standard_normal((R, H))
    if proj is None:
        Ps = [rng.standard_normal((H, H)) / math.sqrt(H) for _ in range(L)]
        proj = lambda l: Ps[l]
    if experts is None:
        Ws = {(l, e): (rng.standard_normal((H, H)) / math.sqrt(H), rng.standard_normal((H, H)) / math.sqrt(H),
                       rng.standard_normal((H, H)) / math.sqrt(H)) for l in range(L) for e in range(E)}
        experts = lambda l, e: Ws[(l, e)]
    return om.StreamOracle(L, K, x0, proj, logits, delays, experts, stop, max_steps, values=values, admit=admit)


def pin_layer_pick():
    assert om.layer_pick([3, 0], [2, 5]) == ("exp", 1)
    assert om.layer_pick([5, 0], [2, 5]) == ("att", 0)      # tie: lower layer first
    assert om.layer_pick([0, 5], [5, 0]) == ("exp", 0)
    assert om.layer_pick([4, 0], [4, 0]) == ("att", 0)      # tie in a layer: attention first
    assert om.layer_pick([4, 0], [1, 0], allow_attention=False) == ("exp", 0)
    assert om.layer_pick([0, 0], [0, 0]) is None


def test_layer_pick():
    pin_layer_pick()


def test_stream_trace_hand_equal_delays():
    delays = np.ones((2, 8), dtype=np.int64)
    s = _mk(R=2, L=2, E=2, K=1, H=3, delays=delays, stop=3, max_steps=8, values=False).run()
    got = [(t.tick, t.kind, t.layer, t.count) for t in s.trace]
    assert got == [(1, "att", 0, 2), (2, "exp", 0, 2), (3, "att", 1, 2), (4, "exp", 1, 2)]
    assert s.n.tolist() == [2, 2] and s.combined == 4
    assert s.done_tick == {(0, 1): 2, (1, 1): 2, (0, 2): 4, (1, 2): 4}


def test_stream_trace_hand_jitter():
    # request 1's first dispatch takes 3 ticks: the queues split and the layers interleave
    delays = np.ones((2, 8), dtype=np.int64)
    delays[1, 0] = 3
    s = _mk(R=2, L=2, E=2, K=1, H=3, delays=delays, stop=4, max_steps=8, values=False).run()
    got = [(t.tick, t.kind, t.layer, t.count) for t in s.trace]
    # t1: att L0 {0,1} -> 0 arrives t2, 1 arrives t4
    # t2: exp L0 {0} -> 0 to att L1            t3: att L1 {0} -> arrives t4
    # t4: both arrive: exp L0 {1} vs exp L1 {0}: tie -> lower layer first
    # t5: exp L1 {0} (depth 1) vs att L1 {1} (depth 1): same layer, attention first
    # t6: exp L1 {0} -> 0 done twice (combined 3); t7: att L0 {0} vs ... see asserts
    assert got[:6] == [(1, "att", 0, 2), (2, "exp", 0, 1), (3, "att", 1, 1), (4, "exp", 0, 1),
                       (5, "att", 1, 1), (6, "exp", 1, 2)]
    assert s.combined >= 4 and all(1 <= n <= 8 for n in s.n)


def pin_stream_scalar_closed_form():
    """H = I = 1, K = 1: x1 = w2 * silu(w1 * a) * (w3 * a) with a = p * x0 / sqrt(x0^2 + eps)."""
    p, w1, w3, w2, x0, eps = 0.7, 1.3, -0.4, 2.1, 0.9, 1e-6
    s = om.StreamOracle(1, 1, np.array([[x0]]), lambda l: np.array([[p]]), lambda r, n: np.array([0.0]),
                        np.ones((1, 4), dtype=np.int64),
                        lambda l, e: (np.array([[w1]]), np.array([[w3]]), np.array([[w2]])), stop=2,
                        max_steps=4).run()
    x = x0
    for _ in range(2):
        a = p * x / math.sqrt(x * x + eps)
        g = w1 * a
        x = w2 * (g / (1.0 + math.exp(-g))) * (w3 * a)
    assert s.n.tolist() == [2]
    assert abs(s.history[0][2][0] - x) < 1e-14


def test_stream_scalar_closed_form():
    pin_stream_scalar_closed_form()


def test_stream_values_independent_of_delays():
    R, L, E, K, H, M = 6, 2, 4, 2, 5, 6
    rng = np.random.default_rng(3)
    outs = []
    for seed in range(3):
        d = np.random.default_rng(seed).integers(1, 5, size=(R, M))
        s = _mk(R, L, E, K, H, d, stop=20, max_steps=M)
        s.run()
        outs.append((s, d))
    ref = outs[0][0]
    for s, _ in outs[1:]:
        for r in range(R):
            m = min(len(s.history[r]), len(ref.history[r]))
            for n in range(m):
                assert np.array_equal(s.history[r][n], ref.history[r][n])


def test_stream_conservation_and_stop():
    R, L, M = 16, 4, 12
    d = np.random.default_rng(5).integers(1, 6, size=(R, M))
    s = _mk(R, L, 8, 2, 4, d, stop=70, max_steps=M, values=False).run()
    assert s.combined == int(s.n.sum())
    assert 70 <= s.combined < 70 + R
    assert len(s.done_tick) == s.combined                  # every (r, n) completed once
    for (r, n), t in s.done_tick.items():
        if n > 1:
            assert s.done_tick[(r, n - 1)] < t            # steps of a request in order
    assert not s.transit and not any(s.pending)
    # once `stop` merges are done at the start of a tick, no attention queue is served
    done = 0
    for t in s.trace:
        if done >= 70:
            assert t.kind != "att"
        if t.kind == "exp":
            done += t.count


def test_stream_pins_catch_planted_mistakes(monkeypatch):
    real = om.layer_pick
    monkeypatch.setattr(om, "layer_pick", lambda a, e, allow_attention=True:
                        real(e, a, allow_attention) and (("att" if real(e, a, allow_attention)[0] == "exp" else "exp"),
                                                         real(e, a, allow_attention)[1]))
    try:
        pin_layer_pick()
        caught = False
    except AssertionError:
        caught = True
    assert caught
    monkeypatch.setattr(om, "layer_pick", real)
    real_rms = om.rmsnorm
    monkeypatch.setattr(om, "rmsnorm", lambda x, eps=1e-6: np.asarray(x, float) / np.sqrt(np.mean(np.asarray(x, float) ** 2, -1, keepdims=True)))
    try:
        pin_stream_scalar_closed_form()
        caught = False
    except AssertionError:
        caught = True
    assert caught


def pin_chain_policies():
    # worked example of the defragmenting score embedded in a 3-layer chain: candidate att_0
    # holds 20 tokens; the next two queues are empty now but drained 100 and 80 recently;
    # an isolated exp_2 holds 60 (no queue after it).  S(att_0) = 20 + .5*100 + .25*80 = 90.
    att, exp = [20, 0, 0], [0, 0, 60]
    drained = [0, 100, 80, 0, 0, 0]
    assert om.chain_pick(att, exp, "defrag", drained=drained, window=2, decay=0.5) == ("att", 0)
    assert om.chain_pick(att, exp, "mtfs") == ("exp", 2)
    assert om.chain_pick(att, exp, "flfs") == ("att", 0)
    assert om.chain_pick([0, 3], [2, 5], "flfs") == ("exp", 0)
    # window 1: S(att_0) = 20 + 0.5 * 100 = 70 > 60 still; decay 0.2: 20 + 20 + 3.2 = 43.2 < 60
    assert om.chain_pick(att, exp, "defrag", drained=drained, window=1, decay=0.5) == ("att", 0)
    assert om.chain_pick(att, exp, "defrag", drained=drained, window=2, decay=0.2) == ("exp", 2)
    # barrier: nothing is served while a dispatch is in flight
    assert om.chain_pick([0, 0], [3, 0], "barrier", in_transit=1) is None
    assert om.chain_pick([0, 2], [3, 0], "barrier", in_transit=0) == ("exp", 0)
    # closed attention queues count as empty
    assert om.chain_pick([9, 0], [1, 0], "defrag", allow_attention=False, drained=[0] * 4) == ("exp", 0)


def test_chain_policies():
    pin_chain_policies()


def pin_defrag_source_variant():
    """StreamEP section 4, the paragraph after the formula: the source averages the queue
    snapshots over the history window and continues the lookahead cyclically along the chain.
    Two layers: chain att_0, exp_0, att_1, exp_1; W = 2, delta = 0.5."""
    # the wrap decides: Q = (8, 1, 2, 6), no history.  Cyclic: S(att_0) = 8 + .5*1 + .25*2 =
    # 9; S(exp_1) = 6 + .5*8 (att_0, wrapped) + .25*1 (exp_0) = 10.25 -> exp_1.  Truncated at
    # the chain end (the paper's version): S(exp_1) = 6 -> att_0.
    att, exp = [8, 2], [1, 6]
    assert om.chain_pick(att, exp, "defrag_src", snap_avg=[0.0] * 4, window=2, decay=0.5) == ("exp", 1)
    assert om.chain_pick(att, exp, "defrag", drained=[0] * 4, window=2, decay=0.5) == ("att", 0)
    # the average decides: Q = (0, 6, 4, 1) and exp_1's snapshots over the window are 20 and 0.
    # Average H = 10: S(exp_0) = 6 + .5*4 + .25*(1 + 10) = 10.75 > S(att_1) = 4 + .5*(1 + 10)
    # = 9.5 -> exp_0.  Summed (H = 20) it would be 13.25 < 14.5 -> att_1.
    att, exp = [0, 4], [6, 1]
    assert om.chain_pick(att, exp, "defrag_src", snap_avg=[0.0, 0.0, 0.0, 10.0], window=2, decay=0.5) == ("exp", 0)
    assert om.chain_pick(att, exp, "defrag_src", snap_avg=[0.0, 0.0, 0.0, 20.0], window=2, decay=0.5) == ("att", 1)


def test_defrag_source_variant():
    pin_defrag_source_variant()


def test_defrag_source_snapshots_are_window_averages():
    """The stream oracle under defrag_src: tick t's decision sees, as H, the average of the
    depth snapshots of the (at most hist_window) ticks before it -- zero before any."""
    R, L, E, K, H, M = 12, 3, 4, 2, 5, 8
    d = np.random.default_rng(5).integers(1, 5, size=(R, M))
    s = _mk(R, L, E, K, H, d, stop=60, max_steps=M, values=False)
    s.policy, s.hist_window = "defrag_src", 3
    seen = []
    real = om.chain_pick

    def spy(*a, **kw):
        seen.append(list(kw["snap_avg"]))
        return real(*a, **kw)
    om.chain_pick = spy
    try:
        s.run()
    finally:
        om.chain_pick = real
    assert len(seen) == len(s.snap_log) == s.tick and seen[0] == [0.0] * (2 * L)
    for t in range(1, s.tick):
        win = s.snap_log[max(0, t - 3):t]
        assert seen[t] == [sum(v[q] for v in win) / len(win) for q in range(2 * L)]
    assert s.combined >= 60 and not s.transit and not any(s.pending)


def test_defrag_source_pins_catch_planted_mistakes(monkeypatch):
    real = om.chain_pick

    def truncated(att, exp, policy, **kw):            # the lookahead stops at the chain end
        if policy != "defrag_src":
            return real(att, exp, policy, **kw)
        Lq = len(att)
        Q = [v for l in range(Lq) for v in (att[l], exp[l])]
        best, best_s = None, None
        for q in [q for q in range(2 * Lq) if Q[q] > 0]:
            look = [(Q[q + j], kw["snap_avg"][q + j]) for j in range(1, kw["window"] + 1) if q + j < 2 * Lq]
            sc = om.defrag_score(Q[q], look, kw["decay"])
            if best is None or sc > best_s:
                best, best_s = q, sc
        return ("att" if best % 2 == 0 else "exp", best // 2)
    monkeypatch.setattr(om, "chain_pick", truncated)
    try:
        pin_defrag_source_variant()
        caught = False
    except AssertionError:
        caught = True
    assert caught


def test_barrier_trace_hand():
    delays = np.ones((2, 8), dtype=np.int64)
    delays[1, 0] = 3
    s = _mk(R=2, L=2, E=2, K=1, H=3, delays=delays, stop=4, max_steps=8, values=False)
    s.policy = "barrier"
    s.run()
    got = [(t.tick, t.kind, t.layer, t.count) for t in s.trace][:6]
    # t1 att L0 {0,1}; t2, t3 idle (request 1 in flight); t4 exp L0 {0,1}; t5 att L1; t6 exp L1
    assert got == [(1, "att", 0, 2), (2, "idle", -1, 0), (3, "idle", -1, 0), (4, "exp", 0, 2),
                   (5, "att", 1, 2), (6, "exp", 1, 2)]


def test_policies_same_values_and_conservation():
    R, L, E, K, H, M = 10, 3, 4, 2, 5, 8
    d = np.random.default_rng(11).integers(1, 5, size=(R, M))
    runs = {}
    for pol in ("mtfs", "flfs", "defrag", "barrier", "defrag_src"):
        s = _mk(R, L, E, K, H, d, stop=40, max_steps=M)
        s.policy = pol
        s.run()
        assert s.combined == int(s.n.sum()) and 40 <= s.combined < 40 + R
        assert not s.transit and not any(s.pending)
        runs[pol] = s
    ref = runs["mtfs"]
    for pol, s in runs.items():
        for r in range(R):
            for n in range(min(len(s.history[r]), len(ref.history[r]))):
                assert np.array_equal(s.history[r][n], ref.history[r][n]), (pol, r, n)


def pin_admission_and_occupancy_hand():
    """Requests 0 and 1 start in layer 0's attention queue, request 2 is admitted at tick 2;
    every dispatch takes one tick, two layers, one expert (E = K = 1), MTFS.
      t1: att_0 {0, 1} (depths att_0 2)            -> 0, 1 in transit to exp_0 (arrive t2)
      t2: admit 2; exp_0 {0, 1} (2) vs att_0 {2} (1) -> exp_0; 0, 1 join att_1
      t3: att_1 {0, 1} (2) vs att_0 {2} (1)          -> att_1; 0, 1 in transit (arrive t4)
      t4: exp_1 {0, 1} (2) vs att_0 {2} (1)          -> exp_1 (stop = 4 merges reached)
      t5: attention closed, nothing in flight: the stream ends with request 2 never served.
    Occupancy seen at the decisions, chain att_0, exp_0, att_1, exp_1 -- t1: (2, 0, 0, 0),
    t2: (1, 2, 0, 0), t3: (1, 0, 2, 0), t4: (1, 0, 0, 2); in transit at a decision: 0 every
    time (arrivals are delivered first); the deepest bucket at service: 2."""
    delays = np.ones((3, 8), dtype=np.int64)
    s = _mk(R=3, L=2, E=1, K=1, H=3, delays=delays, stop=4, max_steps=8, values=False, admit=[0, 0, 2]).run()
    got = [(t.tick, t.kind, t.layer, t.count) for t in s.trace]
    assert got == [(1, "att", 0, 2), (2, "exp", 0, 2), (3, "att", 1, 2), (4, "exp", 1, 2)]
    assert s.n.tolist() == [2, 2, 0] and s.combined == 4
    assert s.peak_q == [2, 2, 2, 2] and s.occ_sum == [5, 2, 2, 2]
    assert s.peak_transit == 0 and s.peak_bucket == 2 and s.to_admit == 0


def test_admission_and_occupancy_hand():
    pin_admission_and_occupancy_hand()


def test_admission_pin_catches_planted_early_admission(monkeypatch):
    """Admitting every request at the start (ignoring the admission ticks) must fail the pin."""
    real = om.StreamOracle.__init__

    def early(self, *a, **kw):
        kw["admit"] = None
        real(self, *a, **kw)
    monkeypatch.setattr(om.StreamOracle, "__init__", early)
    try:
        pin_admission_and_occupancy_hand()
        caught = False
    except AssertionError:
        caught = True
    assert caught


def test_admission_bursts_conserve_and_serve_all():
    """Bursts with no stop: every request is admitted and runs all its steps, each merge is
    counted once, and no request finishes a step before its admission tick."""
    R, L, E, K, H, M = 24, 2, 4, 2, 5, 12
    d = np.random.default_rng(3).integers(1, 4, size=(R, M))
    admit = (np.arange(R) // 6) * 4                     # 6 requests every 4 ticks
    s = _mk(R, L, E, K, H, d, stop=10 ** 6, max_steps=M, values=False, admit=admit).run()
    assert s.to_admit == 0 and s.combined == int(s.n.sum()) == R * M
    first = {r: s.done_tick[(r, 1)] for r in range(R)}
    assert all(first[r] > admit[r] for r in range(R))  # a request's first step ends after it is admitted
