"""ORACLE -- test infrastructure only (see the package docstring).

Plain float64 statement of asynchronous MoE expert execution.  Citations name
the page and the section they follow:

* "SOSP'26 StreamEP" (marsggbo.github.io), section 3: tensors carry metadata
  (RequestID, LayerID = layer / home rank / expert, tensor reference, top-k
  weight); a Receptor puts each arriving token into a token pool and routes it
  to the micro-queue of its target layer and task type; the scheduler picks a
  non-empty queue; the executor gathers the scattered inputs into a contiguous
  batch and runs the expert; results return to the home rank, where the top-k
  merge buffers the first K-1 results and releases the token only when the
  K-th lands; the merge is y = sum_j w_j E_j(x); the shared expert runs on the
  home rank.
* Same page, section 4: MTFS (most tokens first) picks the queue holding the
  most tokens; the defragmenting score S(s) = Q(s) + sum_{j=1..W} delta^j
  [Q(s_j) + H(s_j)] with its worked example (W=2, delta=0.5: 20 + 0.5*100 +
  0.25*80 = 90 against an isolated queue of 60).
* "CascadeEP: Asynchronous Expert Execution for MoE Prefill", abstract:
  expert FFN starts before every replica's tokens are ready, and streamFFN
  batches ready tokens to trade early start against FFN efficiency (read here
  as a minimum batch per expert with a most-tokens-first fallback).
* "asynchronous MoE serving" notes, "inferred obligations": accept exactly the
  selected contributions once (no duplicate accumulation), publish readiness
  only after the payload, and expect arrival-dependent addition order to break
  bitwise equality unless the order is fixed -- hence the combine below sums
  in ascending k order, whatever order the results arrived in.

Readings where the pages are silent (the expert FFN form, the router rule,
tie-breaks, wave timing) are stated at each function.
"""
from dataclasses import dataclass, field
from itertools import combinations

import numpy as np


# ---------------------------------------------------------------- routing ----

def route(logits, K):
    """Top-K routing with renormalised softmax weights.

    StreamEP section 3: each token selects the K experts with the highest
    router scores (128 choose 4 for GPT-OSS-120B).  The router rule itself is
    not on the pages; the reading used is: softmax over all E experts, keep the
    K largest, renormalise their probabilities to sum to one.

    The selection is decided on the logits exactly as given (softmax is
    strictly increasing, so it selects the same set); equal logits go to the
    lower expert index.  The k order of the result is descending score.

    Returns idx [T, K] int64 and w [T, K] float64.
    """
    z = np.asarray(logits, dtype=np.float64)
    T, E = z.shape
    zmax = z.max(axis=1, keepdims=True)
    p = np.exp(z - zmax)
    p = p / p.sum(axis=1, keepdims=True)              # softmax over all E
    idx = np.empty((T, K), dtype=np.int64)
    w = np.empty((T, K), dtype=np.float64)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-z[t, e], e))
        sel = order[:K]
        idx[t] = sel
        w[t] = p[t, sel] / p[t, sel].sum()             # renormalise over the top K
    return idx, w


def route_bruteforce(logits, K):
    """Independent restatement for pinning ``route`` on small inputs.

    Enumerates every K-subset, keeps the one with the largest logit sum (ties:
    the lexicographically smallest subset), orders it by descending logit, and
    computes the weights as a softmax restricted to the subset
    exp(z_j - m) / sum_{i in S} exp(z_i - m).  That is algebraically the same
    as "softmax then renormalise" because the full-softmax denominator cancels.
    """
    z = np.asarray(logits, dtype=np.float64)
    T, E = z.shape
    idx = np.empty((T, K), dtype=np.int64)
    w = np.empty((T, K), dtype=np.float64)
    for t in range(T):
        best, best_sum = None, None
        for S in combinations(range(E), K):
            s = sum(z[t, e] for e in S)
            if best is None or s > best_sum:
                best, best_sum = S, s
        S = sorted(best, key=lambda e: (-z[t, e], e))
        m = max(z[t, e] for e in S)
        num = np.array([np.exp(z[t, e] - m) for e in S])
        idx[t] = S
        w[t] = num / num.sum()
    return idx, w


# ------------------------------------------------------------ expert FFN ----

def silu(a):
    """silu(a) = a * sigmoid(a) = a / (1 + e^-a)."""
    a = np.asarray(a, dtype=np.float64)
    return a / (1.0 + np.exp(-a))


def expert_ffn(X, W1, W3, W2):
    """SwiGLU expert: E(x) = (silu(x W1) * (x W3)) W2.

    The pages name no FFN form; the workload fixes SwiGLU with W1, W3 [H, I]
    and W2 [I, H] and no bias.  X is [n, H]; result [n, H], float64.
    """
    X = np.asarray(X, dtype=np.float64)
    g = X @ np.asarray(W1, dtype=np.float64)
    u = X @ np.asarray(W3, dtype=np.float64)
    return (silu(g) * u) @ np.asarray(W2, dtype=np.float64)


def combine(contribs):
    """Top-k merge, StreamEP section 3: y = sum_{j=1..K} w_j E_j(x).

    ``contribs`` is the list of already-weighted results w_j E_j(x) indexed
    by k; they are added in ascending k order (a fixed order, so the result
    does not depend on which result arrived first)."""
    y = np.zeros_like(np.asarray(contribs[0], dtype=np.float64))
    for c in contribs:
        y = y + c
    return y


def dense_moe(x, idx, w, experts, shared=None):
    """Brute-force dense MoE for pinning: every token through every expert.

    y_t = sum_e m_{t,e} w_{t,e} E_e(x_t) (+ E_shared(x_t)), with m the top-K
    mask.  ``experts(e)`` returns (W1, W3, W2)."""
    x = np.asarray(x, dtype=np.float64)
    T = x.shape[0]
    E = max(int(np.max(idx)) + 1, 1)
    y = np.zeros_like(x)
    for e in range(E):
        out = expert_ffn(x, *experts(e))                # all tokens, masked below
        for t in range(T):
            hit = np.nonzero(idx[t] == e)[0]
            if hit.size:
                y[t] += w[t, hit[0]] * out[t]
    if shared is not None:
        y = y + expert_ffn(x, *shared)
    return y


# -------------------------------------------------------------- policies ----

def mtfs_pick(depths, max_groups=0):
    """MTFS, StreamEP section 4: the queue with the most tokens goes first.

    Applied to the per-expert buckets of one layer's expert queue: non-empty
    buckets ordered by depth, deepest first, equal depth -> lower expert id;
    ``max_groups`` = 0 takes every non-empty bucket (one grouped step)."""
    cand = [(-d, e) for e, d in enumerate(depths) if d > 0]
    cand.sort()
    picks = [e for _, e in cand]
    return picks if max_groups <= 0 else picks[:max_groups]


def threshold_pick(depths, min_batch, max_groups=0, fallback_groups=1):
    """streamFFN reading (CascadeEP abstract): run an expert once it holds at
    least ``min_batch`` ready tokens (deepest first); when none qualifies, fall
    back to MTFS over the non-empty buckets, taking ``fallback_groups``."""
    cand = [(-d, e) for e, d in enumerate(depths) if d >= min_batch]
    cand.sort()
    picks = [e for _, e in cand]
    if picks:
        return picks if max_groups <= 0 else picks[:max_groups]
    return mtfs_pick(depths, fallback_groups)


def rank_pick(depths, ranks, steal=True):
    """Simulated expert-parallel ranks on one device ("asynchronous MoE serving" notes,
    CascadeEP v1: unstarted expert work can be reassigned to an idle helper; StreamEP section
    4 for the pick within a rank).

    Expert e belongs to rank ``e mod ranks``.  Each rank runs its own deepest non-empty
    bucket (equal depth -> lower id).  With ``steal``, every rank that owns no non-empty
    bucket then takes, in rank order, the deepest non-empty bucket that no rank has picked
    (equal depth -> lower id).  Returns the picks in rank order."""
    picks = [None] * ranks
    for r in range(ranks):
        own = [(-depths[e], e) for e in range(r, len(depths), ranks) if depths[e] > 0]
        if own:
            picks[r] = min(own)[1]
    if steal:
        taken = {e for e in picks if e is not None}
        for r in range(ranks):
            if picks[r] is not None:
                continue
            for e in mtfs_pick(depths):
                if e not in taken:
                    picks[r] = e
                    taken.add(e)
                    break
    return [e for e in picks if e is not None]


def defrag_score(q_now, lookahead, delta):
    """Defragmenting score, StreamEP section 4:
    S(s) = Q(s) + sum_{j=1..W} delta^j [Q(s_j) + H(s_j)].

    ``lookahead`` lists (Q(s_j), H(s_j)) for j = 1..W along the execution chain
    attention -> expert -> next attention."""
    s = float(q_now)
    dj = 1.0
    for q, h in lookahead:
        dj = dj * delta                    # delta^j, j = 1..W
        s += dj * (q + h)
    return s


# ----------------------------------------------------- asynchronous layer ----

@dataclass
class StepRecord:
    step: int
    picks: list                      # [(expert, count, sorted ((slot, k), ...))]
    emitted: list                    # token slots whose combine completed this step


@dataclass
class _Slot:
    mask: int = 0                    # which k have been delivered (bit k; bit K = shared)
    results: dict = field(default_factory=dict)   # k -> weighted result (float64 [H])
    landed: int = 0
    combined: int = 0


class AsyncMoEOracle:
    """One MoE layer executed asynchronously, step by step.

    Receptor (StreamEP section 3, steps 1-2): an arriving token is stored in
    the token pool under its RequestID (its combine slot) and each of its
    delivered (expert, k, weight) pairs is appended to that expert's bucket in
    the layer's expert queue.  A token's first delivery also enqueues the
    always-on shared expert (bucket E, weight 1) when the layer has one.

    Step (sections 3-4): the policy picks buckets from their depths; each
    picked bucket is drained whole, its tokens gathered into one contiguous
    batch and run through the expert; every weighted result lands in the
    (slot, k) entry of the top-k merge; a token is emitted once all of its K
    (+1 shared) results have landed, as their sum in ascending k order.

    ``experts(e)`` returns (W1, W3, W2) as float64 arrays, or ``None`` for
    identity experts (E(x) = x).  ``compute`` restricts the float work to a
    set of token slots (the bookkeeping always covers every token).
    """

    def __init__(self, num_experts, top_k, x, experts, has_shared=False, compute=None):
        self.E, self.K = num_experts, top_k
        self.x = np.asarray(x, dtype=np.float64)            # the token pool, by slot
        self.T = self.x.shape[0]
        self.experts = experts
        self.has_shared = has_shared
        self.nb = num_experts + (1 if has_shared else 0)
        self.buckets = [[] for _ in range(self.nb)]
        self.slots = [_Slot() for _ in range(self.T)]
        self.weights = {}                                     # (slot, k) -> w
        self.compute = None if compute is None else set(int(t) for t in compute)
        self.y = {}
        self.emit_step = {}
        self.duplicates = 0
        self.steps = []
        self.nstep = 0

    # Receptor ------------------------------------------------------------
    def deliver(self, tokens, idx, w, rank=None):
        """Deliver the pairs of ``tokens`` (all K, or those of rank (r, n))."""
        for t in np.asarray(tokens, dtype=np.int64):
            t = int(t)
            s = self.slots[t]
            for k in range(self.K):
                e = int(idx[t, k])
                if rank is not None and e % rank[1] != rank[0]:
                    continue
                if s.mask >> k & 1:                            # already accepted once
                    self.duplicates += 1
                    continue
                s.mask |= 1 << k
                self.weights[(t, k)] = float(w[t, k])
                self.buckets[e].append((t, k))
            if self.has_shared and not (s.mask >> self.K & 1):
                s.mask |= 1 << self.K
                self.weights[(t, self.K)] = 1.0
                self.buckets[self.E].append((t, self.K))

    def depths(self):
        return [len(b) for b in self.buckets]

    def snapshot(self):
        """Queue contents: per bucket, the sorted multiset of (slot, k)."""
        return [sorted(b) for b in self.buckets]

    # Scheduler + executor -------------------------------------------------
    def _expert_out(self, e, X):
        if self.experts is None:
            return X.copy()
        return expert_ffn(X, *self.experts(e))

    def step(self, policy):
        """One scheduling step under ``policy`` (a callable depths -> picks)."""
        self.nstep += 1
        picks = policy(self.depths())
        rec = StepRecord(step=self.nstep, picks=[], emitted=[])
        need = self.K + (1 if self.has_shared else 0)
        for e in picks:
            batch = self.buckets[e]
            self.buckets[e] = []
            rec.picks.append((e, len(batch), tuple(sorted(batch))))
            rows = [(t, k) for (t, k) in batch if self.compute is None or t in self.compute]
            if rows:
                X = self.x[[t for t, _ in rows]]               # gather: contiguous batch
                out = self._expert_out(e, X)
                for i, (t, k) in enumerate(rows):
                    self.slots[t].results[k] = self.weights[(t, k)] * out[i]
            for (t, k) in batch:                               # result lands in (t, k)
                s = self.slots[t]
                s.landed += 1
                if s.landed == need:                           # the K-th result: release
                    s.combined += 1
                    self.emit_step[t] = self.nstep
                    rec.emitted.append(t)
                    if self.compute is None or t in self.compute:
                        self.y[t] = combine([s.results[j] for j in sorted(s.results)])
        rec.emitted.sort()
        self.steps.append(rec)
        return rec

    def pending(self):
        return sum(len(b) for b in self.buckets)


def replay_layer(num_experts, top_k, x, idx, w, waves, policy, experts,
                 has_shared=False, compute=None, max_steps=100000):
    """Replay arrival waves against one asynchronous layer on a logical clock.

    One tick per scheduling step; wave i is delivered (in wave order) before
    the first step whose tick is >= its arrival tick; steps continue until
    every delivered pair has been executed.  Arrival delays only shape the
    batches, never the values."""
    sim = AsyncMoEOracle(num_experts, top_k, x, experts, has_shared, compute)
    order = sorted(range(len(waves)), key=lambda i: (waves[i].tick, i))
    nxt = 0
    tick = 0
    while tick < max_steps:
        tick += 1
        while nxt < len(order) and waves[order[nxt]].tick <= tick:
            wv = waves[order[nxt]]
            sim.deliver(wv.tokens, idx, w, wv.rank)
            nxt += 1
        sim.step(policy)
        if nxt == len(order) and sim.pending() == 0:
            break
    return sim


def y_sample(tokens, x, idx, w, experts, shared=None):
    """y for a few tokens straight from the merge formula (no queues).

    StreamEP section 3: y_t = sum_{k} w_{t,k} E_{idx[t,k]}(x_t) in ascending k, plus the
    shared expert E_shared(x_t) with weight one (added last, outside the renormalised
    weights).  Pinned against the brute-force dense MoE on every token of a tiny case and
    against a hand-computed H = I = 1 case, with and without the shared expert."""
    out = {}
    for t in tokens:
        t = int(t)
        xt = np.asarray(x[t], dtype=np.float64)[None, :]
        contribs = [w[t, k] * expert_ffn(xt, *experts(int(idx[t, k])))[0] for k in range(idx.shape[1])]
        if shared is not None:
            contribs.append(expert_ffn(xt, *shared)[0])
        out[t] = combine(contribs)
    return out


# --------------------------------------------------- attention stub (c5) ----

def rmsnorm(x, eps=1e-6):
    """RMSNorm without gain: x / sqrt(mean(x^2) + eps), per row."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def attention_stub(x, P):
    """Stand-in for the attention stage: RMSNorm(x) @ P."""
    return rmsnorm(x) @ np.asarray(P, dtype=np.float64)


def layer_pick(att_depth, exp_depth, allow_attention=True):
    """MTFS over the 2L micro-queues (StreamEP section 3: one attention queue and one expert
    queue per layer; section 4: the queue holding the most tokens goes first).

    Depths count tokens (requests) in both kinds of queue.  Equal depth -> lower layer;
    within a layer the attention queue before the expert queue.  Returns (kind, layer)
    with kind "att" / "exp", or None when every eligible queue is empty."""
    cand = []
    for l, d in enumerate(att_depth):
        if allow_attention and d > 0:
            cand.append((-d, l, 0))
    for l, d in enumerate(exp_depth):
        if d > 0:
            cand.append((-d, l, 1))
    if not cand:
        return None
    _, l, kind = min(cand)
    return ("att" if kind == 0 else "exp", l)


def chain_pick(att_depth, exp_depth, policy, allow_attention=True, drained=None, window=2, decay=0.5,
               in_transit=0, snap_avg=None):
    """Layer-level policies over the 2L micro-queues in chain order att_0, exp_0, att_1, ...

    mtfs    -- most tokens first (``layer_pick``), StreamEP section 4.
    flfs    -- first layer first: the earliest non-empty queue in the chain (section 4).
    defrag  -- the defragmenting score of section 4, S(s) = Q(s) + sum_{j=1..W} delta^j
               [Q(s_j) + H(s_j)], s_j the j-th queue after s along the chain (truncated at
               the last layer, the paper's version); H = tokens drained from a queue over the
               recent ticks (``drained``); highest score first, equal scores -> earlier queue.
    defrag_src -- the same score as StreamEP section 4 describes the source implementation
               (the paragraph after the formula): H(s_j) is the average of queue s_j's depth
               snapshots over the recent window (``snap_avg``), and the lookahead continues
               cyclically along the chain (the queue after the last layer's expert queue is
               layer 0's attention queue) instead of stopping at the last layer.
    barrier -- the synchronous baseline: serve a queue only when nothing is in transit and it
               holds every token still being served (lockstep layers); if tokens are split
               with nothing in transit, serve the earliest queue so progress continues.
    Closed attention queues (after the stop) count as empty everywhere."""
    L = len(att_depth)
    Q = []
    for l in range(L):
        Q.append(att_depth[l] if allow_attention else 0)
        Q.append(exp_depth[l])
    nonempty = [q for q in range(2 * L) if Q[q] > 0]
    if not nonempty:
        return None
    as_pick = lambda q: ("att" if q % 2 == 0 else "exp", q // 2)
    if policy == "mtfs":
        return layer_pick(att_depth, exp_depth, allow_attention)
    if policy == "flfs":
        return as_pick(nonempty[0])
    if policy == "defrag":
        best, best_s = None, None
        for q in nonempty:
            look = [(Q[q + j], drained[q + j]) for j in range(1, window + 1) if q + j < 2 * L]
            s = defrag_score(Q[q], look, decay)
            if best is None or s > best_s:
                best, best_s = q, s
        return as_pick(best)
    if policy == "defrag_src":
        best, best_s = None, None
        for q in nonempty:
            look = [(Q[(q + j) % (2 * L)], snap_avg[(q + j) % (2 * L)]) for j in range(1, window + 1)]
            s = defrag_score(Q[q], look, decay)
            if best is None or s > best_s:
                best, best_s = q, s
        return as_pick(best)
    if policy == "barrier":
        return None if in_transit > 0 else as_pick(nonempty[0])
    raise ValueError(policy)


@dataclass
class TickRecord:
    tick: int
    kind: str                        # "att", "exp" or "idle"
    layer: int
    count: int                       # requests served by the picked queue


class StreamOracle:
    """Streaming multi-layer decode on the 2L micro-queues, tick by tick.

    StreamEP section 3: every request keeps its home (its state lives under its RequestID);
    a layer's attention queue feeds the attention stage, whose output is routed (top-K) and
    dispatched to that layer's expert queue; the merged result returns home and enters the
    next layer's attention queue -- layers advance independently per request, no barrier.
    Readings: the attention stage is the stub a = RMSNorm(x) P_l; x^(n+1) = MoE_l(a), layer
    l = n mod L, no residual; router logits of (request, step) and dispatch delays are given
    (value-independent routing); a dispatch made at tick t arrives at tick t + delay; one
    queue is served per tick (layer_pick); an expert pick drains all of the layer's buckets;
    once `stop` merges have completed (checked at the start of a tick) attention queues are
    no longer served, in-flight work still finishes.

    Per tick: deliver the arrivals due, admit the requests whose admission tick it is into
    layer 0's attention queue (``admit``: per-request tick, None = every request at the start),
    pick a queue, serve it.  ``values`` = False keeps only the integer bookkeeping; ``compute``
    restricts the float chain to some requests.

    Occupancy, for the latency study (StreamEP section 4: queue depths drive the scheduler):
    per queue in chain order the largest depth the scheduler saw at a decision and the sum of
    those depths over the ticks; the largest number of requests in transit; the deepest
    expert bucket at the moment its layer's expert queue was served.
    """

    def __init__(self, L, K, x0, proj, logits, delays, experts, stop, max_steps,
                 values=True, compute=None, policy="mtfs", window=2, decay=0.5, hist_window=8, admit=None):
        self.L, self.K = L, K
        self.policy, self.window, self.decay, self.hist_window = policy, window, decay, hist_window
        self.drain_log = []               # per tick: tokens drained from each of the 2L queues
        self.snap_log = []                # per tick: depth of each of the 2L queues at its decision
        self.R = len(x0)
        self.x0 = np.asarray(x0, dtype=np.float64)
        self.proj, self.logits, self.delays = proj, logits, np.asarray(delays)
        self.experts = experts            # experts(layer, e) -> (W1, W3, W2)
        self.stop, self.max_steps = stop, max_steps
        self.values = values
        self.compute = set(range(self.R)) if compute is None else set(int(r) for r in compute)
        self.n = np.zeros(self.R, dtype=np.int64)
        self.admit = np.zeros(self.R, dtype=np.int64) if admit is None else np.asarray(admit, dtype=np.int64)
        self.att = [set() for _ in range(L)]
        self.att[0] = set(int(r) for r in range(self.R) if self.admit[r] <= 0)
        self.to_admit = int((self.admit > 0).sum())
        self.peak_q = [0] * (2 * L)
        self.occ_sum = [0] * (2 * L)
        self.peak_transit = 0
        self.peak_bucket = 0
        self.transit = {}                 # r -> arrival tick
        self.pending = [set() for _ in range(L)]   # requests whose pairs sit in layer l's queue
        self.a = {}                       # r -> attention output for its current step
        self.route = {}                   # r -> (idx, w) for its current step
        self.x = {r: self.x0[r] for r in self.compute}
        self.history = {r: [self.x0[r]] for r in self.compute}
        self.done_tick = {}               # (r, n) -> tick at which step n completed
        self.combined = 0
        self.tick = 0
        self.trace = []

    def busy(self):
        open_att = self.combined < self.stop and (any(self.att) or self.to_admit > 0)
        return bool(self.transit) or any(self.pending) or open_att

    def step(self):
        self.tick += 1
        for r in sorted(r for r, t in self.transit.items() if t == self.tick):
            del self.transit[r]
            self.pending[int(self.n[r]) % self.L].add(r)
        for r in np.nonzero(self.admit == self.tick)[0]:
            self.att[0].add(int(r))
            self.to_admit -= 1
        recent = self.drain_log[-self.hist_window:] if self.hist_window > 0 else []
        drained = [sum(v[q] for v in recent) for q in range(2 * self.L)]
        snaps = self.snap_log[-self.hist_window:] if self.hist_window > 0 else []
        snap_avg = [sum(v[q] for v in snaps) / len(snaps) if snaps else 0.0 for q in range(2 * self.L)]
        allow = self.combined < self.stop
        att_d, exp_d = [len(a) for a in self.att], [len(p) for p in self.pending]
        pick = chain_pick(att_d, exp_d, self.policy, allow_attention=allow, drained=drained,
                          window=self.window, decay=self.decay, in_transit=len(self.transit),
                          snap_avg=snap_avg)
        snap = [v for l in range(self.L) for v in ((att_d[l] if allow else 0), exp_d[l])]
        self.snap_log.append(snap)
        for q in range(2 * self.L):
            self.peak_q[q] = max(self.peak_q[q], snap[q])
            self.occ_sum[q] += snap[q]
        self.peak_transit = max(self.peak_transit, len(self.transit))
        tick_drain = [0] * (2 * self.L)
        self.drain_log.append(tick_drain)
        if pick is None:
            self.trace.append(TickRecord(self.tick, "idle", -1, 0))
            return
        kind, l = pick
        if kind == "att":
            batch = sorted(self.att[l])
            self.att[l] = set()
            for r in batch:
                n = int(self.n[r])
                idx, w = route(self.logits(r, n)[None, :], self.K)
                self.route[r] = (idx[0], w[0])
                if self.values and r in self.compute:
                    self.a[r] = attention_stub(self.x[r][None, :], self.proj(l))[0]
                self.transit[r] = self.tick + int(self.delays[r, n])
        else:
            batch = sorted(self.pending[l])
            self.pending[l] = set()
            per_expert = {}
            for r in batch:
                for e in self.route[r][0]:
                    per_expert[int(e)] = per_expert.get(int(e), 0) + 1
            self.peak_bucket = max([self.peak_bucket] + list(per_expert.values()))
            for r in batch:
                n = int(self.n[r])
                if self.values and r in self.compute:
                    idx, w = self.route[r]
                    contribs = [w[k] * expert_ffn(self.a[r][None, :], *self.experts(l, int(idx[k])))[0]
                                for k in range(self.K)]
                    self.x[r] = combine(contribs)
                    self.history[r].append(self.x[r])
                self.n[r] = n + 1
                self.done_tick[(r, n + 1)] = self.tick
                self.combined += 1
                if n + 1 < self.max_steps:
                    self.att[(n + 1) % self.L].add(r)
        tick_drain[2 * l + (0 if kind == "att" else 1)] = len(batch)
        self.trace.append(TickRecord(self.tick, kind, l, len(batch)))

    def run(self, max_ticks=1000000):
        while self.busy() and self.tick < max_ticks:
            self.step()
        return self
