"""ORACLE -- test infrastructure only.  A small, exhaustively checkable model of the combine-
slot protocol, with the transition rules of the library's device code.

"asynchronous MoE serving" notes, first research candidate: check a reusable-buffer protocol
on two senders, two receivers, two slots and two selected experts; enumerate delayed
notifications, cancellation and slot-generation wraparound; check ownership, visibility,
exactly-once combine and eventual progress.  CascadeEP (same notes): output readiness is
tracked separately from buffer reclamation; AInfer-PD: an abandoned operation retires its
buffer until a quiescent point.

State per slot: generation, owner request, accepted-pair mask, retired flag, landed count,
the contributions (request, k, input) written into its combine rows, and the token-pool row:
the request whose token vector the row holds (StreamEP section 3: the Receptor stores each
arriving token in the pool; the executor gathers pool rows).  Events:
  deliver(request, k)   a sender's pair, carrying the request's token vector, arrives at the
                        slot the request was given; accepted iff the slot is still owned by
                        that request, not retired, and k not yet accepted (else dropped); the
                        pool row takes the carried vector only when the pair is accepted
  run(expert)           the expert's queue is drained: every queued record reads its slot's
                        pool row and lands on the slot (writes its contribution, bumps the
                        landed count)
  merge(slot)           once all K contributions of the owner have landed: publish
  reclaim(slot)         the published slot is collected and freed (generation + 1)
  cancel(slot)          the owner abandons the request: retire the slot; it is freed only
                        once every accepted record has landed (retire until quiescent)
  assign(slot, request) a free slot takes the next request

The unsafe variant (``reuse_on_cancel=True``) frees a cancelled slot at once -- the bug the
quiescence rule prevents: a late record of the old request then lands on the new owner.
A second unsafe variant (``pool_on_reject=True``) copies every arriving token vector into the
pool row, accepted or not: a late (stale) pair of a cancelled request then replaces the new
owner's input before its records run ("inferred obligations": accept exactly the selected
contributions).
"""
from collections import deque

K = 2


class Model:
    def __init__(self, routes, nslots=2, reuse_on_cancel=False, cancel_requests=(), gen_bits=None,
                 pool_on_reject=False):
        # routes[r] = (expert of k=0, expert of k=1) for request r; requests are assigned to
        # slots in order as slots become free
        self.routes = routes
        self.nslots = nslots
        self.reuse_on_cancel = reuse_on_cancel
        self.pool_on_reject = pool_on_reject
        self.cancel_requests = frozenset(cancel_requests)
        self.gen_bits = gen_bits

    def initial(self):
        slots = []
        nxt = 0
        home = [None] * len(self.routes)
        for s in range(self.nslots):
            owner = nxt if nxt < len(self.routes) else None
            if owner is not None:
                home[owner] = s
            nxt += owner is not None
            # gen, owner, mask, retired, landed, rows, pool row
            slots.append((0, owner, 0, False, 0, frozenset(), None))
        # pending deliveries: (request, k); queues: per expert, tuple of (slot, request, k)
        pend = frozenset((r, k) for r in range(len(self.routes)) for k in range(K))
        queues = (tuple(), tuple())
        return (tuple(slots), pend, queues, nxt, frozenset(), frozenset(), frozenset(), tuple(home))
        # ..., next request to assign, published, cancelled, violations, slot given to each request

    def moves(self, st):
        slots, pend, queues, nxt, pub, canc, bad, home = st
        out = []
        # deliver: the pair goes to the slot its request was given, whoever owns it now
        for (r, k) in sorted(pend):
            if r >= nxt:
                continue                                       # request not assigned yet
            i = home[r]
            slots2 = list(slots)
            q2 = list(queues)
            g, o, m, ret, l, rows, pool = slots[i]
            accepted = o == r and not ret and not (m >> k) & 1
            if accepted:
                slots2[i] = (g, o, m | (1 << k), ret, l, rows, r)
                e = self.routes[r][k]
                q2[e] = q2[e] + ((i, r, k),)
            elif self.pool_on_reject:
                slots2[i] = (g, o, m, ret, l, rows, r)         # the rejected pair's vector lands
            out.append((("deliver", r, k), (tuple(slots2), pend - {(r, k)}, tuple(q2), nxt, pub, canc, bad, home)))
        # run an expert: every queued record reads its pool row and lands
        for e in range(2):
            if not queues[e]:
                continue
            slots2 = list(slots)
            bad2 = set(bad)
            for (i, r, k) in queues[e]:
                g, o, m, ret, l, rows, pool = slots2[i]
                if o != r:
                    bad2.add(("foreign-write", i, r, o))          # a late record hit a reused slot
                slots2[i] = (g, o, m, ret, l + 1, rows | {(r, k, pool)}, pool)
            slots2 = [self._maybe_free(s) for s in slots2]
            q2 = list(queues)
            q2[e] = tuple()
            st2 = self._assign((tuple(slots2), pend, tuple(q2), nxt, pub, canc, frozenset(bad2), home))
            out.append((("run", e), st2))
        # merge when all K of the owner landed
        for i, (g, o, m, ret, l, rows, pool) in enumerate(slots):
            mine = {(r, k, x) for (r, k, x) in rows if r == o}
            if o is not None and not ret and len(mine) == K and o not in pub:
                bad2 = set(bad)
                if rows != mine:
                    bad2.add(("mixed-output", i, o, tuple(sorted(rows, key=repr))))
                if any(x != o for (_, _, x) in mine):
                    bad2.add(("foreign-input", i, o, tuple(sorted(mine, key=repr))))
                if o in canc:
                    bad2.add(("published-after-cancel", o))
                out.append((("merge", i), (slots, pend, queues, nxt, pub | {o}, canc, frozenset(bad2), home)))
        # reclaim a published slot
        for i, (g, o, m, ret, l, rows, pool) in enumerate(slots):
            if o is not None and o in pub and not ret:
                slots2 = list(slots)
                slots2[i] = (self._next_gen(g), None, 0, False, 0, frozenset(), pool)
                out.append((("reclaim", i), self._assign((tuple(slots2), pend, queues, nxt, pub, canc, bad, home))))
        # cancel
        for i, (g, o, m, ret, l, rows, pool) in enumerate(slots):
            if o is not None and o in self.cancel_requests and not ret and o not in pub:
                slots2 = list(slots)
                if self.reuse_on_cancel:
                    slots2[i] = (self._next_gen(g), None, 0, False, 0, frozenset(), pool)
                else:
                    slots2[i] = self._maybe_free((g, o, m, True, l, rows, pool))
                st2 = self._assign((tuple(slots2), pend, queues, nxt, pub, canc | {o}, bad, home))
                out.append((("cancel", i), st2))
        return out

    def _next_gen(self, g):
        return (g + 1) % (1 << self.gen_bits) if self.gen_bits else g + 1

    def _maybe_free(self, s):
        g, o, m, ret, l, rows, pool = s
        if ret and l == bin(m).count("1"):                   # retired and quiescent
            return (self._next_gen(g), None, 0, False, 0, frozenset(), pool)
        return s

    def _assign(self, st):
        slots, pend, queues, nxt, pub, canc, bad, home = st
        slots = list(slots)
        home = list(home)
        for i, s in enumerate(slots):
            if s[1] is None and nxt < len(self.routes):
                slots[i] = (s[0], nxt, 0, False, 0, frozenset(), s[6])
                home[nxt] = i
                nxt += 1
        return (tuple(slots), pend, queues, nxt, pub, canc, bad, tuple(home))

    def explore(self, limit=2000000):
        """Breadth-first over every interleaving.  Returns (states, violations, deadlocks):
        a deadlock is a state with no move in which some request is neither published nor
        cancelled."""
        start = self._assign(self.initial())
        seen = {start}
        dq = deque([start])
        violations, deadlocks = set(), []
        while dq:
            st = dq.popleft()
            violations |= set(st[6])
            mv = self.moves(st)
            if not mv:
                slots, pend, queues, nxt, pub, canc, bad, home = st
                unfinished = [r for r in range(len(self.routes)) if r not in pub and r not in canc]
                if unfinished:
                    deadlocks.append(st)
            for _, st2 in mv:
                if st2 not in seen:
                    seen.add(st2)
                    dq.append(st2)
                    if len(seen) > limit:
                        raise RuntimeError("state space limit")
        return len(seen), violations, deadlocks
