"""Replay of arrival waves on one GPU (the simulated transport).

The pages' multi-GPU transport (CPU metadata message, then NCCL send/recv, "SOSP'26
StreamEP" section 5) is replaced by waves that are already resident in device memory:
each wave is a list of token rows (and, for expert-parallel replays, which of each
token's K pairs it carries).  A logical clock advances one tick per scheduling step;
a wave is delivered before the first step whose tick is >= its arrival tick.  Delays
therefore shape only which tokens are batched together, never the values.
"""
import numpy as np
import torch

from .api import Policy


class LayerReplay:
    """Drives one layer of a ``MoEAsync`` handle through a list of ``Wave`` objects."""

    def __init__(self, moe, waves, num_tokens, device="cuda", idx_host=None, layer=0, max_ticks=None):
        self.moe, self.layer, self.T = moe, layer, num_tokens
        self.waves = sorted(waves, key=lambda w: w.tick)
        self.rows, self.kmask = [], []
        for wv in self.waves:
            rows = torch.as_tensor(np.asarray(wv.tokens, dtype=np.int32), device=device)
            self.rows.append(rows)
            if wv.rank is None:
                self.kmask.append(None)
            else:
                if idx_host is None:
                    raise ValueError("expert-parallel waves need the routing on the host")
                r, n = wv.rank
                sel = (np.asarray(idx_host)[np.asarray(wv.tokens)] % n) == r
                bits = (sel.astype(np.uint64) << np.arange(sel.shape[1], dtype=np.uint64)).sum(1)
                self.kmask.append(torch.as_tensor(bits.astype(np.int64), device=device).to(torch.int32))
        self.last_tick = max((w.tick for w in self.waves), default=0)
        self.max_ticks = max_ticks or (self.last_tick + 1)
        dt = moe.dtype
        self.y_out = torch.empty((num_tokens, moe.H), dtype=dt, device=device)
        self.slot_out = torch.full((num_tokens,), -1, dtype=torch.int32, device=device)
        self.step_out = torch.zeros((num_tokens,), dtype=torch.int32, device=device)
        self.n_out = torch.zeros(1, dtype=torch.int32, device=device)
        self.tick_counts = torch.zeros(4096, dtype=torch.int32, device=device)

    def run_ticks(self, x, idx, w, policy, stream=None, collect_each_step=True, fused=False):
        """Deliver every wave on its tick and run one scheduling step per tick, up to the
        last arrival tick.  No host synchronisation.

        fused: one ``moe_async_tick`` a tick (collect of what the previous steps made ready,
        the tick's last wave, the step); earlier waves of the same tick are enqueued first, and
        a collect after the last tick takes that step's tokens."""
        moe, L = self.moe, self.layer
        self.n_out.zero_()
        nxt = 0
        for tick in range(1, self.last_tick + 1):
            due = []
            while nxt < len(self.waves) and self.waves[nxt].tick <= tick:
                due.append(nxt)
                nxt += 1
            if fused:
                for i in due[:-1]:
                    moe.enqueue(L, x, idx, w, rows=self.rows[i], kmask=self.kmask[i], stream=stream)
                wave = dict(x=x, expert=idx, w=w, rows=self.rows[due[-1]], kmask=self.kmask[due[-1]]) if due else {}
                moe.tick(L, policy, y_out=self.y_out, slot_out=self.slot_out, n_out=self.n_out, append=True,
                         step_out=self.step_out, stream=stream, **wave)
                if tick >= 2:                    # the tokens of steps up to tick - 1
                    self.tick_counts[tick - 2:tick - 1].copy_(self.n_out)
                continue
            for i in due:
                moe.enqueue(L, x, idx, w, rows=self.rows[i], kmask=self.kmask[i], stream=stream)
            moe.schedule_step(L, policy, stream=stream)
            if collect_each_step:
                moe.collect(L, self.y_out, self.slot_out, self.n_out, append=True, stream=stream,
                            step_out=self.step_out)
                self.tick_counts[tick - 1:tick].copy_(self.n_out)
        if fused or not collect_each_step:
            moe.collect(L, self.y_out, self.slot_out, self.n_out, append=True, stream=stream,
                        step_out=self.step_out)
            if self.last_tick >= 1:
                self.tick_counts[self.last_tick - 1:self.last_tick].copy_(self.n_out)
        self.ticks_run = self.last_tick

    def drain(self, policy, max_steps=10000, check_every=8, stream=None):
        """Keep stepping (and collecting) until no token is open; returns the steps taken, or
        -1 if tokens were still open after max_steps (e.g. a pair that never arrived)."""
        moe, L = self.moe, self.layer
        steps = 0
        tick = self.ticks_run
        while True:
            st = moe.stats(stream=stream)
            if st["open_tokens"] == 0 and st["ready"] == 0:
                return steps
            if steps >= max_steps:
                return -1
            for _ in range(check_every):
                tick += 1
                moe.schedule_step(L, policy, stream=stream)
                moe.collect(L, self.y_out, self.slot_out, self.n_out, append=True, stream=stream,
                            step_out=self.step_out)
                if tick - 1 < self.tick_counts.numel():
                    self.tick_counts[tick - 1:tick].copy_(self.n_out)
                steps += 1
            self.ticks_run = tick

    def finish(self, policy, max_steps=10000, stream=None):
        """Drain the way the benchmark does: ``moe_async_wait`` (under MTFS / THRESHOLD one
        device plan of the remaining steps), then one collect.  Returns the wait status."""
        st = self.moe.wait(self.layer, policy, max_steps=max_steps, check_every=32, stream=stream)
        self.moe.collect(self.layer, self.y_out, self.slot_out, self.n_out, append=True, stream=stream,
                         step_out=self.step_out)
        self.finished = True
        return st

    def device_steps(self):
        """Emission step of each collected row, as the device recorded it."""
        n = int(self.n_out.item())
        return self.step_out[:n].cpu().numpy().astype(np.int64)

    def results(self):
        """(y by token [T, H] on the host as float64 or None rows, emission tick per token)."""
        n = int(self.n_out.item())
        slots = self.slot_out[:n].cpu().numpy()
        y = self.y_out[:n].float().cpu().numpy().astype(np.float64)
        counts = self.tick_counts[: self.ticks_run].cpu().numpy()
        emit = np.zeros(n, dtype=np.int64)
        prev = 0
        for t, c in enumerate(counts, start=1):
            emit[prev:c] = t
            prev = max(prev, c)
        return slots, y, emit


def policy_of(spec):
    return Policy.from_spec(spec)
