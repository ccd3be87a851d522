"""Thin Python binding over the C ABI: argument marshalling only.

Every step of the path -- routing, enqueue, scheduling, the expert FFN, the merge,
collection -- runs in the library's CUDA kernels.  torch supplies device memory and
streams; nothing here computes on the data.
"""
import ctypes
from dataclasses import dataclass

import numpy as np
import torch

from . import _native as N

_DT = {torch.float32: N.MOE_F32, torch.bfloat16: N.MOE_BF16}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


@dataclass
class Policy:
    """Scheduling policy of one step (mirrors moe_async_policy)."""
    kind: str = "mtfs"            # "mtfs" | "threshold" | "ranks"
    max_groups: int = 0           # 0 = every qualifying bucket; "ranks": the number of ranks
    min_batch: int = 64
    fallback_groups: int = 1      # "threshold": buckets taken when none qualifies; "ranks": steal

    _KINDS = {"mtfs": N.MOE_POLICY_MTFS, "threshold": N.MOE_POLICY_THRESHOLD, "ranks": N.MOE_POLICY_RANKS}

    def c(self):
        return N.Policy(self._KINDS[self.kind], self.max_groups, self.min_batch, self.fallback_groups)

    @staticmethod
    def from_spec(spec):
        return Policy(spec.policy, spec.max_groups, spec.min_batch, spec.fallback_groups)


def host_writable(t):
    """True if the kernels can write the host tensor `t` directly (pinned host memory mapped
    at the same address), so it can be a collect output."""
    if t.is_cuda:
        return False
    return bool(N.load().moe_async_host_writable(ctypes.c_void_p(t.data_ptr()), t.numel() * t.element_size()))


def route(logits, top_k, idx=None, w=None, stream=None):
    """Top-K router on the device: returns (idx int32 [T,K], w fp32 [T,K])."""
    lib = N.load()
    assert logits.is_cuda and logits.dtype == torch.float32 and logits.is_contiguous()
    T, E = logits.shape
    if idx is None:
        idx = torch.empty((T, top_k), dtype=torch.int32, device=logits.device)
    if w is None:
        w = torch.empty((T, top_k), dtype=torch.float32, device=logits.device)
    N.check(lib.moe_async_route(_ptr(logits), T, E, top_k, _ptr(idx), _ptr(w), _stream(stream)), "route")
    return idx, w


class MoEAsync:
    """One handle of the asynchronous MoE library (see include/moe_async.h)."""

    def __init__(self, num_experts, top_k, hidden, inter, dtype, max_slots, weights=None,
                 num_layers=1, has_shared=False, expert_kind="swiglu", bucket_capacity=0,
                 trace_capacity=0, stream=None):
        self.lib = N.load()
        self.E, self.K, self.H, self.I = num_experts, top_k, hidden, inter
        self.L, self.S = num_layers, max_slots
        self.has_shared = bool(has_shared)
        self.dtype = dtype
        self.KS = top_k + (1 if has_shared else 0)
        cfg = N.Config(num_layers, num_experts, top_k, hidden, inter, _DT[dtype], int(has_shared),
                       max_slots, bucket_capacity,
                       N.MOE_EXPERT_SWIGLU if expert_kind == "swiglu" else N.MOE_EXPERT_IDENTITY,
                       trace_capacity)
        self.trace_capacity = trace_capacity
        arr = ctypes.c_void_p * num_layers

        def ptrs(key):
            if weights is None:
                return None
            for wl in weights:
                t = wl[key]
                assert t.is_cuda and t.dtype == dtype and t.is_contiguous(), key
            return arr(*[wl[key].data_ptr() for wl in weights])

        keep = [ptrs(k) for k in ("w1", "w3", "w2")]
        sh = [ptrs(k) for k in ("sw1", "sw3", "sw2")] if has_shared and weights is not None else [None] * 3
        self.h = ctypes.c_void_p()
        st = self.lib.moe_async_create(ctypes.byref(cfg), *keep, *sh, _stream(stream), ctypes.byref(self.h))
        N.check(st, "moe_async_create")

    # -- the five calls -------------------------------------------------------
    def enqueue(self, layer, x, expert, w, n=None, rows=None, slots=None, kmask=None, gen=None,
                stream=None):
        n = (rows.shape[0] if rows is not None else x.shape[0]) if n is None else n
        st = self.lib.moe_async_enqueue(self.h, layer, n, _ptr(rows), _ptr(slots), _ptr(x), _ptr(expert),
                                        _ptr(w), _ptr(kmask), _ptr(gen), _stream(stream))
        N.check(st, "moe_async_enqueue")

    def schedule_step(self, layer, policy, stream=None):
        p = policy.c()
        N.check(self.lib.moe_async_schedule_step(self.h, layer, ctypes.byref(p), _stream(stream)),
                "moe_async_schedule_step")

    def schedule_steps(self, layer, policy, max_steps, stream=None):
        """Up to `max_steps` consecutive steps in one device plan (MTFS / THRESHOLD)."""
        p = policy.c()
        N.check(self.lib.moe_async_schedule_steps(self.h, layer, ctypes.byref(p), max_steps, _stream(stream)),
                "moe_async_schedule_steps")

    def collect(self, layer, y_out, slot_out, n_out, gen_out=None, append=False, max_out=None, stream=None,
                step_out=None):
        max_out = y_out.shape[0] if max_out is None else max_out
        st = self.lib.moe_async_collect(self.h, layer, max_out, _ptr(y_out), _ptr(slot_out), _ptr(gen_out),
                                        _ptr(step_out), _ptr(n_out), int(append), _stream(stream))
        N.check(st, "moe_async_collect")

    def tick(self, layer, policy, x=None, expert=None, w=None, n=None, rows=None, slots=None, kmask=None, gen=None,
             y_out=None, slot_out=None, n_out=None, gen_out=None, step_out=None, append=False, max_out=None,
             stream=None):
        """One serving tick: collect what was ready (into y_out .. n_out, as `collect`; no
        outputs collects nothing) and enqueue a wave (as `enqueue`; no x enqueues nothing) in
        one control launch, then one scheduling step under `policy`."""
        if x is None:
            n = 0
        else:
            n = (rows.shape[0] if rows is not None else x.shape[0]) if n is None else n
        if y_out is None:
            max_out = 0
        else:
            max_out = y_out.shape[0] if max_out is None else max_out
        p = policy.c()
        st = self.lib.moe_async_tick(self.h, layer, n, _ptr(rows), _ptr(slots), _ptr(x), _ptr(expert), _ptr(w),
                                     _ptr(kmask), _ptr(gen), ctypes.byref(p), max_out, _ptr(y_out), _ptr(slot_out),
                                     _ptr(gen_out), _ptr(step_out), _ptr(n_out), int(append), _stream(stream))
        N.check(st, "moe_async_tick")

    def cancel(self, layer, slots, stream=None):
        """Retire the current request of each slot (int32 device tensor of slot ids)."""
        N.check(self.lib.moe_async_cancel(self.h, layer, slots.numel(), _ptr(slots), _stream(stream)),
                "moe_async_cancel")

    def wait(self, layer, policy, max_steps=1000, check_every=4, stream=None):
        p = policy.c()
        return self.lib.moe_async_wait(self.h, layer, ctypes.byref(p), max_steps, check_every, _stream(stream))

    def sync(self, stream=None):
        return self.lib.moe_async_sync(self.h, _stream(stream))

    def stats(self, stream=None):
        s = N.Stats()
        N.check(self.lib.moe_async_get_stats(self.h, _stream(stream), ctypes.byref(s)), "moe_async_get_stats")
        return {f: getattr(s, f) for f, _ in N.Stats._fields_}

    def trace(self, stream=None):
        cap = max(self.trace_capacity, 1)
        buf = (ctypes.c_int32 * (4 * cap))()
        n = ctypes.c_int32()
        N.check(self.lib.moe_async_get_trace(self.h, _stream(stream), buf, cap, ctypes.byref(n)), "trace")
        return np.frombuffer(buf, dtype=np.int32, count=4 * n.value).reshape(n.value, 4).copy()

    def snapshot(self, layer, cap=None, stream=None):
        nb = self.E + (1 if self.has_shared else 0)
        cap = self.S * self.KS if cap is None else cap
        dep = (ctypes.c_int32 * nb)()
        rec = (ctypes.c_int32 * (2 * cap))()
        n = ctypes.c_int32()
        N.check(self.lib.moe_async_snapshot(self.h, layer, _stream(stream), dep, rec, cap, ctypes.byref(n)),
                "snapshot")
        depths = np.frombuffer(dep, dtype=np.int32, count=nb).copy()
        recs = np.frombuffer(rec, dtype=np.int32, count=2 * n.value).reshape(n.value, 2).copy()
        out, o = [], 0
        for b in range(nb):
            out.append(sorted(map(tuple, recs[o:o + depths[b]].tolist())))
            o += depths[b]
        return depths, out

    # -- streaming multi-layer decode (2L micro-queues) --------------------------
    def stream_setup(self, proj, x0, logits, delays, max_steps, stop, history, done_tick, policy="mtfs",
                     window=2, decay=0.5, hist_window=8, admit=None, stream=None):
        """proj: list of L [H, H] device tensors; x0 [R, H]; logits [R, M, E] fp32; delays
        [R, M] int32; admit [R] int32 admission ticks (None: all at the start); history
        [R, M+1, H] and done_tick [R, M+1] int32 are outputs.
        policy: "mtfs" | "flfs" | "defrag" | "barrier" | "defrag_src" (layer-level queue choice)."""
        R = x0.shape[0]
        arr = ctypes.c_void_p * len(proj)
        self._stream_keep = (logits, delays, admit, history, done_tick)
        cfg = N.StreamConfig(R, max_steps, stop, N.STREAM_POLICIES[policy], window, hist_window, decay)
        st = self.lib.moe_async_stream_setup(self.h, ctypes.byref(cfg), arr(*[p.data_ptr() for p in proj]),
                                             _ptr(x0), _ptr(logits), _ptr(delays), _ptr(admit), _ptr(history),
                                             _ptr(done_tick), _stream(stream))
        N.check(st, "moe_async_stream_setup")

    def stream_stats(self, stream=None):
        """Occupancy of the streaming runtime: ticks, merges, peaks and per-queue sums."""
        out = N.StreamStats()
        N.check(self.lib.moe_async_stream_stats(self.h, _stream(stream), ctypes.byref(out)), "stream_stats")
        nq = out.num_queues
        return {"ticks": out.ticks, "combined": out.combined, "peak_transit": out.peak_transit,
                "peak_bucket": out.peak_bucket, "peak_queue": list(out.peak_queue[:nq]),
                "occupancy_sum": list(out.occupancy_sum[:nq])}

    def stream_run(self, max_ticks=100000, check_every=16, stream=None):
        """Run ticks until the stream is drained; returns (status, ticks, merges)."""
        t, c = ctypes.c_int32(), ctypes.c_int32()
        st = self.lib.moe_async_stream_run(self.h, max_ticks, check_every, ctypes.byref(t), ctypes.byref(c),
                                           _stream(stream))
        return st, t.value, c.value

    def stream_trace(self, cap=1 << 18, stream=None):
        buf = (ctypes.c_int32 * (4 * cap))()
        n = ctypes.c_int32()
        N.check(self.lib.moe_async_stream_trace(self.h, _stream(stream), buf, cap, ctypes.byref(n)), "stream_trace")
        return np.frombuffer(buf, dtype=np.int32, count=4 * n.value).reshape(n.value, 4).copy()

    def profile(self, enable=True):
        """Bracket every later kernel launch with CUDA events (per-kernel timing)."""
        N.check(self.lib.moe_async_profile(self.h, int(enable)), "moe_async_profile")

    def profile_read(self, stream=None):
        """{kind: (total_ms, launches)} for the launches recorded since the last read."""
        n = len(N.KERNEL_KINDS)
        ms = (ctypes.c_double * n)()
        cnt = (ctypes.c_int64 * n)()
        N.check(self.lib.moe_async_profile_read(self.h, _stream(stream), ms, cnt, n), "profile_read")
        return {k: (ms[i], cnt[i]) for i, k in enumerate(N.KERNEL_KINDS)}

    def close(self, stream=None):
        if self.h:
            self.lib.moe_async_destroy(self.h, _stream(stream))
            self.h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
