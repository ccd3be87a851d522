"""Benchmark: routed token-expert pairs/s through asynchronous MoE expert execution.

A step is one pass of the whole hot path over one batch: route the batch's router logits,
deliver its arrival waves on a logical clock (one scheduling step per tick), run every
scheduling step (device-side policy, gathered SwiGLU grouped GEMM, weighted scatter,
readiness-gated merge), drain the queues left after the last arrival, and collect the merged
outputs.  The headline workload is the DeepSeek-style wide layer: 256 routed experts + 1
shared, top-8, H = 7168, I = 2048, bf16, 2048 tokens in 8 Dirichlet(0.5) waves, threshold
scheduling (64 tokens) with a most-tokens-first fallback.  The GPT-OSS decode layer, the Zipf
prefill chunk and the 4-layer streaming decode are measured after it, in the same run, as
sub-records of the same JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c4] [--subconfigs c2,c3,c5]
                  [--impl ours|reference]

Prints one JSON line.  With N > 1 (torchrun) every rank runs an independent replica of the
workload (weak scaling, no data-path collective); the timing is the max over ranks, and the
sub-records are skipped.
"""
import argparse
import ctypes
import dataclasses
import re
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "routed token-expert pairs/sec (expert FFN+combine) at 1 GB300; % of roofline"
UNIT = "pairs/s"


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="c4")
    ap.add_argument("--subconfigs", default="c2,c3,c5",
                    help="workloads measured after the headline one (N = 1 only); '' for none")
    ap.add_argument("--sub-steps", type=int, default=50, help="timed steps of each sub-record")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--fused-tick", action="store_true",
                    help="drive each tick with one moe_async_tick instead of enqueue, schedule_step and collect")
    ap.add_argument("--policy", default="mtfs", choices=["mtfs", "flfs", "defrag", "barrier", "defrag_src"],
                    help="layer-level policy of the streaming workloads (c5, s1)")
    ap.add_argument("--defrag-window", type=int, default=2)
    ap.add_argument("--defrag-decay", type=float, default=0.5)
    ap.add_argument("--history-window", type=int, default=8)
    ap.add_argument("--ranks", type=int, default=0,
                    help="pick policy of the per-layer workloads: R > 0 replaces the workload's policy "
                         "by R simulated expert-parallel ranks (expert e on rank e mod R)")
    ap.add_argument("--no-steal", action="store_true", help="with --ranks: idle ranks do not steal")
    ap.add_argument("--max-groups", type=int, default=-1,
                    help="MTFS / threshold: G >= 0 replaces the workload's bucket limit per step (0 = all)")
    return ap.parse_args(argv)


def policy_name(spec):
    if spec.policy == "ranks":
        return f"ranks (R = {spec.max_groups}, {'with' if spec.fallback_groups else 'no'} stealing)"
    return spec.policy + (f" (G = {spec.max_groups})" if spec.max_groups > 0 else "")


def workload_spec(args, name=None):
    from workloads import get_config
    spec = get_config(name or args.workload)
    if spec.num_layers > 1:
        return spec
    if args.ranks > 0:
        spec = dataclasses.replace(spec, policy="ranks", max_groups=args.ranks,
                                   fallback_groups=0 if args.no_steal else 1)
    elif args.max_groups >= 0:
        spec = dataclasses.replace(spec, max_groups=args.max_groups)
    return spec


# ------------------------------------------------------------------ helpers

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region (every 20 ms)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, interval_ms=20):
        self.gpu = gpu_index
        self.interval = interval_ms
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", str(self.interval)],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.1)                     # the first sample lands before the timed region
        except (OSError, FileNotFoundError):
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        time.sleep(0.05)
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
            out, _ = self.p.communicate()
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            try:
                pw.append(float(f[3]))
            except ValueError:
                pass
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "interval_ms": self.interval, "power_w_max": max(pw) if pw else None,
                "reasons": sorted(reasons)}


KERNEL_SOURCES = ("moe_ffn_tc.cu", "moe_internal.cuh")


def source_hash(files=KERNEL_SOURCES):
    """Hash of the code the FFN kernels are built from (ncu counters go stale when it changes).
    Comments and whitespace are left out, so editing a comment keeps the counters valid."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "asynchronous_expert_execution_gb300", "csrc")
    for f in sorted(files):
        with open(os.path.join(d, f), encoding="utf-8") as fh:
            code = fh.read()
        code = re.sub(r"/\*.*?\*/", " ", code, flags=re.S)        # block comments
        code = re.sub(r"//[^\n]*", " ", code)                       # line comments
        code = " ".join(code.split())
        h.update(f.encode() + code.encode())
    return h.hexdigest()[:16]


def traffic_for(workload, kernel):
    """ncu DRAM bytes per launch of `kernel` on `workload`, if the committed capture matches
    the current kernel source."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("source_hash") != source_hash():
        return None
    k = d.get("workloads", {}).get(workload, {}).get(kernel)
    return None if k is None else k.get("bytes_per_launch")


def aggregate(ms_local, units_per_step, steps, world, device):
    """Whole-job throughput over `world` ranks that each processed `units_per_step` units per
    step for `steps` steps: the slowest rank's time sets the clock (max over ranks), the units
    of all ranks count.  Returns (ms_max, units_per_second)."""
    ms = float(ms_local)
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * units_per_step * steps / (ms / 1e3)


def blas_threads():
    """Threads numpy's BLAS (OpenBLAS) runs with in this process, or None if unknown: read
    from the loaded library through its own query function."""
    seen = set()
    try:
        with open("/proc/self/maps") as f:
            for line in f:
                path = line.split()[-1] if line.split() else ""
                if "openblas" in path.lower() and ".so" in path:
                    seen.add(path)
    except OSError:
        return None
    for path in sorted(seen):
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for sym in ("scipy_openblas_get_num_threads64_", "scipy_openblas_get_num_threads",
                    "openblas_get_num_threads64_", "openblas_get_num_threads"):
            fn = getattr(lib, sym, None)
            if fn is not None:
                fn.restype = ctypes.c_int
                return int(fn())
    return None


# ---------------------------------------------------------------- workload

def build_inputs(spec, seed, dev):
    """Inputs resident in HBM: x, logits, expert weights (generated on the device)."""
    from workloads import make_tokens, make_logits, make_waves
    from workloads.build import expert_weight_slice
    L = spec.layer
    x = make_tokens(spec, seed).to(dev)
    logits = make_logits(spec, seed).to(dev)
    dt = x.dtype
    ws = {}
    for kind, shape in (("w1", (L.hidden, L.inter)), ("w3", (L.hidden, L.inter)), ("w2", (L.inter, L.hidden))):
        t = torch.empty((L.num_experts,) + shape, dtype=dt, device=dev)
        for e in range(L.num_experts):
            t[e] = expert_weight_slice(L, seed, 0, kind, e, device=dev)
        ws[kind] = t
    if L.has_shared:
        from workloads.build import make_layer_weights
        sh = make_layer_weights(L, seed, 0, device=dev, experts=[])
        ws.update({k: sh[k] for k in ("sw1", "sw3", "sw2")})
    return x, logits, ws, make_waves(spec, seed)


# Steps of the drain plan: with nothing arriving, every step takes at least one bucket, so this
# bound never cuts a drain short.
DRAIN_STEPS = 1 << 20


def drain(moe, policy):
    """After the last arrival, the buckets a policy may leave behind run as one device plan of
    consecutive steps (moe_async_schedule_steps, MTFS / threshold), asynchronously like every
    other call of the pass; RANKS steps one at a time through moe_async_wait.  The pass checks
    afterwards that every token was collected."""
    if policy.kind in ("mtfs", "threshold"):
        moe.schedule_steps(0, policy, DRAIN_STEPS)
    else:
        st = moe.wait(0, policy, max_steps=100000, check_every=32)
        assert st == 0, st


class Pass:
    """One full pass of the hot path over the batch (route, waves, steps, drain, collect).

    Each tick: enqueue the tick's waves, one scheduling step, collect what is ready.  fused:
    one ``moe_async_tick`` a tick instead -- the collect of what earlier steps made ready, the
    tick's wave and the step in one control launch, then the step's FFN launches."""

    def __init__(self, pkg, spec, moe, waves, dev, fused=False):
        self.pkg, self.spec, self.moe = pkg, spec, moe
        self.fused = fused
        self.waves = sorted(waves, key=lambda w: w.tick)
        self.rows = [torch.as_tensor(np.asarray(w.tokens, dtype=np.int32), device=dev) for w in self.waves]
        T, L = spec.tokens, spec.layer
        self.idx = torch.empty((T, L.top_k), dtype=torch.int32, device=dev)
        self.w = torch.empty((T, L.top_k), dtype=torch.float32, device=dev)
        self.y = torch.empty((T, L.hidden), dtype=moe.dtype, device=dev)
        self.slots = torch.empty(T, dtype=torch.int32, device=dev)
        self.n = torch.zeros(1, dtype=torch.int32, device=dev)
        self.last_tick = max(w.tick for w in self.waves)
        self.policy = pkg.Policy.from_spec(spec)
        self.drains = self.policy.kind != "mtfs" or self.policy.max_groups > 0

    def __call__(self, x, logits):
        pkg, moe = self.pkg, self.moe
        pkg.route(logits, self.spec.layer.top_k, self.idx, self.w)
        self.n.zero_()
        nxt = 0
        for tick in range(1, self.last_tick + 1):
            due = []
            while nxt < len(self.waves) and self.waves[nxt].tick <= tick:
                due.append(nxt)
                nxt += 1
            if self.fused:
                for i in due[:-1]:
                    moe.enqueue(0, x, self.idx, self.w, rows=self.rows[i])
                wave = dict(x=x, expert=self.idx, w=self.w, rows=self.rows[due[-1]]) if due else {}
                moe.tick(0, self.policy, y_out=self.y, slot_out=self.slots, n_out=self.n, append=True, **wave)
                continue
            for i in due:
                moe.enqueue(0, x, self.idx, self.w, rows=self.rows[i])
            moe.schedule_step(0, self.policy)
            moe.collect(0, self.y, self.slots, self.n, append=True)
        if self.drains:
            drain(moe, self.policy)
        if self.drains or self.fused:
            moe.collect(0, self.y, self.slots, self.n, append=True)


class ArrivalPass:
    """One pass fed from host memory as the waves arrive (the end-to-end measurement): each
    wave's token rows sit packed in pinned host buffers, as a transport delivers them, and a
    side stream copies every wave to the device ahead of need; the router logits of the batch
    are copied and routed first (one launch, as in the resident pass); the tick that delivers
    a wave waits for its rows and enqueues them (slot = token id).  The outputs go to pinned
    host buffers: written there by collect itself when the kernels can address them (each
    merged row crosses the link as it is produced), else copied back after the last collect."""

    def __init__(self, pkg, spec, moe, waves, x_host, logits_host, dev):
        self.pkg, self.spec, self.moe = pkg, spec, moe
        self.waves = sorted(waves, key=lambda w: w.tick)
        T, L = spec.tokens, spec.layer
        tok = [np.asarray(w.tokens, dtype=np.int64) for w in self.waves]
        self.xh = [x_host[torch.as_tensor(t)].contiguous().pin_memory() for t in tok]
        order = torch.as_tensor(np.concatenate(tok))
        self.lh = logits_host[order].contiguous().pin_memory()      # arrival order, like xd
        self.off = np.concatenate([[0], np.cumsum([len(t) for t in tok])]).astype(np.int64)
        self.slot_w = [torch.as_tensor(t.astype(np.int32), device=dev) for t in tok]
        self.xd = torch.empty((T, L.hidden), dtype=x_host.dtype, device=dev)
        self.ld = torch.empty((T, logits_host.shape[1]), dtype=logits_host.dtype, device=dev)
        self.idx = torch.empty((T, L.top_k), dtype=torch.int32, device=dev)
        self.w = torch.empty((T, L.top_k), dtype=torch.float32, device=dev)
        self.y = torch.empty((T, L.hidden), dtype=moe.dtype, device=dev)
        self.slots = torch.empty(T, dtype=torch.int32, device=dev)
        self.n = torch.zeros(1, dtype=torch.int32, device=dev)
        self.yh = torch.empty(self.y.shape, dtype=self.y.dtype).pin_memory()
        self.sh = torch.empty(self.slots.shape, dtype=self.slots.dtype).pin_memory()
        self.last_tick = max(w.tick for w in self.waves)
        self.policy = pkg.Policy.from_spec(spec)
        self.drains = self.policy.kind != "mtfs" or self.policy.max_groups > 0
        self.copy_stream = torch.cuda.Stream(device=dev)
        self.ready = [torch.cuda.Event() for _ in self.waves]
        self.direct = pkg.host_writable(self.yh) and pkg.host_writable(self.sh)

    def h2d_bytes(self):
        return sum(t.numel() * t.element_size() for t in self.xh) + self.lh.numel() * self.lh.element_size()

    def d2h_bytes(self):
        return self.yh.numel() * self.yh.element_size() + self.sh.numel() * self.sh.element_size()

    def __call__(self):
        pkg, moe, K = self.pkg, self.moe, self.spec.layer.top_k
        main = torch.cuda.current_stream()
        cs = self.copy_stream
        cs.wait_stream(main)                     # the previous pass is done with the staging rows
        with torch.cuda.stream(cs):
            for i in range(len(self.waves)):
                a, b = int(self.off[i]), int(self.off[i + 1])
                self.xd[a:b].copy_(self.xh[i], non_blocking=True)
                self.ready[i].record(cs)
        self.ld.copy_(self.lh, non_blocking=True)
        pkg.route(self.ld, K, self.idx, self.w)
        self.n.zero_()
        y_out, s_out = (self.yh, self.sh) if self.direct else (self.y, self.slots)
        nxt = 0
        for tick in range(1, self.last_tick + 1):
            while nxt < len(self.waves) and self.waves[nxt].tick <= tick:
                a, b = int(self.off[nxt]), int(self.off[nxt + 1])
                main.wait_event(self.ready[nxt])
                moe.enqueue(0, self.xd[a:b], self.idx[a:b], self.w[a:b], slots=self.slot_w[nxt])
                nxt += 1
            moe.schedule_step(0, self.policy)
            moe.collect(0, y_out, s_out, self.n, append=True)
        if self.drains:
            drain(moe, self.policy)
            moe.collect(0, y_out, s_out, self.n, append=True)
        if not self.direct:
            self.yh.copy_(self.y, non_blocking=True)
            self.sh.copy_(self.slots, non_blocking=True)


def schedule_independent_bytes(spec, logits):
    """Weight bytes of one pass if every expert the batch touches were read once (the
    schedule-independent bound), from the routing of the batch."""
    from oracle import moe_oracle as om            # routing ids only; the same rule as the kernels
    L = spec.layer
    es = 2 if L.dtype == "bf16" else 4
    idx, _ = om.route(logits.cpu().numpy(), L.top_k)
    touched = len(np.unique(idx)) + (1 if L.has_shared else 0)
    return touched, touched * 3 * L.hidden * L.inter * es


# ------------------------------------------------------------ CPU baseline

def oracle_sample_tokens(spec, logits_host, waves, max_bytes=4 << 30):
    """The first tokens in arrival order whose experts' weights fit `max_bytes` of host copies."""
    from oracle import moe_oracle as om
    L = spec.layer
    idx, _ = om.route(logits_host.numpy(), L.top_k)
    per_expert = 3 * L.hidden * L.inter * (2 if L.dtype == "bf16" else 4)
    tokens, need = [], set()
    for wave in sorted(waves, key=lambda w: w.tick):
        for t in wave.tokens:
            more = need | set(int(e) for e in idx[int(t)])
            if tokens and (len(more) + (1 if L.has_shared else 0)) * per_expert > max_bytes:
                return tokens, need
            tokens.append(int(t))
            need = more
    return tokens, need


def host_weights(ws, experts, has_shared):
    out = {k: {e: ws[k][e].cpu() for e in sorted(experts)} for k in ("w1", "w3", "w2")}
    if has_shared:
        out["shared"] = tuple(ws[k].cpu() for k in ("sw1", "sw3", "sw2"))
    return out


def oracle_sample(spec, x_host, logits_host, wh, tokens, budget_s=0.0):
    """Time the oracle as it stands on a bounded sample of the workload: the sample tokens
    delivered to a fresh oracle and run until every pair is merged under the workload's
    policy, repeated until `budget_s` seconds of oracle time are spent (at least once).  The
    oracle converts the bf16 weights it is handed to float64 itself (inside the timing)."""
    from oracle import moe_oracle as om
    L = spec.layer
    if spec.policy == "ranks":
        pick = lambda d: om.rank_pick(d, spec.max_groups, spec.fallback_groups != 0)
    elif spec.policy == "threshold":
        pick = lambda d: om.threshold_pick(d, spec.min_batch, spec.max_groups, spec.fallback_groups)
    else:
        pick = lambda d: om.mtfs_pick(d, spec.max_groups)
    x64 = x_host.to(torch.float64).numpy()
    z = logits_host.numpy()
    pairs, dt, reps = 0, 0.0, 0
    while reps == 0 or dt < budget_s:
        t0 = time.perf_counter()

        def experts(e):
            if e == L.num_experts:
                return tuple(m.to(torch.float64).numpy() for m in wh["shared"])
            return tuple(wh[k][e].to(torch.float64).numpy() for k in ("w1", "w3", "w2"))
        idx = np.zeros((z.shape[0], L.top_k), dtype=np.int64)
        w = np.zeros((z.shape[0], L.top_k))
        idx[tokens], w[tokens] = om.route(z[tokens], L.top_k)      # only the sample is routed
        sim = om.AsyncMoEOracle(L.num_experts, L.top_k, x64, experts, has_shared=L.has_shared,
                                compute=set(tokens))
        sim.deliver(tokens, idx, w)
        while sim.pending():
            sim.step(pick)
        dt += time.perf_counter() - t0
        pairs += len(tokens) * L.top_k
        reps += 1
        del sim
    threads = blas_threads()
    desc = (f"the first {len(tokens)} arriving tokens ({len(tokens) * L.top_k} routed pairs"
            f"{' + shared' if L.has_shared else ''}), run to completion by a fresh oracle {reps} time(s); "
            f"float64 numpy, BLAS threads: {threads if threads is not None else 'unknown'}")
    return pairs, dt, desc, threads


# ------------------------------------------------------------ measurement

def measure_layer(args, pkg, spec, dev, rank, world, steps, warmup, e2e_steps, with_cpu):
    """Time `steps` passes of a one-layer workload (inputs resident), then a second pass of
    `steps` with every launch bracketed by events (per-kernel times), then `e2e_steps` passes
    end to end from pinned host buffers.  Returns the record of this workload."""
    L = spec.layer
    x, logits, ws, waves = build_inputs(spec, args.seed + rank, dev)
    moe = pkg.MoEAsync(L.num_experts, L.top_k, L.hidden, L.inter, x.dtype, spec.tokens, weights=[ws],
                       has_shared=L.has_shared)
    cpu_in = None
    if with_cpu:
        tokens, need = oracle_sample_tokens(spec, logits.cpu(), waves)
        cpu_in = (tokens, host_weights(ws, need, L.has_shared))
    del ws
    torch.cuda.empty_cache()
    run = Pass(pkg, spec, moe, waves, dev, fused=args.fused_tick)
    drain_by = (None if not run.drains else "moe_async_schedule_steps (one device plan)"
                if run.policy.kind in ("mtfs", "threshold") else "moe_async_wait")

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
            torch.cuda.synchronize()

    for _ in range(warmup):
        run(x, logits)
    assert moe.sync() == 0, "device error during warm-up"
    assert int(run.n.item()) == spec.tokens
    s0 = moe.stats()
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(torch.cuda.current_device())
    barrier()
    clocks.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        run(x, logits)
    ev1.record(stream)
    barrier()
    clk = clocks.stop()
    routed_pairs_step = spec.tokens * L.top_k
    ms, value = aggregate(ev0.elapsed_time(ev1), routed_pairs_step, steps, world, dev)
    s1 = moe.stats()
    assert s1["error"] == 0 and int(run.n.item()) == spec.tokens
    launches = (s1["kernel_launches"] - s0["kernel_launches"]) + steps   # + one route per step

    # per-kernel durations: a second pass of K steps with every launch bracketed by events
    moe.profile(True)
    s2 = moe.stats()
    for _ in range(steps):
        run(x, logits)
    prof = moe.profile_read()
    moe.profile(False)
    s3 = moe.stats()
    runs = (s3["expert_runs"] - s2["expert_runs"]) / steps
    pairs_p = (s3["pairs_executed"] - s2["pairs_executed"]) / steps
    wbytes_step = (s3["weight_bytes"] - s2["weight_bytes"]) / steps
    H, I = L.hidden, L.inter
    es = 2 if L.dtype == "bf16" else 4
    # algorithmic bytes per step of each FFN kernel (weights as scheduled + activations)
    # GEMM2: weights and h in; its bf16 result rows are an implementation cost, and y is
    # written by collect's merge
    alg = {"ffn1": runs * 2 * H * I * es + pairs_p * (H + I) * es,
           "ffn2": runs * H * I * es + pairs_p * I * es}
    kern_ms = {k: prof[k][0] / steps for k in prof}
    dom = max(("ffn1", "ffn2"), key=lambda k: kern_ms[k])
    hbm, tf_burst, tf_sust, src = peaks()
    launches_dom = prof[dom][1] / steps
    achieved = alg[dom] / (kern_ms[dom] / 1e3) / 1e9
    roof = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": achieved / hbm, "peak_source": src,
            "traffic": traffic_for(spec.name, dom),
            "bytes_per_launch": alg[dom] / launches_dom if launches_dom else None,
            "ms_per_launch": kern_ms[dom] / launches_dom if launches_dom else None,
            "launches_per_step": launches_dom}
    # whole FFN + combine path against its roofline: as scheduled (the weights of every expert
    # run of every step) and schedule-independent (each touched expert's weights once)
    flops_step = pairs_p * 6 * H * I
    act_bytes = pairs_p * (H * es + 12) + spec.tokens * H * es      # gathered rows, records, y
    bytes_step = wbytes_step + act_bytes
    touched, w_indep = schedule_independent_bytes(spec, logits)
    t_roof = max(flops_step / (tf_sust * 1e12), bytes_step / (hbm * 1e9))
    t_indep = max(flops_step / (tf_sust * 1e12), (w_indep + act_bytes) / (hbm * 1e9))
    ffn_ms = kern_ms["ffn1"] + kern_ms["ffn2"]
    step_ms = ms / steps
    path = {"t_roof_ms": 1e3 * t_roof, "ffn_combine_ms": ffn_ms, "frac": 1e3 * t_roof / ffn_ms,
            "step_frac": 1e3 * t_roof / step_ms, "weight_bytes_per_step": wbytes_step,
            "expert_runs_per_step": runs, "flops_per_step": flops_step,
            "schedule_independent": {"experts_touched": touched, "weight_bytes": w_indep,
                                     "t_roof_ms": 1e3 * t_indep, "frac": 1e3 * t_indep / ffn_ms,
                                     "step_frac": 1e3 * t_indep / step_ms},
            "weight_reread_factor": wbytes_step / w_indep,
            "kernel_ms_per_step": {k: round(v, 4) for k, v in kern_ms.items()}}

    # end to end through the C ABI from pinned host buffers: every step copies each wave's
    # packed rows and logits to the device as it arrives (side stream, ahead of need) and reads
    # the outputs back after its last collect
    arr = ArrivalPass(pkg, spec, moe, waves, x.cpu(), logits.cpu(), dev)
    arr()                                        # one untimed pass (allocations, first copies)
    barrier()
    assert moe.sync() == 0 and int(arr.n.item()) == spec.tokens
    assert sorted(arr.sh.tolist()) == list(range(spec.tokens))
    # token by token (the completion order may differ), the host copies equal the outputs of
    # the resident pass: the same picks and values
    oa, ob = torch.argsort(arr.sh.long()), torch.argsort(run.slots.cpu().long())
    assert torch.equal(arr.yh[oa], run.y.cpu()[ob]), "end-to-end pass differs from the resident pass"
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        arr()
    e1.record(stream)
    barrier()
    assert moe.sync() == 0 and int(arr.n.item()) == spec.tokens
    e2e_ms, e2e_value = aggregate(e0.elapsed_time(e1), routed_pairs_step, e2e_steps, world, dev)
    e2e = {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": arr.h2d_bytes(),
           "d2h_bytes_per_step": arr.d2h_bytes(), "steps": e2e_steps,
           "copies": "router logits host to device first; each wave's token rows host to device on a "
                     "side stream as it arrives; outputs " + ("written to pinned host memory by collect as "
                     "each token completes" if arr.direct else "device to host after the last collect")}

    cpu = None
    if cpu_in is not None:
        tokens, wh = cpu_in
        p, t, desc, threads = oracle_sample(spec, x.cpu(), logits.cpu(), wh, tokens, budget_s=10.0)
        cpu = {"value": p / t, "unit": UNIT, "cores": threads if threads is not None else os.cpu_count(),
               "host_cores": os.cpu_count(), "kind": "oracle", "sample": desc, "seconds": t}
    moe.close()
    del x, logits, moe, run
    torch.cuda.empty_cache()
    return {"workload": spec.name, "value": value, "unit": UNIT, "steps": steps, "warmup": warmup,
            "ms_per_step": step_ms, "dtype": L.dtype,
            "config": {"workload": spec.name, "experts": L.num_experts, "shared_expert": L.has_shared,
                       "top_k": L.top_k, "hidden": H, "inter": I, "tokens": spec.tokens,
                       "waves": spec.num_waves, "ticks": run_ticks(waves), "policy": policy_name(spec),
                       "routed_pairs_per_step": routed_pairs_step,
                       "ticks_driven_by": "moe_async_tick" if args.fused_tick
                       else "moe_async_enqueue + moe_async_schedule_step + moe_async_collect",
                       "drain": drain_by,
                       "l2": "inputs larger than L2: every step streams the scheduled experts' "
                             f"weights ({wbytes_step / 1e9:.1f} GB) through HBM"},
            "roofline": roof, "path_roofline": path, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": int(launches), "clocks": clk}


def run_ticks(waves):
    return max(w.tick for w in waves)


def measure_stream(args, pkg, spec, dev, steps, warmup, e2e_steps):
    """Streaming multi-layer decode (c5 shape): sustained pairs/s of the device-resident
    runtime under a layer-level policy, with its schedule statistics.  Each step sets the
    stream up again (untimed: projection packing, graph capture) and times the run; the end
    to end figure times the setup and run together with the host copies of the inputs and
    of the outputs (the per-request history and completion ticks)."""
    from workloads import make_stream_inputs
    from workloads.build import make_layer_weights
    lay = spec.layer
    R, H, NL, M = spec.tokens, lay.hidden, spec.num_layers, 64
    wl = make_stream_inputs(spec, args.seed, M, weights=False)
    weights = [make_layer_weights(lay, args.seed, l, device=dev) for l in range(NL)]
    moe = pkg.MoEAsync(lay.num_experts, lay.top_k, H, lay.inter, torch.bfloat16, R, weights=weights,
                       num_layers=NL)
    del weights
    torch.cuda.empty_cache()
    proj = [p.to(dev) for p in wl.proj]
    x0, logits = wl.x0.to(dev), wl.logits.to(dev)
    delays = torch.as_tensor(wl.delays, dtype=torch.int32).to(dev)
    admit = torch.as_tensor(wl.admit, dtype=torch.int32).to(dev) if wl.admit.any() else None
    hist = torch.zeros((R, M + 1, H), dtype=torch.bfloat16, device=dev)
    done = torch.empty((R, M + 1), dtype=torch.int32, device=dev)
    pol = dict(policy=args.policy, window=args.defrag_window, decay=args.defrag_decay,
               hist_window=args.history_window, admit=admit)
    stream = torch.cuda.current_stream()
    times, out = [], None
    clk = None
    clocks = ClockSampler(torch.cuda.current_device())
    for i in range(warmup + steps):
        moe.stream_setup(proj, x0, logits, delays, M, spec.stream_steps, hist, done, **pol)
        s0 = moe.stats()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        if i == warmup:
            clocks.start()
        e0.record(stream)
        st, ticks, comb = moe.stream_run(max_ticks=100000, check_every=16)
        e1.record(stream)
        torch.cuda.synchronize()
        assert st == 0, st
        s1 = moe.stats()
        if i >= warmup:
            times.append(e0.elapsed_time(e1))
            out = (ticks, comb, s1["expert_runs"] - s0["expert_runs"], s1["weight_bytes"] - s0["weight_bytes"],
                   s1["kernel_launches"] - s0["kernel_launches"])
    clk = clocks.stop()
    tr = moe.stream_trace()
    occ = moe.stream_stats()
    dn = done.cpu().numpy()
    # end to end: inputs from pinned host memory, setup + run, outputs back to pinned memory
    x0h, lh, dh = x0.cpu().pin_memory(), logits.cpu().pin_memory(), delays.cpu().pin_memory()
    hh = torch.empty(hist.shape, dtype=hist.dtype).pin_memory()
    doh = torch.empty(done.shape, dtype=done.dtype).pin_memory()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    comb_e2e = 0
    for _ in range(e2e_steps):
        x0.copy_(x0h, non_blocking=True)
        logits.copy_(lh, non_blocking=True)
        delays.copy_(dh, non_blocking=True)
        moe.stream_setup(proj, x0, logits, delays, M, spec.stream_steps, hist, done, **pol)
        st, _, c = moe.stream_run(max_ticks=100000, check_every=16)
        assert st == 0, st
        hh.copy_(hist, non_blocking=True)
        doh.copy_(done, non_blocking=True)
        comb_e2e += c
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0
    moe.close()
    ticks, comb, runs, wbytes, launches = out
    lat, req_mean, req_steps = [], [], []
    for r in range(R):
        ts = [int(wl.admit[r])] + [int(t) for t in dn[r, 1:] if t >= 0]
        d = np.diff(ts)
        lat += list(d)
        req_steps.append(len(d))
        req_mean.append(float(np.mean(d)) if len(d) else None)
    ms = float(np.median(times))
    pairs = comb * lay.top_k
    hbm, tf_burst, tf_sust, src = peaks()
    exp_passes = int((tr[:, 1] == 2).sum())
    att_passes = int((tr[:, 1] == 1).sum())
    t_roof = (wbytes + att_passes * H * H * 2) / (hbm * 1e9)
    # schedule-independent (lockstep) bound: a cohort of R requests advances one layer per
    # expert pass, so ceil(merges / R) passes each read every touched expert of the layer once
    passes_lockstep = -(-comb // R)
    w_lockstep = passes_lockstep * lay.num_experts * 3 * H * lay.inter * 2
    t_lock = (w_lockstep + passes_lockstep * H * H * 2) / (hbm * 1e9)
    del proj, x0, logits, delays, hist, done
    torch.cuda.empty_cache()
    return {"workload": spec.name, "value": pairs / (ms / 1e3), "unit": UNIT, "steps": steps, "warmup": warmup,
            "ms_per_step": ms, "dtype": "bf16",
            "config": {"workload": spec.name, "layers": NL, "requests": R, "stop_merges": spec.stream_steps,
                       "policy": args.policy, "defrag_window": args.defrag_window,
                       "defrag_decay": args.defrag_decay, "history_window": args.history_window},
            "schedule": {"ticks": ticks, "merges": comb, "expert_passes": exp_passes, "attention_passes": att_passes,
                         "expert_runs": runs, "weight_bytes": wbytes,
                         "reread_vs_lockstep": exp_passes / max(1, passes_lockstep),
                         "step_latency_ticks_mean": float(np.mean(lat)),
                         "step_latency_ticks_p99": float(np.percentile(lat, 99))},
            "path_roofline": {"t_roof_ms": 1e3 * t_roof, "frac": 1e3 * t_roof / ms, "peak": hbm,
                              "peak_source": src,
                              "schedule_independent": {"lockstep_passes": passes_lockstep,
                                                       "weight_bytes": w_lockstep, "t_roof_ms": 1e3 * t_lock,
                                                       "frac": 1e3 * t_lock / ms},
                              "weight_reread_factor": wbytes / w_lockstep},
            "e2e": {"value": comb_e2e * lay.top_k / e2e_s, "unit": UNIT,
                    "h2d_bytes_per_step": x0h.numel() * 2 + lh.numel() * 4 + dh.numel() * 4,
                    "d2h_bytes_per_step": hh.numel() * 2 + doh.numel() * 4, "steps": e2e_steps,
                    "includes": "stream setup (projection packing, graph capture) and run, host copies"},
            "study": stream_study(spec, lay, ticks, comb, lat, req_mean, req_steps, tr, occ, ms, pairs,
                                  1e3 * t_roof / ms),
            "gpu_launches": int(launches), "clocks": clk}


SLO_TICKS = 8      # per-step latency target of the study's goodput (ticks, mean over a request)


def stream_study(spec, lay, ticks, comb, lat, req_mean, req_steps, tr, occ, ms, pairs, roof_frac):
    """The latency study's figures for one streaming run ("asynchronous MoE serving" notes,
    second research candidate): accepted load, goodput under a per-step latency target, tail
    step latency, request completion, queue and bucket occupancy, and how busy the GPU was."""
    R = spec.tokens
    ms_tick = ms / max(1, ticks)
    ok = [r for r in range(R) if req_mean[r] is not None and req_mean[r] <= SLO_TICKS]
    busy_ticks = int((tr[:, 1] != 0).sum()) if len(tr) else 0
    nq = len(occ["peak_queue"])
    return {
        "accepted_load": {"merges_per_tick": comb / max(1, ticks), "pairs_per_s": pairs / (ms / 1e3)},
        "step_latency_ticks": {"mean": float(np.mean(lat)), "p50": float(np.percentile(lat, 50)),
                               "p99": float(np.percentile(lat, 99)), "max": int(np.max(lat))},
        "step_latency_ms_gpu": {"p50": float(np.percentile(lat, 50)) * ms_tick,
                                "p99": float(np.percentile(lat, 99)) * ms_tick},
        "goodput": {"slo_mean_step_ticks": SLO_TICKS, "requests_meeting_frac": len(ok) / R,
                    "pairs_per_s": sum(req_steps[r] for r in ok) * lay.top_k / (ms / 1e3),
                    "merges_per_tick": sum(req_steps[r] for r in ok) / max(1, ticks)},
        "completion": {"steps_min": int(min(req_steps)), "steps_median": float(np.median(req_steps)),
                       "steps_max": int(max(req_steps)), "requests_served_frac": sum(1 for n in req_steps if n) / R},
        "occupancy": {"peak_queue": occ["peak_queue"],
                      "mean_queue": [round(v / max(1, occ["ticks"]), 2) for v in occ["occupancy_sum"]],
                      "peak_in_transit": occ["peak_transit"], "peak_bucket": occ["peak_bucket"],
                      "queues": [f"{'att' if q % 2 == 0 else 'exp'}_{q // 2}" for q in range(nq)]},
        "busy_ticks_frac": busy_ticks / max(1, ticks),
        "gpu_roofline_frac": roof_frac,
        "ms_per_tick": ms_tick}


# -------------------------------------------------------------------- main

def run_reference(args, rank, world):
    """The oracle on the host cores: each step a bounded sample of the workload."""
    spec = workload_spec(args)
    if rank != 0:
        return
    if spec.num_layers > 1:
        print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the oracle on the "
                          "one-layer workloads; pass --workload c1..c4"}), flush=True)
        return
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    x, logits, ws, waves = build_inputs(spec, args.seed, dev)
    tokens, need = oracle_sample_tokens(spec, logits.cpu(), waves)
    wh = host_weights(ws, need, spec.layer.has_shared)
    del ws
    xh, lh = x.cpu(), logits.cpu()
    for _ in range(args.warmup):
        oracle_sample(spec, xh, lh, wh, tokens)
    tot_p, tot_t, desc, threads = 0, 0.0, "", None
    for _ in range(args.steps):
        p, t, desc, threads = oracle_sample(spec, xh, lh, wh, tokens)
        tot_p += p
        tot_t += t
    value = tot_p / tot_t
    cores = threads if threads is not None else os.cpu_count()
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": spec.name, "experts": spec.layer.num_experts, "top_k": spec.layer.top_k,
                       "hidden": spec.layer.hidden, "inter": spec.layer.inter, "tokens": spec.tokens,
                       "waves": spec.num_waves, "policy": policy_name(spec), "sample": desc},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "host_cores": os.cpu_count(),
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    assert args.warmup >= 3, "at least 3 warm-up steps"
    import __graft_entry__ as g
    g.build()
    import asynchronous_expert_execution_gb300 as pkg

    assert torch.cuda.is_available(), "bench.py needs a CUDA device"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    spec = workload_spec(args)
    if spec.num_layers > 1:
        rec = measure_stream(args, pkg, spec, dev, args.steps, args.warmup, args.e2e_steps)
    else:
        rec = measure_layer(args, pkg, spec, dev, rank, world, args.steps, args.warmup, args.e2e_steps,
                            with_cpu=rank == 0 and not args.no_cpu_baseline)
    subs = {}
    if world == 1 and args.subconfigs:
        for name in [n for n in args.subconfigs.split(",") if n and n != args.workload]:
            sp = workload_spec(args, name)
            if sp.num_layers > 1:
                subs[name] = measure_stream(args, pkg, sp, dev, max(1, args.sub_steps // 5), args.warmup,
                                            max(1, args.e2e_steps // 10))
            else:
                subs[name] = measure_layer(args, pkg, sp, dev, rank, world, args.sub_steps, args.warmup,
                                           args.e2e_steps, with_cpu=False)
    if rank == 0:
        line = {"metric": METRIC, "value": rec["value"], "unit": UNIT, "n_gpus": world, "steps": rec["steps"],
                "warmup": rec["warmup"], "ms_per_step": rec["ms_per_step"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": rec["dtype"], "data": "synthetic",
                "config": dict(rec["config"], parallelism=f"replicas x{world}")}
        for k, v in rec.items():                     # roofline, e2e, cpu_baseline, clocks, schedule, study ...
            if k not in line and k not in ("workload",):
                line[k] = v
        if subs:
            line["subconfigs"] = subs
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
