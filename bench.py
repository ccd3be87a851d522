"""Benchmark: routed token-expert pairs/s through asynchronous MoE expert execution.

A step is one pass of the whole hot path over one batch: route the batch's router logits,
deliver its arrival waves on a logical clock (one scheduling step per tick), run every
scheduling step (device-side policy, gathered SwiGLU grouped GEMM, weighted scatter,
readiness-gated merge) and collect the merged outputs.  The workload is the GPT-OSS-120B
shaped decode layer: 128 experts, top-4, H = I = 2880, bf16, 256 tokens in 16 waves with
exponential arrival delays, most-tokens-first scheduling.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c2] [--impl ours|reference]

Prints one JSON line.  With N > 1 (torchrun) every rank runs an independent replica of the
workload (weak scaling, no data-path collective); the timing is the max over ranks.
"""
import argparse
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


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="c2")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--policy", default="mtfs", choices=["mtfs", "flfs", "defrag", "barrier"],
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
    return ap.parse_args()


def policy_name(spec):
    if spec.policy == "ranks":
        return f"ranks (R = {spec.max_groups}, {'with' if spec.fallback_groups else 'no'} stealing)"
    return spec.policy + (f" (G = {spec.max_groups})" if spec.max_groups > 0 else "")


def workload_spec(args):
    from workloads import get_config
    spec = get_config(args.workload)
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
    """nvidia-smi clock/throttle sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        time.sleep(0.25)
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
            out, _ = self.p.communicate()
        sm, mx, reasons = [], [], set()
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
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
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


def traffic_for(kernel):
    """ncu DRAM bytes per launch for `kernel`, if the committed capture matches this source."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("source_hash") != source_hash():
        return None
    k = d.get("kernels", {}).get(kernel)
    return None if k is None else k.get("bytes_per_launch_full_size")


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


class Pass:
    """One full pass of the hot path over the batch (route, waves, steps, collect)."""

    def __init__(self, pkg, spec, moe, waves, dev):
        self.pkg, self.spec, self.moe = pkg, spec, moe
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
        self.route_launches = 0

    def __call__(self, x, logits):
        pkg, moe = self.pkg, self.moe
        pkg.route(logits, self.spec.layer.top_k, self.idx, self.w)
        self.route_launches += 1
        self.n.zero_()
        nxt = 0
        for tick in range(1, self.last_tick + 1):
            while nxt < len(self.waves) and self.waves[nxt].tick <= tick:
                moe.enqueue(0, x, self.idx, self.w, rows=self.rows[nxt])
                nxt += 1
            moe.schedule_step(0, self.policy)
            moe.collect(0, self.y, self.slots, self.n, append=True)
        if self.policy.kind != "mtfs" or self.policy.max_groups > 0:
            # a policy that may leave buckets behind after the last arrival keeps stepping
            # until every token is merged; the host reads the device counters every 32 steps
            # (measured on the DeepSeek-wide threshold workload: every 8 steps -1.4%, every
            # 128 steps about the same as 32, the extra empty steps costing what fewer reads save)
            st = moe.wait(0, self.policy, max_steps=100000, check_every=32)
            assert st == 0, st
            moe.collect(0, self.y, self.slots, self.n, append=True)


# ------------------------------------------------------------ CPU baseline

def oracle_sample(spec, x_host, logits_host, ws_host, waves, budget_s=0.0):
    """Time the oracle as it stands on a bounded sample of the workload: the waves in arrival
    order, each delivered to a fresh oracle and run until its pairs are merged, until
    `budget_s` seconds of oracle time are spent (at least the first wave; only waves whose
    experts are in `ws_host`)."""
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
    pairs, dt, n_waves, n_tokens = 0, 0.0, 0, 0
    for wave in sorted(waves, key=lambda w: w.tick):
        tokens = np.asarray(wave.tokens)
        if len(tokens) == 0:
            continue
        if n_waves > 0 and dt >= budget_s:
            break
        cache = {}

        def experts(e, cache=cache):
            if e not in cache:
                cache[e] = tuple(ws_host[k][e].to(torch.float64).numpy() for k in ("w1", "w3", "w2"))
            return cache[e]

        t0 = time.perf_counter()
        idx, w = om.route(z, L.top_k)
        if not all(int(e) in ws_host["w1"] for e in np.unique(idx[tokens])):
            break                                   # experts not copied to the host: sample ends
        sim = om.AsyncMoEOracle(L.num_experts, L.top_k, x64, experts, has_shared=False,
                                compute=set(tokens.tolist()))
        sim.deliver(tokens, idx, w)
        while sim.pending():
            sim.step(pick)
        dt += time.perf_counter() - t0
        pairs += len(tokens) * L.top_k
        n_waves += 1
        n_tokens += len(tokens)
        del cache, sim
    return pairs, dt, (f"first {n_waves} arriving wave(s): {n_tokens} tokens = {pairs} routed pairs "
                       f"(oracle, float64)")


def host_weights_for_sample(ws, waves, logits_host, K, max_waves=1, max_bytes=8 << 30):
    """Host copies of the experts the first `max_waves` arriving waves route to (the first
    wave always; later waves while the copies stay under `max_bytes`)."""
    from oracle import moe_oracle as om
    idx, _ = om.route(logits_host.numpy(), K)
    per_expert = sum(ws[k][0].numel() * ws[k][0].element_size() for k in ("w1", "w3", "w2"))
    need = set()
    for i, wave in enumerate(sorted(waves, key=lambda w: w.tick)[:max_waves]):
        more = need | set(idx[np.asarray(wave.tokens, dtype=np.int64)].ravel().tolist())
        if i > 0 and len(more) * per_expert > max_bytes:
            break
        need = more
    out = {k: {} for k in ("w1", "w3", "w2")}
    for k in out:
        for e in sorted(need):
            out[k][e] = ws[k][e].cpu()
    return out


# -------------------------------------------------------------------- main

def run_reference(args, rank, world):
    """The oracle on the host cores: each step a bounded sample of the workload."""
    from workloads import get_config, make_tokens, make_logits, make_waves
    spec = workload_spec(args)
    if rank != 0:
        return
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    x, logits, ws, waves = build_inputs(spec, args.seed, dev)
    wh = host_weights_for_sample(ws, waves, logits.cpu(), spec.layer.top_k)
    del ws
    xh, lh = x.cpu(), logits.cpu()
    for _ in range(args.warmup):
        oracle_sample(spec, xh, lh, wh, waves)
    tot_p, tot_t, desc = 0, 0.0, ""
    for _ in range(args.steps):
        p, t, desc = oracle_sample(spec, xh, lh, wh, waves)
        tot_p += p
        tot_t += t
    value = tot_p / tot_t
    cores = os.cpu_count()
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": spec.name, "experts": spec.layer.num_experts, "top_k": spec.layer.top_k,
                       "hidden": spec.layer.hidden, "inter": spec.layer.inter, "tokens": spec.tokens,
                       "waves": spec.num_waves, "policy": policy_name(spec), "sample": desc},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_stream(args, pkg, dev):
    """Streaming multi-layer decode (c5 shape): sustained pairs/s of the device-resident
    runtime under a layer-level policy, with its schedule statistics.  Each step sets the
    stream up again (untimed: projection packing, graph capture) and times the run."""
    from workloads import get_config, make_stream_inputs
    from workloads.build import make_layer_weights
    spec = workload_spec(args)
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
    hist = torch.zeros((R, M + 1, H), dtype=torch.bfloat16, device=dev)
    done = torch.empty((R, M + 1), dtype=torch.int32, device=dev)
    pol = dict(policy=args.policy, window=args.defrag_window, decay=args.defrag_decay,
               hist_window=args.history_window)
    stream = torch.cuda.current_stream()
    times, out = [], None
    for i in range(args.warmup + args.steps):
        moe.stream_setup(proj, x0, logits, delays, M, spec.stream_steps, hist, done, **pol)
        s0 = moe.stats()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        st, ticks, comb = moe.stream_run(max_ticks=100000, check_every=16)
        e1.record(stream)
        torch.cuda.synchronize()
        assert st == 0, st
        s1 = moe.stats()
        if i >= args.warmup:
            times.append(e0.elapsed_time(e1))
            out = (ticks, comb, s1["expert_runs"] - s0["expert_runs"], s1["weight_bytes"] - s0["weight_bytes"],
                   s1["kernel_launches"] - s0["kernel_launches"])
    tr = moe.stream_trace()
    dn = done.cpu().numpy()
    moe.close()
    ticks, comb, runs, wbytes, launches = out
    lat = []
    for r in range(R):
        ts = [0] + [int(t) for t in dn[r, 1:] if t >= 0]
        lat += list(np.diff(ts))
    ms = float(np.median(times))
    pairs = comb * lay.top_k
    hbm, tf_burst, tf_sust, src = peaks()
    exp_passes = int((tr[:, 1] == 2).sum())
    att_passes = int((tr[:, 1] == 1).sum())
    t_roof = (wbytes + att_passes * H * H * 2) / (hbm * 1e9)
    line = {"metric": METRIC, "value": pairs / (ms / 1e3), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": spec.name, "layers": NL, "requests": R, "stop_merges": spec.stream_steps,
                       "policy": args.policy, "defrag_window": args.defrag_window,
                       "defrag_decay": args.defrag_decay, "history_window": args.history_window},
            "schedule": {"ticks": ticks, "merges": comb, "expert_passes": exp_passes, "attention_passes": att_passes,
                         "expert_runs": runs, "weight_bytes": wbytes,
                         "reread_vs_lockstep": exp_passes / max(1, -(-comb // R)),
                         "step_latency_ticks_mean": float(np.mean(lat)),
                         "step_latency_ticks_p99": float(np.percentile(lat, 99))},
            "path_roofline": {"t_roof_ms": 1e3 * t_roof, "frac": 1e3 * t_roof / ms, "peak": hbm,
                              "peak_source": src},
            "gpu_launches": int(launches)}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    from workloads import get_config as _gc
    if _gc(args.workload).num_layers > 1:
        import __graft_entry__ as g
        g.build()
        import asynchronous_expert_execution_gb300 as pkg
        torch.cuda.set_device(local)
        return run_stream(args, pkg, torch.device("cuda", local))

    import __graft_entry__ as g
    g.build()
    import asynchronous_expert_execution_gb300 as pkg
    from workloads import get_config

    assert torch.cuda.is_available(), "bench.py needs a CUDA device"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    spec = workload_spec(args)
    L = spec.layer
    assert args.warmup >= 3, "at least 3 warm-up steps"

    x, logits, ws, waves = build_inputs(spec, args.seed + rank, dev)
    weights = [{k: v for k, v in ws.items()}]
    moe = pkg.MoEAsync(L.num_experts, L.top_k, L.hidden, L.inter, x.dtype, spec.tokens, weights=weights,
                       has_shared=L.has_shared)
    cpu_ws = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu_ws = host_weights_for_sample(ws, waves, logits.cpu(), L.top_k, max_waves=len(waves))
    del weights, ws
    torch.cuda.empty_cache()
    run = Pass(pkg, spec, moe, waves, dev)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
            torch.cuda.synchronize()

    for _ in range(args.warmup):
        run(x, logits)
    assert moe.sync() == 0, "device error during warm-up"
    assert int(run.n.item()) == spec.tokens
    s0 = moe.stats()
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(local)
    barrier()
    clocks.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        run(x, logits)
    ev1.record(stream)
    barrier()
    clk = clocks.stop()
    routed_pairs_step = spec.tokens * L.top_k
    ms, value = aggregate(ev0.elapsed_time(ev1), routed_pairs_step, args.steps, world, dev)
    s1 = moe.stats()
    assert s1["error"] == 0 and int(run.n.item()) == spec.tokens
    pairs_step = (s1["pairs_executed"] - s0["pairs_executed"]) / args.steps
    launches = (s1["kernel_launches"] - s0["kernel_launches"]) + args.steps   # + one route per step

    # per-kernel durations: a second pass of K steps with every launch bracketed by events
    moe.profile(True)
    s2 = moe.stats()
    for _ in range(args.steps):
        run(x, logits)
    prof = moe.profile_read()
    moe.profile(False)
    s3 = moe.stats()
    runs = (s3["expert_runs"] - s2["expert_runs"]) / args.steps
    pairs_p = (s3["pairs_executed"] - s2["pairs_executed"]) / args.steps
    wbytes_step = (s3["weight_bytes"] - s2["weight_bytes"]) / args.steps
    H, I = L.hidden, L.inter
    es = 2 if L.dtype == "bf16" else 4
    # algorithmic bytes per step of each FFN kernel (weights as scheduled + activations)
    alg = {"ffn1": runs * 2 * H * I * es + pairs_p * (H + I) * es,
           "ffn2": runs * H * I * es + pairs_p * I * es + spec.tokens * H * es}
    kern_ms = {k: prof[k][0] / args.steps for k in prof}
    dom = max(("ffn1", "ffn2"), key=lambda k: kern_ms[k])
    hbm, tf_burst, tf_sust, src = peaks()
    launches_dom = prof[dom][1] / args.steps
    achieved = alg[dom] / (kern_ms[dom] / 1e3) / 1e9
    roof = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": achieved / hbm, "peak_source": src,
            "traffic": traffic_for(dom),
            "bytes_per_launch": alg[dom] / launches_dom if launches_dom else None,
            "ms_per_launch": kern_ms[dom] / launches_dom if launches_dom else None}
    # whole FFN + combine path against its as-scheduled roofline
    flops_step = pairs_p * 6 * H * I
    bytes_step = wbytes_step + pairs_p * 2 * H * es + spec.tokens * H * es
    t_roof = max(flops_step / (tf_sust * 1e12), bytes_step / (hbm * 1e9))
    ffn_ms = kern_ms["ffn1"] + kern_ms["ffn2"]
    path = {"t_roof_ms": 1e3 * t_roof, "ffn_combine_ms": ffn_ms, "frac": 1e3 * t_roof / ffn_ms,
            "step_frac": 1e3 * t_roof / (ms / args.steps), "weight_bytes_per_step": wbytes_step,
            "expert_runs_per_step": runs, "flops_per_step": flops_step,
            "kernel_ms_per_step": {k: round(v, 4) for k, v in kern_ms.items()}}

    # end to end through the C ABI from pinned host buffers (H2D inputs, D2H outputs per step)
    xh = x.cpu().pin_memory()
    lh = logits.cpu().pin_memory()
    yh = torch.empty(run.y.shape, dtype=run.y.dtype).pin_memory()
    sh = torch.empty(run.slots.shape, dtype=run.slots.dtype).pin_memory()
    xd, ld = torch.empty_like(x), torch.empty_like(logits)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        xd.copy_(xh, non_blocking=True)
        ld.copy_(lh, non_blocking=True)
        run(xd, ld)
        yh.copy_(run.y, non_blocking=True)
        sh.copy_(run.slots, non_blocking=True)
    e1.record(stream)
    barrier()
    e2e_ms, e2e_value = aggregate(e0.elapsed_time(e1), routed_pairs_step, args.e2e_steps, world, dev)
    h2d = xh.numel() * xh.element_size() + lh.numel() * lh.element_size()
    d2h = yh.numel() * yh.element_size() + sh.numel() * sh.element_size()
    e2e = {"value": e2e_value, "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": args.e2e_steps}

    cpu = None
    if rank == 0 and cpu_ws is not None:
        p, t, desc = oracle_sample(spec, x.cpu(), logits.cpu(), cpu_ws, waves, budget_s=10.0)
        cpu = {"value": p / t, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle", "sample": desc,
               "seconds": t}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": L.dtype, "data": "synthetic",
                "config": {"workload": spec.name, "experts": L.num_experts, "top_k": L.top_k,
                           "hidden": H, "inter": I, "tokens": spec.tokens, "waves": spec.num_waves,
                           "ticks": run.last_tick, "policy": policy_name(spec),
                           "routed_pairs_per_step": routed_pairs_step,
                           "l2": "inputs larger than L2: every step streams the scheduled experts' "
                                 f"weights ({wbytes_step / 1e9:.1f} GB) through HBM",
                           "parallelism": f"replicas x{world}"},
                "roofline": roof, "path_roofline": path, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": int(launches), "clocks": clk}
        print(json.dumps(line), flush=True)
    moe.close()
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
