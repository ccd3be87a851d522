"""Materialise a workload: token vectors, router logits, expert weights, waves.

Weights use the storage convention of the tiny exactness case: W1 and W3 are
[H, I] and W2 is [I, H] per expert (so an expert computes with x @ W1), with
entries N(0, sd = 1/sqrt(fan_in)), fan_in = H for W1/W3 and I for W2.
"""
from dataclasses import dataclass, field
import math

import numpy as np
import torch

from .generators import counter_normal, counter_uniform, to_dtype_exact
from .configs import WorkloadSpec

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}

# stream ids: one per (layer, tensor kind); experts are contiguous counter ranges
_S_X, _S_LOGIT, _S_W1, _S_W3, _S_W2, _S_SW1, _S_SW3, _S_SW2, _S_PROJ = range(9)


def _stream(layer, kind):
    return layer * 32 + kind


@dataclass
class Wave:
    """One arrival wave of routed pairs (a simulated rank's delivery).

    tick   -- logical arrival time: the wave is delivered before the first
              scheduling step whose tick is >= this value.
    tokens -- int64 array of token ids (= request / combine-slot ids) carried.
    rank   -- None: every top-k pair of each carried token is delivered.
              (r, n): only the pairs whose expert e has e % n == r (expert
              parallelism with experts striped over n simulated ranks).
    """
    tick: int
    tokens: np.ndarray
    rank: tuple = None


@dataclass
class Workload:
    spec: WorkloadSpec
    seed: int
    x: torch.Tensor                 # [T, H] workload dtype
    logits: torch.Tensor            # [T, E] float32
    weights: list                   # per layer: dict(w1, w3, w2[, sw1, sw3, sw2])
    waves: list = field(default_factory=list)


def expert_weight_slice(spec_layer, seed, layer, kind, expert, device="cpu"):
    """One expert's weight matrix, regenerated from its counter range."""
    H, I = spec_layer.hidden, spec_layer.inter
    if kind in ("w1", "w3"):
        rows, cols, fan_in = H, I, H
        stream = _stream(layer, _S_W1 if kind == "w1" else _S_W3)
    elif kind == "w2":
        rows, cols, fan_in = I, H, I
        stream = _stream(layer, _S_W2)
    else:
        raise ValueError(kind)
    n = rows * cols
    v = counter_normal(seed, stream, n, offset=expert * n, device=device) / math.sqrt(fan_in)
    return to_dtype_exact(v, spec_layer.dtype).view(rows, cols)


def make_layer_weights(spec_layer, seed, layer=0, device="cpu", experts=None):
    """All routed-expert weights of one layer (generated expert by expert)."""
    E, H, I = spec_layer.num_experts, spec_layer.hidden, spec_layer.inter
    dt = TORCH_DTYPE[spec_layer.dtype]
    ex = range(E) if experts is None else experts
    out = {}
    for kind, shape in (("w1", (H, I)), ("w3", (H, I)), ("w2", (I, H))):
        t = torch.empty((len(ex),) + shape, dtype=dt, device=device)
        for j, e in enumerate(ex):
            t[j] = expert_weight_slice(spec_layer, seed, layer, kind, e, device)
        out[kind] = t
    if spec_layer.has_shared:
        Is = spec_layer.shared_inter
        for kind, shape, stream, fan in (("sw1", (H, Is), _S_SW1, H), ("sw3", (H, Is), _S_SW3, H),
                                         ("sw2", (Is, H), _S_SW2, Is)):
            n = shape[0] * shape[1]
            v = counter_normal(seed, _stream(layer, stream), n, device=device) / math.sqrt(fan)
            out[kind] = to_dtype_exact(v, spec_layer.dtype).view(shape)
    return out


def make_tokens(spec, seed, n=None, offset_tokens=0, device="cpu", layer=0):
    H = spec.layer.hidden
    n = spec.tokens if n is None else n
    v = counter_normal(seed, _stream(layer, _S_X), n * H, offset=offset_tokens * H, device=device)
    return to_dtype_exact(v, spec.layer.dtype).view(n, H)


def make_logits(spec, seed, device="cpu", layer=0):
    """Router logits [T, E] (float32).

    normal : N(0, 1) iid
    uniform: U(0, 1) iid
    zipf   : log p_e + N(0, 1), with expert popularity p_e proportional to
             rank_e^-s and ranks assigned by a seeded permutation of experts.
    """
    T, E = spec.tokens, spec.layer.num_experts
    st = _stream(layer, _S_LOGIT)
    if spec.router == "uniform":
        v = counter_uniform(seed, st, T * E, device=device)
    elif spec.router == "normal":
        v = counter_normal(seed, st, T * E, device=device)
    elif spec.router == "zipf":
        rng = np.random.default_rng([seed, 101, layer])
        ranks = rng.permutation(E) + 1
        p = ranks.astype(np.float64) ** (-spec.zipf_s)
        p /= p.sum()
        logp = torch.tensor(np.log(p), dtype=torch.float64, device=device)
        v = counter_normal(seed, st, T * E, device=device).view(T, E) + logp
    else:
        raise ValueError(spec.router)
    return v.to(torch.float32).view(T, E)


def _largest_remainder(total, fracs):
    raw = np.asarray(fracs, dtype=np.float64) * total
    base = np.floor(raw).astype(np.int64)
    rem = int(total - base.sum())
    order = sorted(range(len(raw)), key=lambda i: (-(raw[i] - base[i]), i))
    for i in order[:rem]:
        base[i] += 1
    return base


def make_waves(spec, seed):
    """Arrival waves for single-layer workloads (see ``Wave``)."""
    T, n = spec.tokens, spec.num_waves
    rng = np.random.default_rng([seed, 202])
    perm = rng.permutation(T)
    if spec.waves == "even":
        groups = np.array_split(perm, n)
    elif spec.waves == "straggler":
        ns = int(round(spec.straggler_frac * T))
        groups = np.array_split(perm[: T - ns], n - 1) + [perm[T - ns:]]
    elif spec.waves == "dirichlet":
        fr = rng.dirichlet(np.full(n, spec.dirichlet_alpha))
        sizes = _largest_remainder(T, fr)
        groups = np.split(perm, np.cumsum(sizes)[:-1])
    elif spec.waves == "ep_rank":
        groups = [np.arange(T) for _ in range(n)]
    else:
        raise ValueError(spec.waves)

    if spec.arrival == "permute":
        ticks = rng.permutation(n) + 1
    elif spec.arrival == "exp":
        ticks = np.maximum(1, np.ceil(rng.exponential(1.0, size=n) * 4.0)).astype(np.int64)
        if spec.waves == "straggler":
            ticks[-1] = ticks[:-1].max() + 1
    elif spec.arrival == "index":
        ticks = np.arange(n) + 1
    else:
        raise ValueError(spec.arrival)

    waves = []
    for i, g in enumerate(groups):
        rank = (i, n) if spec.waves == "ep_rank" else None
        waves.append(Wave(tick=int(ticks[i]), tokens=np.sort(np.asarray(g, dtype=np.int64)), rank=rank))
    return waves


def make_workload(spec, seed=0, device="cpu", weights=True):
    """Single-layer workload: x, logits, weights and waves, all seeded."""
    x = make_tokens(spec, seed, device=device)
    logits = make_logits(spec, seed, device=device)
    ws = [make_layer_weights(spec.layer, seed, 0, device)] if weights else []
    return Workload(spec=spec, seed=seed, x=x, logits=logits, weights=ws, waves=make_waves(spec, seed))


_S_DELAY = 10


@dataclass
class StreamWorkload:
    """Inputs of the streaming multi-layer decode (config c5 and its smaller variants).

    x0      [R, H]        initial request states, N(0, 1)
    proj    [L] x [H, H]  attention-stub projections, N(0, sd 1/sqrt(H))
    weights [L] x dict    routed experts of every layer (as make_layer_weights)
    logits  [R, M, E]     router logits of (request r, step n): U(0, 1) like c2, or with the
                          "zipf" stream router log p + N(0, 1), p the Zipf popularity of the
                          step's layer (n mod L), one seeded expert order per layer
    delays  [R, M]        dispatch delay in ticks: ceil(LogNormal(0, sigma)), at least 1;
                          x slow_factor for requests homed (r mod stream_ranks) on a slow rank
    admit   [R]           tick at which request r enters layer 0's attention queue (0 = at
                          start; bursts of admit_burst requests every admit_gap ticks)
    """
    spec: WorkloadSpec
    seed: int
    max_steps: int
    x0: torch.Tensor
    proj: list
    weights: list
    logits: torch.Tensor
    delays: np.ndarray
    admit: np.ndarray = None


def make_stream_inputs(spec, seed, max_steps, device="cpu", weights=True, requests=None, delay_seed=None):
    L, lay = spec.num_layers, spec.layer
    R = spec.tokens if requests is None else requests
    H, E = lay.hidden, lay.num_experts
    x0 = make_tokens(spec, seed, n=R, device=device)
    proj = []
    for l in range(L):
        v = counter_normal(seed, _stream(l, _S_PROJ), H * H, device=device) / math.sqrt(H)
        proj.append(to_dtype_exact(v, lay.dtype).view(H, H))
    ws = [make_layer_weights(lay, seed, l, device) for l in range(L)] if weights else []
    if spec.stream_router == "zipf":
        noise = counter_normal(seed, _stream(0, _S_LOGIT) + 7, R * max_steps * E, device=device).view(R, max_steps, E)
        logp = torch.empty((L, E), dtype=torch.float64, device=device)
        for l in range(L):
            ranks = np.random.default_rng([seed, 101, l]).permutation(E) + 1
            p = ranks.astype(np.float64) ** (-spec.zipf_s)
            logp[l] = torch.tensor(np.log(p / p.sum()), dtype=torch.float64, device=device)
        layer_of_step = torch.arange(max_steps, device=device) % L
        logits = (noise + logp[layer_of_step][None, :, :]).to(torch.float32)
    else:
        logits = counter_uniform(seed, _stream(0, _S_LOGIT) + 7, R * max_steps * E, device=device)
        logits = logits.to(torch.float32).view(R, max_steps, E)
    z = counter_normal(seed if delay_seed is None else delay_seed, _stream(0, _S_DELAY), R * max_steps).numpy()
    delays = np.maximum(1, np.ceil(np.exp(spec.stream_sigma * z))).astype(np.int32).reshape(R, max_steps)
    if spec.slow_ranks > 0:
        slow = (np.arange(R) % spec.stream_ranks) < spec.slow_ranks
        delays[slow] *= np.int32(spec.slow_factor)
    admit = np.zeros(R, dtype=np.int32)
    if spec.admit_burst > 0:
        admit = ((np.arange(R) // spec.admit_burst) * spec.admit_gap).astype(np.int32)
    return StreamWorkload(spec=spec, seed=seed, max_steps=max_steps, x0=x0, proj=proj, weights=ws,
                          logits=logits, delays=delays, admit=admit)


def shuffled_waves(waves, seed):
    """Same deliveries, re-ordered arrival ticks (for arrival-order invariance)."""
    rng = np.random.default_rng([seed, 303])
    ticks = [w.tick for w in waves]
    perm = rng.permutation(len(waves))
    return [Wave(tick=int(ticks[perm[i]]), tokens=w.tokens.copy(), rank=w.rank) for i, w in enumerate(waves)]


def repartitioned_waves(T, n, seed, first_tick=1):
    """A different partition of all T tokens into n waves at ticks first_tick.. ."""
    rng = np.random.default_rng([seed, 404])
    perm = rng.permutation(T)
    cuts = np.sort(rng.choice(np.arange(1, T), size=n - 1, replace=False)) if n > 1 else []
    groups = np.split(perm, cuts)
    return [Wave(tick=first_tick + i, tokens=np.sort(g.astype(np.int64))) for i, g in enumerate(groups)]
