"""Workload descriptions: shapes, distributions and arrival structure.

The five named workloads follow the synthetic configurations the build is
measured on (a tiny fp32 exactness case, a GPT-OSS-120B-shaped decode layer, a
skewed prefill chunk with a straggler wave, a DeepSeek-style wide layer with a
shared expert, and a streaming multi-layer decode).  The ``TEST_CONFIGS`` are
smaller cases for element-by-element parity: they span several GEMM tiles in
every dimension and leave ragged tails (H and 2I not multiples of 128, H and I
not multiples of 64).
"""
from dataclasses import dataclass, replace


@dataclass(frozen=True)
class LayerSpec:
    num_experts: int          # E routed experts
    top_k: int                # K
    hidden: int               # H
    inter: int                # I (SwiGLU intermediate)
    dtype: str                # "f32" | "bf16"
    has_shared: bool = False  # one always-on shared expert, weight 1
    shared_inter: int = 0     # its intermediate size (must equal `inter`)


@dataclass(frozen=True)
class WorkloadSpec:
    name: str
    layer: LayerSpec
    tokens: int                       # T tokens (one per request slot)
    router: str                       # "normal" | "uniform" | "zipf"
    zipf_s: float = 1.2
    waves: str = "even"               # "even" | "straggler" | "dirichlet" | "ep_rank"
    num_waves: int = 4
    arrival: str = "permute"          # "permute" | "exp" | "index"
    straggler_frac: float = 0.30
    dirichlet_alpha: float = 0.5
    policy: str = "mtfs"              # "mtfs" | "threshold" | "ranks" (max_groups = ranks, fallback_groups != 0 = steal)
    min_batch: int = 64
    max_groups: int = 0               # 0 = all qualifying buckets
    fallback_groups: int = 1
    num_layers: int = 1
    # streaming multi-layer decode (config "c5")
    stream_steps: int = 0             # stop after this many combined token-layer steps
    stream_ranks: int = 16
    stream_sigma: float = 1.0
    # delay regimes of the streaming decode: burst admission of requests (admit_burst requests
    # every admit_gap ticks; 0 = all at tick 0), skewed expert load (router "zipf": logits =
    # log-popularity + N(0, 1), one popularity order per layer), and delayed simulated ranks
    # (the requests homed on the first slow_ranks of stream_ranks ranks get slow_factor x
    # their dispatch delays)
    stream_router: str = "uniform"
    admit_burst: int = 0
    admit_gap: int = 0
    slow_ranks: int = 0
    slow_factor: int = 1
    notes: str = ""


GPT_OSS_LAYER = LayerSpec(num_experts=128, top_k=4, hidden=2880, inter=2880, dtype="bf16")

CONFIGS = {
    "c1": WorkloadSpec(
        name="c1_tiny_fp32", layer=LayerSpec(8, 2, 64, 128, "f32"), tokens=32,
        router="normal", waves="even", num_waves=4, arrival="permute", policy="mtfs",
        notes="1 MoE layer, 8 experts, top-2, H=64, I=128, fp32, 32 tokens, 4 random-order waves"),
    "c2": WorkloadSpec(
        name="c2_gptoss_decode", layer=GPT_OSS_LAYER, tokens=256,
        router="uniform", waves="even", num_waves=16, arrival="exp", policy="mtfs",
        notes="128 experts top-4 H=I=2880 bf16, 256 decode tokens, 16 waves, exp delays, MTFS"),
    "c3": WorkloadSpec(
        name="c3_gptoss_prefill_zipf", layer=GPT_OSS_LAYER, tokens=4096,
        router="zipf", zipf_s=1.2, waves="straggler", num_waves=16, arrival="exp",
        straggler_frac=0.30, policy="mtfs",
        notes="4096-token prefill chunk, Zipf(1.2) popularity, 15 waves + a 30% straggler last"),
    "c4": WorkloadSpec(
        name="c4_deepseek_wide_shared",
        layer=LayerSpec(256, 8, 7168, 2048, "bf16", has_shared=True, shared_inter=2048),
        tokens=2048, router="normal", waves="dirichlet", num_waves=8, arrival="index",
        dirichlet_alpha=0.5, policy="threshold", min_batch=64, fallback_groups=1,
        notes="256 routed + 1 shared expert, top-8, H=7168, I=2048, 2048 tokens, Dirichlet(0.5) waves"),
    "c5": WorkloadSpec(
        name="c5_streaming_4layer", layer=GPT_OSS_LAYER, tokens=512, router="uniform",
        waves="stream", num_waves=16, arrival="lognormal", policy="mtfs", num_layers=4,
        stream_steps=10000, stream_ranks=16, stream_sigma=1.0,
        notes="4 layers of the c2 shape, 512 requests, RMSNorm+projection attention stub"),
    # the streaming decode under three delay regimes (its policy and latency study)
    "c5b": WorkloadSpec(
        name="c5b_streaming_burst", layer=GPT_OSS_LAYER, tokens=512, router="uniform",
        waves="stream", num_waves=16, arrival="lognormal", policy="mtfs", num_layers=4,
        stream_steps=10000, stream_ranks=16, stream_sigma=1.0, admit_burst=128, admit_gap=8,
        notes="c5 with requests admitted in bursts of 128 every 8 ticks"),
    "c5s": WorkloadSpec(
        name="c5s_streaming_skewed", layer=GPT_OSS_LAYER, tokens=512, router="uniform",
        waves="stream", num_waves=16, arrival="lognormal", policy="mtfs", num_layers=4,
        stream_steps=10000, stream_ranks=16, stream_sigma=1.0, stream_router="zipf",
        notes="c5 with Zipf(1.2) expert popularity per layer"),
    "c5d": WorkloadSpec(
        name="c5d_streaming_delayed_ranks", layer=GPT_OSS_LAYER, tokens=512, router="uniform",
        waves="stream", num_waves=16, arrival="lognormal", policy="mtfs", num_layers=4,
        stream_steps=10000, stream_ranks=16, stream_sigma=1.0, slow_ranks=2, slow_factor=4,
        notes="c5 with 2 of 16 simulated ranks delivering 4x later"),
}

# Smaller cases for element-by-element parity (several tiles + ragged tails).
TEST_CONFIGS = {
    # bf16, GEMM1 M = 2I = 416 (3 tiles + 32), K = H = 584 (9 k-blocks + 8);
    # GEMM2 M = H = 584 (4 tiles + 72), K = I = 208 (3 k-blocks + 16).
    "m1": WorkloadSpec(
        name="m1_bf16_ragged", layer=LayerSpec(16, 4, 584, 208, "bf16"), tokens=200,
        router="normal", waves="even", num_waves=5, arrival="exp", policy="mtfs"),
    # bf16 with a shared expert and the threshold policy; one expert gets > 256 rows.
    "m2": WorkloadSpec(
        name="m2_bf16_shared_threshold",
        layer=LayerSpec(24, 6, 320, 192, "bf16", has_shared=True, shared_inter=192),
        tokens=600, router="zipf", zipf_s=1.2, waves="dirichlet", num_waves=6,
        arrival="index", policy="threshold", min_batch=40, fallback_groups=1),
    # fp32 with ragged shapes (SIMT path), pairs split across waves by EP rank.
    "m3": WorkloadSpec(
        name="m3_f32_ep_rank", layer=LayerSpec(12, 3, 136, 80, "f32"), tokens=96,
        router="normal", waves="ep_rank", num_waves=4, arrival="permute", policy="mtfs"),
    # profiling-sized slice of the GPT-OSS layer: 32 experts of H = I = 2880 (1.6 GB of
    # weights, well above L2), 64 decode tokens in 4 waves -- same kernels, same tile shapes.
    "p1": WorkloadSpec(
        name="p1_gptoss_slice", layer=GPT_OSS_LAYER.__class__(32, 4, 2880, 2880, "bf16"), tokens=64,
        router="uniform", waves="even", num_waves=4, arrival="index", policy="mtfs"),
    # profiling-sized slice of the skewed prefill layer: 32 GPT-OSS experts, Zipf(1.2)
    # popularity, 2048 tokens -- the popular experts get hundreds of rows per step.
    "p3": WorkloadSpec(
        name="p3_gptoss_prefill_slice", layer=GPT_OSS_LAYER.__class__(32, 4, 2880, 2880, "bf16"), tokens=2048,
        router="zipf", zipf_s=1.2, waves="even", num_waves=4, arrival="index", policy="mtfs"),
    # profiling-sized slice of the DeepSeek-wide layer: 32 of its experts + the shared expert
    # (2.9 GB of weights, well above L2), 320 tokens so each routed expert gets ~80, one wave,
    # threshold 64 -- the shapes of that layer's big step in one launch pair.
    "p4": WorkloadSpec(
        name="p4_deepseek_wide_slice",
        layer=LayerSpec(32, 8, 7168, 2048, "bf16", has_shared=True, shared_inter=2048), tokens=320,
        router="normal", waves="even", num_waves=1, arrival="index", policy="threshold", min_batch=64,
        fallback_groups=1),
    # streaming multi-layer decode, small: 4 layers, ragged H (2.5 tiles of 128), 48 requests.
    "s1": WorkloadSpec(
        name="s1_stream_small", layer=LayerSpec(16, 4, 320, 192, "bf16"), tokens=48, router="uniform",
        waves="stream", num_waves=16, arrival="lognormal", policy="mtfs", num_layers=4,
        stream_steps=150, stream_ranks=16, stream_sigma=1.0),
    # the small stream with all three regimes at once: bursts of 12 requests every 5 ticks,
    # Zipf routing, ranks 0-2 of 8 four times slower
    "s1x": WorkloadSpec(
        name="s1x_stream_small_regimes", layer=LayerSpec(16, 4, 320, 192, "bf16"), tokens=48,
        router="uniform", waves="stream", num_waves=16, arrival="lognormal", policy="mtfs", num_layers=4,
        stream_steps=150, stream_ranks=8, stream_sigma=1.0, stream_router="zipf", admit_burst=12,
        admit_gap=5, slow_ranks=3, slow_factor=4),
    # deep K, split over K chunks when a step has few tiles: H = 6136 (96 k-blocks, the last
    # 56 wide -> 4 chunks of 24), I = 3088 (49 k-blocks, the last 16 wide -> 2 chunks of
    # 24/25), 2I = 6176 (48 tiles + 32 rows), H = 47 tiles + 120 rows.
    "k1": WorkloadSpec(
        name="k1_bf16_deep_k", layer=LayerSpec(8, 2, 6136, 3088, "bf16"), tokens=32,
        router="normal", waves="even", num_waves=1, arrival="index", policy="mtfs"),
    # wide token tiles: 2 experts, top-2, so each item holds every token (256 >= the wide
    # threshold of 128); H = 1000 and 2I = 992 leave ragged M and K tails.
    "w1": WorkloadSpec(
        name="w1_bf16_wide_tiles", layer=LayerSpec(2, 2, 1000, 496, "bf16"), tokens=256,
        router="normal", waves="even", num_waves=1, arrival="index", policy="mtfs"),
    # the m1 layer under simulated expert-parallel ranks: 4 ranks with work stealing, and 5
    # ranks (uneven ownership) without.
    "r1": WorkloadSpec(
        name="r1_bf16_ranks_steal", layer=LayerSpec(16, 4, 584, 208, "bf16"), tokens=200,
        router="normal", waves="even", num_waves=5, arrival="exp", policy="ranks", max_groups=4,
        fallback_groups=1),
    "r2": WorkloadSpec(
        name="r2_bf16_ranks_no_steal", layer=LayerSpec(16, 4, 584, 208, "bf16"), tokens=200,
        router="normal", waves="even", num_waves=5, arrival="exp", policy="ranks", max_groups=5,
        fallback_groups=0),
    # degenerate rank counts: one rank (one bucket a step, deepest first) and more ranks than
    # buckets (every non-empty bucket runs on its owner; the extra ranks find nothing to steal)
    "r3": WorkloadSpec(
        name="r3_bf16_one_rank", layer=LayerSpec(16, 4, 584, 208, "bf16"), tokens=200,
        router="normal", waves="even", num_waves=5, arrival="exp", policy="ranks", max_groups=1,
        fallback_groups=1),
    "r4": WorkloadSpec(
        name="r4_bf16_more_ranks_than_buckets", layer=LayerSpec(16, 4, 584, 208, "bf16"), tokens=200,
        router="normal", waves="even", num_waves=5, arrival="exp", policy="ranks", max_groups=24,
        fallback_groups=1),
    # bf16 decode-like: many experts, few tokens each.
    "m4": WorkloadSpec(
        name="m4_bf16_decode", layer=LayerSpec(64, 4, 1024, 512, "bf16"), tokens=64,
        router="uniform", waves="even", num_waves=8, arrival="exp", policy="mtfs"),
}


def get_config(name, **overrides):
    spec = CONFIGS.get(name) or TEST_CONFIGS.get(name)
    if spec is None:
        raise KeyError(name)
    return replace(spec, **overrides) if overrides else spec
