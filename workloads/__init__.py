"""Seeded synthetic inputs for asynchronous MoE expert execution.

This module is shared by the CPU oracle and by the GPU harness (tests and the
benchmark).  It holds *no* arithmetic of the method itself: no routing, no
expert FFN, no combine, no scheduling.  It only draws the raw inputs -- token
vectors, expert weights, router logits and the arrival-wave schedule -- in the
shapes and distributions of the workloads the pages describe (GPT-OSS-120B's
128-expert top-4 hidden-2880 layer as in "SOSP'26 StreamEP", section 3; a
DeepSeek-style wide layer; a tiny exactness case).

Float inputs come from a counter-based generator written with plain torch
integer/float64 ops, so the same element index yields the same value on the
CPU and on a CUDA device.  That lets a GPU run generate multi-gigabyte weight
tensors in place while the oracle regenerates (or copies) just the slices it
needs.  Discrete schedule draws (permutations, wave sizes, arrival ticks) use
numpy's PCG64 on the host.
"""
from .generators import counter_uniform, counter_normal, to_dtype_exact  # noqa: F401
from .configs import (  # noqa: F401
    LayerSpec, WorkloadSpec, CONFIGS, TEST_CONFIGS, get_config,
)
from .build import (  # noqa: F401
    Workload, Wave, make_workload, make_layer_weights, expert_weight_slice, make_tokens,
    make_logits, make_waves, shuffled_waves, repartitioned_waves, StreamWorkload, make_stream_inputs,
)
