"""ORACLE -- test infrastructure, not part of the product path.

A plain, slow, obviously-correct CPU statement of what asynchronous MoE expert
execution computes, written from the pages' description ("SOSP'26 StreamEP"
sections 3-4; the CascadeEP abstract's streamFFN) and kept free of any code
shared with the CUDA library: no common kernels, headers, helpers or constant
tables.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline may import it.  Arithmetic is float64 on the exact input values.

Every function here is pinned by ``tests/test_oracle_pins.py`` against facts
that do not come from the oracle itself (values printed on the pages,
brute-force enumeration, closed forms, invariants).
"""
from .moe_oracle import (  # noqa: F401
    route, route_bruteforce, silu, expert_ffn, combine, dense_moe,
    mtfs_pick, threshold_pick, defrag_score, AsyncMoEOracle, StepRecord,
    rmsnorm, attention_stub, replay_layer, y_sample, layer_pick, chain_pick, StreamOracle, TickRecord,
)
