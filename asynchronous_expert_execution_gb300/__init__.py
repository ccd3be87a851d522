"""Asynchronous MoE expert execution on GB300 (sm_103a).

Routed token vectors arrive in waves tagged (RequestID, LayerID, expert, top-k
weight), are bucketed into per-expert micro-queues, picked by a device-side
scheduler (most-tokens-first or a minimum batch), gathered and run through the
expert SwiGLU FFN as a grouped GEMM, and merged y = sum_j w_j E_j(x) once all K
results of a token have landed ("SOSP'26 StreamEP" sections 3-4; the CascadeEP
abstract's streamFFN).  The compute lives in ``libmoe_async.so`` (C ABI in
``include/moe_async.h``); this package is its thin binding.
"""
from ._native import MoEError, load  # noqa: F401
from .api import MoEAsync, Policy, host_writable, route  # noqa: F401
from .replay import LayerReplay  # noqa: F401
