"""Cases for the bounds-checked build (libmoe_async_debug.so).  Not collected on their own:
tests/test_gpu_debug_bounds.py runs them, with a few parity tests, in a child process whose
environment sets MOE_DEBUG_BOUNDS=1 so that the bounds-checked library is the one loaded.

A record planted with an out-of-range slot or k is rejected by every kernel family that reads
records (tcgen05 bf16, CUDA-core fp32, identity): MOE_ERR_BOUNDS is latched, nothing out of
range is read or written, and every real token still comes out equal to the oracle."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as om
from workloads import LayerSpec, WorkloadSpec, make_workload
from tests.gpu_helpers import TOL, rel_err, expert_getter, by_token

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import asynchronous_expert_execution_gb300 as p
    from asynchronous_expert_execution_gb300 import _native as N
    assert N.DEBUG_BOUNDS and N.LIB_PATH.endswith("libmoe_async_debug.so"), "run with MOE_DEBUG_BOUNDS=1"
    return p


@pytest.mark.parametrize("dtype,kind,shared,via", [("bf16", "swiglu", False, "step"), ("bf16", "swiglu", True, "step"),
                                                   ("f32", "swiglu", False, "step"), ("f32", "identity", False, "step"),
                                                   ("bf16", "swiglu", True, "tick")])
def test_planted_out_of_range_records_are_rejected(pkg, dtype, kind, shared, via):
    from asynchronous_expert_execution_gb300 import _native as N
    T, E, K, H, I = 48, 8, 2, 136, 80
    spec = WorkloadSpec(name="bounds", layer=LayerSpec(E, K, H, I, dtype, has_shared=shared, shared_inter=I),
                        tokens=T, router="normal", waves="even", num_waves=1, arrival="index", policy="mtfs")
    wl = make_workload(spec, seed=6)
    ws = [{k: v.cuda().contiguous() for k, v in wl.weights[0].items()}] if kind == "swiglu" else None
    S = T + 8                                                      # room in h for the planted rows
    moe = pkg.MoEAsync(E, K, H, I, wl.x.dtype, S, weights=ws, has_shared=shared, expert_kind=kind)
    x = wl.x.cuda().contiguous()
    idx, w = pkg.route(wl.logits.cuda().contiguous(), K)
    moe.enqueue(0, x, idx, w)
    KS = K + (1 if shared else 0)
    bad = [((S + 3) << 5) | 0,            # slot beyond max_slots
           (0 << 5) | 31,                 # a real slot with k beyond K (+ shared)
           ((1 << 25) << 5) | 1]          # slot far beyond (still a positive int32)
    for b, rec in zip((0, 3, E - 1), bad):
        N.check(moe.lib.moe_async_debug_append_record(moe.h, 0, b, rec, None), "append")
    if via == "tick":                                              # the step from moe_async_tick
        moe.tick(0, pkg.Policy())
    else:
        moe.schedule_step(0, pkg.Policy())
    y = torch.empty((T, H), dtype=x.dtype, device="cuda")
    slots = torch.empty(T, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.collect(0, y, slots, n)
    assert moe.sync() == N.MOE_ERR_BOUNDS
    assert int(n.item()) == T                                     # every real token completed
    got = by_token(slots.cpu().numpy(), y.float().cpu().numpy().astype(np.float64), T, H)
    ii, ww = idx.cpu().numpy().astype(np.int64), w.cpu().numpy().astype(np.float64)
    xs = wl.x.double().numpy()
    if kind == "identity":
        want = (ww.sum(1) + (1.0 if shared else 0.0))[:, None] * xs
    else:
        get = expert_getter(wl.weights[0], E)
        want = om.dense_moe(xs, ii, ww, get, shared=get(E) if shared else None)
    assert rel_err(got, want) <= TOL[dtype], rel_err(got, want)
    # the scheduler halts after the error: a later step picks nothing
    moe.enqueue(0, x, idx, w, rows=torch.tensor([0], dtype=torch.int32, device="cuda"),
                gen=torch.ones(1, dtype=torch.int32, device="cuda"))
    before = moe.stats()["pairs_executed"]
    moe.schedule_step(0, pkg.Policy())
    assert moe.stats()["pairs_executed"] == before
    moe.close()


def test_step_rows_beyond_activation_buffer_are_rejected(pkg):
    """An in-range record planted once too often (a second copy of a real pair) makes the
    step's gathered rows exceed the h buffer of max_slots x K rows: the scheduler latches
    MOE_ERR_BOUNDS and runs nothing instead of writing past h."""
    from asynchronous_expert_execution_gb300 import _native as N
    T, E, K, H, I = 32, 4, 2, 64, 64
    spec = WorkloadSpec(name="bounds_h", layer=LayerSpec(E, K, H, I, "bf16"), tokens=T, router="normal",
                        waves="even", num_waves=1, arrival="index", policy="mtfs")
    wl = make_workload(spec, seed=7)
    ws = [{k: v.cuda().contiguous() for k, v in wl.weights[0].items()}]
    moe = pkg.MoEAsync(E, K, H, I, wl.x.dtype, T, weights=ws)
    x = wl.x.cuda().contiguous()
    idx, w = pkg.route(wl.logits.cuda().contiguous(), K)
    moe.enqueue(0, x, idx, w)                                      # T x K rows: h is full
    e0 = int(idx[0, 0].item())
    N.check(moe.lib.moe_async_debug_append_record(moe.h, 0, e0, (0 << 5) | 0, None), "append")
    moe.schedule_step(0, pkg.Policy())
    assert moe.sync() == N.MOE_ERR_BOUNDS
    st = moe.stats()
    assert st["pairs_executed"] == 0 and st["tokens_combined"] == 0
    moe.close()
