"""moe_async_forward_noalloc: the allocation-free layer forward, for callers that cannot call
cudaMalloc where they run the layer.  Its output must match the regular asynchronous path
(create / enqueue / schedule / collect) on the same routed batch, on two calls in a row
(the scratch array keeps the previous call's contents)."""
import ctypes

import numpy as np
import pytest
import torch

from workloads import get_config, make_workload

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 2e-2}


def _rel(a, b):
    return float(np.abs(a - b).max() / np.abs(b).max())


@pytest.mark.parametrize("name", ["c1", "m4"])
def test_forward_noalloc_matches_async_path(name):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as g
    g.build()
    import asynchronous_expert_execution_gb300 as pkg
    from asynchronous_expert_execution_gb300 import _native as N
    lib = N.load()
    f = lib.moe_async_forward_noalloc
    f.argtypes = [ctypes.c_int32] * 6 + [ctypes.c_void_p] * 8
    f.restype = ctypes.c_int

    spec = get_config(name)
    L = spec.layer
    T, H = spec.tokens, L.hidden
    wl = make_workload(spec, seed=11)
    dt = wl.x.dtype
    ws = {k: v.cuda().contiguous() for k, v in wl.weights[0].items()}
    x = wl.x.cuda().contiguous()
    idx, w = pkg.route(wl.logits.cuda().contiguous(), L.top_k)

    # the existing entry points: every token delivered at once, run to completion, collected
    moe = pkg.MoEAsync(L.num_experts, L.top_k, H, L.inter, dt, T, weights=[ws])
    moe.enqueue(0, x, idx, w)
    assert moe.wait(0, pkg.Policy(), max_steps=8) == 0
    y_async = torch.empty((T, H), dtype=dt, device="cuda")
    slots = torch.empty(T, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.collect(0, y_async, slots, n)
    assert int(n.item()) == T
    ref = np.empty((T, H))
    ref[slots.cpu().numpy()] = y_async.float().cpu().numpy()
    moe.close()

    dcode = N.MOE_F32 if L.dtype == "f32" else N.MOE_BF16
    for call in range(2):
        y = torch.full((T, H), float("nan"), dtype=dt, device="cuda")
        st = f(T, L.num_experts, L.top_k, H, L.inter, dcode, x.data_ptr(), idx.data_ptr(), w.data_ptr(),
               ws["w1"].data_ptr(), ws["w3"].data_ptr(), ws["w2"].data_ptr(), y.data_ptr(),
               torch.cuda.current_stream().cuda_stream)
        assert st == N.MOE_OK, (call, st)
        torch.cuda.synchronize()
        got = y.float().cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        assert _rel(got, ref) <= TOL[L.dtype], (call, _rel(got, ref))

    # beyond the fixed scratch: rejected, nothing launched
    big = (16 << 20) // (4 * L.top_k * L.inter) + 1
    st = f(big, L.num_experts, L.top_k, H, L.inter, dcode, x.data_ptr(), idx.data_ptr(), w.data_ptr(),
           ws["w1"].data_ptr(), ws["w3"].data_ptr(), ws["w2"].data_ptr(), y.data_ptr(),
           torch.cuda.current_stream().cuda_stream)
    assert st == N.MOE_ERR_CAPACITY
