"""moe_async_forward_noalloc: the allocation-free layer forward, for callers that cannot call
cudaMalloc where they run the layer (a memory pool that owns the device, an allocation-free
runtime, a plugin handed only its buffers).  Its output is compared with the CPU oracle,
element by element (or on a seeded token sample at the GPT-OSS decode shape), on two calls in
a row: the scratch array is shared by every call and keeps the previous call's contents.

This file is collected last, so a run that stops at its first failure has already run every
other test; it passes alone in a fresh process and after the others."""
import ctypes

import numpy as np
import pytest
import torch

from oracle import moe_oracle as om
from workloads import LayerSpec, WorkloadSpec, get_config, make_workload, make_tokens, make_logits
from workloads.build import expert_weight_slice

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 2e-2}
SCRATCH_BYTES = 16 << 20


def _rel(a, b):
    return float(np.abs(a - b).max() / np.abs(b).max())


@pytest.fixture(scope="module")
def api():
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
    return pkg, N, f


def _call(api, T, L, x, idx, w, ws, y):
    pkg, N, f = api
    dcode = N.MOE_F32 if L.dtype == "f32" else N.MOE_BF16
    return f(T, L.num_experts, L.top_k, L.hidden, L.inter, dcode, x.data_ptr(), idx.data_ptr(), w.data_ptr(),
             ws["w1"].data_ptr(), ws["w3"].data_ptr(), ws["w2"].data_ptr(), y.data_ptr(),
             torch.cuda.current_stream().cuda_stream)


def _two_calls(api, spec, x, idx, w, ws, want, rows=None):
    """Two calls in a row, each compared with the oracle rows `want` (all rows, or `rows`)."""
    pkg, N, f = api
    L = spec.layer
    T, H = spec.tokens, L.hidden
    for call in range(2):
        y = torch.full((T, H), float("nan"), dtype=x.dtype, device="cuda")
        st = _call(api, T, L, x, idx, w, ws, y)
        assert st == N.MOE_OK, (call, st)
        torch.cuda.synchronize()
        got = y.float().cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        if rows is not None:
            got = got[rows]
        assert _rel(got, want) <= TOL[L.dtype], (call, _rel(got, want))


def _small_spec(name, E, K, H, I, T, dtype):
    return WorkloadSpec(name=name, layer=LayerSpec(E, K, H, I, dtype), tokens=T, router="normal",
                        waves="even", num_waves=1, arrival="index", policy="mtfs")


@pytest.mark.parametrize("case", ["c1", "m4", "ragged_f32", "ragged_bf16", "grid_loops"])
def test_forward_noalloc_matches_oracle(api, case):
    pkg, N, f = api
    if case in ("c1", "m4"):
        spec = get_config(case)
    elif case == "ragged_f32":
        spec = _small_spec("ragged", 6, 2, 200, 72, 40, "f32")        # H, I not multiples of 128
    elif case == "ragged_bf16":
        spec = _small_spec("ragged", 6, 3, 200, 72, 40, "bf16")
    else:
        # T * K pairs above the 65535 grid rows of the first kernel and T above those of the
        # second, so both kernels' row loops run more than once; T*K*I*4 = 13.4 MB fits
        spec = _small_spec("grid", 4, 2, 16, 24, 70000, "f32")
    L = spec.layer
    wl = make_workload(spec, seed=11)
    ws = {k: v.cuda().contiguous() for k, v in wl.weights[0].items()}
    x = wl.x.cuda().contiguous()
    idx, w = pkg.route(wl.logits.cuda().contiguous(), L.top_k)
    ii, ww = idx.cpu().numpy().astype(np.int64), w.cpu().numpy().astype(np.float64)
    if case == "ragged_f32":
        # an expert id outside [0, E) contributes nothing (no handle holds an error here)
        idx[0, 1] = -1
        idx[1, 0] = L.num_experts
        ww = ww.copy()
        ww[0, 1] = 0.0
        ww[1, 0] = 0.0
    ex = lambda e: tuple(wl.weights[0][k][e].double().numpy() for k in ("w1", "w3", "w2"))
    want = om.dense_moe(wl.x.double().numpy(), ii, ww, ex)
    _two_calls(api, spec, x, idx, w, ws, want)


def test_forward_noalloc_gpt_oss_decode_shape(api):
    """The GPT-OSS decode shape (256 tokens, top-4 of 128 experts, H = I = 2880, bf16) fills
    11.8 of the 16 MiB of scratch; the oracle computes a seeded sample of tokens one by one."""
    pkg, N, f = api
    spec = get_config("c2")
    L = spec.layer
    T = spec.tokens
    assert T * L.top_k * L.inter * 4 <= SCRATCH_BYTES
    ws = {}
    for kind, shape in (("w1", (L.hidden, L.inter)), ("w3", (L.hidden, L.inter)), ("w2", (L.inter, L.hidden))):
        t = torch.empty((L.num_experts,) + shape, dtype=torch.bfloat16, device="cuda")
        for e in range(L.num_experts):
            t[e] = expert_weight_slice(L, 0, 0, kind, e, device="cuda")
        ws[kind] = t
    xh = make_tokens(spec, 0)
    x = xh.cuda().contiguous()
    idx, w = pkg.route(make_logits(spec, 0).cuda().contiguous(), L.top_k)
    ii, ww = idx.cpu().numpy().astype(np.int64), w.cpu().numpy().astype(np.float64)
    sample = sorted(np.random.default_rng(5).choice(T, size=12, replace=False).tolist())
    experts = lambda e: tuple(ws[k][e].to("cpu", torch.float64).numpy() for k in ("w1", "w3", "w2"))
    ys = om.y_sample(sample, xh.double().numpy(), ii, ww, experts)
    want = np.stack([ys[t] for t in sample])
    _two_calls(api, spec, x, idx, w, ws, want, rows=sample)
    del ws
    torch.cuda.empty_cache()


def test_forward_noalloc_rejects_beyond_scratch(api):
    """T*K*I*4 bytes above the fixed scratch: MOE_ERR_CAPACITY, nothing launched, and the
    next call that fits still works."""
    pkg, N, f = api
    spec = get_config("m4")
    L = spec.layer
    wl = make_workload(spec, seed=3)
    ws = {k: v.cuda().contiguous() for k, v in wl.weights[0].items()}
    x = wl.x.cuda().contiguous()
    idx, w = pkg.route(wl.logits.cuda().contiguous(), L.top_k)
    y = torch.empty((spec.tokens, L.hidden), dtype=x.dtype, device="cuda")
    big = SCRATCH_BYTES // (4 * L.top_k * L.inter) + 1
    assert _call(api, big, L, x, idx, w, ws, y) == N.MOE_ERR_CAPACITY
    ii, ww = idx.cpu().numpy().astype(np.int64), w.cpu().numpy().astype(np.float64)
    ex = lambda e: tuple(wl.weights[0][k][e].double().numpy() for k in ("w1", "w3", "w2"))
    want = om.dense_moe(wl.x.double().numpy(), ii, ww, ex)
    _two_calls(api, spec, x, idx, w, ws, want)
