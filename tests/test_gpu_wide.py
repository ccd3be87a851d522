"""GPU: items of many tokens run in wide token tiles (128 tokens), small ones in narrow tiles.

A token's output must not depend on the width of the tile it ran in.  Checked on a two-expert
top-2 layer (ragged M and K tails): all 256 tokens in one step (two items of 256 tokens: wide
tiles in both GEMMs), steps of 40 tokens (items of 33..63 tokens: one wide tile, its MMA only
as wide as the item, in both GEMMs) and steps of 32 (narrow tiles in both) give bitwise equal
outputs, and they match the float64 oracle within the bf16 bound.
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as om
from workloads import get_config, make_tokens, make_logits
from workloads.build import make_layer_weights
from tests.gpu_helpers import TOL, rel_err, expert_getter

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as g
    g.build()
    import asynchronous_expert_execution_gb300 as p
    return p


def _run(pkg, spec, wdev, x, idx, w, batch):
    L = spec.layer
    T = spec.tokens
    moe = pkg.MoEAsync(L.num_experts, L.top_k, L.hidden, L.inter, torch.bfloat16, T, weights=[wdev],
                       trace_capacity=4096)
    y = torch.empty(T, L.hidden, dtype=torch.bfloat16, device="cuda")
    sl = torch.empty(T, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    for t0 in range(0, T, batch):
        rows = torch.arange(t0, min(T, t0 + batch), dtype=torch.int32, device="cuda")
        moe.enqueue(0, x, idx, w, rows=rows)
        moe.schedule_step(0, pkg.Policy("mtfs"))
    moe.collect(0, y, sl, n)
    assert moe.sync() == 0
    trace = moe.trace()
    moe.close()
    k = int(n.item())
    assert k == T
    out = np.zeros((T, L.hidden), dtype=np.float32)
    out[sl[:k].cpu().numpy()] = y[:k].float().cpu().numpy()
    return out, trace


def test_wide_tiles_bitwise_equal_to_narrow_and_oracle(pkg):
    spec = get_config("w1")
    L = spec.layer
    T = spec.tokens
    wdev = make_layer_weights(L, 0, device="cuda")
    x = make_tokens(spec, 0, device="cuda").contiguous()
    ii, ww = om.route(make_logits(spec, 0).numpy(), L.top_k)
    idx = torch.tensor(ii, dtype=torch.int32, device="cuda")
    w = torch.tensor(ww, dtype=torch.float32, device="cuda")

    y_wide, tr_wide = _run(pkg, spec, wdev, x, idx, w, T)
    y_mixed, tr_mixed = _run(pkg, spec, wdev, x, idx, w, 40)
    y_narrow, tr_narrow = _run(pkg, spec, wdev, x, idx, w, 32)
    # the premise: one step of two 256-token items; items of 33..63 tokens (one wide tile
    # each, from the wide threshold of 33); items of at most 32 tokens
    assert sorted(c for _, _, _, c in tr_wide.tolist()) == [T, T]
    assert all(33 <= c < 64 for _, _, _, c in tr_mixed.tolist()[:-2])
    assert max(c for _, _, _, c in tr_narrow.tolist()) <= 32

    assert np.array_equal(y_wide.view(np.uint32), y_mixed.view(np.uint32))
    assert np.array_equal(y_wide.view(np.uint32), y_narrow.view(np.uint32))

    ex = expert_getter({k: v.cpu() for k, v in wdev.items()}, L.num_experts)
    ys = om.y_sample(range(T), x.cpu().double().numpy(), ii, ww, ex)
    want = np.stack([ys[t] for t in range(T)])
    err = rel_err(y_wide.astype(np.float64), want)
    assert err <= TOL["bf16"], err
