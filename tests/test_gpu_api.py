"""GPU: API surface around the hot path -- a handle with two layers used through the
per-layer calls (each layer its own weights, queues and outputs), and the combinations the
library rejects (cancellation on a handle running the streaming runtime)."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as om
from workloads import get_config, make_tokens, make_logits, make_stream_inputs
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


def _collect(pkg, moe, layer, T, H):
    y = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    sl = torch.empty(T, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.collect(layer, y, sl, n)
    assert moe.sync() == 0
    k = int(n.item())
    out = np.full((T, H), np.nan)
    out[sl[:k].cpu().numpy()] = y[:k].float().cpu().numpy()
    return k, out


def test_two_layer_handle_layers_independent(pkg):
    spec = get_config("m4")                       # 64 experts, top-4, H 1024, I 512, bf16
    L = spec.layer
    T, H = spec.tokens, L.hidden
    w = [make_layer_weights(L, 0, layer=l, device="cuda") for l in range(2)]
    xs = [make_tokens(spec, 0, layer=l, device="cuda").contiguous() for l in range(2)]
    routes = [om.route(make_logits(spec, 0, layer=l).numpy(), L.top_k) for l in range(2)]

    def run(layers):
        moe = pkg.MoEAsync(L.num_experts, L.top_k, H, L.inter, torch.bfloat16, T, weights=w, num_layers=2)
        for l in layers:
            ii, ww = routes[l]
            moe.enqueue(l, xs[l], torch.tensor(ii, dtype=torch.int32, device="cuda"),
                        torch.tensor(ww, dtype=torch.float32, device="cuda"))
        for l in layers:
            moe.schedule_step(l, pkg.Policy("mtfs"))
        out = {l: _collect(pkg, moe, l, T, H) for l in (0, 1)}
        moe.close()
        return out

    both = run([0, 1])
    only0 = run([0])
    for l in (0, 1):
        k, got = both[l]
        assert k == T
        ii, ww = routes[l]
        ex = expert_getter({kk: v.cpu() for kk, v in w[l].items()}, L.num_experts)
        ys = om.y_sample(range(T), xs[l].cpu().double().numpy(), ii, ww, ex)
        want = np.stack([ys[t] for t in range(T)])
        assert rel_err(got, want) <= TOL["bf16"]
    # layer 0's results do not depend on layer 1's traffic; an unused layer emits nothing
    assert np.array_equal(both[0][1].view(np.uint64), only0[0][1].view(np.uint64))
    assert only0[1][0] == 0


def test_stream_mode_rejects_cancel(pkg):
    spec = get_config("s1")
    lay = spec.layer
    R, H, NL, M = spec.tokens, lay.hidden, spec.num_layers, 4
    wl = make_stream_inputs(spec, 0, M, weights=False)
    weights = [make_layer_weights(lay, 0, l, device="cuda") for l in range(NL)]
    moe = pkg.MoEAsync(lay.num_experts, lay.top_k, H, lay.inter, torch.bfloat16, R, weights=weights,
                       num_layers=NL)
    hist = torch.zeros((R, M + 1, H), dtype=torch.bfloat16, device="cuda")
    done = torch.empty((R, M + 1), dtype=torch.int32, device="cuda")
    moe.stream_setup([p.cuda() for p in wl.proj], wl.x0.cuda(), wl.logits.cuda(),
                     torch.as_tensor(wl.delays, dtype=torch.int32).cuda(), M, spec.stream_steps, hist, done)
    with pytest.raises(pkg.MoEError) as ei:
        moe.cancel(0, torch.zeros(1, dtype=torch.int32, device="cuda"))
    assert ei.value.status == 7                    # MOE_ERR_UNSUPPORTED
    st, ticks, comb = moe.stream_run(max_ticks=100000, check_every=16)
    assert st == 0 and comb > 0                    # the handle is still usable
    moe.close()
