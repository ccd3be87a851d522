"""GPU: steps with few tiles split each tile over its K chunks across CTAs.

Every tile's product is the ascending-order sum of fixed K-chunk partials, whether its chunks
ran on one CTA or on several, so a token's output must not depend on the step it ran in.
Checked here on a deep-K layer (4 / 2 chunks, ragged K and M tails): the same tokens run in
one wide step (too many tiles to split) and in one-expert steps (split) give bitwise equal
outputs, and both match the float64 oracle within the bf16 bound.
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as om
from workloads import get_config, make_tokens, make_logits
from workloads.build import make_layer_weights
from tests.gpu_helpers import TOL, rel_err, expert_getter

pytestmark = pytest.mark.gpu

# the kernels' rules: a contraction of nk 64-wide k-blocks has 1, 2 or 4 chunks of >= 24
# k-blocks; a launch of n tiles on G CTAs splits all its tiles when n <= 2 G and
# ceil(n c / G) < ceil(n / G) c
def _chunks(nk):
    q = nk // 24
    return 4 if q >= 4 else 2 if q >= 2 else 1


def _split(n, G, c):
    return c > 1 and n <= 2 * G and -(-n * c // G) < -(-n // G) * c


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as g
    g.build()
    import asynchronous_expert_execution_gb300 as p
    return p


def _run(pkg, spec, wdev, x, idx, w, policy):
    L = spec.layer
    T = spec.tokens
    moe = pkg.MoEAsync(L.num_experts, L.top_k, L.hidden, L.inter, torch.bfloat16, T, weights=[wdev],
                       trace_capacity=4096)
    moe.enqueue(0, x, idx, w)
    assert moe.wait(0, policy, max_steps=1000, check_every=1) == 0
    y = torch.empty(T, L.hidden, dtype=torch.bfloat16, device="cuda")
    sl = torch.empty(T, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.collect(0, y, sl, n)
    assert moe.sync() == 0
    trace = moe.trace()
    moe.close()
    k = int(n.item())
    assert k == T
    out = np.zeros((T, L.hidden), dtype=np.float32)
    out[sl[:k].cpu().numpy()] = y[:k].float().cpu().numpy()
    return out, trace


def test_split_k_bitwise_equal_to_whole_and_oracle(pkg):
    spec = get_config("k1")
    L = spec.layer
    T, H, I = spec.tokens, L.hidden, L.inter
    wdev = make_layer_weights(L, 0, device="cuda")
    x = make_tokens(spec, 0, device="cuda").contiguous()
    logits = make_logits(spec, 0)
    ii, ww = om.route(logits.numpy(), L.top_k)
    idx = torch.tensor(ii, dtype=torch.int32, device="cuda")
    w = torch.tensor(ww, dtype=torch.float32, device="cuda")

    y_whole, tr_whole = _run(pkg, spec, wdev, x, idx, w, pkg.Policy("mtfs"))
    y_split, tr_split = _run(pkg, spec, wdev, x, idx, w, pkg.Policy("mtfs", max_groups=1))

    # the premise: the wide step has too many tiles to split, the one-expert steps split
    G = torch.cuda.get_device_properties(0).multi_processor_count
    m1, m2 = -(-2 * I // 128), -(-H // 128)
    c1, c2 = _chunks(-(-H // 64)), _chunks(-(-I // 64))
    assert (c1, c2) == (4, 2)
    steps_w = {}
    for s, _, e, c in tr_whole.tolist():
        steps_w.setdefault(s, []).append(c)
    assert len(steps_w) == 1
    n1 = sum(-(-c // 32) for c in next(iter(steps_w.values()))) * m1
    n2 = n1 // m1 * m2
    assert not _split(n1, G, c1) and not _split(n2, G, c2), (n1, n2)
    per_step = {}
    for s, _, e, c in tr_split.tolist():
        per_step.setdefault(s, []).append(c)
    assert all(len(v) == 1 for v in per_step.values()) and len(per_step) > 1
    for v in per_step.values():
        nt = -(-v[0] // 32)
        assert _split(nt * m1, G, c1) and _split(nt * m2, G, c2)

    assert np.array_equal(y_whole.view(np.uint32), y_split.view(np.uint32))

    ex = expert_getter({k: v.cpu() for k, v in wdev.items()}, L.num_experts)
    ys = om.y_sample(range(T), x.cpu().double().numpy(), ii, ww, ex)
    want = np.stack([ys[t] for t in range(T)])
    err = rel_err(y_split.astype(np.float64), want)
    assert err <= TOL["bf16"], err
