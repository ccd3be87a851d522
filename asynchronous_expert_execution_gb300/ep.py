"""Expert-parallel exchange across ranks: the multi-GPU split of the path.

"SOSP'26 StreamEP" section 3: a token lives on its home rank, which routes it; each of its K
(expert, weight) pairs goes to the rank holding that expert; the result w * E(x) returns home,
where the top-k merge holds the first K-1 results and releases y = sum_k w_k E_k(x) only when
the K-th has landed.  Section 5: ranks exchange a small metadata message first (how many
pairs, and which (token, k, expert, weight) each carries), then the tensor payload, so every
receiver sizes its buffers before any data arrives.

This module is that exchange on torch.distributed (NCCL between GPUs, gloo on the CPU):

* experts are split over ranks in contiguous ranges, expert e on rank e * world // E;
* ``dispatch`` sends each rank's home pairs to their owners: counts, then metadata, then the
  token rows (three collectives, in that order);
* ``give_back`` returns the owners' weighted results along the reversed splits;
* ``Readiness`` is the home side's gate: each (token, k) result is accepted exactly once, and
  a token is released once all K have landed, never earlier.

The arithmetic is not here: the owner's expert FFN and the home merge are the caller's (on a
GPU, the library's grouped GEMM and merge; in the CPU test, the oracle's).  Every run of this
build has one GPU, so the module is exercised by two gloo ranks on the CPU only.
"""
import torch
import torch.distributed as dist

# metadata columns of one pair
META_HOME, META_TOKEN, META_K, META_EXPERT, META_W = range(5)
META_COLS = 5


def owner_of(expert, num_experts, world):
    """Rank holding expert `expert` (contiguous ranges: rank r holds [r E / world, (r+1) E / world))."""
    return (expert * world) // num_experts


def local_experts(rank, num_experts, world):
    """Experts held by `rank`, in ascending order."""
    return [e for e in range(num_experts) if owner_of(e, num_experts, world) == rank]


class EPExchange:
    """The pair exchange of one expert-parallel layer among the ranks of `group`."""

    def __init__(self, num_experts, top_k, hidden, group=None):
        self.E, self.K, self.H = num_experts, top_k, hidden
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)

    def _a2a(self, out, inp, out_splits, in_splits):
        dist.all_to_all_single(out, inp, out_splits, in_splits, group=self.group)

    def dispatch(self, tokens, x, idx, w, kmask=None):
        """Send the home pairs of `tokens` (global ids [n]; rows x [n, H], idx / w [n, K]) to the
        ranks owning their experts; `kmask` [n, K] bool selects the pairs carried (a wave may
        carry some of a token's pairs).  Returns what this rank received as owner: metadata
        [m, 5] float64 (home rank, token, k, expert, weight), rows [m, H], and the per-source
        counts (needed to send the results back)."""
        n = tokens.shape[0]
        sel = torch.ones((n, self.K), dtype=torch.bool) if kmask is None else kmask.bool()
        t_idx, k_idx = torch.nonzero(sel, as_tuple=True)
        experts = idx[t_idx, k_idx].long()
        dest = (experts * self.world) // self.E
        order = torch.argsort(dest, stable=True)               # grouped by destination rank
        t_idx, k_idx, experts, dest = t_idx[order], k_idx[order], experts[order], dest[order]
        meta = torch.stack([torch.full_like(experts, self.rank, dtype=torch.float64), tokens[t_idx].double(),
                            k_idx.double(), experts.double(), w[t_idx, k_idx].double()], dim=1)
        rows = x[t_idx].contiguous()
        # phase 1: how many pairs go to each rank
        send_counts = torch.bincount(dest, minlength=self.world).to(torch.int64)
        recv_counts = torch.empty_like(send_counts)
        self._a2a(recv_counts, send_counts, [1] * self.world, [1] * self.world)
        s_split, r_split = send_counts.tolist(), recv_counts.tolist()
        # phase 2: the metadata of every pair
        recv_meta = torch.empty((sum(r_split), META_COLS), dtype=torch.float64)
        self._a2a(recv_meta, meta, r_split, s_split)
        # phase 3: the payload (token rows)
        recv_rows = torch.empty((sum(r_split), self.H), dtype=x.dtype)
        self._a2a(recv_rows, rows, r_split, s_split)
        return recv_meta, recv_rows, (r_split, s_split)

    def give_back(self, recv_meta, results, splits):
        """Return the owner's weighted results ([m, H], in the order of `recv_meta`) to the home
        ranks.  Returns the metadata and rows this rank receives back as home."""
        r_split, s_split = splits
        back_meta = torch.empty((sum(s_split), META_COLS), dtype=torch.float64)
        self._a2a(back_meta, recv_meta.contiguous(), s_split, r_split)
        back_rows = torch.empty((sum(s_split), self.H), dtype=results.dtype)
        self._a2a(back_rows, results.contiguous(), s_split, r_split)
        return back_meta, back_rows


class Readiness:
    """Home-side top-k merge gate: each (token, k) result is accepted once; a token is released
    when all K have landed (its results, by k, are handed to the caller's merge)."""

    def __init__(self, tokens, top_k):
        self.K = top_k
        self.results = {int(t): {} for t in tokens}
        self.released = set()
        self.duplicates = 0

    def land(self, token, k, row):
        """Accept the result of (token, k); returns True when this landing completes the token."""
        token, k = int(token), int(k)
        got = self.results[token]
        if k in got or token in self.released:
            self.duplicates += 1                  # exactly once: a second copy is dropped
            return False
        got[k] = row
        if len(got) == self.K:
            self.released.add(token)
            return True
        return False

    def rows(self, token):
        """The token's K results in ascending k (for the merge)."""
        got = self.results[int(token)]
        return [got[k] for k in sorted(got)]
