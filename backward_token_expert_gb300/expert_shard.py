"""Expert-parallel partition of the recalibration path: the host-side plan
and the exchanges between ranks.

LRMoE trains with the experts spread over GPUs (expert parallelism, LRMoE
sec. 1 and 2): every rank holds a block of tokens (their logits, routing,
output gradients and saved projection inputs) and owns a block of experts
(their weights and weight gradients).  Selection must see all candidates of
an expert, and it runs before the compacted rows travel (LRMoE Alg. 1:
score and select, then compact and exchange), so that only retained rows
cross the network, the smaller payload the paper argues for (LRMoE sec. 1).
The exchanges, in path order:

1. routing statistics: an all-reduce of the per-expert routed counts n_e and
   of the summed gate probabilities sum_t p_t,e (2E numbers); every rank then
   applies the quota rule to the global counts itself;
2. candidates: every token owner sends (u, e_u, R_u) of each of its pairs to
   the owner of expert e_u (three 8-byte numbers per pair);
3. selection runs at the expert owner on all candidates of its experts;
4. requests: the owner sends each retained pair id u back to the owner of
   token u div k;
5. rows: token owners compact the requested rows (delta_u = alpha_u g_t and
   phi_u) and send them to the expert owner, which holds them in its
   selection order;
6. the grouped GEMMs run at the owner on its experts' segments;
7. the input-gradient rows go back to the token owners (the combine), which
   put them at their pairs' rows (the inverse mapping).

Ranks own contiguous blocks: expert block r is [r E / W, (r+1) E / W) and
token block r is [r T / W, (r+1) T / W) for W ranks.  Pair ids are global,
u = t k + j.  All exchanges are ``all_to_all_single`` calls with split sizes
exchanged first, so they run on NCCL (GPU tensors) and gloo (CPU tensors)
alike.  The arithmetic of every step is not here: the caller passes the
tensors its kernels produced, and gets back what the next step needs.
"""

from __future__ import annotations

import dataclasses

import torch
import torch.distributed as dist


@dataclasses.dataclass(frozen=True)
class ShardPlan:
    """Which rank owns which experts and tokens."""

    T: int
    E: int
    k: int
    world: int
    rank: int

    def expert_range(self, r: int | None = None) -> tuple[int, int]:
        r = self.rank if r is None else r
        return r * self.E // self.world, (r + 1) * self.E // self.world

    def token_range(self, r: int | None = None) -> tuple[int, int]:
        r = self.rank if r is None else r
        return r * self.T // self.world, (r + 1) * self.T // self.world

    def pair_range(self, r: int | None = None) -> tuple[int, int]:
        t0, t1 = self.token_range(r)
        return t0 * self.k, t1 * self.k

    def expert_owner(self, e: torch.Tensor) -> torch.Tensor:
        """Rank that owns each expert id of `e`."""
        starts = torch.tensor([self.expert_range(r)[0] for r in range(1, self.world)], dtype=torch.int64,
                              device=e.device)
        return torch.bucketize(e.to(torch.int64), starts, right=True)

    def token_owner_of_pair(self, u: torch.Tensor) -> torch.Tensor:
        """Rank that holds the token of each pair id of `u`."""
        starts = torch.tensor([self.token_range(r)[0] for r in range(1, self.world)], dtype=torch.int64,
                              device=u.device)
        return torch.bucketize(torch.div(u.to(torch.int64), self.k, rounding_mode="floor"), starts, right=True)


def _counts_by_rank(dest: torch.Tensor, world: int) -> list[int]:
    return torch.bincount(dest, minlength=world).tolist()


def exchange(send: torch.Tensor, send_counts: list[int], group=None) -> tuple[torch.Tensor, list[int]]:
    """All-to-all of the rows of `send`, grouped by destination rank (the
    first send_counts[0] rows to rank 0, ...).  Returns the received rows,
    grouped by source rank in rank order, and how many came from each.  Rows
    travel as raw bytes (int32 words when a row is a multiple of 4 bytes), so
    every dtype goes through every backend unchanged."""
    world = len(send_counts)
    sc = torch.tensor(send_counts, dtype=torch.int64, device=send.device)
    rc = torch.empty(world, dtype=torch.int64, device=send.device)
    dist.all_to_all_single(rc, sc, group=group)
    recv_counts = rc.tolist()
    row_shape = tuple(send.shape[1:])
    raw = send.contiguous().reshape(send.shape[0], -1).view(torch.uint8)
    word = torch.int32 if raw.shape[1] % 4 == 0 else torch.uint8
    raw = raw.view(word)
    recv = torch.empty((sum(recv_counts), raw.shape[1]), dtype=word, device=send.device)
    dist.all_to_all_single(recv, raw, output_split_sizes=recv_counts, input_split_sizes=send_counts, group=group)
    return recv.view(torch.uint8).view(send.dtype).reshape((sum(recv_counts),) + row_shape), recv_counts


def global_route_counts(plan: ShardPlan, expert_idx_local: torch.Tensor, psum_local: torch.Tensor,
                        group=None) -> tuple[torch.Tensor, torch.Tensor]:
    """Exchange 1: the routed counts n_e of the whole batch and the gate
    probabilities summed over all tokens, from this rank's tokens (its
    [T_r, k] expert ids and its per-expert sums of the softmax rows)."""
    counts = torch.bincount(expert_idx_local.reshape(-1).to(torch.int64), minlength=plan.E)
    psum = psum_local.to(torch.float64).clone()
    dist.all_reduce(counts, group=group)
    dist.all_reduce(psum, group=group)
    return counts, psum


@dataclasses.dataclass
class Candidates:
    """All candidates of the experts this rank owns, in ascending pair id."""

    u: torch.Tensor  # [n] int64 global pair ids
    e: torch.Tensor  # [n] int64 expert of each pair
    R: torch.Tensor  # [n] float64 score of each pair (exactly the sender's value)


def exchange_candidates(plan: ShardPlan, R_local: torch.Tensor, expert_idx_local: torch.Tensor,
                        group=None) -> Candidates:
    """Exchange 2: every pair's (u, e_u, R_u) to the owner of e_u.  The sent
    scores are converted to float64, exactly for fp32 or fp64 inputs; pair ids
    and expert ids are below 2^53, so they travel exactly too."""
    p0, p1 = plan.pair_range()
    u = torch.arange(p0, p1, dtype=torch.int64, device=R_local.device)
    e = expert_idx_local.reshape(-1).to(torch.int64)
    dest = plan.expert_owner(e)
    order = torch.sort(dest, stable=True).indices  # ascending u within each destination
    payload = torch.stack([u[order].to(torch.float64), e[order].to(torch.float64),
                           R_local.reshape(-1)[order].to(torch.float64)], dim=1)
    recv, _ = exchange(payload, _counts_by_rank(dest, plan.world), group)
    # sources arrive in rank order and token blocks ascend with the rank, so
    # the received pair ids already ascend
    return Candidates(u=recv[:, 0].to(torch.int64), e=recv[:, 1].to(torch.int64), R=recv[:, 2])


@dataclasses.dataclass
class Requests:
    """Exchange 4 seen from both sides."""

    asked_u: torch.Tensor  # token-owner side: requested pair ids, grouped by requesting rank
    asked_counts: list[int]  # how many each rank asked for
    order: torch.Tensor  # owner side: permutation that grouped its retained ids by token owner
    sent_counts: list[int]  # owner side: how many ids went to each token owner


def request_rows(plan: ShardPlan, sel_u: torch.Tensor, group=None) -> Requests:
    """Exchange 4: the owner's retained pair ids (expert-major, ascending u
    within an expert) to the owners of their tokens."""
    sel_u = sel_u.to(torch.int64)
    dest = plan.token_owner_of_pair(sel_u)
    order = torch.sort(dest, stable=True).indices
    sent_counts = _counts_by_rank(dest, plan.world)
    asked, asked_counts = exchange(sel_u[order], sent_counts, group)
    return Requests(asked_u=asked, asked_counts=asked_counts, order=order, sent_counts=sent_counts)


def send_rows(req: Requests, rows: torch.Tensor, group=None) -> torch.Tensor:
    """Exchange 5: the token owner's rows for ``req.asked_u`` (one per asked
    id, in the same order) to the ranks that asked; returns, at the asking
    rank, its rows in its own selection order."""
    got, _ = exchange(rows, req.asked_counts, group)
    out = torch.empty_like(got)
    out[req.order] = got
    return out


def return_rows(req: Requests, rows_in_sel_order: torch.Tensor, group=None) -> torch.Tensor:
    """Exchange 7: rows computed at the expert owner (one per retained pair,
    in its selection order) back to the token owners; returns, at each token
    owner, the rows for ``req.asked_u`` in that order."""
    back, _ = exchange(rows_in_sel_order[req.order], req.sent_counts, group)
    return back
