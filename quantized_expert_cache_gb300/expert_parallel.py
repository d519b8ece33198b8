"""Expert parallelism across processes, one GPU each.

neurall/llama.cpp README, "More GPUs": every GPU keeps its own expert cache
in its own memory, so more GPUs cache more experts.  The pages do not say how
the experts are split between the GPUs; this module's reading is expert
parallelism: rank r of N holds a contiguous range of every layer's experts
(``shard_range``) in its own context (``moe_set_expert_shard``), with its own
pool, pointer tables, miss log and promotion pass, so the ranks cache
disjoint experts and their pools add up.

Two exchange patterns, through ``torch.distributed`` (NCCL between GPUs,
gloo for the host logic on CPU):

- replicated tokens (batch-1 decode: every rank holds the same x and the
  same router logits): every rank routes every token over all experts, its
  context computes the partial sum over its own experts (the other ranks'
  assignments are left out in the kernels), and one sum all-reduce of
  y [T][H] fp32 gives the layer's output on every rank (``allreduce_partial``);
- distributed tokens (prompt passes: rank r holds its own T_r tokens, routed
  over all experts): one all-to-all sends each token row (x, its k global
  expert ids and weights) to every rank that owns one of its picks
  (``dispatch``); each rank runs its experts over the rows it received with
  the clock of the whole step (``moe_ffn_forward_rows``); a second all-to-all
  returns the partial rows, which the token's home rank sums in rank order
  (``combine``).  ``prefill_layer`` chains the three.

The packing around the collectives (row gathers, the rank-ordered sum) is
plain tensor indexing on the caller's device; on GPUs run it on the
context's stream (``with torch.cuda.stream(...)``) so that it is ordered
with the library's kernels.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import moe_ffn_forward_rows


def shard_range(n_experts: int, rank: int, world: int) -> tuple[int, int]:
    """(first expert, number of experts) of rank `rank`: experts
    [E r / N, E (r + 1) / N) (integer division), so shard sizes differ by at
    most one and every expert has exactly one owner."""
    if not (0 <= rank < world) or n_experts < world:
        raise ValueError("need 0 <= rank < world <= n_experts")
    base = n_experts * rank // world
    return base, n_experts * (rank + 1) // world - base


def owners(idx: torch.Tensor, n_experts: int, world: int) -> torch.Tensor:
    """Rank that owns each global expert id of `idx` (same shape, int64)."""
    starts = torch.tensor([n_experts * r // world for r in range(1, world)], dtype=torch.int64, device=idx.device)
    return torch.bucketize(idx.to(torch.int64), starts, right=True)


def allreduce_partial(y: torch.Tensor, group=None) -> torch.Tensor:
    """Replicated tokens: y (this rank's partial sum, fp32 [T][H]) becomes the
    sum over every rank's partial, in place."""
    dist.all_reduce(y, op=dist.ReduceOp.SUM, group=group)
    return y


class DispatchHandle:
    """What `combine` needs to bring the partial rows home."""

    def __init__(self, order, send_counts, recv_counts, n_tokens, hidden):
        self.order = order              # token ids sent, grouped by destination rank (ascending within)
        self.send_counts = send_counts  # rows sent to each rank
        self.recv_counts = recv_counts  # rows received from each rank
        self.n_tokens = n_tokens        # this rank's tokens
        self.hidden = hidden


def dispatch(x: torch.Tensor, idx: torch.Tensor, w: torch.Tensor, n_experts: int, group=None):
    """Distributed tokens: send every token row to each rank that owns one of
    its k picks.  x fp32 [T][H], idx int32 [T][k] global ids, w fp32 [T][k]
    (this rank's tokens).  Returns (x_rows, idx_rows, w_rows, step_tokens,
    handle): the rows this rank received (from rank 0's tokens first, each
    source's rows in token order), and the number of tokens of the step over
    all ranks (the clock a rank's pool hits are stamped with)."""
    if x.dtype != torch.float32 or w.dtype != torch.float32 or idx.dtype != torch.int32:
        raise TypeError("dispatch: x and w must be float32 and idx int32 (the payload carries the ids' bits)")
    world = dist.get_world_size(group)
    T, k = idx.shape
    H = x.shape[1]
    dev = x.device
    own = owners(idx, n_experts, world)
    rows = [torch.nonzero((own == s).any(dim=1)).flatten() for s in range(world)]
    send_counts = [int(r.numel()) for r in rows]
    meta = torch.tensor([[c, T] for c in send_counts], dtype=torch.int64, device=dev)
    meta_in = torch.empty_like(meta)
    dist.all_to_all_single(meta_in, meta, group=group)
    recv_counts = [int(c) for c in meta_in[:, 0].tolist()]
    step_tokens = int(meta_in[:, 1].sum().item())
    order = torch.cat(rows) if rows else torch.empty(0, dtype=torch.int64, device=dev)
    # one payload row: x, then the k ids (their bits carried as fp32), then w
    payload = torch.cat([x[order], idx[order].contiguous().view(torch.float32), w[order]], dim=1).contiguous()
    recv = torch.empty((sum(recv_counts), H + 2 * k), dtype=torch.float32, device=dev)
    dist.all_to_all_single(recv, payload, output_split_sizes=recv_counts, input_split_sizes=send_counts,
                           group=group)
    x_r = recv[:, :H].contiguous()
    idx_r = recv[:, H:H + k].contiguous().view(torch.int32)
    w_r = recv[:, H + k:].contiguous()
    return x_r, idx_r, w_r, step_tokens, DispatchHandle(order, send_counts, recv_counts, T, H)


def combine(y_rows: torch.Tensor, handle: DispatchHandle, group=None) -> torch.Tensor:
    """Return the partial rows to their home ranks and sum them: y[t] =
    sum over the owning ranks s = 0, 1, ... of rank s's partial row of t
    (0 for a token with no row anywhere, which cannot happen with k >= 1)."""
    h = handle
    back = torch.empty((sum(h.send_counts), h.hidden), dtype=torch.float32, device=y_rows.device)
    dist.all_to_all_single(back, y_rows.contiguous(), output_split_sizes=h.send_counts,
                           input_split_sizes=h.recv_counts, group=group)
    y = torch.zeros((h.n_tokens, h.hidden), dtype=torch.float32, device=y_rows.device)
    off = 0
    for c in h.send_counts:  # owners in rank order; token ids are distinct within one
        if c:
            y[h.order[off:off + c]] += back[off:off + c]
        off += c
    return y


def rows_forward(ctx, layer: int, stream=None):
    """This rank's part of a prompt layer: its context's experts over the
    received rows, stamped with the step's clock."""

    def run(x_rows, idx_rows, w_rows, step_tokens):
        y = torch.empty_like(x_rows)
        moe_ffn_forward_rows(ctx, layer, x_rows, x_rows.shape[0], idx_rows, w_rows, y, step_tokens, stream)
        return y

    return run


def prefill_layer(x, idx, w, n_experts: int, local_forward, group=None):
    """dispatch -> local_forward(x_rows, idx_rows, w_rows, step_tokens) ->
    combine: the layer's output for this rank's tokens, and the step's token
    count (for cache_step)."""
    x_r, idx_r, w_r, step_tokens, handle = dispatch(x, idx, w, n_experts, group)
    y_r = local_forward(x_r, idx_r, w_r, step_tokens)
    return combine(y_r, handle, group), step_tokens
