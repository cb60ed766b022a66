"""Binned sums and cumulative sums of an input split across ranks.

Each rank holds one contiguous shard of the input, in rank order.  The
exchange step is the one the binned method has ("SyclReproSum", "How It
Works": per-thread states merge exactly, then convert once): every rank
deposits its shard into a binned state (32 + 16 K bytes, no pointers),
the states are gathered from all ranks, and
  - the sum: every rank merges all states and converts, so every rank gets
    the bits a single-GPU sum of the whole input gives;
  - the cumulative sum: rank r merges the states of ranks 0..r-1 and runs
    its shard's cumulative sum from that state, so its outputs are the
    whole input's cumulative sum at its positions.
Scalar partial sums would not do: splitting an input and adding the chunk
results loses reproducibility ("Accumulator capacity").

The gather goes through torch.distributed: with the gloo backend the state
bytes travel through host memory, with NCCL as CUDA tensors.  The
arithmetic (deposit, merge, conversion, cumulative sum) runs in the
library's kernels.  `ops` exists for tests: it replaces the device calls
(state_new, state_deposit, state_merge, state_finalize, cumsum_from_state)
with others of the same meaning.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from compensated_bit_reproducible_gb300 import api


class _DeviceOps:
    state_new = staticmethod(api.state_new)
    state_deposit = staticmethod(api.state_deposit)
    state_merge = staticmethod(api.state_merge)
    state_finalize = staticmethod(api.state_finalize)
    cumsum_from_state = staticmethod(api.repro_cumsum_from_state)


def gather_states(state: torch.Tensor, group=None) -> list[torch.Tensor]:
    """All ranks' states (uint8 tensors of equal length), in rank order, on
    the device of `state`."""
    ws = dist.get_world_size(group)
    backend = dist.get_backend(group)
    send = state if backend == "nccl" else state.cpu()
    parts = [torch.empty_like(send) for _ in range(ws)]
    dist.all_gather(parts, send, group=group)
    return [p.to(state.device) for p in parts]


def _shard_state(x: torch.Tensor, K: int, ops) -> torch.Tensor:
    st = ops.state_new(x.dtype, K, device=x.device)
    if x.numel():
        ops.state_deposit(st, x, K)
    return st


def sum(x: torch.Tensor, K: int = 3, group=None, ops=None) -> torch.Tensor:
    """Binned sum of the whole input, of which this rank holds the contiguous
    shard x; the same one-element tensor (same bits) on every rank."""
    ops = ops or _DeviceOps
    states = gather_states(_shard_state(x, K, ops), group)
    acc = ops.state_new(x.dtype, K, device=x.device)
    for st in states:
        ops.state_merge(acc, st, x.dtype, K)
    return ops.state_finalize(acc, x.dtype, K)


def cumsum(x: torch.Tensor, K: int = 3, group=None, out: torch.Tensor | None = None, ops=None) -> torch.Tensor:
    """This rank's part of the binned cumulative sum of the whole input (x is
    this rank's contiguous shard; shards in rank order)."""
    ops = ops or _DeviceOps
    rank = dist.get_rank(group)
    states = gather_states(_shard_state(x, K, ops), group)
    carry = ops.state_new(x.dtype, K, device=x.device)
    for st in states[:rank]:
        ops.state_merge(carry, st, x.dtype, K)
    if out is None:
        out = torch.empty_like(x)
    if x.numel():
        ops.cumsum_from_state(x, carry, K, out=out)
    return out
