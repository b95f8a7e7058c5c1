"""Vocabulary-sharded decode step over several GPUs (one process per GPU).

The step is memory-bound (arXiv 2401.10774, abstract): at batch 1 every
weight byte is read once per step and replicas do not help.  Splitting the
vocabulary rows of the head projections (W2) and of lm_head over G GPUs cuts
the bytes each GPU reads by about the share of those rows, at the cost of one
small exchange per step:

    medusa_shard_partial   on every GPU: heads and per-head top-k over its
                           rows, tree attention, verification over its rows;
                           writes one record (top-k lists with global ids,
                           per-node score states, typical-mode candidate scores)
    exchange               one all-gather of the records (rank order)
    medusa_shard_finish    on every GPU: the records combined into the global
                           top-k lists, the tree, the node results and the
                           acceptance -- the same answer on every GPU

The exchange is the only collective; it moves a few KB per step.
"""
from __future__ import annotations

import torch


def exchange(record: torch.Tensor, records: torch.Tensor, group=None) -> None:
    """All-gather of one flat record per rank into records[world][...] in rank
    order (NCCL for device tensors, gloo for host tensors)."""
    import torch.distributed as dist
    dist.all_gather_into_tensor(records.view(-1), record.view(-1), group=group)


def bounds(vocab: int, n_shards: int):
    """Contiguous row ranges [v0, v1) of n_shards near-equal shards."""
    return [(vocab * s // n_shards, vocab * (s + 1) // n_shards) for s in range(n_shards)]


def shard_weights(W2: torch.Tensor, lm_head: torch.Tensor, v0: int, v1: int):
    """A shard's rows of every head projection ([K][v1-v0][H], contiguous) and of lm_head."""
    return W2[:, v0:v1].contiguous(), lm_head[v0:v1].contiguous()


class ShardedStep:
    """One GPU's part of the vocabulary-sharded step: its config (with its row
    range), its record and the gathered records of every rank."""

    def __init__(self, shape, n_shards: int, shard: int, device="cuda", row_ranges=None, **over):
        """row_ranges: the shards' [v0, v1) in rank order (default: bounds())."""
        from . import medusa as M
        self.M = M
        self.ranges = list(row_ranges) if row_ranges is not None else bounds(shape.vocab, n_shards)
        v0, v1 = self.ranges[shard]
        self.cfg = M.make_config(shape, vocab_begin=v0, vocab_rows=v1 - v0, **over)
        self.n = n_shards
        nbytes = M.shard_record_bytes(self.cfg)
        self.record = torch.zeros(nbytes, dtype=torch.uint8, device=device)
        self.records = torch.zeros((n_shards, nbytes), dtype=torch.uint8, device=device)
        self.ws = M.alloc_workspace(self.cfg, device)

    def partial(self, io, stream=None) -> None:
        self.M.medusa_shard_partial(self.cfg, io, self.record, self.ws, stream)

    def finish(self, io, stream=None) -> None:
        self.M.medusa_shard_finish(self.cfg, io, self.records, self.n, self.ws, stream)

    def step(self, io, group=None, stream=None) -> None:
        """partial, one all-gather of the records, finish."""
        self.partial(io, stream)
        exchange(self.record, self.records, group)
        self.finish(io, stream)
