"""Vocabulary shards (CPU): what one shard computes over its rows of the head
projections and of lm_head, combined over the shards, equals the unsplit step
(the oracle's shard functions pinned against its own unsplit functions, for
ragged splits into 2 and 3 shards); and the combination carried out across
two gloo ranks, each computing its shard and exchanging its partial result
with the library's exchange helper, gives the same answer on every rank."""
from __future__ import annotations

import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from medusa_head_tree_heads_b300 import synth
from oracle import medusa_oracle as O
from tests import util as U

SPLITS = {2: [0.37], 3: [0.21, 0.64]}  # cut points as fractions of the vocabulary (ragged)


def _bounds(V, S):
    cuts = [int(f * V) for f in SPLITS[S]]
    b = [0] + cuts + [V]
    return list(zip(b[:-1], b[1:]))


def _unsplit(n, s, o_flat):
    z = O.head_hidden(n["h"], n["W1"], n["b1"])
    idx, val = O.topk_lists(O.head_logits(z, n["W2"]), list(s.topk))
    st = O.verify_stats(o_flat, n["lm_head"], s.temperature if s.accept == "typical" else None)
    return z, idx, val, st


def check_shards_match_unsplit(M, name, S) -> None:
    s, inp = U.planned_inputs(name)
    n = U.np_inputs(inp)
    rng = np.random.default_rng(7)
    o_flat = O.round_to_storage(rng.standard_normal((9, s.hidden)) / np.sqrt(s.hidden), s.dtype)
    z, idx, val, st = _unsplit(n, s, o_flat)
    temp = s.temperature if s.accept == "typical" else None
    parts, states = [], []
    for v0, v1 in _bounds(s.vocab, S):
        parts.append(M.shard_topk(z, n["W2"][:, v0:v1], v0, list(s.topk)))
        states.append(M.shard_node_states(o_flat, n["lm_head"][v0:v1], v0, temp))
    midx, mval, src = M.merge_topk(parts, list(s.topk))
    np.testing.assert_array_equal(midx, idx)
    live = idx >= 0
    np.testing.assert_allclose(mval[live], val[live], rtol=1e-12)
    for b, k, r in zip(*np.nonzero(live)):  # each entry traced to the shard and rank it came from
        si, j = src[b, k, r]
        assert parts[si][0][b, k, j] == idx[b, k, r]
    res = M.merge_node_states(states, temp)
    np.testing.assert_array_equal(res["argmax"], st["argmax"])
    np.testing.assert_allclose(res["maxlogit"], st["maxlogit"], rtol=1e-12)
    if temp is not None:
        np.testing.assert_allclose(res["lse"], st["lse"], rtol=1e-12)
        np.testing.assert_allclose(res["entropy"], st["entropy"], rtol=1e-10)


@pytest.mark.parametrize("S", [2, 3])
@pytest.mark.parametrize("name", ["7b-mini", "gqa-mini", "tiny-fp32-gqa"])
def test_shards_match_the_unsplit_step(name, S):
    check_shards_match_unsplit(O, name, S)


def _free_port() -> int:
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _rank_main(rank, world, port, name, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank))
    import torch.distributed as dist
    from medusa_head_tree_heads_b300 import shards as SH
    dist.init_process_group("gloo")
    try:
        s, inp = U.planned_inputs(name)
        n = U.np_inputs(inp)
        rng = np.random.default_rng(7)
        o_flat = O.round_to_storage(rng.standard_normal((9, s.hidden)) / np.sqrt(s.hidden), s.dtype)
        temp = s.temperature if s.accept == "typical" else None
        v0, v1 = _bounds(s.vocab, world)[rank]
        z = O.head_hidden(n["h"], n["W1"], n["b1"])
        idx, val = O.shard_topk(z, n["W2"][:, v0:v1], v0, list(s.topk))
        st = O.shard_node_states(o_flat, n["lm_head"][v0:v1], v0, temp)
        # this rank's partial result as one flat record, exchanged as the
        # library exchanges the device records (one all-gather, rank order)
        rec = torch.from_numpy(np.concatenate([idx.ravel().astype(np.float64), val.ravel(), st["m"], st["i"],
                                               st["z"], st["s"]]))
        allrec = torch.empty((world, rec.numel()), dtype=rec.dtype)
        SH.exchange(rec, allrec)
        nt = idx.size
        parts, states = [], []
        for r in range(world):
            x = allrec[r].numpy()
            parts.append((x[:nt].astype(np.int32).reshape(idx.shape), x[nt:2 * nt].reshape(idx.shape)))
            m = x[2 * nt:].reshape(4, -1)
            states.append({"m": m[0], "i": m[1].astype(np.int64), "z": m[2], "s": m[3]})
        midx, _, _ = O.merge_topk(parts, list(s.topk))
        res = O.merge_node_states(states, temp)
        ref_idx, _ = O.topk_lists(O.head_logits(z, n["W2"]), list(s.topk))
        ref = O.verify_stats(o_flat, n["lm_head"], temp)
        ok = bool(np.array_equal(midx, ref_idx) and np.array_equal(res["argmax"], ref["argmax"]))
        if temp is not None:
            ok = ok and bool(np.allclose(res["lse"], ref["lse"], rtol=1e-12))
        q.put((rank, ok))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("name", ["7b-mini", "gqa-mini"])
def test_two_gloo_ranks_combine_their_shards(name):
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, name, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert res == [(0, True), (1, True)]
