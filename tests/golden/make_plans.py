"""Writes tests/golden/plans.json: for every workload, which inputs to redraw
and which (node, token) pairs to plant so that the oracle's acceptance depth
is the planted one and every decision the tests compare exactly has a margin.

Calls only the oracle and the seeded input generator.  Run from the repo root:
    python tests/golden/make_plans.py [shape ...]

Per sequence b:
  1. draw h_b (redraw number r = 0, 1, ...) until, for every head, the gap
     between consecutive logits at each top-k boundary (ranks 1..k and k+1)
     is at least rel_head * max|logit|;
  2. draw the planted depth d (fixed, or uniform in [lo, hi]) and one rank per
     depth; the path nodes p_0 = root .. p_d follow those ranks;
  3. plant, at p_{j-1}, the head-j candidate of that rank (j = 1..d), and at
     p_d a stop token that is not among the depth-(d+1) candidates (any token
     when d is the full depth) -- it becomes the bonus token;
  4. (reduced workloads) redraw the q row of any other node whose top-2 base
     scores are closer than rel_node * max|score| (a q row changes only its
     own node's output);
  5. check with the oracle that the acceptance length is d, that the accepted
     tokens and bonus are the planted ones, and (typical acceptance) that
     every child of a path node clears or misses its threshold by at least
     0.05 in log space.
"""
from __future__ import annotations

import json
import math
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from medusa_head_tree_heads_b300 import synth  # noqa: E402
from oracle import medusa_oracle as O  # noqa: E402

REL_HEAD = {"bf16": 1e-3, "f32": 1e-4}
REL_NODE = {"bf16": 2e-3, "f32": 1e-4}
TYPICAL_LOG_MARGIN = 0.05


def to_np(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def head_gaps_ok(lg: np.ndarray, topk, rel: float) -> bool:
    """lg [K,V] logits of one sequence."""
    for k in range(lg.shape[0]):
        n = topk[k] if k < len(topk) else 1
        srt = np.sort(lg[k])[::-1]
        g = rel * np.abs(lg[k]).max()
        for j in range(n):
            if srt[j] - srt[j + 1] < g:
                return False
    return True


def build_plan(s: synth.Shape, log=print) -> dict:
    rng = np.random.Generator(np.random.PCG64(s.seed * 31 + 7))
    W = synth.make_weights(s)
    Wn = {k: to_np(v) for k, v in W.items()}
    B, D, T = s.batch, s.depth, s.n_nodes
    topk = list(s.topk)
    tree = O.Tree.for_shape(s)

    # 1. h redraws until the head top-k boundaries have margins
    redraw = [0] * B
    pending = list(range(B))
    topk_idx = np.zeros((B, s.n_heads, max(topk + [1])), dtype=np.int32)
    while pending:
        hrows = torch.stack([synth.draw_h_row(s, b, redraw[b]) for b in pending])
        z = O.head_hidden(to_np(hrows), Wn["W1"], Wn["b1"])
        lg = O.head_logits(z, Wn["W2"])
        idx, _ = O.topk_lists(lg, topk)
        nxt = []
        for j, b in enumerate(pending):
            if head_gaps_ok(lg[j], topk, REL_HEAD[s.dtype]):
                topk_idx[b] = idx[j]
            else:
                redraw[b] += 1
                nxt.append(b)
        pending = nxt
        log(f"  {s.name}: head-margin redraws pending {len(pending)}")

    # 2-3. planted paths
    seqs = []
    for b in range(B):
        if s.planted[0] == "fixed":
            d = s.planted[1]
        else:
            d = int(rng.integers(s.planted[1], s.planted[2] + 1))
        path = [0]
        plant = []
        for j in range(1, d + 1):
            kids = tree.children[path[-1]]
            if not kids:  # an explicit tree's leaf above the drawn depth ends the path
                d = j - 1
                break
            child = kids[int(rng.integers(0, len(kids)))]
            plant.append([path[-1], int(topk_idx[b, j - 1, tree.rank[child]])])
            path.append(child)
        excluded = set(topk_idx[b, d, :topk[d]].tolist()) if d < D else set()
        while True:
            stop = int(rng.integers(0, s.vocab))
            if stop not in excluded:
                break
        plant.append([path[-1], stop])
        seqs.append({"depth": d, "plant": plant, "nodes": path, "tokens": [p[1] for p in plant[:-1]],
                     "bonus": stop})

    plan = {"h_redraws": redraw, "q_redraws": [], "seqs": seqs}
    inp = synth.make_inputs(s, plan)
    n = {k: to_np(v) for k, v in inp.items()}

    # 4. node margins (reduced workloads: every node; full-size: path nodes only)
    planted_nodes = {b: {p[0] for p in seqs[b]["plant"]} for b in range(B)}
    q_red = {}
    nodes_only = None if not s.full_size else {b: sorted(planted_nodes[b]) for b in range(B)}
    for it in range(50):
        res = O.step(n, s, nodes_only=nodes_only)
        bad = []
        for b in range(B):
            for i in range(T):
                if nodes_only is not None and i not in nodes_only[b]:
                    continue
                m1, m2 = res["maxlogit"][b, i], res["second"][b, i]
                gap = m1 - m2
                if gap < REL_NODE[s.dtype] * max(abs(m1), abs(m2)):
                    if i in planted_nodes[b]:
                        raise RuntimeError(f"{s.name}: planted node {b},{i} lacks a margin")
                    bad.append((b, i))
        if not bad:
            break
        for b, i in bad:
            q_red[(b, i)] = q_red.get((b, i), 0) + 1
            inp["q"][b, i] = synth.draw_q_row(s, b, i, q_red[(b, i)])
        n["q"] = to_np(inp["q"])
        log(f"  {s.name}: node-margin redraws {len(bad)}")
    else:
        raise RuntimeError("node margins did not converge")
    plan["q_redraws"] = [[b, i, r] for (b, i), r in sorted(q_red.items())]

    # 5. the oracle must realise the planted acceptance
    for b in range(B):
        sq = seqs[b]
        assert res["accept_len"][b] == sq["depth"], (s.name, b, res["accept_len"][b], sq["depth"])
        assert res["acc_tokens"][b] == sq["tokens"], (s.name, b)
        assert res["acc_nodes"][b] == sq["nodes"], (s.name, b)
        if s.accept == "typical-sample":  # the bonus is the draw at the last kept node: keep it, with its margin
            last = sq["nodes"][-1]
            dm, d2 = res["draw_max"][b, last], res["draw_second"][b, last]
            assert dm - d2 >= REL_NODE[s.dtype] * max(1.0, abs(dm)), (s.name, b, "draw margin")
            sq["bonus"] = int(res["bonus"][b])
        assert res["bonus"][b] == sq["bonus"], (s.name, b)
        assert [int(x) for x in res["topk_idx"][b].ravel()] == [int(x) for x in topk_idx[b].ravel()]
        if s.accept in ("typical", "typical-sample"):
            flat = res["attn_out"].reshape(B * T, -1)
            for p in sq["nodes"]:
                thr = O.typical_threshold(res["entropy"][b, p], s.eps, s.delta)
                for c in tree.children[p]:
                    lp = O.token_logprob(flat[b * T + p], n["lm_head"], int(res["tokens"][b, c]), s.temperature,
                                         res["lse"][b, p])
                    assert abs(lp - math.log(thr)) >= TYPICAL_LOG_MARGIN, (s.name, b, p, c)
    return plan


def main(names):
    path = synth.PLANS_PATH
    plans = {}
    if os.path.exists(path):
        with open(path) as f:
            plans = json.load(f)
    for name in names:
        s = synth.SHAPES[name]
        print(f"building plan for {name}")
        plans[name] = build_plan(s)
        with open(path, "w") as f:
            json.dump(plans, f, indent=1, sort_keys=True)
            f.write("\n")


if __name__ == "__main__":
    main(sys.argv[1:] or list(synth.SHAPES))
