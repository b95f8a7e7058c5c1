"""Round after round of Medusa decoding on the GPU, over a table backbone.

One round ("Medusa Heads", "Attenzione sull'albero e accettazione": the heads
propose, the tree is verified in one pass, the kept branch is appended and
the next round starts from it) is these calls of the C ABI, all enqueued on
one stream with no host synchronisation between rounds:

    medusa_heads_topk      heads + per-head top-k on the hidden state
    medusa_tree_build      the candidate tree and its tokens
    (backbone)             the tree's queries, keys and values
    medusa_tree_attn_lens  tree attention over each sequence's grown cache
    medusa_verify_accept   verification and greedy acceptance
    medusa_kv_commit       the kept branch (root first) into the cache
    medusa_next_inputs     next hidden state and next root

The backbone stand-in looks each tree token up in per-token tables
(synth.make_toy): a row gather on the device, no part of the method.  Every
round's root, accept length, tokens, nodes and bonus are kept in device
history buffers, read back once at the end.
"""
from __future__ import annotations

from typing import Dict

import torch

from . import medusa as M


class DecodeLoop:
    def __init__(self, shape, toy: Dict[str, torch.Tensor], device="cuda"):
        self.s = shape
        self.cfg = M.make_config(shape)
        self.dev = {k: v.to(device) for k, v in toy.items()}
        d = self.dev
        # the loop owns its mutable state (caches, lengths, hidden state, root);
        # the initial values stay aside for reset()
        self.init = {k: d[k] for k in ("k_cache", "v_cache", "kv_lens", "h", "root_token")}
        for k in self.init:
            d[k] = d[k].clone()
        self.ws = M.alloc_workspace(self.cfg, device)
        self.out = M.alloc_outputs(self.cfg, device)
        B, T = shape.batch, shape.n_nodes
        dt = shape.torch_dtype
        self.q = torch.empty((B, T, shape.n_q_heads, shape.head_dim), dtype=dt, device=device)
        self.kt = torch.empty((B, T, shape.n_kv_heads, shape.head_dim), dtype=dt, device=device)
        self.vt = torch.empty_like(self.kt)
        R, D = shape.rounds, shape.depth
        i32 = dict(dtype=torch.int32, device=device)
        self.hist = {"root": torch.empty((R, B), **i32), "accept_len": torch.empty((R, B), **i32),
                     "acc_tokens": torch.empty((R, B, max(D, 1)), **i32),
                     "acc_nodes": torch.empty((R, B, D + 1), **i32), "bonus": torch.empty((R, B), **i32)}

    def backbone(self) -> None:
        tok = self.out["tree"]["token"].view(-1).long()
        d = self.dev
        torch.index_select(d["Qtab"], 0, tok, out=self.q.view(-1, *d["Qtab"].shape[1:]))
        torch.index_select(d["Ktab"], 0, tok, out=self.kt.view(-1, *d["Ktab"].shape[1:]))
        torch.index_select(d["Vtab"], 0, tok, out=self.vt.view(-1, *d["Vtab"].shape[1:]))

    def round(self, r: int) -> None:
        cfg, d, o, ws, hist = self.cfg, self.dev, self.out, self.ws, self.hist
        M.medusa_heads_topk(cfg, d["h"], d["W1"], d["b1"], d["W2"], o["topk_idx"], o["topk_val"], ws)
        M.medusa_tree_build(cfg, o["topk_idx"], d["root_token"], o["tree"])
        self.backbone()
        M.medusa_tree_attn_lens(cfg, self.q, self.kt, self.vt, d["k_cache"], d["v_cache"], d["kv_lens"], o["tree"],
                                o["attn_out"], ws)
        res = {"node_argmax": o["node_argmax"], "node_maxlogit": o["node_maxlogit"], "node_lse": o["node_lse"],
               "node_entropy": o["node_entropy"], "accept_len": hist["accept_len"][r],
               "acc_tokens": hist["acc_tokens"][r], "acc_nodes": hist["acc_nodes"][r], "bonus": hist["bonus"][r]}
        M.medusa_verify_accept(cfg, o["attn_out"], d["lm_head"], o["tree"], res, ws)
        hist["root"][r].copy_(d["root_token"])
        M.medusa_kv_commit(cfg, res["acc_nodes"], res["accept_len"], self.kt, self.vt, d["k_cache"], d["v_cache"],
                           d["kv_lens"], ws)
        M.medusa_next_inputs(cfg, o["attn_out"], res["acc_nodes"], res["accept_len"], res["bonus"], d["h"],
                             d["root_token"], ws)

    def reset(self) -> None:
        """Back to the state before the first round (device copies)."""
        for k, v in self.init.items():
            self.dev[k].copy_(v)

    def run(self, rounds: int = None) -> None:
        for r in range(self.s.rounds if rounds is None else rounds):
            self.round(r)

    def tokens(self) -> int:
        """Tokens the rounds run so far emitted (each keeps its accepted
        candidates and the root it started from)."""
        return int((self.hist["accept_len"] + 1).sum().item())

    def history(self) -> Dict[str, list]:
        """Per round and sequence: root, accept_len, acc_tokens (first
        accept_len entries), acc_nodes (first accept_len + 1) and bonus."""
        h = {k: v.cpu() for k, v in self.hist.items()}
        R, B = h["root"].shape
        out = {"root": h["root"].tolist(), "accept_len": h["accept_len"].tolist(), "bonus": h["bonus"].tolist(),
               "acc_tokens": [], "acc_nodes": []}
        for r in range(R):
            n = out["accept_len"][r]
            out["acc_tokens"].append([h["acc_tokens"][r, b, :n[b]].tolist() for b in range(B)])
            out["acc_nodes"].append([h["acc_nodes"][r, b, :n[b] + 1].tolist() for b in range(B)])
        return out
