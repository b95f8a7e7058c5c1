"""Seeded synthetic inputs for one Medusa decode step.

This module only draws random numbers and lays them out; it holds none of the
step's arithmetic (no head FFN, no projection, no top-k, no tree, no
attention, no acceptance).  Both the CUDA path (tests, benchmark) and the CPU
oracle (tests) take their inputs from here.

Workload shapes follow the method's description in "Medusa Heads"
(ultralytics glossary): K heads read the final hidden state ``h``; each head
is a residual SiLU feed-forward layer followed by a vocabulary projection
that starts as a copy of ``lm_head`` ("Come le teste prevedono i token
successivi").  The candidate tree is the Cartesian product of the per-depth
top-k lists ("Attenzione sull'albero e accettazione").

Distributions (``N(0, s)`` below gives the standard deviation):
  lm_head  ~ N(0, 1/sqrt(H))        (variance 1/H, fan-in scale)
  W2_k     = lm_head + N(0, 0.01)   (zero-init variant: an exact copy)
  W1_k, b1 ~ N(0, 0.02)             (zero-init variant: zeros)
  h, q, k, v (tree and cache) ~ N(0, 1)
  root_token ~ uniform over the vocabulary
Every tensor is drawn in fp32 from its own seeded ``torch.Generator`` and then
rounded (RNE) to the workload's storage type.

Planting.  A plant list ``[(node, token), ...]`` per sequence overwrites the
tree q/k/v rows of those nodes so that the base model's top token at that
node is ``token`` with a large margin: every q head of kv group g becomes
``2*sqrt(Dh)*u_g`` and the node's own key ``15*u_g`` (self score 30 against
cache scores of spread ~2), and the node's value for group g is
``24 * M_g[token] / |M_g[token]|`` with ``M_g`` the sum of the lm_head column
slices of the q heads in group g.  Which nodes and tokens to plant (and how
many times to redraw ``h_b`` or a node's q row) is decided offline and stored
with the tests; this module only applies it.
"""
from __future__ import annotations

import dataclasses
import json
import math
import os
from typing import Dict, List, Optional, Sequence, Tuple

import torch

PLANT_GAMMA_Q = 2.0  # q = PLANT_GAMMA_Q * sqrt(Dh) * u
PLANT_GAMMA_K = 15.0  # k_self = PLANT_GAMMA_K * u
PLANT_ALPHA_V = 24.0  # |v| = PLANT_ALPHA_V


@dataclasses.dataclass(frozen=True)
class Shape:
    """One workload: sizes, storage type, acceptance rule and seed."""

    name: str
    dtype: str  # "f32" or "bf16"
    hidden: int
    vocab: int
    n_heads: int
    batch: int
    topk: Tuple[int, ...]  # top-k per tree depth (depth = len(topk))
    kv_len: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    accept: str  # "greedy", "typical", "sample" or "typical-sample"
    planted: Tuple  # ("fixed", d) or ("uniform", lo, hi)
    seed: int
    kv_capacity: int = 0  # cache rows per sequence; 0 means kv_len
    temperature: float = 0.7
    eps: float = 0.3
    delta: float = 0.09
    full_size: bool = False  # the oracle checks every node only when False
    sparse_nodes: int = 0  # > 0: an explicit tree of that many non-root nodes (see explicit_tree)
    sample_seed: Tuple[int, int] = (0x1234567, 0x89ABCDE)  # sampling verification: Philox key and step
    sample_step: int = 0

    @property
    def depth(self) -> int:
        return len(self.topk)

    @property
    def n_nodes(self) -> int:
        """Tree rows including the root (sizes of the level products, summed;
        for an explicit tree its node count)."""
        if self.sparse_nodes:
            return self.sparse_nodes + 1
        total, level = 1, 1
        for k in self.topk:
            level *= k
            total += level
        return total

    @property
    def tree_parent(self) -> Optional[Tuple[int, ...]]:
        return explicit_tree(self.topk, self.sparse_nodes)[0] if self.sparse_nodes else None

    @property
    def tree_rank(self) -> Optional[Tuple[int, ...]]:
        return explicit_tree(self.topk, self.sparse_nodes)[1] if self.sparse_nodes else None

    @property
    def cap(self) -> int:
        return self.kv_capacity if self.kv_capacity else self.kv_len

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


_TREES: Dict[Tuple, Tuple] = {}


def explicit_tree(topk: Sequence[int], n: int) -> Tuple[Tuple[int, ...], Tuple[int, ...]]:
    """A sparse candidate tree of n non-root nodes taken from the Cartesian
    tree of ``topk`` (a workload definition, the pages fix no rule): every
    node scores the product of 1/(rank+1) along its path (a head's lower-ranked
    candidates are less likely to be right) and the n best nodes are kept,
    ties to the lower node id, so every kept node's parent is kept.  Returns
    (parent, rank) in (depth, parent, rank) order, node 0 the root."""
    key = (tuple(topk), n)
    if key in _TREES:
        return _TREES[key]
    parent, rank, score = [-1], [0], [1.0]
    level = [0]
    for d in range(1, len(topk) + 1):
        nxt = []
        for p in level:
            for r in range(topk[d - 1]):
                parent.append(p)
                rank.append(r)
                score.append(score[p] / (r + 1))
                nxt.append(len(parent) - 1)
        level = nxt
    if n > len(parent) - 1:
        raise ValueError("more nodes than the Cartesian tree has")
    order = sorted(range(1, len(parent)), key=lambda i: (-score[i], i))
    keep = sorted([0] + order[:n])
    new_id = {old: i for i, old in enumerate(keep)}
    out = (tuple(-1 if i == 0 else new_id[parent[i]] for i in keep), tuple(rank[i] for i in keep))
    _TREES[key] = out
    return out


# The five stated workloads, then reduced variants that keep every structural
# feature (head count, tree shape, GQA ratio, acceptance rule) at sizes the
# oracle finishes in seconds, with ragged vocabulary and cache lengths.
SHAPES: Dict[str, Shape] = {}


def _add(s: Shape) -> None:
    SHAPES[s.name] = s


_add(Shape("tiny-fp32", "f32", 256, 1000, 3, 1, (2, 3), 128, 4, 4, 64, "greedy", ("fixed", 2), 1000))
_add(Shape("7b-bf16", "bf16", 4096, 32000, 5, 1, (4, 3, 2, 2, 1), 1024, 32, 32, 128, "greedy", ("fixed", 3), 1001,
           full_size=True))
_add(Shape("13b-bf16", "bf16", 5120, 32000, 5, 8, (3, 2, 2, 1), 2048, 40, 40, 128, "greedy", ("uniform", 0, 4), 1002,
           full_size=True))
_add(Shape("gqa128k-bf16", "bf16", 4096, 128256, 4, 16, (4, 3, 2, 2), 4096, 32, 8, 128, "typical", ("uniform", 0, 4),
           1003, full_size=True))
_add(Shape("33b-bf16", "bf16", 6656, 32000, 5, 32, (4, 3, 2, 2, 2), 8192, 52, 52, 128, "greedy", ("uniform", 0, 5),
           1004, full_size=True))
# reduced variants
_add(Shape("7b-mini", "bf16", 640, 3001, 5, 1, (4, 3, 2, 2, 1), 300, 5, 5, 128, "greedy", ("fixed", 3), 2001,
           kv_capacity=333))
_add(Shape("13b-mini", "bf16", 384, 2500, 5, 3, (3, 2, 2, 1), 200, 3, 3, 128, "greedy", ("uniform", 0, 4), 2002,
           kv_capacity=211))
_add(Shape("gqa-mini", "bf16", 512, 4099, 4, 2, (4, 3, 2, 2), 257, 4, 2, 128, "typical", ("uniform", 0, 4), 2003,
           kv_capacity=260))
_add(Shape("33b-mini", "bf16", 256, 1500, 5, 3, (4, 3, 2, 2, 2), 129, 2, 2, 128, "greedy", ("uniform", 0, 5), 2004))
_add(Shape("tiny-fp32-gqa", "f32", 256, 777, 3, 2, (3, 2), 70, 4, 2, 64, "typical", ("uniform", 0, 2), 2005,
           kv_capacity=75))
# batched reduced variants for the tensor-core heads (batch 5..32): odd batch,
# a GQA typical batch of 16, a batch of 32 with half-tile hidden and ragged
# reduction, and 7B-wide heads whose tile counts make the heads' work split
# (124 CTAs on 148 SMs) cut tiles between CTAs in both the layer and the projection
_add(Shape("b5-mini", "bf16", 256, 777, 3, 5, (3, 2), 70, 2, 1, 128, "greedy", ("uniform", 0, 2), 2006))
_add(Shape("gqa-b16-mini", "bf16", 512, 4099, 4, 16, (4, 3, 2, 2), 257, 4, 2, 128, "typical", ("uniform", 0, 4), 2007,
           kv_capacity=260))
_add(Shape("33b-b32-mini", "bf16", 320, 1500, 5, 32, (4, 3, 2, 2, 2), 129, 5, 5, 64, "greedy", ("uniform", 0, 5), 2008))
_add(Shape("13b-b8-split", "bf16", 4096, 5000, 5, 8, (3, 2, 2, 1), 200, 32, 32, 128, "greedy", ("uniform", 0, 4), 2009,
           kv_capacity=211))
# explicit (sparse) trees: subsets of the Cartesian tree chosen by explicit_tree,
# with leaves at several depths -- reduced greedy / typical / fp32 variants,
# the GQA workload with its stated 76 nodes, and the 7B shapes with 64 nodes
_add(Shape("sparse-mini", "bf16", 256, 777, 4, 3, (4, 3, 2, 2), 70, 2, 1, 128, "greedy", ("uniform", 0, 4), 2010,
           sparse_nodes=24))
_add(Shape("sparse-typical-mini", "bf16", 512, 1500, 4, 2, (4, 3, 2, 2), 100, 4, 2, 128, "typical",
           ("uniform", 0, 4), 2011, sparse_nodes=40))
_add(Shape("sparse-f32", "f32", 256, 600, 3, 2, (3, 3, 2), 40, 4, 2, 64, "greedy", ("uniform", 0, 3), 2012,
           sparse_nodes=10))
_add(Shape("gqa76-bf16", "bf16", 4096, 128256, 4, 16, (4, 3, 2, 2), 4096, 32, 8, 128, "typical", ("uniform", 0, 4),
           1005, full_size=True, sparse_nodes=76))
_add(Shape("7b-sparse64", "bf16", 4096, 32000, 5, 1, (4, 3, 2, 2, 1), 1024, 32, 32, 128, "greedy", ("fixed", 3),
           1006, full_size=True, sparse_nodes=64))
# sampling verification: reduced variants (a low temperature keeps the planted
# draws far from ties) and the 7B shapes at temperature 0.7
_add(Shape("sample-mini", "bf16", 640, 3001, 5, 2, (4, 3, 2, 2, 1), 300, 5, 5, 128, "sample", ("uniform", 0, 3),
           2013, kv_capacity=333, temperature=0.3))
_add(Shape("sample-sparse-mini", "bf16", 256, 777, 4, 3, (4, 3, 2, 2), 70, 2, 1, 128, "sample", ("uniform", 0, 4),
           2014, sparse_nodes=24, temperature=0.3, sample_seed=(7, 11), sample_step=3))
_add(Shape("7b-sample", "bf16", 4096, 32000, 5, 1, (4, 3, 2, 2, 1), 1024, 32, 32, 128, "sample", ("fixed", 3),
           1007, full_size=True))
# typical acceptance whose bonus token is drawn (the GQA reduced shapes; 4 x 89 nodes take two node tiles)
_add(Shape("typical-sample-mini", "bf16", 512, 4099, 4, 4, (4, 3, 2, 2), 257, 4, 2, 128, "typical-sample",
           ("uniform", 0, 4), 2015, kv_capacity=260, sample_seed=(21, 22), sample_step=5))
# profiling case: the 7B shapes with a quarter-sized vocabulary (still far
# larger than L2) so that counter replays stay small
_add(Shape("7b-prof", "bf16", 4096, 8192, 5, 1, (4, 3, 2, 2, 1), 1024, 32, 32, 128, "greedy", ("fixed", 3), 4001,
           full_size=True))
# profiling case of the tensor-bound verification: the GQA workload's batch,
# tree and widths with a 32000-row vocabulary (lm_head 262 MB, still past L2)
_add(Shape("gqa-prof", "bf16", 4096, 32000, 4, 16, (4, 3, 2, 2), 1024, 32, 8, 128, "typical", ("uniform", 0, 4), 4002,
           full_size=True))
# profiling case of the tensor-bound attention: the 33B workload with 4 sequences
_add(Shape("33b-prof", "bf16", 6656, 32000, 5, 4, (4, 3, 2, 2, 2), 8192, 52, 52, 128, "greedy", ("uniform", 0, 5), 4003,
           full_size=True))
# edge cases: a chain tree (the mask is causal), a root-only tree, an empty
# cache, the widest tree under the 512-node limit, and the deepest tree
_add(Shape("chain-bf16", "bf16", 256, 999, 3, 2, (1, 1, 1), 64, 2, 2, 128, "greedy", ("uniform", 0, 3), 3001))
_add(Shape("rootonly-f32", "f32", 128, 500, 1, 2, (), 40, 2, 1, 64, "greedy", ("fixed", 0), 3002))
_add(Shape("nocache-bf16", "bf16", 256, 700, 2, 2, (3, 2), 0, 2, 2, 128, "typical", ("uniform", 0, 2), 3003))
_add(Shape("wide-bf16", "bf16", 256, 1200, 3, 1, (8, 8, 6), 100, 2, 1, 128, "greedy", ("fixed", 3), 3004))
_add(Shape("deep-bf16", "bf16", 192, 600, 8, 2, (2, 2, 2, 2, 2, 2, 2, 2), 33, 3, 1, 64, "greedy", ("uniform", 0, 8),
           3005))
# the per-depth list limit (16 entries): the tensor-core heads and the merged
# tree at kmax 16, heads deeper than the tree; the fp32 streaming heads and
# typical acceptance over 16 children per node
_add(Shape("k16-bf16", "bf16", 256, 1200, 3, 2, (16, 16), 60, 2, 1, 128, "greedy", ("uniform", 0, 2), 3006))
_add(Shape("k16-f32", "f32", 128, 800, 2, 2, (16, 9), 40, 2, 1, 64, "typical", ("uniform", 0, 2), 3007))

# tensor tags for seed derivation
_TAG = {"lm_head": 1, "W2": 2, "W1": 3, "b1": 4, "h": 5, "root": 6, "q": 7, "k_tree": 8, "v_tree": 9,
        "k_cache": 10, "v_cache": 11, "u": 12, "q_redraw": 13}


def seed_for(base: int, tag: str, index: int = 0, redraw: int = 0) -> int:
    """Deterministic 63-bit seed for one tensor (or one row of one)."""
    x = (base * 1_000_003 + _TAG[tag] * 7_919 + index * 104_729 + redraw * 15_485_863) & 0x7FFF_FFFF_FFFF_FFFF
    return x


def _randn(shape, seed: int) -> torch.Tensor:
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32)


def _cast(x: torch.Tensor, s: Shape) -> torch.Tensor:
    return x.to(s.torch_dtype)


def draw_h_row(s: Shape, b: int, redraw: int = 0) -> torch.Tensor:
    """Row b of the final hidden state, redraw number ``redraw`` (0 = first)."""
    return _cast(_randn((s.hidden,), seed_for(s.seed, "h", b, redraw)), s)


def draw_q_row(s: Shape, b: int, node: int, redraw: int) -> torch.Tensor:
    """A fresh q row [Hq, Dh] for (b, node); redraw >= 1."""
    return _cast(_randn((s.n_q_heads, s.head_dim), seed_for(s.seed, "q_redraw", b * s.n_nodes + node, redraw)), s)


def make_weights(s: Shape, zero_init: bool = False) -> Dict[str, torch.Tensor]:
    """lm_head [V,H], W1 [K,H,H] (out,in), b1 [K,H], W2 [K,V,H]."""
    H, V, K = s.hidden, s.vocab, s.n_heads
    lm = _cast(_randn((V, H), seed_for(s.seed, "lm_head")) * (1.0 / math.sqrt(H)), s)
    W2 = torch.empty((K, V, H), dtype=s.torch_dtype)
    W1 = torch.empty((K, H, H), dtype=s.torch_dtype)
    b1 = torch.empty((K, H), dtype=s.torch_dtype)
    lm32 = lm.to(torch.float32)
    for k in range(K):
        if zero_init:
            W2[k] = lm
            W1[k].zero_()
            b1[k].zero_()
        else:
            W2[k] = _cast(lm32 + 0.01 * _randn((V, H), seed_for(s.seed, "W2", k)), s)
            W1[k] = _cast(0.02 * _randn((H, H), seed_for(s.seed, "W1", k)), s)
            b1[k] = _cast(0.02 * _randn((H,), seed_for(s.seed, "b1", k)), s)
    del lm32
    return {"lm_head": lm, "W1": W1, "b1": b1, "W2": W2}


def make_activations(s: Shape, h_redraws: Optional[Sequence[int]] = None) -> Dict[str, torch.Tensor]:
    """h [B,H], root_token [B] int32, tree q [B,T,Hq,Dh], k/v tree [B,T,Hkv,Dh],
    k/v cache [B,cap,Hkv,Dh] (rows >= kv_len are filled too but never read)."""
    B, T = s.batch, s.n_nodes
    h = torch.stack([draw_h_row(s, b, (h_redraws[b] if h_redraws else 0)) for b in range(B)])
    g = torch.Generator().manual_seed(seed_for(s.seed, "root"))
    root = torch.randint(0, s.vocab, (B,), generator=g, dtype=torch.int64).to(torch.int32)
    q = _cast(_randn((B, T, s.n_q_heads, s.head_dim), seed_for(s.seed, "q")), s)
    kt = _cast(_randn((B, T, s.n_kv_heads, s.head_dim), seed_for(s.seed, "k_tree")), s)
    vt = _cast(_randn((B, T, s.n_kv_heads, s.head_dim), seed_for(s.seed, "v_tree")), s)
    kc = torch.empty((B, max(s.cap, 1), s.n_kv_heads, s.head_dim), dtype=s.torch_dtype)
    vc = torch.empty_like(kc)
    for b in range(B):  # per sequence, to bound the fp32 temporary
        kc[b] = _cast(_randn((max(s.cap, 1), s.n_kv_heads, s.head_dim), seed_for(s.seed, "k_cache", b)), s)
        vc[b] = _cast(_randn((max(s.cap, 1), s.n_kv_heads, s.head_dim), seed_for(s.seed, "v_cache", b)), s)
    return {"h": h, "root_token": root, "q": q, "k_tree": kt, "v_tree": vt, "k_cache": kc, "v_cache": vc}


def plant(s: Shape, inputs: Dict[str, torch.Tensor], b: int, node: int, token: int) -> None:
    """Overwrite the tree q/k/v rows of (b, node) so that the base model's top
    token at that node is ``token`` (construction in the module docstring)."""
    Dh, Hq, Hkv = s.head_dim, s.n_q_heads, s.n_kv_heads
    G = Hq // Hkv
    lm_row = inputs["lm_head"][token].to(torch.float64)  # [H]
    for g in range(Hkv):
        u = _randn((Dh,), seed_for(s.seed, "u", (b * s.n_nodes + node) * Hkv + g)).to(torch.float64)
        u = u / u.norm()
        m = torch.zeros(Dh, dtype=torch.float64)
        for hh in range(g * G, (g + 1) * G):
            m += lm_row[hh * Dh:(hh + 1) * Dh]
        inputs["k_tree"][b, node, g] = (PLANT_GAMMA_K * u).to(s.torch_dtype)
        inputs["v_tree"][b, node, g] = (PLANT_ALPHA_V * m / m.norm()).to(s.torch_dtype)
        for hh in range(g * G, (g + 1) * G):
            inputs["q"][b, node, hh] = (PLANT_GAMMA_Q * math.sqrt(Dh) * u).to(s.torch_dtype)


def apply_plan(s: Shape, inputs: Dict[str, torch.Tensor], plan: dict) -> None:
    """Apply a stored plan: q-row redraws, then the planted (node, token) pairs."""
    for b, node, r in plan.get("q_redraws", []):
        inputs["q"][b, node] = draw_q_row(s, b, node, r)
    for b, seq in enumerate(plan["seqs"]):
        for node, token in seq["plant"]:
            plant(s, inputs, b, node, token)


def make_inputs(s: Shape, plan: Optional[dict] = None, zero_init: bool = False) -> Dict[str, torch.Tensor]:
    """All step inputs on the CPU; with ``plan`` the stored redraws and plants are applied."""
    out = make_weights(s, zero_init=zero_init)
    out.update(make_activations(s, plan.get("h_redraws") if plan else None))
    if plan:
        apply_plan(s, out, plan)
    return out


PLANS_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "tests", "golden",
                          "plans.json")


def load_plans(path: str = PLANS_PATH) -> dict:
    with open(path) as f:
        return json.load(f)


# ----------------------------------------------------------------------------
# Toy backbone for multi-round decoding.
#
# The decode step's inputs around the path (the tree's queries, keys and
# values, the next hidden state) come from a base model.  For a loop of many
# rounds a stand-in model is needed whose greedy continuation is known and
# whose heads are right part of the time.  This toy draws, per token x:
#   u[x, g]  a random unit vector per kv group g, key K[x, g] = a * u[x, g] and
#            query Q[x, h] = a * u[x, h // G] with a^2 / sqrt(Dh) = 30, so every
#            token attends almost only to its own key (a cache key scores ~N(0, 2)
#            against it),
#   Vt[x, g] a random N(0, 1) value, so the hidden state at token x is close
#            to hv[x] = [Vt[x, h // G] for each q head h] (length H);
# a random cyclic permutation pi of the vocabulary is the greedy continuation:
#   lm_head[pi(x)] = hv[x] / |hv[x]|;
# heads (W1 = b1 = 0, so z = h) with row W2_d[pi^(d+1)(x)] = +hv[x] / |hv[x]|
# when head d is right about x (probability head_acc[d], drawn per (d, x)), else
# -hv[x] / |hv[x]| (the true token then scores lowest and leaves the list).
# These are random draws and row arrangements only: none of the step's
# arithmetic happens here.


@dataclasses.dataclass(frozen=True)
class ToyShape:
    """A toy backbone and the loop run on it (field names as in Shape, so the
    same config builder applies)."""

    name: str
    hidden: int
    vocab: int
    n_heads: int
    batch: int
    topk: Tuple[int, ...]
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    kv_len: int  # cache rows before the first round
    rounds: int
    head_acc: Tuple[float, ...]  # per head depth: chance that the head is right about a token
    seed: int
    dtype: str = "bf16"
    accept: str = "greedy"
    temperature: float = 0.7
    eps: float = 0.3
    delta: float = 0.09

    @property
    def depth(self) -> int:
        return len(self.topk)

    @property
    def kv_capacity(self) -> int:
        """Room for every round's commit (at most depth + 1 rows per round)."""
        return self.kv_len + self.rounds * (self.depth + 1)

    cap = kv_capacity

    @property
    def n_nodes(self) -> int:
        total, level = 1, 1
        for k in self.topk:
            level *= k
            total += level
        return total

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


TOYS: Dict[str, ToyShape] = {}
for _t in (
    ToyShape("toy-mini", 256, 997, 4, 3, (3, 2, 2, 1), 2, 1, 128, 40, 12, (0.9, 0.8, 0.7, 0.6), 5001),
    ToyShape("toy-gqa-mini", 512, 1201, 4, 2, (4, 3, 2), 4, 2, 128, 70, 10, (0.85, 0.7, 0.55, 0.4), 5002),
    ToyShape("toy-7b", 4096, 32000, 5, 1, (4, 3, 2, 2, 1), 32, 32, 128, 1024, 64, (0.9, 0.8, 0.7, 0.6, 0.5),
             5003),
):
    TOYS[_t.name] = _t

_TOY_TAG = {"perm": 1, "u": 2, "v": 3, "right": 4, "cache_k": 5, "cache_v": 6, "root": 7}


def _toy_seed(t: ToyShape, tag: str, index: int = 0) -> int:
    return (t.seed * 1_000_003 + _TOY_TAG[tag] * 7_919 + index * 104_729) & 0x7FFF_FFFF_FFFF_FFFF


def make_toy(t: ToyShape) -> Dict[str, torch.Tensor]:
    """The toy's tables, weights and first-round inputs (CPU tensors):
    Qtab [V,Hq,Dh], Ktab / Vtab [V,Hkv,Dh], lm_head [V,H], W1 [K,H,H], b1 [K,H],
    W2 [K,V,H], k_cache / v_cache [B,cap,Hkv,Dh] (the first kv_len rows drawn,
    the rest zero), kv_lens [B], root_token [B], h [B,H] (the hidden state whose
    greedy continuation is the root), perm [V] (pi) and right [K,V] (1 where
    head k is right about a token)."""
    V, H, K, B = t.vocab, t.hidden, t.n_heads, t.batch
    Hq, Hkv, Dh = t.n_q_heads, t.n_kv_heads, t.head_dim
    G = Hq // Hkv
    dt = t.torch_dtype
    g = torch.Generator().manual_seed(_toy_seed(t, "perm"))
    order = torch.randperm(V, generator=g)
    perm = torch.empty(V, dtype=torch.int64)
    perm[order] = torch.roll(order, -1)  # one cycle through every token
    u = _randn((V, Hkv, Dh), _toy_seed(t, "u"))
    u = u / u.norm(dim=-1, keepdim=True)
    a = math.sqrt(30.0 * math.sqrt(Dh))
    Ktab = (a * u).to(dt)
    Qtab = (a * u).repeat_interleave(G, dim=1).to(dt)
    Vtab = _randn((V, Hkv, Dh), _toy_seed(t, "v")).to(dt)
    hv = Vtab.to(torch.float32).repeat_interleave(G, dim=1).reshape(V, H)
    unit = hv / hv.norm(dim=-1, keepdim=True)
    lm = torch.empty((V, H), dtype=torch.float32)
    lm[perm] = unit
    W2 = torch.empty((K, V, H), dtype=dt)
    right_all = torch.zeros((K, V), dtype=torch.int8)
    step = perm.clone()  # pi^(d+1)
    for d in range(K):
        step = perm[step] if d > 0 else perm[perm]
        acc = t.head_acc[d] if d < len(t.head_acc) else 0.0
        right = torch.rand(V, generator=torch.Generator().manual_seed(_toy_seed(t, "right", d))) < acc
        right_all[d] = right.to(torch.int8)
        rows = torch.where(right[:, None], unit, -unit)
        W2d = torch.empty((V, H), dtype=torch.float32)
        W2d[step] = rows
        W2[d] = W2d.to(dt)
    cap = t.kv_capacity
    kc = torch.zeros((B, cap, Hkv, Dh), dtype=dt)
    vc = torch.zeros((B, cap, Hkv, Dh), dtype=dt)
    for b in range(B):
        kc[b, :t.kv_len] = _randn((t.kv_len, Hkv, Dh), _toy_seed(t, "cache_k", b)).to(dt)
        vc[b, :t.kv_len] = _randn((t.kv_len, Hkv, Dh), _toy_seed(t, "cache_v", b)).to(dt)
    gr = torch.Generator().manual_seed(_toy_seed(t, "root"))
    root = torch.randint(0, V, (B,), generator=gr, dtype=torch.int64)
    inv = torch.empty(V, dtype=torch.int64)
    inv[perm] = torch.arange(V)
    h = hv[inv[root]].to(dt)
    return {"Qtab": Qtab, "Ktab": Ktab, "Vtab": Vtab, "lm_head": lm.to(dt), "W1": torch.zeros((K, H, H), dtype=dt),
            "b1": torch.zeros((K, H), dtype=dt), "W2": W2, "k_cache": kc, "v_cache": vc,
            "kv_lens": torch.full((B,), t.kv_len, dtype=torch.int32), "root_token": root.to(torch.int32), "h": h,
            "perm": perm.to(torch.int32), "right": right_all}
