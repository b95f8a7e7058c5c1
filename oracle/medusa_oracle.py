"""Plain CPU oracle for one Medusa speculative decode step.

TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the benchmark's
CPU-baseline / reference arm may import this module; the CUDA library never
does, and the two share no code.  It is deliberately slow and literal: every
step is the definition written out in float64 (inputs decoded exactly from
their stored fp32 or bf16 values), with a library matmul where the definition
is a matrix product and plain loops elsewhere.

Sources (page title -- section):
  [P1] "Medusa Heads", ultralytics glossary (Italian):
       "Come le teste prevedono i token successivi" -- head structure, the
       zero-initialised head snippet and its printed result;
       "Attenzione sull'albero e accettazione" -- Cartesian candidate tree,
       ancestor-only mask, one verification pass, greedy and typical
       acceptance.
  [P2] "Tetes de decodage Medusa", aiunderstanding.org -- "Plongee profonde"
       (tree attention mask, longest matching prefix, typical acceptance is
       not distribution-exact).
  [P3] "Medusa: Simple LLM Inference Acceleration Framework with Multiple
       Decoding Heads", arXiv 2401.10774 -- abstract.

Readings where the pages leave a step open (each is also listed with the
design notes):
  R1  head k (1-based) scores position t+k+1; the root of the tree is the base
      model's token for t+1, given as input (P1 first section).
  R2  "its own ancestors" includes the node itself, so a chain tree gives the
      causal mask.
  R3  attention scale 1/sqrt(Dh); no rotary embedding; q head h reads kv head
      floor(h / (Hq/Hkv)).
  R4  lm_head is applied directly to the concatenated attention output of a
      node (there is no backbone block in this step).
  R5  ties in top-k and argmax go to the lower token index.
  R6  heads deeper than the tree still run; their top-1 is reported.
  R7  typical acceptance: p = softmax(logits / temperature); entropy in nats;
      threshold min(eps, delta * exp(-H)); a child is kept when p(token) is
      strictly greater than the threshold; the longest accepted path wins,
      ties to the lowest node index at the first divergence; the bonus token
      is the argmax at the last accepted node.
  R8  the attention output is rounded to its storage type (bf16 or fp32)
      before the verification projection reads it.
  R15 typical acceptance with a sampled bonus: the acceptance as R7, the
      bonus token drawn from softmax(logits / temperature) at the last kept
      node with the sampling mode's Gumbel-max draw (same noise keying).
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence

import numpy as np


# ----------------------------------------------------------------- decoding --

def decode(a: np.ndarray) -> np.ndarray:
    """Exact float64 value of stored data.  uint16 arrays hold bf16 bit
    patterns (the upper half of an fp32); float arrays are widened."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 (ties to even), returned as
    float64.  bf16 keeps 8 exponent bits and 7 stored mantissa bits."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    ax = np.abs(x)
    tiny = ax < 2.0 ** -126  # bf16 subnormal range: spacing 2^-133
    q = x[tiny] / 2.0 ** -133
    out[tiny] = np.round(q) * 2.0 ** -133  # np.round rounds halves to even
    xn = x[~tiny]
    bits = xn.view(np.uint64)
    keep = (bits >> np.uint64(45)) & np.uint64(1)
    bits = (bits + np.uint64((1 << 44) - 1) + keep) & ~np.uint64((1 << 45) - 1)
    out[~tiny] = bits.view(np.float64)
    return out


def round_to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """R8: the value the step stores for the attention output."""
    if dtype == "bf16":
        return round_to_bf16(x)
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


# ---------------------------------------------------------------- the heads --

def silu(x: np.ndarray) -> np.ndarray:
    """SiLU(x) = x * sigmoid(x)  [P1, "Come le teste prevedono..."]."""
    return x / (1.0 + np.exp(-x))


def head_hidden(h, W1, b1) -> np.ndarray:
    """z[b,k] = h[b] + SiLU(W1_k h[b] + b1_k): the residual SiLU feed-forward
    layer of each Medusa head [P1, "Come le teste prevedono i token
    successivi"].  h [B,H], W1 [K,H,H] (out, in), b1 [K,H] -> z [B,K,H]."""
    h = decode(h)
    K = W1.shape[0]
    B, H = h.shape
    z = np.empty((B, K, H))
    for k in range(K):
        Wk = decode(W1[k])
        bk = decode(b1[k])
        a = h @ Wk.T + bk  # [B,H]
        z[:, k, :] = h + silu(a)
    return z


def head_logits(z: np.ndarray, W2, heads: Optional[Sequence[int]] = None) -> np.ndarray:
    """logits[b,k,v] = W2_k[v] . z[b,k]: the vocabulary projection of each head
    (no bias) [P1, same section].  z [B,K,H], W2 [K,V,H] -> [B,K,V]."""
    B, K, H = z.shape
    V = W2.shape[1]
    ks = range(K) if heads is None else heads
    out = np.full((B, K, V), np.nan)
    for k in ks:
        out[:, k, :] = z[:, k, :] @ decode(W2[k]).T
    return out


def base_logits(h, lm_head) -> np.ndarray:
    """lm_head(h): the base model's next-token scores [P1, same section]."""
    return decode(h) @ decode(lm_head).T


def topk_lists(logits: np.ndarray, topk: Sequence[int]):
    """Per-head top-k (R5, R6): head d (0-based) keeps topk[d] tokens when
    d < depth, else 1; order is descending logit, ties to the lower index.
    Returns idx int32 [B,K,kmax] (pad -1) and val float64 [B,K,kmax] (pad -inf)."""
    B, K, V = logits.shape
    kmax = max(list(topk) + [1])
    idx = np.full((B, K, kmax), -1, dtype=np.int32)
    val = np.full((B, K, kmax), -np.inf)
    ids = np.arange(V)
    for b in range(B):
        for k in range(K):
            n = topk[k] if k < len(topk) else 1
            # library sort on the key (-logit, token id): primary key last
            order = np.lexsort((ids, -logits[b, k]))[:n]
            idx[b, k, :n] = order
            val[b, k, :n] = logits[b, k, order]
    return idx, val


# ----------------------------------------------------------------- the tree --

class Tree:
    """Candidate tree [P1, "Attenzione sull'albero e accettazione"]: the
    heads' top-k lists combined by Cartesian product, prefixes shared -- or,
    given ``parent``/``rank``, an explicit subset of that tree (fewer
    branches, same structure).  Nodes are numbered breadth-first: node 0 is the
    root; the nodes of depth d follow those of depth d-1, ordered by parent,
    then by rank in the head-d list.  A node of rank r at depth d carries head
    d's r-th candidate."""

    def __init__(self, topk: Sequence[int], parent: Optional[Sequence[int]] = None,
                 rank: Optional[Sequence[int]] = None):
        self.topk = list(topk)
        self.depth_max = len(self.topk)
        if parent is None:
            parent, depth, rank = [-1], [0], [0]
            level = [0]
            for d in range(1, self.depth_max + 1):
                nxt = []
                for p in level:
                    for r in range(self.topk[d - 1]):
                        parent.append(p)
                        depth.append(d)
                        rank.append(r)
                        nxt.append(len(parent) - 1)
                level = nxt
        else:
            parent, rank = list(parent), list(rank)
            assert parent[0] == -1 and rank[0] == 0
            depth = [0]
            for i in range(1, len(parent)):
                assert 0 <= parent[i] < i
                depth.append(depth[parent[i]] + 1)
                assert depth[i] <= self.depth_max and 0 <= rank[i] < self.topk[depth[i] - 1]
                assert (depth[i - 1], parent[i - 1], rank[i - 1]) < (depth[i], parent[i], rank[i])
        self.parent = np.array(parent, dtype=np.int32)
        self.depth = np.array(depth, dtype=np.int32)
        self.rank = np.array(rank, dtype=np.int32)
        self.T = len(parent)
        self.children: List[List[int]] = [[] for _ in range(self.T)]
        for i in range(1, self.T):
            self.children[parent[i]].append(i)
        self.leaves = [i for i in range(self.T) if not self.children[i]]
        # R2: node i sees exactly the nodes on its chain to the root, itself included
        self.mask = np.zeros((self.T, self.T), dtype=bool)
        for i in range(self.T):
            j = i
            while j >= 0:
                self.mask[i, j] = True
                j = parent[j]
        # root-to-leaf node ids, -1 after a leaf shallower than the tree depth
        self.paths = np.array([self.chain(l) + [-1] * (self.depth_max + 1 - len(self.chain(l)))
                               for l in self.leaves], dtype=np.int32).reshape(len(self.leaves), self.depth_max + 1)

    @classmethod
    def for_shape(cls, shape) -> "Tree":
        """The workload's tree: Cartesian, or its explicit parent/rank lists."""
        return cls(shape.topk, getattr(shape, "tree_parent", None), getattr(shape, "tree_rank", None))

    def chain(self, i: int) -> List[int]:
        """Nodes from the root down to i."""
        out = []
        while i >= 0:
            out.append(i)
            i = int(self.parent[i])
        return out[::-1]

    def tokens(self, topk_idx: np.ndarray, root_token: Sequence[int]) -> np.ndarray:
        """token[b,0] = root token (R1); token[b,i] = head (depth_i)'s candidate
        of rank rank_i."""
        B = topk_idx.shape[0]
        tok = np.zeros((B, self.T), dtype=np.int32)
        for b in range(B):
            tok[b, 0] = root_token[b]
            for i in range(1, self.T):
                tok[b, i] = topk_idx[b, self.depth[i] - 1, self.rank[i]]
        return tok


# --------------------------------------------------------- tree attention ---

def tree_attention(q, k_tree, v_tree, k_cache, v_cache, kv_len, mask: np.ndarray,
                   nodes: Optional[Sequence[int]] = None, batches: Optional[Sequence[int]] = None) -> np.ndarray:
    """Every tree node attends, in one pass, to the whole KV cache and to the
    tree nodes its mask row allows [P1, "Attenzione sull'albero e
    accettazione"; P2, "Plongee profonde"]:
        o[b,i,h] = sum_j softmax_j(q[b,i,h] . k_j / sqrt(Dh)) v_j
    over j in cache[0..kv_len) and {tree node j : mask[i,j]}, with kv head
    floor(h/G) (R3).  ``kv_len`` is one length or one per sequence.  Shapes:
    q [B,T,Hq,Dh], k/v tree [B,T,Hkv,Dh], k/v cache [B,cap,Hkv,Dh].  Returns
    o [B,T,Hq*Dh] in float64; rows outside ``nodes`` / ``batches`` are NaN."""
    B, T, Hq, Dh = q.shape
    Hkv = k_tree.shape[2]
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(Dh)
    nodes = list(range(T)) if nodes is None else list(nodes)
    batches = list(range(B)) if batches is None else list(batches)
    o = np.full((B, T, Hq * Dh), np.nan)
    lens = [int(kv_len)] * B if np.ndim(kv_len) == 0 else [int(x) for x in kv_len]
    for b in batches:
        L = lens[b]
        for g in range(Hkv):
            Kc = decode(k_cache[b, :L, g, :])
            Vc = decode(v_cache[b, :L, g, :])
            Kt = decode(k_tree[b, :, g, :])
            Vt = decode(v_tree[b, :, g, :])
            for h in range(g * G, (g + 1) * G):
                Q = decode(q[b, nodes, h, :])  # [n,Dh]
                s_cache = (Q @ Kc.T) * scale  # [n,L]
                s_tree = (Q @ Kt.T) * scale  # [n,T]
                s_tree = np.where(mask[nodes, :], s_tree, -np.inf)
                s = np.concatenate([s_cache, s_tree], axis=1)
                s = s - s.max(axis=1, keepdims=True)
                p = np.exp(s)
                p = p / p.sum(axis=1, keepdims=True)
                out = p[:, :L] @ Vc + p[:, L:] @ Vt
                o[b, nodes, h * Dh:(h + 1) * Dh] = out
    return o


# -------------------------------------------------------------- verification -

def verify_stats(o_stored: np.ndarray, lm_head, temperature: Optional[float] = None,
                 rows: Optional[Sequence[int]] = None, chunk: int = 256) -> Dict[str, np.ndarray]:
    """Base-model scores of every tree node, lm_head . o_i (R4), and their
    summaries [P1, "Attenzione sull'albero e accettazione"]:
      argmax (R5) and max logit, for greedy acceptance;
      with a temperature: log-partition lse = log sum exp(logit/temp) and
      entropy H = -sum p log p of p = softmax(logit/temp), for typical
      acceptance;
      'second', the runner-up score, used only to check input margins.
    o_stored [N,H] (already rounded to storage, R8).  Returns float64 arrays of
    length N (NaN / -1 outside ``rows``), plus 'logits' for the rows when N is
    small enough to keep them."""
    N = o_stored.shape[0]
    rows = list(range(N)) if rows is None else list(rows)
    W = decode(lm_head)
    res = {"argmax": np.full(N, -1, dtype=np.int64), "maxlogit": np.full(N, np.nan),
           "second": np.full(N, np.nan), "lse": np.full(N, np.nan), "entropy": np.full(N, np.nan)}
    for c in range(0, len(rows), chunk):
        rr = rows[c:c + chunk]
        L = o_stored[rr] @ W.T  # [n,V]
        res["argmax"][rr] = np.argmax(L, axis=1)  # first maximum = lowest index
        res["maxlogit"][rr] = L.max(axis=1)
        res["second"][rr] = np.sort(L, axis=1)[:, -2]  # runner-up score (margin checks)
        if temperature is not None:
            x = L / temperature
            m = x.max(axis=1, keepdims=True)
            e = np.exp(x - m)
            Z = e.sum(axis=1, keepdims=True)
            p = e / Z
            res["lse"][rr] = (m + np.log(Z))[:, 0]
            with np.errstate(divide="ignore", invalid="ignore"):
                plogp = np.where(p > 0, p * np.log(p), 0.0)
            res["entropy"][rr] = -plogp.sum(axis=1)
    return res


# Counter-based noise for sampling verification.  Philox4x32-10 (Salmon,
# Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11):
# ten rounds over a 128-bit counter; each round multiplies two counter words
# by fixed constants, the high halves are xored with the other two words and
# the key, and the key advances by a Weyl sequence between rounds.
PHILOX_MUL = (0xD2511F53, 0xCD9E8D57)
PHILOX_WEYL = (0x9E3779B9, 0xBB67AE85)
_U32 = 0xFFFFFFFF


def philox4x32_10(c0, c1, c2, c3, k0: int, k1: int):
    """Vectorised over numpy arrays of counter words (held as uint64 < 2^32)."""
    c = [np.asarray(x, dtype=np.uint64) for x in (c0, c1, c2, c3)]
    k0, k1 = np.uint64(k0), np.uint64(k1)
    for r in range(10):
        if r:
            k0 = (k0 + np.uint64(PHILOX_WEYL[0])) & np.uint64(_U32)
            k1 = (k1 + np.uint64(PHILOX_WEYL[1])) & np.uint64(_U32)
        p0 = np.uint64(PHILOX_MUL[0]) * c[0]
        p1 = np.uint64(PHILOX_MUL[1]) * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & np.uint64(_U32)
        hi1, lo1 = p1 >> np.uint64(32), p1 & np.uint64(_U32)
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
    return c


def gumbel_noise(seed: Sequence[int], step: int, node: int, V: int) -> np.ndarray:
    """Noise of vocabulary rows 0..V-1 at global node n (= b*T + i): Philox
    word n % 4 of counter (v, n // 4, step, 0) under key (seed0, seed1); its top
    24 bits give u = (w >> 8 + 1/2) / 2^24 in (0, 1) and g = -ln(-ln u), a
    standard Gumbel variable."""
    v = np.arange(V, dtype=np.uint64)
    z = np.zeros(V, dtype=np.uint64)
    words = philox4x32_10(v, z + np.uint64(node // 4), z + np.uint64(step), z, int(seed[0]), int(seed[1]))
    u = ((words[node % 4] >> np.uint64(8)).astype(np.float64) + 0.5) / 16777216.0
    return -np.log(-np.log(u))


def sample_stats(o_stored: np.ndarray, lm_head, temperature: float, seed: Sequence[int], step: int,
                 rows: Optional[Sequence[int]] = None,
                 node_ids: Optional[Sequence[int]] = None) -> Dict[str, np.ndarray]:
    """Sampling verification: each node draws its token from softmax(logit /
    temperature) by the Gumbel-max rule, argmax_v(logit_v / temperature + g_v)
    (ties to the lower id).  Row r of ``o_stored`` is global node node_ids[r]
    (default r) for the noise.  Returns 'argmax' (the draw), 'maxlogit' (the
    winning perturbed score) and 'second' (the runner-up, for margin checks)."""
    N = o_stored.shape[0]
    rows = list(range(N)) if rows is None else list(rows)
    node_ids = list(range(N)) if node_ids is None else list(node_ids)
    W = decode(lm_head)
    res = {"argmax": np.full(N, -1, dtype=np.int64), "maxlogit": np.full(N, np.nan), "second": np.full(N, np.nan),
           "lse": np.full(N, np.nan), "entropy": np.full(N, np.nan)}
    for n in rows:
        x = (o_stored[n] @ W.T) / temperature + gumbel_noise(seed, step, node_ids[n], W.shape[0])
        res["argmax"][n] = int(np.argmax(x))
        srt = np.sort(x)
        res["maxlogit"][n], res["second"][n] = srt[-1], srt[-2]
    return res


def token_logprob(o_stored_row: np.ndarray, lm_head, token: int, temperature: float, lse: float) -> float:
    """log p(token) under softmax(lm_head . o / temperature)."""
    return float(o_stored_row @ decode(lm_head[token])) / temperature - lse


def typical_threshold(entropy: float, eps: float, delta: float) -> float:
    """Entropy-tied acceptance threshold (R7): min(eps, delta * exp(-H))."""
    return min(eps, delta * math.exp(-entropy))


# ---------------------------------------------------------------- acceptance -

def accept_greedy(tree: Tree, tokens_b: np.ndarray, argmax_b: np.ndarray):
    """Greedy acceptance [P1, "Attenzione sull'albero e accettazione"]: a
    candidate is kept when it equals the base model's top choice at its
    parent; walk from the root while some child matches (tokens of one
    top-k list are distinct, so at most one does).  Returns
    (length, tokens, nodes incl. root, bonus = top choice at the last node)."""
    cur, nodes, toks = 0, [0], []
    for _ in range(tree.depth_max):
        nxt = None
        for c in tree.children[cur]:
            if tokens_b[c] == argmax_b[cur]:
                nxt = c
                break
        if nxt is None:
            break
        nodes.append(nxt)
        toks.append(int(tokens_b[nxt]))
        cur = nxt
    return len(toks), toks, nodes, int(argmax_b[cur])


def accept_rejection(tree: Tree, tokens_b: np.ndarray, probs, uniform):
    """Rejection sampling against the base model over the tree's fixed
    candidates [P2: exact rejection sampling verifies the candidates against
    the base model's distribution, so the output keeps that distribution]:
    at the current node its children are tried in rank order; child i's token
    is accepted with its base probability renormalised over the tokens not
    yet rejected, p(t_i) / (1 - sum_{j<i} p(t_j)) (a candidate of probability
    one is the whole remaining mass); if one is accepted the walk continues
    from it, else the bonus token is drawn from p with the rejected tokens
    removed.  ``probs(node)`` is the base distribution at a node (length V),
    ``uniform()`` a draw from U(0, 1).  Returns (length, tokens, nodes incl.
    root, bonus)."""
    cur, nodes, toks = 0, [0], []
    while True:
        p = np.array(probs(cur), dtype=np.float64)
        rest = 1.0
        nxt = None
        for c in tree.children[cur]:
            t = int(tokens_b[c])
            if rest > 0 and uniform() * rest < p[t]:
                nxt = c
                break
            rest -= p[t]
            p[t] = 0.0
        if nxt is None:
            q = p / p.sum()
            bonus = int(np.searchsorted(np.cumsum(q), uniform() * q.sum(), side="right"))
            return len(toks), toks, nodes, min(bonus, len(q) - 1)
        nodes.append(nxt)
        toks.append(int(tokens_b[nxt]))
        cur = nxt


def accept_typical(tree: Tree, tokens_b: np.ndarray, argmax_b: np.ndarray, keep_edge):
    """Typical acceptance (R7): ``keep_edge(parent, child)`` says whether the
    child's token clears its parent's entropy-tied threshold; the longest
    chain of kept edges from the root wins, ties to the lowest node index at
    the first divergence (a depth-first walk in node order keeps the first
    longest chain it meets)."""
    best = [0]

    def walk(path):
        nonlocal best
        if len(path) > len(best):
            best = list(path)
        for c in tree.children[path[-1]]:
            if keep_edge(path[-1], c):
                walk(path + [c])

    walk([0])
    toks = [int(tokens_b[n]) for n in best[1:]]
    return len(toks), toks, best, int(argmax_b[best[-1]])


# ------------------------------------------------ around the step (commit) --

def kv_commit(k_cache, v_cache, k_tree, v_tree, acc_nodes, accept_len, kv_lens):
    """The kept branch is appended for the next round [P1, "Attenzione
    sull'albero e accettazione"]: for each sequence b, the key / value rows of
    its accepted nodes acc_nodes[b][0..n] (root first, n = accept_len[b]) go
    to cache rows kv_lens[b] .. kv_lens[b] + n, and the length grows by n + 1.
    Returns new (k_cache, v_cache, kv_lens); the inputs are not modified."""
    kc, vc = np.array(k_cache, copy=True), np.array(v_cache, copy=True)
    lens = [int(x) for x in kv_lens]
    for b in range(len(lens)):
        n = int(accept_len[b])
        for d in range(n + 1):
            node = int(acc_nodes[b][d])
            kc[b, lens[b] + d] = k_tree[b, node]
            vc[b, lens[b] + d] = v_tree[b, node]
        lens[b] += n + 1
    return kc, vc, np.array(lens, dtype=np.int32)


def next_inputs(attn_out_stored, acc_nodes, accept_len, bonus):
    """The next round starts from the last accepted node: its attention output
    (what the base lm_head scored, R4) is the next hidden state and the bonus
    token the next root (R1).  Returns (h_next [B,H], root_next [B])."""
    B = attn_out_stored.shape[0]
    h = np.stack([attn_out_stored[b, int(acc_nodes[b][int(accept_len[b])])] for b in range(B)])
    return h, np.array([int(x) for x in bonus], dtype=np.int32)


# ------------------------------------------------------ vocabulary shards --
# The step is memory-bound [P3, abstract], so at batch 1 only a split of the
# weights cuts the bytes each GPU reads: shard s holds vocabulary rows
# [v0, v1) of every head projection and of lm_head, computes what those rows
# give, and the shards' small partial results are combined.  These functions
# state that split on the CPU: what one shard computes, and the combination,
# whose result must equal the unsplit step.

def shard_topk(z: np.ndarray, W2_shard, v0: int, topk: Sequence[int]):
    """One shard's per-head top-k (R5, R6) over its rows: W2_shard [K,Vs,H]
    holds rows v0 .. v0+Vs-1 of every head.  Token ids are global (local row
    + v0; ties still go to the lower id).  Returns idx [B,K,kmax] (pad -1),
    val [B,K,kmax] (pad -inf)."""
    idx, val = topk_lists(head_logits(z, W2_shard), topk)
    return np.where(idx >= 0, idx + v0, -1).astype(np.int32), val


def merge_topk(parts: Sequence, topk: Sequence[int]):
    """Global per-head top-k from the shards' lists [(idx, val), ...]: the
    union of the candidates, again by descending value, ties to the lower
    id; also the (shard, rank in that shard's list) each entry came from."""
    B, K, kmax = parts[0][0].shape
    idx = np.full((B, K, kmax), -1, dtype=np.int32)
    val = np.full((B, K, kmax), -np.inf)
    src = np.full((B, K, kmax, 2), -1, dtype=np.int32)
    for b in range(B):
        for k in range(K):
            n = topk[k] if k < len(topk) else 1
            cand = [(-float(pv[b, k, j]), int(pi[b, k, j]), si, j) for si, (pi, pv) in enumerate(parts)
                    for j in range(kmax) if pi[b, k, j] >= 0]
            cand.sort()
            for r, (nv, t, si, j) in enumerate(cand[:n]):
                idx[b, k, r], val[b, k, r], src[b, k, r] = t, -nv, (si, j)
    return idx, val, src


def shard_node_states(o_stored: np.ndarray, lm_shard, v0: int, temperature: Optional[float] = None):
    """One shard's scores of every node over its lm_head rows, reduced to a
    state that combines across shards: the maximum m and its (global, lowest)
    id, and with a temperature T, z = sum_v exp(t_v) and s = sum_v exp(t_v) t_v
    with t_v = (logit_v - m) / T (so log-partition = m / T + ln z, entropy =
    ln z - s / z).  Returns arrays m, i, z, s over the nodes."""
    L = o_stored @ decode(lm_shard).T  # [N, Vs]
    m = L.max(axis=1)
    i = np.argmax(L, axis=1) + v0  # first maximum = lowest id
    if temperature is None:
        return {"m": m, "i": i, "z": np.ones_like(m), "s": np.zeros_like(m)}
    t = (L - m[:, None]) / temperature
    e = np.exp(t)
    return {"m": m, "i": i, "z": e.sum(axis=1), "s": (e * t).sum(axis=1)}


def merge_node_states(parts: Sequence[Dict[str, np.ndarray]], temperature: Optional[float] = None):
    """Combination of the shards' node states: the larger maximum wins (ties
    to the lower id); with a temperature each shard's sums are brought to the
    common maximum, z = sum_s z_s e^(d_s) and s = sum_s e^(d_s) (s_s + z_s d_s)
    with d_s = (m_s - m) / T.  Returns argmax, maxlogit and (with T) lse and
    entropy, as verify_stats names them."""
    m = np.max(np.stack([p["m"] for p in parts]), axis=0)
    i = np.full(m.shape, np.iinfo(np.int64).max)
    for p in parts:
        i = np.where(p["m"] == m, np.minimum(i, p["i"]), i)
    res = {"argmax": i, "maxlogit": m}
    if temperature is not None:
        z = np.zeros_like(m)
        ss = np.zeros_like(m)
        for p in parts:
            d = (p["m"] - m) / temperature
            z += p["z"] * np.exp(d)
            ss += np.exp(d) * (p["s"] + p["z"] * d)
        res["lse"] = m / temperature + np.log(z)
        res["entropy"] = np.log(z) - ss / z
    return res


# ------------------------------------------------------- rounds of decoding --

def decode_rounds(toy: Dict[str, np.ndarray], shape, rounds: int) -> Dict[str, list]:
    """Round after round of Medusa decoding over a table backbone [P1,
    "Attenzione sull'albero e accettazione": the kept branch is appended and
    the next round starts from it].  A round: heads and top-k on the hidden
    state, the candidate tree, the tree's queries / keys / values looked up
    per token in the backbone's tables (Qtab [V,Hq,Dh], Ktab / Vtab
    [V,Hkv,Dh]), tree attention over each sequence's grown cache, greedy
    verification and acceptance, then the commit of the kept branch (root
    first) and the next inputs (hidden state of the last kept node, the bonus
    as the next root).  ``toy`` holds numpy arrays (bf16 as uint16 bit
    patterns) as synth.make_toy lays them out.  Returns per round the root,
    accept_len, acc_tokens, acc_nodes and bonus of every sequence."""
    topk = list(shape.topk)
    tree = Tree(topk)
    kc, vc = toy["k_cache"], toy["v_cache"]
    lens = [int(x) for x in toy["kv_lens"]]
    h, root = toy["h"], [int(x) for x in toy["root_token"]]
    out = {k: [] for k in ("root", "accept_len", "acc_tokens", "acc_nodes", "bonus")}
    for _ in range(rounds):
        z = head_hidden(h, toy["W1"], toy["b1"])
        idx, _ = topk_lists(head_logits(z, toy["W2"]), topk)
        tok = tree.tokens(idx, root)
        B, T = tok.shape
        q, kt, vt = toy["Qtab"][tok], toy["Ktab"][tok], toy["Vtab"][tok]
        o = round_to_storage(tree_attention(q, kt, vt, kc, vc, lens, tree.mask), shape.dtype)
        am = verify_stats(o.reshape(B * T, -1), toy["lm_head"])["argmax"].reshape(B, T)
        acc = [accept_greedy(tree, tok[b], am[b]) for b in range(B)]
        n = [a[0] for a in acc]
        nodes = [a[2] for a in acc]
        out["root"].append(list(root))
        out["accept_len"].append(n)
        out["acc_tokens"].append([a[1] for a in acc])
        out["acc_nodes"].append(nodes)
        out["bonus"].append([a[3] for a in acc])
        kc, vc, lens = kv_commit(kc, vc, kt, vt, nodes, n, lens)
        lens = [int(x) for x in lens]
        h, root = next_inputs(o, nodes, n, [a[3] for a in acc])
        root = [int(x) for x in root]
    return out


# -------------------------------------------------------------- whole step --

def step(inp: Dict[str, np.ndarray], shape, nodes_only: Optional[Dict[int, Sequence[int]]] = None) -> Dict:
    """One decode step, stages in order: heads, top-k, tree, tree attention,
    verification, acceptance.  ``inp`` holds numpy arrays (bf16 as uint16
    bit patterns); ``shape`` carries sizes and the acceptance rule.  With
    ``nodes_only`` = {b: [nodes]} the attention and verification run only on
    those nodes (acceptance then must not leave them)."""
    topk = list(shape.topk)
    z = head_hidden(inp["h"], inp["W1"], inp["b1"])
    logits = head_logits(z, inp["W2"])
    idx, val = topk_lists(logits, topk)
    tree = Tree.for_shape(shape)
    tok = tree.tokens(idx, inp["root_token"])
    B, T = tok.shape
    H = shape.hidden
    o = np.full((B, T, H), np.nan)
    for b in range(B):
        nb = None if nodes_only is None else nodes_only[b]
        ob = tree_attention(inp["q"], inp["k_tree"], inp["v_tree"], inp["k_cache"], inp["v_cache"],
                            shape.kv_len, tree.mask, nodes=nb, batches=[b])
        o[b] = ob[b]
    o_st = round_to_storage(o, shape.dtype)
    typical = shape.accept in ("typical", "typical-sample")
    flat = o_st.reshape(B * T, H)
    rows = None
    if nodes_only is not None:
        rows = [b * T + i for b in range(B) for i in nodes_only[b]]
    if shape.accept == "sample":
        stats = sample_stats(flat, inp["lm_head"], shape.temperature, shape.sample_seed, shape.sample_step, rows=rows)
    else:
        stats = verify_stats(flat, inp["lm_head"], shape.temperature if typical else None, rows=rows)
    argmax = stats["argmax"].reshape(B, T)
    res = {"z": z, "head_logits": logits, "topk_idx": idx, "topk_val": val, "tree": tree, "tokens": tok,
           "attn_out": o_st, "argmax": argmax, "maxlogit": stats["maxlogit"].reshape(B, T),
           "second": stats["second"].reshape(B, T), "lse": stats["lse"].reshape(B, T), "entropy": stats["entropy"].reshape(B, T),
           "accept_len": [], "acc_tokens": [], "acc_nodes": [], "bonus": []}
    if shape.accept == "typical-sample":  # R15: the bonus is a draw from the base distribution
        draws = sample_stats(flat, inp["lm_head"], shape.temperature, shape.sample_seed, shape.sample_step,
                             rows=rows)
        res["draw"] = draws["argmax"].reshape(B, T)
        res["draw_max"] = draws["maxlogit"].reshape(B, T)
        res["draw_second"] = draws["second"].reshape(B, T)
    for b in range(B):
        if typical:
            def keep(p, c, b=b):
                row = flat[b * T + p]
                if np.isnan(row).any():
                    return False
                lp = token_logprob(row, inp["lm_head"], int(tok[b, c]), shape.temperature, stats["lse"][b * T + p])
                thr = typical_threshold(stats["entropy"][b * T + p], shape.eps, shape.delta)
                return math.exp(lp) > thr
            n, tk, nd, bonus = accept_typical(tree, tok[b], argmax[b], keep)
            if shape.accept == "typical-sample":
                bonus = int(res["draw"][b, nd[-1]])
        else:
            n, tk, nd, bonus = accept_greedy(tree, tok[b], argmax[b])
        res["accept_len"].append(n)
        res["acc_tokens"].append(tk)
        res["acc_nodes"].append(nd)
        res["bonus"].append(bonus)
    return res
