"""Planted mistakes in a copy of the oracle (CPU only) must fail the pins:
evidence that the pins would catch a dropped term, a wrong sign or index, or
a transposed operand in the oracle itself."""
from __future__ import annotations

import math
import types

import numpy as np
import pytest

from oracle import medusa_oracle as O
from tests import test_oracle_pins as P


def mutant(**repl):
    m = types.ModuleType("oracle_mutant")
    m.__dict__.update({k: v for k, v in O.__dict__.items() if not k.startswith("__")})
    m.__dict__.update(repl)
    return m


def _no_residual(h, W1, b1):
    h = O.decode(h)
    z = np.empty((h.shape[0], W1.shape[0], h.shape[1]))
    for k in range(W1.shape[0]):
        z[:, k] = O.silu(h @ O.decode(W1[k]).T + O.decode(b1[k]))
    return z


def _no_bias(h, W1, b1):
    h = O.decode(h)
    z = np.empty((h.shape[0], W1.shape[0], h.shape[1]))
    for k in range(W1.shape[0]):
        z[:, k] = h + O.silu(h @ O.decode(W1[k]).T)
    return z


def _transposed_w1(h, W1, b1):
    h = O.decode(h)
    z = np.empty((h.shape[0], W1.shape[0], h.shape[1]))
    for k in range(W1.shape[0]):
        z[:, k] = h + O.silu(h @ O.decode(W1[k]) + O.decode(b1[k]))
    return z


def _silu_sign(x):
    return x / (1.0 + np.exp(x))


def _topk_high_tie(logits, topk):
    B, K, V = logits.shape
    idx = np.full((B, K, max(topk)), -1, dtype=np.int32)
    val = np.full((B, K, max(topk)), -np.inf)
    for b in range(B):
        for k in range(K):
            n = topk[k] if k < len(topk) else 1
            order = np.lexsort((-np.arange(V), -logits[b, k]))[:n]
            idx[b, k, :n] = order
            val[b, k, :n] = logits[b, k, order]
    return idx, val


class _DescTree(O.Tree):
    """mask transposed: a node sees its descendants instead of its ancestors"""

    def __init__(self, topk, parent=None, rank=None):
        super().__init__(topk, parent, rank)
        self.mask = self.mask.T.copy()


class _NoSelfTree(O.Tree):
    """mask without the node itself"""

    def __init__(self, topk, parent=None, rank=None):
        super().__init__(topk, parent, rank)
        np.fill_diagonal(self.mask, False)
        self.mask[0, 0] = True


class _DeepLeavesTree(O.Tree):
    """shallow leaves of an explicit tree dropped (paths only at full depth)"""

    def __init__(self, topk, parent=None, rank=None):
        super().__init__(topk, parent, rank)
        keep = [i for i, l in enumerate(self.leaves) if self.depth[l] == self.depth_max]
        self.leaves = [self.leaves[i] for i in keep]
        self.paths = self.paths[keep]


def _typical_last_longest(tree, tokens_b, argmax_b, keep_edge):
    # ties to the LAST longest chain met (the highest node at the first divergence)
    best = [0]

    def walk(path):
        nonlocal best
        if len(path) >= len(best):
            best = list(path)
        for c in tree.children[path[-1]]:
            if keep_edge(path[-1], c):
                walk(path + [c])

    walk([0])
    toks = [int(tokens_b[n]) for n in best[1:]]
    return len(toks), toks, best, int(argmax_b[best[-1]])


def _commit_off_by_one(k_cache, v_cache, k_tree, v_tree, acc_nodes, accept_len, kv_lens):
    # rows written one position past the cache end
    return O.kv_commit(k_cache, v_cache, k_tree, v_tree, acc_nodes, accept_len, [l + 1 for l in kv_lens])


def _attn_uniform_len(q, k_tree, v_tree, k_cache, v_cache, kv_len, mask, nodes=None, batches=None):
    # per-sequence lengths ignored: the first one for every sequence
    L = kv_len if np.ndim(kv_len) == 0 else int(kv_len[0])
    return O.tree_attention(q, k_tree, v_tree, k_cache, v_cache, L, mask, nodes, batches)


def _gumbel_sign(seed, step, node, V):
    return -O.gumbel_noise(seed, step, node, V)  # -g is not Gumbel-max noise


def _gumbel_one_word(seed, step, node, V):
    return O.gumbel_noise(seed, step, node - node % 4, V)  # word 0 for every node of a counter


def _philox(rounds=10, mul=O.PHILOX_MUL, weyl=O.PHILOX_WEYL, bump_first=False, order=(0, 1, 2, 3)):
    """A Philox4x32 variant with one planted mistake."""
    U = 0xFFFFFFFF

    def f(c0, c1, c2, c3, k0, k1):
        c = [np.asarray(x, dtype=np.uint64) for x in (c0, c1, c2, c3)]
        k0, k1 = np.uint64(k0), np.uint64(k1)
        for r in range(rounds):
            if r or bump_first:
                k0 = (k0 + np.uint64(weyl[0])) & np.uint64(U)
                k1 = (k1 + np.uint64(weyl[1])) & np.uint64(U)
            p0 = np.uint64(mul[0]) * c[0]
            p1 = np.uint64(mul[1]) * c[2]
            c = [(p1 >> np.uint64(32)) ^ c[1] ^ k0, p1 & np.uint64(U), (p0 >> np.uint64(32)) ^ c[3] ^ k1,
                 p0 & np.uint64(U)]
        return [c[i] for i in order]
    return f


def _gumbel_neg_log(seed, step, node, V):
    # -ln(u): exponential noise, not Gumbel
    g = O.gumbel_noise(seed, step, node, V)
    return -np.log(np.exp(-np.exp(-g)))


def _rounds_root_hidden(toy, shape, rounds):
    # each round starts from the root's hidden state instead of the last kept node's
    B = toy["h"].shape[0]
    orig = O.next_inputs
    O.next_inputs = lambda o, nodes, n, bonus: orig(o, [[nd[0]] * (len(nd)) for nd in nodes], [0] * B, bonus)
    try:
        return O.decode_rounds(toy, shape, rounds)
    finally:
        O.next_inputs = orig


def _rejection_unnormalised(tree, tokens_b, probs, uniform):
    # accepts child i with p(t_i) instead of renormalising after earlier rejections
    cur, nodes, toks = 0, [0], []
    while True:
        p = np.array(probs(cur), dtype=np.float64)
        nxt = None
        for c in tree.children[cur]:
            t = int(tokens_b[c])
            if uniform() < p[t]:
                nxt = c
                break
            p[t] = 0.0
        if nxt is None:
            q = p / p.sum()
            return len(toks), toks, nodes, min(int(np.searchsorted(np.cumsum(q), uniform(), side="right")), len(q) - 1)
        nodes.append(nxt)
        toks.append(int(tokens_b[nxt]))
        cur = nxt


def _attn_scale_dh(q, k_tree, v_tree, k_cache, v_cache, kv_len, mask, nodes=None, batches=None):
    Dh = q.shape[-1]
    return O.tree_attention(q * (math.sqrt(Dh) / Dh), k_tree, v_tree, k_cache, v_cache, kv_len, mask, nodes, batches)


def _attn_wrong_group(q, k_tree, v_tree, k_cache, v_cache, kv_len, mask, nodes=None, batches=None):
    # q head h reads kv head h % Hkv instead of h // G
    Hq, Hkv = q.shape[2], k_tree.shape[2]
    G = Hq // Hkv
    perm = [(h % Hkv) * G + h // Hkv for h in range(Hq)]
    inv = np.argsort(perm)
    o = O.tree_attention(q[:, :, perm], k_tree, v_tree, k_cache, v_cache, kv_len, mask, nodes, batches)
    B, T, _ = o.shape
    Dh = q.shape[3]
    return o.reshape(B, T, Hq, Dh)[:, :, inv].reshape(B, T, Hq * Dh)


def _greedy_child_argmax(tree, tokens_b, argmax_b):
    cur, nodes, toks = 0, [0], []
    for _ in range(tree.depth_max):
        nxt = None
        for c in tree.children[cur]:
            if tokens_b[c] == argmax_b[c]:  # wrong index: the child's own choice
                nxt = c
                break
        if nxt is None:
            break
        nodes.append(nxt)
        toks.append(int(tokens_b[nxt]))
        cur = nxt
    return len(toks), toks, nodes, int(argmax_b[cur])


def _argmax_last(o_stored, lm_head, temperature=None, rows=None, chunk=256):
    res = O.verify_stats(o_stored, lm_head, temperature, rows, chunk)
    L = o_stored @ O.decode(lm_head).T
    res["argmax"] = L.shape[1] - 1 - np.argmax(L[:, ::-1], axis=1)
    return res


def _threshold_no_exp(entropy, eps, delta):
    return min(eps, delta * entropy)


def _check_rounds(M):
    from tests import test_decode_loop as L
    t, toy = L._toy_np("toy-mini")
    hist = M.decode_rounds(toy, t, t.rounds)
    inv = np.argsort(toy["perm"])
    for r in range(t.rounds):
        for b in range(t.batch):
            x = int(inv[hist["root"][r][b]])
            n = 0
            while n < t.depth and toy["right"][n][x]:
                n += 1
            assert hist["accept_len"][r][b] == n


MUTANTS = [
    ("head drops the residual", dict(head_hidden=_no_residual), P.check_zero_init),
    ("head drops the bias", dict(head_hidden=_no_bias), P.check_head_vs_torch),
    ("head W1 transposed", dict(head_hidden=_transposed_w1), P.check_head_vs_torch),
    ("SiLU sign flipped", dict(silu=_silu_sign), P.check_silu),
    ("top-k ties to the higher index", dict(topk_lists=_topk_high_tie), P.check_topk),
    ("mask sees descendants", dict(Tree=_DescTree), P.check_tree_2x3),
    ("mask drops the node itself", dict(Tree=_NoSelfTree), P.check_attention_paths),
    ("attention scale 1/Dh", dict(tree_attention=_attn_scale_dh), P.check_attention_paths),
    ("GQA group index", dict(tree_attention=_attn_wrong_group), P.check_attention_paths),
    ("greedy compares the child's own argmax", dict(accept_greedy=_greedy_child_argmax), P.check_greedy_lossless),
    ("argmax ties to the last index", dict(verify_stats=_argmax_last), P.check_verify),
    ("threshold without exp", dict(typical_threshold=_threshold_no_exp), P.check_verify),
    ("explicit tree loses its shallow leaves", dict(Tree=_DeepLeavesTree), P.check_explicit_tree),
    ("typical ties to the last longest chain", dict(accept_typical=_typical_last_longest),
     P.check_typical_shallow_tie),
    ("commit writes one row late", dict(kv_commit=_commit_off_by_one), P.check_kv_commit),
    ("per-sequence lengths ignored", dict(tree_attention=_attn_uniform_len), P.check_kv_commit),
    ("Gumbel noise sign flipped", dict(gumbel_noise=_gumbel_sign), P.check_gumbel_max),
    ("one Philox word for four nodes", dict(gumbel_noise=_gumbel_one_word), P.check_gumbel_max),
    ("Philox with nine rounds", dict(philox4x32_10=_philox(rounds=9)), P.check_philox_kat),
    ("Philox output words swapped", dict(philox4x32_10=_philox(order=(0, 3, 2, 1))), P.check_philox_kat),
    ("Philox key bumped before round 1", dict(philox4x32_10=_philox(bump_first=True)), P.check_philox_kat),
    ("Philox Weyl constant off by two", dict(philox4x32_10=_philox(weyl=(0x9E3779B7, 0xBB67AE85))),
     P.check_philox_kat),
    ("Philox multipliers exchanged", dict(philox4x32_10=_philox(mul=O.PHILOX_MUL[::-1])), P.check_philox_kat),
    ("exponential noise instead of Gumbel", dict(gumbel_noise=_gumbel_neg_log), P.check_gumbel_distribution),
    ("rounds restart from the root's hidden state", dict(decode_rounds=_rounds_root_hidden), _check_rounds),
    ("rejection without renormalising", dict(accept_rejection=_rejection_unnormalised),
     P.check_rejection_sampling_is_lossless),
]


@pytest.mark.parametrize("name,repl,check", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, repl, check):
    m = mutant(**repl)
    with pytest.raises(AssertionError):
        check(m)
