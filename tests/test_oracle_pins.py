"""Pins of the CPU oracle to facts fixed by the pages and by mathematics
(no GPU).  Every check is written as a function of the oracle module so that
tests/test_oracle_mutants.py can show that planted mistakes fail them."""
from __future__ import annotations

import math
import os

import numpy as np
import pytest
import torch

from medusa_head_tree_heads_b300 import synth
from oracle import medusa_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def to_np(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


# --------------------------------------------------------------- checks ------

def check_zero_init(M) -> None:
    """Zero-initialised heads reproduce lm_head exactly ("Medusa Heads",
    "Come le teste prevedono i token successivi": printed [True, True, True])."""
    fx = {}
    with open(os.path.join(GOLDEN, "zero_init_heads.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            k, *v = line.split()
            fx[k] = v
    H, V, K = int(fx["hidden_size"][0]), int(fx["vocab_size"][0]), int(fx["num_heads"][0])
    s = synth.SHAPES["tiny-fp32"]
    assert (s.hidden, s.vocab, s.n_heads) == (H, V, K)
    w = synth.make_weights(s, zero_init=True)
    h = synth.draw_h_row(s, 0)[None, :]
    z = M.head_hidden(to_np(h), to_np(w["W1"]), to_np(w["b1"]))
    lg = M.head_logits(z, to_np(w["W2"]))
    base = M.base_logits(to_np(h), to_np(w["lm_head"]))
    printed = [np.array_equal(lg[:, k, :], base) for k in range(K)]
    assert printed == [x == "True" for x in fx["printed"]], printed


def check_head_vs_torch(M) -> None:
    """Head FFN + projection against torch.nn.functional (float64, CPU)."""
    g = torch.Generator().manual_seed(7)
    B, K, H, V = 3, 2, 24, 40
    h = torch.randn(B, H, generator=g, dtype=torch.float64)
    W1 = torch.randn(K, H, H, generator=g, dtype=torch.float64) * 0.3
    b1 = torch.randn(K, H, generator=g, dtype=torch.float64) * 0.3
    W2 = torch.randn(K, V, H, generator=g, dtype=torch.float64)
    z = M.head_hidden(h.numpy(), W1.numpy(), b1.numpy())
    lg = M.head_logits(z, W2.numpy())
    for k in range(K):
        zt = h + torch.nn.functional.silu(torch.nn.functional.linear(h, W1[k], b1[k]))
        lt = torch.nn.functional.linear(zt, W2[k])
        np.testing.assert_allclose(z[:, k], zt.numpy(), rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(lg[:, k], lt.numpy(), rtol=1e-12, atol=1e-12)


def check_topk(M) -> None:
    """Per-head top-k: descending, ties to the lower index (reading R5), heads
    past the tree depth keep 1; brute force and torch.topk on small inputs."""
    rng = np.random.default_rng(3)
    B, K, V = 2, 4, 50
    lg = rng.integers(0, 12, size=(B, K, V)).astype(np.float64)  # many ties
    topk = (3, 2, 4)
    idx, val = M.topk_lists(lg, topk)
    for b in range(B):
        for k in range(K):
            n = topk[k] if k < len(topk) else 1
            brute = sorted(range(V), key=lambda v: (-lg[b, k, v], v))[:n]
            assert idx[b, k, :n].tolist() == brute
            assert (idx[b, k, n:] == -1).all()
            tv = torch.topk(torch.from_numpy(lg[b, k]), n).values.numpy()
            np.testing.assert_array_equal(val[b, k, :n], tv)


def check_tree_2x3(M) -> None:
    """The worked example: head-1 top-2 x head-2 top-3 gives 6 candidates in a
    prefix-sharing tree ("Attenzione sull'albero e accettazione")."""
    rows, paths, fx = [], [], {}
    with open(os.path.join(GOLDEN, "tree_2x3.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            p = line.split()
            if p[0] == "path":
                paths.append([int(x) for x in p[1:]])
            elif p[0].isdigit():
                rows.append([int(x) for x in p])
            else:
                fx[p[0]] = int(p[1])
    t = M.Tree((2, 3))
    assert len(t.leaves) == fx["candidates"] == 6
    assert t.T == fx["nodes_including_root"] == 9
    for r in rows:
        i, parent, depth, rank = r[:4]
        assert (t.parent[i], t.depth[i], t.rank[i]) == (parent, depth, rank)
        assert sorted(np.nonzero(t.mask[i])[0].tolist()) == sorted(r[4:])
    assert t.paths.tolist() == paths


def check_tree_invariants(M) -> None:
    """Node counts sum_d prod_{j<=d} k_j for the five workloads; every branch at
    depth d takes the same head-d list; a chain gives the causal mask; each
    mask row holds exactly depth+1 nodes, all on the node's root path."""
    for topk, n in [((2, 3), 8), ((4, 3, 2, 2, 1), 136), ((3, 2, 2, 1), 33), ((4, 3, 2, 2), 88),
                    ((4, 3, 2, 2, 2), 184)]:
        t = M.Tree(topk)
        assert t.T - 1 == n
        assert len(t.leaves) == int(np.prod(topk))
    t = M.Tree((3, 2, 2))
    idx = np.array([[[11, 12, 13], [21, 22, -1], [31, 32, -1], [41, -1, -1]]], dtype=np.int32)
    tok = t.tokens(idx, [5])[0]
    assert tok[0] == 5
    for i in range(t.T):
        kids = [tok[c] for c in t.children[i]]
        if t.depth[i] < 3:
            assert kids == [idx[0, t.depth[i], r] for r in range(t.topk[t.depth[i]])]
    chain = M.Tree((1, 1, 1, 1, 1))
    np.testing.assert_array_equal(chain.mask, np.tril(np.ones((6, 6), dtype=bool)))
    for i in range(t.T):
        assert t.mask[i].sum() == t.depth[i] + 1
        assert set(np.nonzero(t.mask[i])[0].tolist()) == set(t.chain(i))


def _rand_attn_inputs(seed, B, T, Hq, Hkv, Dh, L, cap):
    g = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(*s, generator=g, dtype=torch.float64).numpy()
    return r(B, T, Hq, Dh), r(B, T, Hkv, Dh), r(B, T, Hkv, Dh), r(B, cap, Hkv, Dh), r(B, cap, Hkv, Dh)


def check_attention_paths(M) -> None:
    """Tree attention equals, at every node of every root-to-leaf path, causal
    attention over (cache ++ path) computed by torch's scaled_dot_product_attention
    (one pass over all branches gives what each branch alone would) -- for a
    Cartesian tree and for a sparse one with leaves at several depths."""
    topk = (3, 2, 2)
    parent, rank = synth.explicit_tree(topk, 7)
    for t in (M.Tree(topk), M.Tree(topk, parent, rank)):
        _attention_paths_one(M, t)


def _attention_paths_one(M, t) -> None:
    B, Hq, Hkv, Dh, L, cap = 2, 4, 2, 16, 11, 13
    q, kt, vt, kc, vc = _rand_attn_inputs(1, B, t.T, Hq, Hkv, Dh, L, cap)
    o = M.tree_attention(q, kt, vt, kc, vc, L, t.mask)
    G = Hq // Hkv
    for b in range(B):
        for row in t.paths:
            path = [int(x) for x in row if x >= 0]
            n = len(path)
            for h in range(Hq):
                g = h // G
                Q = torch.from_numpy(q[b, path, h])[None, None]  # [1,1,n,Dh]
                Kp = np.concatenate([kc[b, :L, g], kt[b, path, g]])
                Vp = np.concatenate([vc[b, :L, g], vt[b, path, g]])
                allow = torch.ones(n, L + n, dtype=torch.bool)
                allow[:, L:] = torch.tril(torch.ones(n, n, dtype=torch.bool))
                ref = torch.nn.functional.scaled_dot_product_attention(
                    Q, torch.from_numpy(Kp)[None, None], torch.from_numpy(Vp)[None, None], attn_mask=allow)[0, 0]
                np.testing.assert_allclose(o[b, path, h * Dh:(h + 1) * Dh], ref.numpy(), rtol=1e-12, atol=1e-12)


def check_attention_single_node(M) -> None:
    """Empty cache and a root-only tree: the output is the root's value."""
    t = M.Tree(())
    q, kt, vt, kc, vc = _rand_attn_inputs(2, 1, 1, 4, 2, 8, 0, 3)
    o = M.tree_attention(q, kt, vt, kc, vc, 0, t.mask)
    for h in range(4):
        np.testing.assert_array_equal(o[0, 0, h * 8:(h + 1) * 8], vt[0, 0, h // 2])


def check_verify(M) -> None:
    """argmax / max against torch on random scores (first maximum wins);
    uniform scores: entropy = log-partition = ln V (closed form)."""
    rng = np.random.default_rng(5)
    N, H, V = 7, 12, 33
    o = rng.standard_normal((N, H))
    W = rng.standard_normal((V, H))
    st = M.verify_stats(o, W, temperature=0.7)
    lg = torch.from_numpy(o) @ torch.from_numpy(W).T
    assert st["argmax"].tolist() == torch.argmax(lg, dim=1).tolist()
    np.testing.assert_allclose(st["maxlogit"], lg.max(dim=1).values.numpy(), rtol=1e-14)
    ref_lse = torch.logsumexp(lg / 0.7, dim=1).numpy()
    np.testing.assert_allclose(st["lse"], ref_lse, rtol=1e-12)
    p = torch.softmax(lg / 0.7, dim=1)
    np.testing.assert_allclose(st["entropy"], torch.distributions.Categorical(probs=p).entropy().numpy(), rtol=1e-10)
    W2 = np.zeros((V, H))
    W2[3] = 1.0
    W2[9] = 1.0  # exact tie between tokens 3 and 9
    st = M.verify_stats(np.ones((1, H)), W2)
    assert st["argmax"][0] == 3
    st = M.verify_stats(np.zeros((2, H)), W, temperature=0.7)
    np.testing.assert_allclose(st["entropy"], math.log(V), rtol=1e-14)
    np.testing.assert_allclose(st["lse"], math.log(V), rtol=1e-14)
    assert M.typical_threshold(math.log(V), 0.3, 0.09) == pytest.approx(0.09 / V, rel=1e-14)
    assert M.typical_threshold(0.0, 0.3, 0.09) == 0.09
    assert M.typical_threshold(0.0, 0.05, 0.09) == 0.05


# toy one-layer model for the lossless check: tokens embed to q/k/v, the
# base model's next token is argmax(lm_head . attention output)
class Toy:
    def __init__(self, seed, V=64, Hq=2, Hkv=1, Dh=8, L=9):
        g = torch.Generator().manual_seed(seed)
        r = lambda *s: torch.randn(*s, generator=g, dtype=torch.float64)
        self.V, self.Hq, self.Hkv, self.Dh, self.L = V, Hq, Hkv, Dh, L
        H = Hq * Dh
        self.E = r(V, H)
        self.Wq = r(Hq * Dh, H) / math.sqrt(H)
        self.Wk = r(Hkv * Dh, H) / math.sqrt(H)
        self.Wv = r(Hkv * Dh, H) / math.sqrt(H)
        self.lm = r(V, H) * 3.0
        self.kc = r(1, L, Hkv, Dh)
        self.vc = r(1, L, Hkv, Dh)

    def qkv(self, tokens):
        x = self.E[tokens]
        return ((x @ self.Wq.T).reshape(-1, self.Hq, self.Dh), (x @ self.Wk.T).reshape(-1, self.Hkv, self.Dh),
                (x @ self.Wv.T).reshape(-1, self.Hkv, self.Dh))

    def sequential_greedy(self, root, n):
        """Plain autoregressive greedy decoding, one token per step, with
        torch's attention: returns the n tokens after root."""
        seq, out = [root], []
        G = self.Hq // self.Hkv
        for _ in range(n):
            q, k, v = self.qkv(seq)
            o = []
            for h in range(self.Hq):
                K = torch.cat([self.kc[0, :, h // G], k[:, h // G]])
                Vv = torch.cat([self.vc[0, :, h // G], v[:, h // G]])
                o.append(torch.nn.functional.scaled_dot_product_attention(q[-1:, h][None], K[None], Vv[None])[0, 0])
            nxt = int(torch.argmax(self.lm @ torch.cat(o)))
            out.append(nxt)
            seq.append(nxt)
        return out


def check_greedy_lossless(M) -> None:
    """Greedy acceptance is lossless: accepted tokens + bonus equal plain
    sequential greedy decoding ("Attenzione sull'albero e accettazione";
    "Plongee profonde").  The sequential tokens are planted into the head
    lists at seeded ranks; cutting one list cuts the accepted prefix there."""
    topk = (3, 2, 2, 1)
    D = len(topk)
    for seed in range(6):
        toy = Toy(100 + seed)
        rng = np.random.default_rng(seed)
        root = int(rng.integers(0, toy.V))
        want = toy.sequential_greedy(root, D + 1)
        cut = D if seed % 2 == 0 else int(rng.integers(1, D + 1))  # depth whose list misses the token
        idx = np.full((1, D, max(topk)), -1, dtype=np.int32)
        for d in range(D):
            others = [x for x in rng.permutation(toy.V).tolist() if x != want[d]][:topk[d]]
            lst = others[:topk[d]]
            if d + 1 != cut or seed % 2 == 0:
                lst[int(rng.integers(0, topk[d]))] = want[d]
            idx[0, d, :topk[d]] = lst
        t = M.Tree(topk)
        tok = t.tokens(idx, [root])
        q, k, v = toy.qkv(torch.from_numpy(tok[0]).long())
        o = M.tree_attention(q.numpy()[None], k.numpy()[None], v.numpy()[None], toy.kc.numpy(), toy.vc.numpy(),
                             toy.L, t.mask)
        st = M.verify_stats(o[0], toy.lm.numpy())
        n, toks, nodes, bonus = M.accept_greedy(t, tok[0], st["argmax"])
        exp_n = D if seed % 2 == 0 else cut - 1
        assert n == exp_n, (seed, n, exp_n)
        assert toks == want[:n]
        assert bonus == want[n]
        assert [int(tok[0, x]) for x in nodes[1:]] == toks


def check_typical_special_cases(M) -> None:
    """delta = 0 keeps every candidate (threshold 0); a uniform base
    distribution keeps every candidate (1/V > delta/V); both give the full
    depth.  A distribution peaked away from every candidate keeps none."""
    topk = (2, 3, 2)
    t = M.Tree(topk)
    tok = t.tokens(np.array([[[1, 2, 0], [3, 4, 5], [6, 7, 0]]], dtype=np.int32), [9])[0]
    V = 10
    am = np.zeros(t.T, dtype=np.int64)
    H_unif = math.log(V)
    n, *_ = M.accept_typical(t, tok, am, lambda p, c: (1.0 / V) > M.typical_threshold(5.0, 0.3, 0.0))
    assert n == 3
    n, toks, nodes, _ = M.accept_typical(t, tok, am, lambda p, c: (1.0 / V) > M.typical_threshold(H_unif, 0.3, 0.09))
    assert n == 3 and nodes == [0, 1, 3, 9]  # lowest index at every divergence
    n, *_ = M.accept_typical(t, tok, am, lambda p, c: 1e-9 > M.typical_threshold(0.01, 0.3, 0.09))
    assert n == 0


def check_explicit_tree(M) -> None:
    """An explicit parent/rank tree: the explicit form of a Cartesian tree is
    that tree; for a sparse subset, every node's depth is the length of its
    chain of parents, its mask row is that chain, the leaves are the nodes no
    node names as parent (some shallower than the tree depth) and every path
    row is a leaf's chain followed by -1."""
    for topk in [(2, 3), (3, 2, 2), (1, 1, 1), ()]:
        t = M.Tree(topk)
        e = M.Tree(topk, t.parent.tolist(), t.rank.tolist())
        for f in ("parent", "depth", "rank", "mask", "paths"):
            np.testing.assert_array_equal(getattr(e, f), getattr(t, f))
        assert e.leaves == t.leaves
    topk = (4, 3, 2, 2)
    parent, rank = synth.explicit_tree(topk, 24)
    t = M.Tree(topk, parent, rank)

    def walk(i):
        out = []
        while i >= 0:
            out.append(i)
            i = parent[i]
        return out[::-1]

    for i in range(len(parent)):
        ch = walk(i)
        assert t.depth[i] == len(ch) - 1
        assert set(np.nonzero(t.mask[i])[0].tolist()) == set(ch)
    leaves = [i for i in range(len(parent)) if i not in set(parent[1:])]
    assert t.leaves == leaves and len({int(t.depth[l]) for l in leaves}) > 1
    assert len(t.paths) == len(leaves)
    for row, l in zip(t.paths.tolist(), leaves):
        ch = walk(l)
        assert row == ch + [-1] * (len(topk) + 1 - len(ch))


def check_typical_shallow_tie(M) -> None:
    """Equal kept lengths go to the lower node at the first divergence, also
    when the other branch ends in a shallower leaf with a lower node id."""
    t = M.Tree((2, 2), [-1, 0, 0, 1], [0, 0, 1, 0])  # node 2 is a depth-1 leaf, node 3 a child of node 1
    tok = np.array([9, 1, 2, 3], dtype=np.int32)
    n, toks, nodes, _ = M.accept_typical(t, tok, np.zeros(4, dtype=np.int64), lambda p, c: c != 3)
    assert n == 1 and nodes == [0, 1] and toks == [1]


def check_ragged_lengths(M) -> None:
    """Per-sequence cache lengths: each sequence's output equals the one-length
    call for that sequence alone (0, a middle value and the full capacity)."""
    t = M.Tree((2, 2))
    B, Hq, Hkv, Dh, cap = 3, 4, 2, 8, 9
    q, kt, vt, kc, vc = _rand_attn_inputs(5, B, t.T, Hq, Hkv, Dh, cap, cap)
    lens = [0, 4, cap]
    o = M.tree_attention(q, kt, vt, kc, vc, lens, t.mask)
    for b, L in enumerate(lens):
        ob = M.tree_attention(q, kt, vt, kc, vc, L, t.mask, batches=[b])
        np.testing.assert_array_equal(o[b], ob[b])


def check_kv_commit(M) -> None:
    """After the accepted chain is committed, plain attention (torch SDPA) of
    the last accepted node's query over the grown cache alone reproduces that
    node's tree-attention output: the committed rows are exactly what the node
    saw in the tree.  Rows past the old lengths other than the committed ones
    and the other sequences' rows stay as they were."""
    topk = (3, 2, 2)
    t = M.Tree(topk)
    B, Hq, Hkv, Dh, cap = 3, 4, 2, 16, 20
    q, kt, vt, kc, vc = _rand_attn_inputs(7, B, t.T, Hq, Hkv, Dh, cap, cap)
    lens = [5, 0, 9]
    o = M.tree_attention(q, kt, vt, kc, vc, lens, t.mask)
    leaf_rows = t.paths.tolist()
    acc_nodes = [leaf_rows[4][:4], leaf_rows[0][:2] + [-1, -1], leaf_rows[11][:3] + [-1]]
    accept_len = [3, 1, 2]
    kc2, vc2, lens2 = M.kv_commit(kc, vc, kt, vt, acc_nodes, accept_len, lens)
    assert lens2.tolist() == [l + n + 1 for l, n in zip(lens, accept_len)]
    G = Hq // Hkv
    for b in range(B):
        last = acc_nodes[b][accept_len[b]]
        for h in range(Hq):
            g = h // G
            Q = torch.from_numpy(q[b, [last], h])[None, None]
            K = torch.from_numpy(kc2[b, :lens2[b], g])[None, None]
            V = torch.from_numpy(vc2[b, :lens2[b], g])[None, None]
            ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V)[0, 0, 0].numpy()
            np.testing.assert_allclose(o[b, last, h * Dh:(h + 1) * Dh], ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_array_equal(kc2[b, :lens[b]], kc[b, :lens[b]])
        np.testing.assert_array_equal(kc2[b, lens2[b]:], kc[b, lens2[b]:])
    h_next, root_next = M.next_inputs(o, acc_nodes, accept_len, [7, 8, 9])
    for b in range(B):
        np.testing.assert_array_equal(h_next[b], o[b, acc_nodes[b][accept_len[b]]])
    assert root_next.tolist() == [7, 8, 9]


def check_philox(M) -> None:
    """Philox4x32-10 words: uniform (chi-square over 64 bins for each of the 4
    words of 2^15 consecutive counters), all distinct (the rounds are a
    bijection of the counter for a fixed key), and one flipped counter bit
    changes half of the 128 output bits on average (avalanche)."""
    n = 1 << 15
    c = np.arange(n, dtype=np.uint64)
    z = np.zeros(n, dtype=np.uint64)
    words = M.philox4x32_10(c, z + np.uint64(5), z, z, 0x1234, 0xABCD)
    for w in words:
        counts = np.bincount((w >> np.uint64(26)).astype(np.int64), minlength=64)
        chi2 = ((counts - n / 64) ** 2 / (n / 64)).sum()
        assert chi2 < 120, chi2  # 63 degrees of freedom
    packed = set(zip(*[w.tolist() for w in words]))
    assert len(packed) == n
    flips = []
    for i in range(400):
        a = M.philox4x32_10(np.uint64(i), np.uint64(9), np.uint64(0), np.uint64(0), 3, 4)
        b = M.philox4x32_10(np.uint64(i ^ (1 << (i % 32))), np.uint64(9), np.uint64(0), np.uint64(0), 3, 4)
        flips.append(sum(bin(int(x) ^ int(y)).count("1") for x, y in zip(a, b)))
    assert abs(np.mean(flips) - 64) < 3, np.mean(flips)


def check_philox_kat(M) -> None:
    """Philox4x32-10 reproduces the generator's published known-answer
    vectors (fixture tests/golden/philox4x32_10_kat.txt: the Random123
    library's test file for the SC'11 generator), word for word: a dropped
    or extra round, a wrong multiplier or Weyl constant, a key bumped before
    the first round or output words in another order all change them."""
    path = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")
    rows = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 3
    for r in rows:
        c = [np.uint64(int(x, 16)) for x in r[0:4]]
        k0, k1 = int(r[4], 16), int(r[5], 16)
        want = [int(x, 16) for x in r[6:10]]
        got = [int(np.asarray(w).ravel()[0]) for w in M.philox4x32_10(*c, k0, k1)]
        assert got == want, (r, ["%08x" % g for g in got])


def check_gumbel_distribution(M) -> None:
    """The noise is standard Gumbel: over 2^14 vocabulary rows of one node the
    empirical CDF stays within the Kolmogorov-Smirnov bound (p ~ 1e-3) of
    exp(-exp(-g)); its mean is the Euler-Mascheroni constant and its
    variance pi^2/6 (within 5 standard errors)."""
    n = 1 << 14
    g = np.sort(M.gumbel_noise((5, 6), 3, 7, n))
    cdf = np.exp(-np.exp(-g))
    emp_hi = np.arange(1, n + 1) / n
    emp_lo = np.arange(0, n) / n
    ks = max(np.max(emp_hi - cdf), np.max(cdf - emp_lo))
    assert ks < 1.95 / math.sqrt(n), ks
    assert abs(g.mean() - 0.5772156649015329) < 5 * math.sqrt(math.pi ** 2 / 6 / n), g.mean()
    assert abs(g.var() - math.pi ** 2 / 6) < 5 * 2.2 / math.sqrt(n), g.var()


def check_gumbel_max(M) -> None:
    """Gumbel-max draws follow softmax(logit / temperature): over 40000 steps
    of a 5-token vocabulary the draw frequencies pass a chi-square test (4
    degrees of freedom, bound at p ~ 1e-4); and the four nodes that share one
    Philox counter (different words) draw independently (with equal logits
    they agree about 1/5 of the time, not always)."""
    logits = np.array([2.0, 1.0, 0.5, 0.0, -1.0])
    temp = 0.7
    p = np.exp(logits / temp)
    p /= p.sum()
    steps = 40000
    draws = np.array([int(np.argmax(logits / temp + M.gumbel_noise((11, 12), s, 6, 5))) for s in range(steps)])
    counts = np.bincount(draws, minlength=5)
    chi2 = ((counts - steps * p) ** 2 / (steps * p)).sum()
    assert chi2 < 23.5, (counts, chi2)
    same = 0
    for s in range(2000):
        d = [int(np.argmax(M.gumbel_noise((1, 2), s, n, 5))) for n in range(4)]
        same += d[0] == d[1]
    assert abs(same / 2000 - 0.2) < 0.04, same


def check_plans(M) -> None:
    """On every reduced workload the oracle realises the planted acceptance."""
    plans = synth.load_plans()
    for name in ["tiny-fp32", "tiny-fp32-gqa", "7b-mini", "13b-mini", "gqa-mini", "33b-mini", "sparse-mini",
                 "sparse-typical-mini", "sparse-f32", "sample-mini", "sample-sparse-mini", "typical-sample-mini"]:
        s = synth.SHAPES[name]
        inp = {k: to_np(v) for k, v in synth.make_inputs(s, plans[name]).items()}
        res = M.step(inp, s)
        for b, sq in enumerate(plans[name]["seqs"]):
            assert res["accept_len"][b] == sq["depth"], (name, b)
            assert res["acc_tokens"][b] == sq["tokens"]
            assert res["acc_nodes"][b] == sq["nodes"]
            assert res["bonus"][b] == sq["bonus"]


def check_bf16_rounding(M) -> None:
    """fp64 -> bf16 rounding: agrees with torch's fp32->bf16 on fp32 inputs and
    with nearest-of-neighbours brute force (ties to even) on fp64 inputs."""
    rng = np.random.default_rng(9)
    x32 = (rng.standard_normal(20000) * np.exp(rng.uniform(-30, 30, 20000))).astype(np.float32)
    ref = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(M.round_to_bf16(x32.astype(np.float64)), ref)
    x = rng.standard_normal(3000) * np.exp(rng.uniform(-5, 5, 3000))
    got = M.round_to_bf16(x)
    for xi, gi in zip(x, got):
        e = math.floor(math.log2(abs(xi)))
        ulp = 2.0 ** (e - 7)
        lo = math.floor(xi / ulp) * ulp
        cands = [lo, lo + ulp]
        best = min(cands, key=lambda c: (abs(c - xi), int(round(c / ulp)) % 2))
        assert gi == best, (xi, gi, best)
    # exact halfway points go to the even neighbour
    assert M.round_to_bf16(np.array([1.0 + 2.0 ** -8]))[0] == 1.0
    assert M.round_to_bf16(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 1.0 + 2 * 2.0 ** -7


def check_silu(M) -> None:
    """SiLU special values and the identity silu(x) - silu(-x) = x."""
    assert M.silu(np.array([0.0]))[0] == 0.0
    assert M.silu(np.array([1.0]))[0] == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)
    x = np.linspace(-20, 20, 101)
    np.testing.assert_allclose(M.silu(x) - M.silu(-x), x, atol=1e-13)
    assert M.silu(np.array([40.0]))[0] == pytest.approx(40.0, rel=1e-15)


CHECKS = [check_zero_init, check_head_vs_torch, check_topk, check_tree_2x3, check_tree_invariants,
          check_attention_paths, check_attention_single_node, check_verify, check_greedy_lossless,
          check_typical_special_cases, check_plans, check_bf16_rounding, check_silu, check_explicit_tree,
          check_typical_shallow_tie, check_ragged_lengths, check_kv_commit, check_philox, check_gumbel_max,
          check_philox_kat, check_gumbel_distribution]


@pytest.mark.parametrize("check", CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(O)


def _sampling_tree_case():
    """A 2x2 tree over a 5-token vocabulary with fixed base distributions per
    node, and the exact distribution of what sequential sampling emits."""
    V = 5
    tree_topk = (2, 2)
    rng = np.random.default_rng(3)
    T = 1 + 2 + 4
    P = rng.dirichlet(np.ones(V) * 0.8, size=T)
    tokens = np.array([0, 1, 3, 2, 4, 0, 3])  # root, depth-1 children, depth-2 children
    return V, tree_topk, P, tokens


def _exact_emission(tree, tokens, P):
    """P(accepted tokens + bonus) for plain sequential sampling from the base
    distributions: draw at the current node; a draw equal to a child's token
    moves there, any other draw ends the walk as the bonus."""
    out = {}

    def walk(node, pref, pr):
        for x in range(P.shape[1]):
            kid = [c for c in tree.children[node] if tokens[c] == x]
            if kid:
                walk(kid[0], pref + (x,), pr * P[node, x])
            else:
                out[pref + ("bonus", x)] = out.get(pref + ("bonus", x), 0.0) + pr * P[node, x]

    walk(0, (), 1.0)
    return out


def check_rejection_sampling_is_lossless(M) -> None:
    """Both sampling verifications emit what sequential sampling from the base
    model emits: the rejection walk over the fixed candidates and the
    Gumbel-max draw per node with a candidate kept when it equals its
    parent's draw (the library's sampling mode).  Over 30000 trials each, the
    emitted (tokens, bonus) frequencies pass a chi-square test against the
    exact distribution computed by enumeration (bound at p ~ 1e-4)."""
    V, topk, P, tokens = _sampling_tree_case()
    tree = M.Tree(topk)
    exact = _exact_emission(tree, tokens, P)
    keys = sorted(exact, key=str)
    n = 30000
    rng = np.random.default_rng(11)
    counts_r = {k: 0 for k in keys}
    counts_g = {k: 0 for k in keys}
    for trial in range(n):
        k, toks, _, bonus = M.accept_rejection(tree, tokens, lambda node: P[node], rng.random)
        counts_r[tuple(toks) + ("bonus", bonus)] += 1
        g = -np.log(-np.log(rng.random((tree.T, V))))
        draw = np.argmax(np.log(P) + g, axis=1)
        k, toks, _, bonus = M.accept_greedy(tree, tokens, draw)  # keep a child equal to its parent's draw
        counts_g[tuple(toks) + ("bonus", bonus)] += 1
    dof = len(keys) - 1
    bound = dof + 4.3 * math.sqrt(2 * dof)
    for counts in (counts_r, counts_g):
        chi2 = sum((counts[k] - n * exact[k]) ** 2 / (n * exact[k]) for k in keys)
        assert chi2 < bound, (chi2, bound)


CHECKS.append(check_rejection_sampling_is_lossless)
