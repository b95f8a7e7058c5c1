"""Round after round of decoding over a table backbone (the steps around the
path: commit of the kept branch, next inputs, next round).

CPU: the oracle's rounds emit exactly the tokens of plain sequential greedy
decoding of the same backbone ("Attenzione sull'albero e accettazione":
greedy acceptance keeps only what the base model would have produced; the
kept branch feeds the next round), over many rounds.  The sequential side is
written here from the backbone's definition (attention over the cache and
every earlier token, then the base lm_head), sharing nothing with the
oracle's tree code.

GPU: the library's rounds (decode_loop.DecodeLoop, all C-ABI calls, no host
synchronisation between rounds) equal the oracle's round for round, bit for
bit: roots, accept lengths, accepted tokens and nodes, bonus tokens and the
final cache lengths and contents."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from medusa_head_tree_heads_b300 import synth
from oracle import medusa_oracle as O
from tests import util as U

TOYS = ["toy-mini", "toy-gqa-mini"]


def _toy_np(name):
    t = synth.TOYS[name]
    return t, {k: U.to_np(v) for k, v in synth.make_toy(t).items()}


def _f64(a):
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    return a.astype(np.float64)


def sequential_greedy(t, toy, b, n_tokens):
    """Plain autoregressive greedy decoding of the backbone for sequence b:
    each token attends (every q head to its kv group) over the first kv_len
    cache rows and the keys of all tokens so far, itself included; the
    output, stored in the backbone's type, goes through lm_head; the next
    token is the argmax (ties to the lower id).  Returns n_tokens tokens
    starting with the root."""
    Q, K, Vt, lm = _f64(toy["Qtab"]), _f64(toy["Ktab"]), _f64(toy["Vtab"]), _f64(toy["lm_head"])
    G = t.n_q_heads // t.n_kv_heads
    keys = list(_f64(toy["k_cache"][b, :t.kv_len]))
    vals = list(_f64(toy["v_cache"][b, :t.kv_len]))
    x = int(toy["root_token"][b])
    out = [x]
    while len(out) < n_tokens:
        keys.append(K[x])
        vals.append(Vt[x])
        Ka, Va = np.stack(keys), np.stack(vals)  # [n, Hkv, Dh]
        o = []
        for h in range(t.n_q_heads):
            s = Ka[:, h // G] @ Q[x, h] / math.sqrt(t.head_dim)
            p = np.exp(s - s.max())
            o.append((p / p.sum()) @ Va[:, h // G])
        o = torch.from_numpy(np.concatenate(o)).to(torch.bfloat16).to(torch.float64).numpy()
        x = int(np.argmax(lm @ o))
        out.append(x)
    return out


def _streams(hist, B):
    s = [[] for _ in range(B)]
    for r in range(len(hist["root"])):
        for b in range(B):
            s[b] += [hist["root"][r][b]] + list(hist["acc_tokens"][r][b])
    return s


@pytest.mark.parametrize("name", TOYS)
def test_oracle_rounds_equal_sequential_greedy(name):
    t, toy = _toy_np(name)
    hist = O.decode_rounds(toy, t, t.rounds)
    streams = _streams(hist, t.batch)
    total = 0
    for b in range(t.batch):
        want = sequential_greedy(t, toy, b, len(streams[b]) + 1)
        assert streams[b] == want[:-1], b
        # every round's bonus is the next round's root, the last one the next token
        assert hist["bonus"][-1][b] == want[-1]
        total += len(streams[b])
    # the heads are right often enough that rounds keep several tokens
    assert total / (t.batch * t.rounds) > 1.5


@pytest.mark.parametrize("name", TOYS)
def test_oracle_accept_lengths_follow_the_heads(name):
    """By the backbone's construction a round whose hidden state belongs to
    token x keeps exactly as many candidates as heads 1, 2, ... are right
    about x in a row (a right head ranks the true continuation first, a wrong
    one ranks it last), so every accept length is known in advance: this
    pins the chaining of rounds (next hidden state from the last kept node,
    next root from the bonus) and the heads' place in the tree."""
    t, toy = _toy_np(name)
    hist = O.decode_rounds(toy, t, t.rounds)
    inv = np.argsort(toy["perm"])
    for r in range(t.rounds):
        for b in range(t.batch):
            x = int(inv[hist["root"][r][b]])  # the token whose hidden state starts the round
            n = 0
            while n < t.depth and toy["right"][n][x]:
                n += 1
            assert hist["accept_len"][r][b] == n, (r, b)


def test_oracle_rounds_follow_the_backbone_cycle():
    """The toy's greedy continuation is its permutation, by construction."""
    t, toy = _toy_np("toy-mini")
    hist = O.decode_rounds(toy, t, t.rounds)
    perm = toy["perm"]
    for s in _streams(hist, t.batch):
        assert all(int(perm[a]) == b for a, b in zip(s, s[1:]))


@pytest.mark.gpu
@pytest.mark.parametrize("name", TOYS)
def test_gpu_rounds_match_the_oracle(name):
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the gpu-marked tests")
    from medusa_head_tree_heads_b300 import decode_loop
    from medusa_head_tree_heads_b300 import medusa as M
    t = synth.TOYS[name]
    toy_t = synth.make_toy(t)
    toy = {k: U.to_np(v) for k, v in toy_t.items()}
    loop = decode_loop.DecodeLoop(t, toy_t)
    loop.run()
    torch.cuda.synchronize()
    assert M.medusa_get_device_error(loop.ws) == 0
    got = loop.history()
    ref = O.decode_rounds(toy, t, t.rounds)
    for key in ("root", "accept_len", "bonus"):
        assert got[key] == [[int(x) for x in row] for row in ref[key]], key
    for key in ("acc_tokens", "acc_nodes"):
        assert got[key] == [[[int(x) for x in seq] for seq in row] for row in ref[key]], key
    # the caches: every committed row, and the lengths
    lens = [t.kv_len] * t.batch
    for r in range(t.rounds):
        lens = [lens[b] + ref["accept_len"][r][b] + 1 for b in range(t.batch)]
    assert loop.dev["kv_lens"].cpu().tolist() == lens
    tok = _streams(ref, t.batch)
    for b in range(t.batch):
        kc = U.to_np(loop.dev["k_cache"][b])
        np.testing.assert_array_equal(kc[:t.kv_len], toy["k_cache"][b, :t.kv_len])
        np.testing.assert_array_equal(kc[t.kv_len:lens[b]], toy["Ktab"][tok[b]])
