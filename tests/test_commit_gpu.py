"""The steps around the hot path on the GPU: per-sequence cache lengths in the
tree attention, the KV commit of the accepted branch and the next round's
inputs, each against the oracle on the same seeded inputs (attention within
the float tolerance, data movement bit-exact), plus a two-step loop."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from medusa_head_tree_heads_b300 import synth
from oracle import medusa_oracle as O
from tests import util as U

pytestmark = pytest.mark.gpu


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the gpu-marked tests")


def _lens(s, seed):
    """Seeded per-sequence lengths covering 0, the full capacity and values between."""
    cap = s.cap
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, cap + 1, size=s.batch)
    lens[0] = 0
    if s.batch > 1:
        lens[-1] = cap
    return lens.astype(np.int32)


# tensor-core kernel (Dh 128; sparse tree), mma.sync kernel (Dh 64), fp32 kernel
@pytest.mark.parametrize("name", ["7b-mini", "gqa-b16-mini", "sparse-mini", "33b-b32-mini", "tiny-fp32-gqa"])
def test_ragged_cache_lengths_match_the_oracle(name):
    _need_gpu()
    from medusa_head_tree_heads_b300 import medusa as M
    s, inp = U.planned_inputs(name)
    d = {k: v.cuda() for k, v in inp.items()}
    n = U.np_inputs(inp)
    cfg = M.make_config(s)
    ws = M.alloc_workspace(cfg)
    out = M.alloc_outputs(cfg)
    lens = _lens(s, 11)
    dlens = torch.from_numpy(lens).cuda()
    zeros = torch.zeros(s.batch, s.n_heads, max(list(s.topk) + [1]), dtype=torch.int32, device="cuda")
    M.medusa_tree_build(cfg, zeros, d["root_token"], out["tree"])  # tokens do not enter the attention
    M.medusa_tree_attn_lens(cfg, d["q"], d["k_tree"], d["v_tree"], d["k_cache"], d["v_cache"], dlens,
                            out["tree"], out["attn_out"], ws)
    torch.cuda.synchronize()
    assert M.medusa_get_device_error(ws) == 0
    tree = O.Tree.for_shape(s)
    ref = O.tree_attention(n["q"], n["k_tree"], n["v_tree"], n["k_cache"], n["v_cache"], lens, tree.mask)
    got = out["attn_out"].float().cpu().numpy().astype(np.float64)
    U.assert_close(got, O.round_to_storage(ref, s.dtype), s.dtype, f"{name} attn_out")


def test_out_of_range_length_sets_the_device_error():
    _need_gpu()
    from medusa_head_tree_heads_b300 import medusa as M
    s, inp = U.planned_inputs("7b-mini")
    d = {k: v.cuda() for k, v in inp.items()}
    cfg = M.make_config(s)
    ws = M.alloc_workspace(cfg)
    out = M.alloc_outputs(cfg)
    zeros = torch.zeros(s.batch, s.n_heads, max(s.topk), dtype=torch.int32, device="cuda")
    M.medusa_tree_build(cfg, zeros, d["root_token"], out["tree"])
    bad = torch.full((s.batch,), s.cap + 1, dtype=torch.int32, device="cuda")  # past the capacity: clamped
    M.medusa_tree_attn_lens(cfg, d["q"], d["k_tree"], d["v_tree"], d["k_cache"], d["v_cache"], bad,
                            out["tree"], out["attn_out"], ws)
    torch.cuda.synchronize()
    assert M.medusa_get_device_error(ws) == -5


@pytest.mark.parametrize("name", ["7b-mini", "gqa-b16-mini", "sparse-f32"])
def test_kv_commit_and_next_inputs_are_bit_exact(name):
    _need_gpu()
    from medusa_head_tree_heads_b300 import medusa as M
    s, inp = U.planned_inputs(name)
    n = U.np_inputs(inp)
    cfg = M.make_config(s)
    ws = M.alloc_workspace(cfg)
    tree = O.Tree.for_shape(s)
    rng = np.random.default_rng(3)
    D = s.depth
    acc_nodes = np.full((s.batch, D + 1), -1, dtype=np.int32)
    accept_len = np.zeros(s.batch, dtype=np.int32)
    for b in range(s.batch):  # a seeded kept prefix of a seeded leaf path
        row = [x for x in tree.paths[rng.integers(len(tree.paths))] if x >= 0]
        k = int(rng.integers(0, len(row)))
        acc_nodes[b, :k + 1] = row[:k + 1]
        accept_len[b] = k
    lens = np.array([int(rng.integers(0, s.cap - D)) for _ in range(s.batch)], dtype=np.int32)
    kc, vc = inp["k_cache"].clone().cuda(), inp["v_cache"].clone().cuda()
    dl = torch.from_numpy(lens.copy()).cuda()
    M.medusa_kv_commit(cfg, torch.from_numpy(acc_nodes).cuda(), torch.from_numpy(accept_len).cuda(),
                       inp["k_tree"].cuda(), inp["v_tree"].cuda(), kc, vc, dl, ws)
    torch.cuda.synchronize()
    assert M.medusa_get_device_error(ws) == 0
    rkc, rvc, rl = O.kv_commit(n["k_cache"], n["v_cache"], n["k_tree"], n["v_tree"], acc_nodes, accept_len, lens)
    np.testing.assert_array_equal(U.to_np(kc), rkc)
    np.testing.assert_array_equal(U.to_np(vc), rvc)
    np.testing.assert_array_equal(dl.cpu().numpy(), rl)
    # next inputs from a seeded stand-in for the attention output (same bits on both sides)
    attn = synth._cast(torch.randn(s.batch, s.n_nodes, s.hidden, generator=torch.Generator().manual_seed(5)), s)
    bonus = rng.integers(0, s.vocab, size=s.batch).astype(np.int32)
    h_next = torch.empty(s.batch, s.hidden, dtype=s.torch_dtype, device="cuda")
    root_next = torch.empty(s.batch, dtype=torch.int32, device="cuda")
    M.medusa_next_inputs(cfg, attn.cuda(), torch.from_numpy(acc_nodes).cuda(), torch.from_numpy(accept_len).cuda(),
                         torch.from_numpy(bonus).cuda(), h_next, root_next, ws)
    torch.cuda.synchronize()
    rh, rr = O.next_inputs(U.to_np(attn), acc_nodes, accept_len, bonus)
    np.testing.assert_array_equal(U.to_np(h_next), rh)
    np.testing.assert_array_equal(root_next.cpu().numpy(), rr)


def test_commit_without_room_changes_nothing():
    _need_gpu()
    from medusa_head_tree_heads_b300 import medusa as M
    s, inp = U.planned_inputs("7b-mini")
    cfg = M.make_config(s)
    ws = M.alloc_workspace(cfg)
    acc_nodes = torch.tensor([[0, 1, 5, -1, -1, -1]], dtype=torch.int32, device="cuda")
    accept_len = torch.tensor([2], dtype=torch.int32, device="cuda")
    lens = torch.tensor([s.cap - 2], dtype=torch.int32, device="cuda")  # three rows needed, two free
    kc, vc = inp["k_cache"].clone().cuda(), inp["v_cache"].clone().cuda()
    M.medusa_kv_commit(cfg, acc_nodes, accept_len, inp["k_tree"].cuda(), inp["v_tree"].cuda(), kc, vc, lens, ws)
    torch.cuda.synchronize()
    assert M.medusa_get_device_error(ws) == -5
    assert torch.equal(kc.cpu(), inp["k_cache"]) and torch.equal(vc.cpu(), inp["v_cache"])
    assert lens.item() == s.cap - 2


@pytest.mark.parametrize("schedule", ["serial", "overlap"])
def test_two_step_loop_commits_and_chains(schedule):
    """Step 1 (planted acceptance, bit-exact with the oracle), commit, next
    inputs, step 2 on the grown per-sequence caches: the committed rows and
    lengths equal the oracle's commit of its own step-1 acceptance, and step
    2's attention equals the oracle's over those caches."""
    _need_gpu()
    from medusa_head_tree_heads_b300 import medusa as M
    s, inp = U.planned_inputs("13b-mini")
    n = U.np_inputs(inp)
    d = {k: v.cuda() for k, v in inp.items()}
    d["k_cache"], d["v_cache"] = d["k_cache"].clone(), d["v_cache"].clone()
    cfg = M.make_config(s, schedule={"serial": M.SERIAL, "overlap": M.OVERLAP}[schedule])
    ws = M.alloc_workspace(cfg)
    out = M.alloc_outputs(cfg)
    lens = torch.full((s.batch,), s.kv_len, dtype=torch.int32, device="cuda")
    M.medusa_step(cfg, M.step_io(d, out, lens), ws)
    ref1 = O.step(n, s)
    M.medusa_kv_commit(cfg, out["acc_nodes"], out["accept_len"], d["k_tree"], d["v_tree"], d["k_cache"],
                       d["v_cache"], lens, ws)
    h2 = torch.empty_like(d["h"])
    root2 = torch.empty_like(d["root_token"])
    M.medusa_next_inputs(cfg, out["attn_out"], out["acc_nodes"], out["accept_len"], out["bonus"], h2, root2, ws)
    d2 = dict(d, h=h2, root_token=root2)
    out2 = M.alloc_outputs(cfg)
    M.medusa_step(cfg, M.step_io(d2, out2, lens), ws)
    torch.cuda.synchronize()
    assert M.medusa_get_device_error(ws) == 0
    np.testing.assert_array_equal(out["accept_len"].cpu().numpy(), ref1["accept_len"])
    acc = np.full((s.batch, s.depth + 1), -1, dtype=np.int32)
    for b in range(s.batch):
        acc[b, :len(ref1["acc_nodes"][b])] = ref1["acc_nodes"][b]
    rkc, rvc, rl = O.kv_commit(n["k_cache"], n["v_cache"], n["k_tree"], n["v_tree"], acc,
                               np.array(ref1["accept_len"]), [s.kv_len] * s.batch)
    np.testing.assert_array_equal(lens.cpu().numpy(), rl)
    np.testing.assert_array_equal(U.to_np(d["k_cache"]), rkc)
    np.testing.assert_array_equal(U.to_np(d["v_cache"]), rvc)
    assert torch.equal(root2.cpu(), out["bonus"].cpu())
    tree = O.Tree.for_shape(s)
    ref_o = O.tree_attention(n["q"], n["k_tree"], n["v_tree"], rkc, rvc, rl, tree.mask)
    U.assert_close(out2["attn_out"].float().cpu().numpy().astype(np.float64), O.round_to_storage(ref_o, s.dtype),
                   s.dtype, "step-2 attn_out")
