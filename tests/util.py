"""Shared test helpers: input conversion, the oracle side and the CUDA side of
one step, and the comparison rules (bit-exact for integers, a stated
tolerance for floats)."""
from __future__ import annotations

import functools
import math
from typing import Dict

import numpy as np
import torch

from medusa_head_tree_heads_b300 import synth

# float tolerance: max |gpu - oracle| <= TOL * max |oracle| over the compared
# block (bf16 storage with fp32 accumulation; fp32 config without TF32)
TOL = {"bf16": 2e-2, "f32": 1e-5}


def to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def np_inputs(inp: Dict[str, torch.Tensor]) -> Dict[str, np.ndarray]:
    return {k: to_np(v) for k, v in inp.items()}


@functools.lru_cache(maxsize=None)
def plans():
    return synth.load_plans()


def planned_inputs(name: str):
    s = synth.SHAPES[name]
    return s, synth.make_inputs(s, plans()[name])


def pack_mask(mask: np.ndarray) -> np.ndarray:
    """bool [T,T] -> uint32 words [T, ceil(T/32)] (bit j%32 of word j/32)."""
    T = mask.shape[0]
    W = (T + 31) // 32
    out = np.zeros((T, W), dtype=np.uint32)
    for i in range(T):
        for j in np.nonzero(mask[i])[0]:
            out[i, j // 32] |= np.uint32(1) << np.uint32(j % 32)
    return out


def assert_close(got, ref, dtype: str, what: str) -> None:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    finite = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), finite), f"{what}: non-finite pattern differs"
    if not finite.any():
        return
    scale = np.abs(ref[finite]).max()
    err = np.abs(got[finite] - ref[finite]).max()
    assert err <= TOL[dtype] * scale, f"{what}: max|d|={err:.3e} > {TOL[dtype]}*{scale:.3e}"


# ------------------------------------------------------------------ GPU side --

def to_device(inp: Dict[str, torch.Tensor], device="cuda") -> Dict[str, torch.Tensor]:
    return {k: v.to(device) for k, v in inp.items()}


def gpu_step(s, dinp: Dict[str, torch.Tensor], fused: bool = True, **over) -> Dict[str, torch.Tensor]:
    """One step through the C ABI (fused medusa_step, or the four stage calls);
    `over` sets config fields (e.g. schedule)."""
    from medusa_head_tree_heads_b300 import medusa as M
    cfg = M.make_config(s, **over)
    ws = M.alloc_workspace(cfg)
    out = M.alloc_outputs(cfg)
    if fused:
        io = M.step_io(dinp, out)
        M.medusa_step(cfg, io, ws)
    else:
        M.medusa_heads_topk(cfg, dinp["h"], dinp["W1"], dinp["b1"], dinp["W2"], out["topk_idx"], out["topk_val"], ws)
        M.medusa_tree_build(cfg, out["topk_idx"], dinp["root_token"], out["tree"])
        M.medusa_tree_attn(cfg, dinp["q"], dinp["k_tree"], dinp["v_tree"], dinp["k_cache"], dinp["v_cache"],
                           out["tree"], out["attn_out"], ws)
        M.medusa_verify_accept(cfg, out["attn_out"], dinp["lm_head"], out["tree"], out, ws)
    torch.cuda.synchronize()
    err = M.medusa_get_device_error(ws)
    assert err == 0, f"device error word {err}"
    res = {k: v.cpu() for k, v in out.items() if k != "tree"}
    res["tree"] = {k: v.cpu() for k, v in out["tree"].items()}
    return res


# --------------------------------------------------------------- comparison --

def compare_step(s, res: Dict, ref: Dict, check_all_nodes: bool = True) -> None:
    """GPU step outputs vs the oracle's, stage by stage."""
    from oracle import medusa_oracle as O
    B, T, D = s.batch, s.n_nodes, s.depth
    # heads: top-k ids bit-exact, values within tolerance
    np.testing.assert_array_equal(res["topk_idx"].numpy(), ref["topk_idx"], err_msg="topk_idx")
    live = ref["topk_idx"] >= 0
    assert_close(res["topk_val"].numpy()[live], ref["topk_val"][live], s.dtype, "topk_val")
    # tree: bit-exact
    tree = ref["tree"]
    t = res["tree"]
    np.testing.assert_array_equal(t["token"].numpy(), ref["tokens"], err_msg="tree token")
    np.testing.assert_array_equal(t["parent"].numpy(), tree.parent, err_msg="tree parent")
    np.testing.assert_array_equal(t["depth"].numpy(), tree.depth, err_msg="tree depth")
    np.testing.assert_array_equal(t["rank"].numpy(), tree.rank, err_msg="tree rank")
    np.testing.assert_array_equal(t["mask"].numpy().view(np.uint32), pack_mask(tree.mask), err_msg="tree mask")
    np.testing.assert_array_equal(t["paths"].numpy(), tree.paths, err_msg="tree paths")
    np.testing.assert_array_equal(t["pos"].numpy(), s.kv_len + tree.depth, err_msg="tree pos")
    # attention output
    got_o = res["attn_out"].float().numpy().astype(np.float64)
    if check_all_nodes:
        assert_close(got_o, ref["attn_out"], s.dtype, "attn_out")
        np.testing.assert_array_equal(res["node_argmax"].numpy(), ref["argmax"], err_msg="node_argmax")
        assert_close(res["node_maxlogit"].numpy(), ref["maxlogit"], s.dtype, "node_maxlogit")
        if s.accept in ("typical", "typical-sample"):
            assert_close(res["node_lse"].numpy(), ref["lse"], s.dtype, "node_lse")
            assert_close(res["node_entropy"].numpy(), ref["entropy"], s.dtype, "node_entropy")
    # acceptance: bit-exact
    for b in range(B):
        n = ref["accept_len"][b]
        assert int(res["accept_len"][b]) == n, ("accept_len", b)
        assert res["acc_tokens"][b, :n].tolist() == ref["acc_tokens"][b], ("acc_tokens", b)
        assert (res["acc_tokens"][b, n:D] == -1).all()
        assert res["acc_nodes"][b, :n + 1].tolist() == ref["acc_nodes"][b], ("acc_nodes", b)
        assert (res["acc_nodes"][b, n + 1:] == -1).all()
        assert int(res["bonus"][b]) == ref["bonus"][b], ("bonus", b)


def _sample_nodes(s, plan, b, rng, extra=8):
    """Every node of the first sequence; elsewhere the planted nodes and
    `extra` seeded random ones."""
    if b == 0:
        return list(range(s.n_nodes))
    planted = [p[0] for p in plan["seqs"][b]["plant"]]
    rand = rng.choice(s.n_nodes, size=min(extra, s.n_nodes), replace=False).tolist()
    return sorted(set(planted) | set(rand))


def compare_full_size(s, inp: Dict, res: Dict) -> None:
    """A full-size step against the oracle: heads, top-k and tree everywhere;
    the planted acceptance bit for bit; attention output and the base model's
    choice on sampled nodes (an unplanted node's choice may trail the oracle's
    best only by what rounding and the stored attention output allow)."""
    from oracle import medusa_oracle as O
    plan = plans()[s.name]
    n = np_inputs(inp)
    # heads and top-k: every sequence, every head
    z = O.head_hidden(n["h"], n["W1"], n["b1"])
    idx, val = O.topk_lists(O.head_logits(z, n["W2"]), list(s.topk))
    np.testing.assert_array_equal(res["topk_idx"].numpy(), idx)
    live = idx >= 0
    assert_close(res["topk_val"].numpy()[live], val[live], s.dtype, "topk_val")
    # the tree: everything
    tree = O.Tree.for_shape(s)
    np.testing.assert_array_equal(res["tree"]["token"].numpy(), tree.tokens(idx, n["root_token"]))
    np.testing.assert_array_equal(res["tree"]["parent"].numpy(), tree.parent)
    np.testing.assert_array_equal(res["tree"]["mask"].numpy().view(np.uint32), pack_mask(tree.mask))
    np.testing.assert_array_equal(res["tree"]["paths"].numpy(), tree.paths)
    # acceptance: the planted result, bit-exact
    for b, sq in enumerate(plan["seqs"]):
        assert int(res["accept_len"][b]) == sq["depth"], b
        assert res["acc_tokens"][b, :sq["depth"]].tolist() == sq["tokens"], b
        assert res["acc_nodes"][b, :sq["depth"] + 1].tolist() == sq["nodes"], b
        assert int(res["bonus"][b]) == sq["bonus"], b
    # sampled nodes: attention output and the base model's choice
    rng = np.random.default_rng(s.seed)
    bs = sorted({0, s.batch - 1} | set(rng.choice(s.batch, size=min(2, s.batch), replace=False).tolist()))
    typical = s.accept == "typical"
    for b in bs:
        nodes = _sample_nodes(s, plan, b, rng)
        o = O.tree_attention(n["q"], n["k_tree"], n["v_tree"], n["k_cache"], n["v_cache"], s.kv_len, tree.mask,
                             nodes=nodes, batches=[b])
        o_st = O.round_to_storage(o[b, nodes], s.dtype)
        got = res["attn_out"][b, nodes].float().numpy()
        assert_close(got, o_st, s.dtype, f"attn_out b={b}")
        sample = s.accept == "sample"
        ids = [b * s.n_nodes + i for i in nodes]
        if sample:
            st = O.sample_stats(o_st, n["lm_head"], s.temperature, s.sample_seed, s.sample_step, node_ids=ids)
        else:
            st = O.verify_stats(o_st, n["lm_head"], s.temperature if typical else None)
        assert_close(res["node_maxlogit"][b, nodes].numpy(), st["maxlogit"], s.dtype, "maxlogit")
        planted = {p[0] for p in plan["seqs"][b]["plant"]}
        lm = n["lm_head"]
        for j, i in enumerate(nodes):
            g = int(res["node_argmax"][b, i])
            r = int(st["argmax"][j])
            if i in planted or g == r:
                assert g == r, (b, i)
            else:  # an unplanted node: the GPU's choice must tie the best within rounding
                wg, wr = O.decode(lm[g]), O.decode(lm[r])
                lg = float(o_st[j] @ wg)
                # Two sources of difference.  (1) The GPU scores its own stored
                # attention output, which differs from the oracle's by the
                # attention's rounding (checked above within its tolerance):
                # a logit moves by at most |w| |o_gpu - o_oracle|, so the
                # oracle's score of the GPU's choice may trail the best by
                # (|w_g| + |w_r|) |o_gpu - o_oracle|.  (2) Accumulation
                # rounding, bounded relative to the best score's magnitude
                # (at least 1 for sampled scores: the Gumbel noise of order 1
                # can put the best near 0 while the rounding of the logit
                # part does not shrink with it).
                drift = (np.linalg.norm(wg) + np.linalg.norm(wr)) * float(np.linalg.norm(got[j] - o_st[j]))
                scale = abs(st["maxlogit"][j])
                if sample:
                    lg = lg / s.temperature + float(O.gumbel_noise(s.sample_seed, s.sample_step, ids[j],
                                                                   s.vocab)[g])
                    drift /= s.temperature
                    scale = max(1.0, scale)
                assert st["maxlogit"][j] - lg <= 2e-3 * scale + drift, (b, i, g, r)
        if typical:
            assert_close(res["node_lse"][b, nodes].numpy(), st["lse"], s.dtype, "lse")
            assert_close(res["node_entropy"][b, nodes].numpy(), st["entropy"], s.dtype, "entropy")
