"""CUDA path vs the CPU oracle, through the C ABI (needs a B300).

Reduced workloads: every output compared -- integers bit-exact, floats
within the stated tolerance.  Full-size workloads (the launch shapes the
benchmark times): all head top-k lists, the whole tree and the acceptance
bit-exact, plus attention outputs and base-model choices at sampled nodes
(every planted node and seeded random ones) computed by the oracle one by
one."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from medusa_head_tree_heads_b300 import synth
from oracle import medusa_oracle as O
from tests import util as U

pytestmark = pytest.mark.gpu

SMALL = [n for n, s in synth.SHAPES.items() if not s.full_size]
FULL = [n for n, s in synth.SHAPES.items() if s.full_size]


@pytest.fixture(scope="module", autouse=True)
def cuda():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the gpu-marked tests")
    from medusa_head_tree_heads_b300 import medusa as M
    M.lib()  # fails loudly when the library is missing


@pytest.mark.parametrize("name", SMALL)
def test_step_matches_oracle(name):
    s, inp = U.planned_inputs(name)
    ref = O.step(U.np_inputs(inp), s)
    res = U.gpu_step(s, U.to_device(inp))
    U.compare_step(s, res, ref)
    for b, sq in enumerate(U.plans()[name]["seqs"]):  # the planted acceptance
        assert int(res["accept_len"][b]) == sq["depth"]
        assert int(res["bonus"][b]) == sq["bonus"]


# bf16, head dim 128, batch <= 32: shapes the overlap schedule accepts (greedy,
# typical, sample; sparse and wide trees; no cache; a depth-1 chain; 16-entry lists)
OVERLAP_OK = ["7b-mini", "13b-mini", "gqa-mini", "gqa-b16-mini", "sample-mini", "sparse-mini",
              "sparse-typical-mini", "wide-bf16", "nocache-bf16", "b5-mini", "chain-bf16", "13b-b8-split", "k16-bf16",
              "typical-sample-mini"]


@pytest.mark.parametrize("name", OVERLAP_OK)
def test_overlap_schedule_matches_oracle(name):
    """The attention issued beside the head projection (unsplit, no waits),
    the candidate merge waiting on the projection's completion count: every
    output against the oracle, as in the serial order."""
    from medusa_head_tree_heads_b300 import medusa as M
    s, inp = U.planned_inputs(name)
    ref = O.step(U.np_inputs(inp), s)
    res = U.gpu_step(s, U.to_device(inp), schedule=M.OVERLAP)
    U.compare_step(s, res, ref)
    for b, sq in enumerate(U.plans()[name]["seqs"]):
        assert int(res["accept_len"][b]) == sq["depth"]
        assert int(res["bonus"][b]) == sq["bonus"]


@pytest.mark.parametrize("name", ["7b-mini", "gqa-b16-mini"])
def test_overlap_schedule_graph_replays_are_identical(name):
    """One CUDA graph of the overlap step replayed back to back: the completion
    count resets itself each step, and every replay gives the integers of an
    eager serial step bit for bit."""
    from medusa_head_tree_heads_b300 import medusa as M
    s, inp = U.planned_inputs(name)
    d = U.to_device(inp)
    serial = U.gpu_step(s, d, schedule=M.SERIAL)
    cfg = M.make_config(s, schedule=M.OVERLAP)
    ws = M.alloc_workspace(cfg)
    out = M.alloc_outputs(cfg)
    io = M.step_io(d, out)
    M.medusa_step(cfg, io, ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        M.medusa_step(cfg, io, ws)
    for _ in range(3):
        for k in ("topk_idx", "node_argmax", "accept_len", "acc_nodes", "bonus"):
            out[k].fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        assert M.medusa_get_device_error(ws) == 0
        for k in ("topk_idx", "node_argmax", "accept_len", "acc_nodes", "acc_tokens", "bonus"):
            assert torch.equal(out[k].cpu(), serial[k]), k
        U.assert_close(out["attn_out"].float().cpu().numpy(), serial["attn_out"].float().numpy(), s.dtype,
                       "attn_out")


@pytest.mark.parametrize("name", ["tiny-fp32", "gqa-mini", "33b-mini", "deep-bf16", "k16-bf16", "k16-f32"])
def test_stage_calls_equal_fused_step(name):
    s, inp = U.planned_inputs(name)
    d = U.to_device(inp)
    a = U.gpu_step(s, d, fused=True)
    b = U.gpu_step(s, d, fused=False)
    # integers bit-exact; floats within the stated tolerance (the fused step may
    # pick a different attention launch shape, hence another summation order)
    for k in a:
        if k == "tree":
            for t in a[k]:
                assert torch.equal(a[k][t], b[k][t]), t
        elif a[k].dtype in (torch.int32, torch.int64):
            assert torch.equal(a[k], b[k]), k
        elif k not in ("node_lse", "node_entropy") or s.accept in ("typical", "typical-sample"):
            U.assert_close(a[k].float().numpy(), b[k].float().numpy(), s.dtype, k)


@pytest.mark.parametrize("name", ["7b-mini", "33b-mini"])
def test_profiled_step_equals_step(name):
    """medusa_step_profiled (sequential stage order, events between stages)
    gives the same results as medusa_step (overlapped order)."""
    from medusa_head_tree_heads_b300 import medusa as M
    s, inp = U.planned_inputs(name)
    d = U.to_device(inp)
    cfg = M.make_config(s)
    ws = M.alloc_workspace(cfg)
    a, b = M.alloc_outputs(cfg), M.alloc_outputs(cfg)
    M.medusa_step(cfg, M.step_io(d, a), ws)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * len(M.STEP_KERNELS))]
    for e in evs:
        e.record()
    M.medusa_step_profiled(cfg, M.step_io(d, b), ws, evs)
    torch.cuda.synchronize()
    for k in ("topk_idx", "node_argmax", "accept_len", "acc_nodes", "bonus"):
        assert torch.equal(a[k], b[k]), k
    for k in ("node_maxlogit", "attn_out", "topk_val"):
        U.assert_close(a[k].float().cpu().numpy(), b[k].float().cpu().numpy(), s.dtype, k)


@pytest.mark.parametrize("name", ["tiny-fp32", "tiny-fp32-gqa", "k16-f32", "sparse-f32"])
def test_forked_fp32_step_in_a_graph_equals_the_serial_step(name):
    """The fp32 step runs its tree attention and verification on a second
    stream beside the heads; captured in a CUDA graph (two branches) and
    replayed, it gives the profiled step's results (one stream, stage order)
    bit for bit: the same kernels with the same launch shapes."""
    from medusa_head_tree_heads_b300 import medusa as M
    s, inp = U.planned_inputs(name)
    assert s.dtype == "f32"
    d = U.to_device(inp)
    cfg = M.make_config(s)
    ws = M.alloc_workspace(cfg)
    a, b = M.alloc_outputs(cfg), M.alloc_outputs(cfg)
    io = M.step_io(d, a)
    M.medusa_step(cfg, io, ws)  # eager once (creates the side stream outside the capture)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        M.medusa_step(cfg, io, ws)
    def fill(outs):  # the same sentinel wherever a step leaves an output entry unwritten
        for v in outs.values():
            for t in (v.values() if isinstance(v, dict) else [v]):
                t.fill_(-7)

    for _ in range(3):
        fill(a)
        g.replay()
    fill(b)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * len(M.STEP_KERNELS))]
    for e in evs:
        e.record()
    M.medusa_step_profiled(cfg, M.step_io(d, b), ws, evs)
    torch.cuda.synchronize()
    assert M.medusa_get_device_error(ws) == 0
    for k in a:
        if k == "tree":
            for t in a[k]:
                assert torch.equal(a[k][t], b[k][t]), t
        else:
            assert torch.equal(a[k], b[k]), k


def test_fp32_step_captured_on_a_threads_first_call():
    """A host thread whose first fp32 step is inside a graph capture gets no
    second stream (creating one could break the capture): the capture
    succeeds, the step runs in one stream and matches the forked step."""
    import threading

    from medusa_head_tree_heads_b300 import medusa as M
    s, inp = U.planned_inputs("tiny-fp32-gqa")
    d = U.to_device(inp)
    cfg = M.make_config(s)
    ws = M.alloc_workspace(cfg)
    a, b = M.alloc_outputs(cfg), M.alloc_outputs(cfg)
    for outs in (a, b):  # the same sentinel wherever a step leaves an output entry unwritten
        for v in outs.values():
            for x in (v.values() if isinstance(v, dict) else [v]):
                x.fill_(-7)
    M.medusa_step(cfg, M.step_io(d, b), ws)  # this thread: forked
    torch.cuda.synchronize()
    err = []

    def run():
        try:
            torch.cuda.set_device(d["h"].device)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                M.medusa_step(cfg, M.step_io(d, a), ws)
            g.replay()
            torch.cuda.synchronize()
        except Exception as e:  # reported below
            err.append(e)

    t = threading.Thread(target=run)
    t.start()
    t.join()
    assert not err, err
    assert M.medusa_get_device_error(ws) == 0
    for k in a:
        if k == "tree":
            for x in a[k]:
                assert torch.equal(a[k][x], b[k][x]), x
        else:
            assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("name", ["7b-mini", "gqa-mini"])
def test_repeated_steps_are_identical(name):
    """The workspace tickets reset themselves: back-to-back steps agree bitwise."""
    from medusa_head_tree_heads_b300 import medusa as M
    s, inp = U.planned_inputs(name)
    d = U.to_device(inp)
    cfg = M.make_config(s)
    ws = M.alloc_workspace(cfg)
    outs = []
    for _ in range(3):
        out = M.alloc_outputs(cfg)
        M.medusa_step(cfg, M.step_io(d, out), ws)
        torch.cuda.synchronize()
        outs.append(out)
    for k in ("topk_idx", "node_argmax", "accept_len", "acc_nodes", "bonus", "node_maxlogit"):
        assert torch.equal(outs[0][k], outs[1][k]) and torch.equal(outs[0][k], outs[2][k]), k


@pytest.mark.parametrize("name", ["tiny-fp32", "7b-mini"])
def test_zero_init_heads_reproduce_lm_head(name):
    """"Medusa Heads", "Come le teste prevedono i token successivi": with the
    head layer zeroed and the projection a copy of lm_head every head gives
    lm_head's prediction; on the GPU every head's top-k (ids and values) is
    bitwise the same, and equals the oracle's lm_head(h) top-k."""
    from medusa_head_tree_heads_b300 import medusa as M
    s = synth.SHAPES[name]
    inp = synth.make_inputs(s, zero_init=True)
    d = U.to_device(inp)
    cfg = M.make_config(s)
    ws = M.alloc_workspace(cfg)
    out = M.alloc_outputs(cfg)
    M.medusa_heads_topk(cfg, d["h"], d["W1"], d["b1"], d["W2"], out["topk_idx"], out["topk_val"], ws)
    torch.cuda.synchronize()
    idx, val = out["topk_idx"].cpu(), out["topk_val"].cpu()
    for k in range(1, s.n_heads):
        m = min(s.topk[k] if k < s.depth else 1, s.topk[0])  # common prefix of the two lists
        assert torch.equal(idx[:, k, :m], idx[:, 0, :m])
        assert torch.equal(val[:, k, :m], val[:, 0, :m])
    base = O.base_logits(U.to_np(inp["h"]), U.to_np(inp["lm_head"]))
    ridx, _ = O.topk_lists(base[:, None, :], [s.topk[0]])
    np.testing.assert_array_equal(idx[:, 0, :s.topk[0]].numpy(), ridx[:, 0, :s.topk[0]])


def test_typical_delta_zero_accepts_full_depth():
    """delta = 0 makes the threshold 0: every candidate is kept (full depth)."""
    from medusa_head_tree_heads_b300 import medusa as M
    s, inp = U.planned_inputs("gqa-mini")
    d = U.to_device(inp)
    cfg = M.make_config(s, delta=0.0)
    ws = M.alloc_workspace(cfg)
    out = M.alloc_outputs(cfg)
    M.medusa_step(cfg, M.step_io(d, out), ws)
    torch.cuda.synchronize()
    assert (out["accept_len"].cpu() == s.depth).all()
    assert (out["acc_nodes"].cpu()[:, :] == torch.tensor([0, 1, 5, 17, 41], dtype=torch.int32)).all()


def test_out_of_range_token_sets_device_error():
    """A tree token outside the vocabulary is caught by the acceptance
    kernel's own bounds check: the error word is set, nothing is read."""
    from medusa_head_tree_heads_b300 import medusa as M
    s, inp = U.planned_inputs("gqa-mini")
    d = U.to_device(inp)
    cfg = M.make_config(s)
    ws = M.alloc_workspace(cfg)
    out = M.alloc_outputs(cfg)
    M.medusa_step(cfg, M.step_io(d, out), ws)
    torch.cuda.synchronize()
    assert M.medusa_get_device_error(ws) == 0
    out["tree"]["token"][0, 3] = s.vocab + 5
    M.medusa_verify_accept(cfg, out["attn_out"], d["lm_head"], out["tree"], out, ws)
    torch.cuda.synchronize()
    assert M.medusa_get_device_error(ws) == -5
    assert M.medusa_get_device_error(ws) == 0  # read clears it


def test_bounded_wait_reports_timeout_and_context_survives():
    """Failure detection without a fault: a wait on an mbarrier nothing
    completes gives up after its budget, records MEDUSA_ERR_TIMEOUT, and the
    context keeps working (a full step afterwards matches the oracle)."""
    from medusa_head_tree_heads_b300 import medusa as M
    s, inp = U.planned_inputs("7b-mini")
    cfg = M.make_config(s)
    ws = M.alloc_workspace(cfg)
    M.medusa_check_bounded_wait(ws, 2000)
    torch.cuda.synchronize()
    assert M.medusa_get_device_error(ws) == -4
    assert M.medusa_get_device_error(ws) == 0
    ref = O.step(U.np_inputs(inp), s)
    res = U.gpu_step(s, U.to_device(inp))
    U.compare_step(s, res, ref)


@pytest.mark.parametrize("name,schedule", [(n, "auto") for n in FULL] +
                         [(n, "serial") for n in ("7b-bf16", "13b-bf16", "gqa128k-bf16", "33b-bf16")])
def test_full_size_sampled(name, schedule):
    """Full size in the launch configuration the benchmark times (AUTO: the
    overlap order wherever it is supported), plus the tensor-core shapes in
    the serial order."""
    from medusa_head_tree_heads_b300 import medusa as M
    s, inp = U.planned_inputs(name)
    res = U.gpu_step(s, U.to_device(inp), schedule={"auto": M.AUTO, "serial": M.SERIAL, "overlap": M.OVERLAP}[schedule])
    U.compare_full_size(s, inp, res)
