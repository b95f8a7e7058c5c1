"""The vocabulary-sharded step through the C ABI, its shards emulated one
after another on one GPU: every shard's medusa_shard_partial on its own rows
of W2 and lm_head (ragged row counts, not multiples of any tile), the records
copied side by side as the all-gather would lay them out, then
medusa_shard_finish.  The result must equal the oracle's unsplit step: ids,
tree, node choices and acceptance bit for bit, floats within the tolerance
(the combination only reorders sums)."""
from __future__ import annotations

import pytest
import torch

from oracle import medusa_oracle as O
from tests import util as U

pytestmark = pytest.mark.gpu

CASES = [("7b-mini", 2), ("7b-mini", 3), ("gqa-mini", 2), ("gqa-b16-mini", 3), ("sample-mini", 3),
         ("13b-b8-split", 2), ("33b-b32-mini", 2), ("tiny-fp32", 2), ("tiny-fp32-gqa", 3), ("sparse-typical-mini", 2),
         ("k16-f32", 2)]


def sharded_run(name, S):
    from medusa_head_tree_heads_b300 import medusa as M
    from medusa_head_tree_heads_b300 import shards as SH
    s, inp = U.planned_inputs(name)
    d = U.to_device(inp)
    # ragged cuts: the first shard takes a little more than its share
    cuts = [0] + [int(s.vocab * (k + 0.31) / S) for k in range(1, S)] + [s.vocab]
    ranges = list(zip(cuts[:-1], cuts[1:]))
    steps = [SH.ShardedStep(s, S, k, row_ranges=ranges) for k in range(S)]
    out = M.alloc_outputs(steps[0].cfg)
    io = None
    for k, st in enumerate(steps):
        W2s, lms = SH.shard_weights(d["W2"], d["lm_head"], *ranges[k])
        io = M.step_io(dict(d, W2=W2s, lm_head=lms), out)
        st.partial(io)
        steps[0].records[k].copy_(st.record)
    steps[0].finish(io)
    torch.cuda.synchronize()
    for st in steps:
        assert M.medusa_get_device_error(st.ws) == 0
    res = {k: v.cpu() for k, v in out.items() if k != "tree"}
    res["tree"] = {k: v.cpu() for k, v in out["tree"].items()}
    return s, inp, res


@pytest.mark.parametrize("name,S", CASES)
def test_sharded_step_matches_the_oracle(name, S):
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the gpu-marked tests")
    s, inp, res = sharded_run(name, S)
    ref = O.step(U.np_inputs(inp), s)
    U.compare_step(s, res, ref)


def test_misordered_shards_set_the_device_error():
    """Records in the wrong order do not tile the vocabulary: the combination
    reports MEDUSA_ERR_DEVICE (its own check, nothing out of bounds)."""
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the gpu-marked tests")
    from medusa_head_tree_heads_b300 import medusa as M
    from medusa_head_tree_heads_b300 import shards as SH
    s, inp = U.planned_inputs("7b-mini")
    d = U.to_device(inp)
    steps = [SH.ShardedStep(s, 2, k) for k in range(2)]
    out = M.alloc_outputs(steps[0].cfg)
    for k, st in enumerate(steps):
        W2s, lms = SH.shard_weights(d["W2"], d["lm_head"], *SH.bounds(s.vocab, 2)[k])
        io = M.step_io(dict(d, W2=W2s, lm_head=lms), out)
        st.partial(io)
        steps[0].records[1 - k].copy_(st.record)
    steps[0].finish(io)
    torch.cuda.synchronize()
    assert M.medusa_get_device_error(steps[0].ws) == -5


@pytest.mark.parametrize("name,S", [("7b-bf16", 2), ("gqa76-bf16", 4)])
def test_sharded_full_size_matches_the_oracle(name, S):
    """Full size, ragged shards: compared with the oracle the way the fused
    full-size step is (heads, top-k, tree everywhere; planted acceptance bit
    for bit; attention and the base model's choice on sampled nodes)."""
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the gpu-marked tests")
    s, inp, res = sharded_run(name, S)
    U.compare_full_size(s, inp, res)
