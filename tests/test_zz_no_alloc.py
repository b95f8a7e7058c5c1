"""medusa_heads_topk_noalloc: the heads stage for callers that cannot
allocate device memory (no workspace argument; the library's fixed device
scratch array is used instead).  Its results must match medusa_heads_topk,
the entry point that takes a caller workspace, call after call.

This file is collected last on purpose: the variant shares one device array
across calls, so it is checked both in a fresh process and after every other
test has used the library."""
from __future__ import annotations

import pytest
import torch

from medusa_head_tree_heads_b300 import synth
from tests import util as U

pytestmark = pytest.mark.gpu


def _reference(name):
    """Inputs on the device and the workspace entry point's results."""
    from medusa_head_tree_heads_b300 import medusa as M
    s, inp = U.planned_inputs(name)
    d = U.to_device(inp)
    cfg = M.make_config(s)
    ws = M.alloc_workspace(cfg)
    ref = M.alloc_outputs(cfg)
    M.medusa_heads_topk(cfg, d["h"], d["W1"], d["b1"], d["W2"], ref["topk_idx"], ref["topk_val"], ws)
    torch.cuda.synchronize()
    return s, cfg, d, ref


def _check_noalloc(s, cfg, d, ref, what):
    from medusa_head_tree_heads_b300 import medusa as M
    out = M.alloc_outputs(cfg)
    out["topk_idx"].fill_(-7)
    out["topk_val"].fill_(float("nan"))
    M.medusa_heads_topk_noalloc(cfg, d["h"], d["W1"], d["b1"], d["W2"], out["topk_idx"], out["topk_val"])
    torch.cuda.synchronize()
    assert torch.equal(out["topk_idx"], ref["topk_idx"]), what
    live = ref["topk_idx"] >= 0
    U.assert_close(out["topk_val"][live].cpu().numpy(), ref["topk_val"][live].cpu().numpy(), s.dtype,
                   f"topk_val {what}")


# gqa-b16-mini (batch 16, 89 nodes) fits only because the heads stage packs
# its own scratch: counted to the end of the whole step's workspace it would
# need the verification partials too (over 16 MiB)
@pytest.mark.parametrize("name", ["tiny-fp32", "7b-mini", "13b-mini", "gqa-mini", "gqa-b16-mini"])
def test_noalloc_matches_workspace_entry_point(name):
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the gpu-marked tests")
    s, cfg, d, ref = _reference(name)
    for call in range(2):  # the shared scratch keeps the previous call's contents
        _check_noalloc(s, cfg, d, ref, (name, call))


def test_noalloc_configs_in_turn():
    """Configs of different batch, width and list length one after another:
    each call lays the shared array out differently, so an earlier call's z
    pairs, cut-tile partials and candidates lie where the next call keeps its
    boundary tickets.  Every call must still equal the workspace entry point
    (the entry point clears both ticket arrays before its kernels run)."""
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the gpu-marked tests")
    names = ["33b-b32-mini", "13b-b8-split", "7b-mini", "gqa-b16-mini", "b5-mini", "k16-bf16"]
    refs = {n: _reference(n) for n in names}
    for i, n in enumerate(names + names[::-1]):
        s, cfg, d, ref = refs[n]
        _check_noalloc(s, cfg, d, ref, (i, n))


def test_noalloc_rejects_configs_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the gpu-marked tests")
    from medusa_head_tree_heads_b300 import medusa as M
    # 64 sequences x 8 heads x 8192 hidden of fp32 activations alone exceed the fixed 16 MiB
    cfg = M.make_config(synth.SHAPES["7b-mini"], batch=64, hidden=8192, n_q_heads=64, n_kv_heads=64, n_heads=8)
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros(16, dtype=torch.int32, device="cuda")
    val = torch.zeros(16, dtype=torch.float32, device="cuda")
    with pytest.raises(M.MedusaError) as e:
        M.medusa_heads_topk_noalloc(cfg, x, x, x, x, idx, val)
    assert e.value.code == -2
