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


@pytest.mark.parametrize("name", ["tiny-fp32", "7b-mini", "13b-mini", "gqa-mini"])
def test_noalloc_matches_workspace_entry_point(name):
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the gpu-marked tests")
    from medusa_head_tree_heads_b300 import medusa as M
    s, inp = U.planned_inputs(name)
    d = U.to_device(inp)
    cfg = M.make_config(s)
    ws = M.alloc_workspace(cfg)
    ref = M.alloc_outputs(cfg)
    M.medusa_heads_topk(cfg, d["h"], d["W1"], d["b1"], d["W2"], ref["topk_idx"], ref["topk_val"], ws)
    torch.cuda.synchronize()
    for call in range(2):  # the shared scratch keeps the previous call's contents
        out = M.alloc_outputs(cfg)
        out["topk_idx"].fill_(-7)
        out["topk_val"].fill_(float("nan"))
        M.medusa_heads_topk_noalloc(cfg, d["h"], d["W1"], d["b1"], d["W2"], out["topk_idx"], out["topk_val"])
        torch.cuda.synchronize()
        assert torch.equal(out["topk_idx"], ref["topk_idx"]), (name, call)
        live = ref["topk_idx"] >= 0
        U.assert_close(out["topk_val"][live].cpu().numpy(), ref["topk_val"][live].cpu().numpy(), s.dtype,
                       f"topk_val call {call}")


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
