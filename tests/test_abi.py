"""C-ABI checks that need no GPU: the library loads, exports every function
include/medusa.h declares, sizes its workspace and tree, and rejects bad
arguments on the host before any launch."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from medusa_head_tree_heads_b300 import build as B
from medusa_head_tree_heads_b300 import medusa as M
from medusa_head_tree_heads_b300 import synth

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "medusa.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not B.up_to_date():
        B.build()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(medusa_\w+)\s*\(", src, flags=re.M)))


def test_header_lists_the_binding_exports():
    assert declared_functions() == sorted(M.EXPORTS)


def test_library_exports_every_declared_function():
    L = ctypes.CDLL(M.LIB_PATH)
    for name in declared_functions():
        assert hasattr(L, name), name


@pytest.mark.parametrize("name", sorted(synth.SHAPES))
def test_tree_size_closed_form(name):
    s = synth.SHAPES[name]
    cfg = M.make_config(s)
    T, NL, W = M.tree_size(cfg)
    assert T == s.n_nodes
    if s.tree_parent is None:  # Cartesian: the product of the list sizes
        n = 1
        for k in s.topk:
            n *= k
    else:  # explicit: the nodes that are nobody's parent
        n = T - len(set(s.tree_parent[1:]))
    assert NL == n
    assert W == (T + 31) // 32
    assert M.workspace_bytes(cfg) > 0


def test_workspace_is_modest_at_full_size():
    # the workspace holds partial results only (no weight-sized buffers)
    for name in ("7b-bf16", "13b-bf16", "gqa128k-bf16", "33b-bf16"):
        assert M.workspace_bytes(M.make_config(synth.SHAPES[name])) < 256 << 20


BAD = [
    (dict(batch=0), -1), (dict(hidden=100), -2), (dict(head_dim=96), -2), (dict(n_kv_heads=3), -1),
    (dict(kv_capacity=10), -1), (dict(dtype=7), -1), (dict(accept_mode=5), -1), (dict(n_heads=9), -2),
    (dict(depth=6), -2), (dict(temperature=0.0, accept_mode=1), -1), (dict(schedule=3), -1),
    (dict(schedule=M.OVERLAP, dtype=M.F32), -2), (dict(schedule=M.OVERLAP, head_dim=64, n_q_heads=10), -2),
    (dict(schedule=M.OVERLAP, batch=33), -2),
]


@pytest.mark.parametrize("over,code", BAD)
def test_invalid_configs_are_rejected_on_the_host(over, code):
    cfg = M.make_config(synth.SHAPES["7b-mini"], **over)
    assert M.workspace_bytes(cfg) == 0
    r = M.lib().medusa_tree_size(ctypes.byref(cfg), None, None, None)
    assert r == code, (over, r)


def test_topk_and_node_limits():
    cfg = M.make_config(synth.SHAPES["7b-mini"])
    cfg.topk[0] = 17  # above the per-depth limit
    assert M.lib().medusa_tree_size(ctypes.byref(cfg), None, None, None) == -2
    cfg = M.make_config(synth.SHAPES["wide-bf16"])
    cfg.topk[2] = 8  # 8 + 64 + 512 nodes: above 512
    assert M.lib().medusa_tree_size(ctypes.byref(cfg), None, None, None) == -2


BAD_TREES = [  # (parent, rank) for topk (2, 2): each breaks one rule of the explicit tree
    ([0, 0, 0], [0, 0, 1]),          # root's parent is not -1
    ([-1, 0, 1, 0], [0, 0, 0, 1]),   # (depth, parent, rank) order broken: depth 2 before depth 1
    ([-1, 0, 0], [0, 1, 0]),         # ranks under one parent out of order
    ([-1, 0, 0], [0, 0, 0]),         # the same child twice
    ([-1, 0, 3, 0], [0, 0, 0, 1]),   # parent after the node
    ([-1, 0, 0], [0, 0, 2]),         # rank beyond the depth-1 list (k = 2)
    ([-1, 0, 1, 2], [0, 0, 0, 0]),   # depth 3 in a depth-2 tree
]


@pytest.mark.parametrize("parent,rank", BAD_TREES)
def test_invalid_explicit_trees_are_rejected(parent, rank):
    s = synth.SHAPES["7b-mini"]
    cfg = M.make_config(s, depth=2)
    cfg.topk[0], cfg.topk[1] = 2, 2
    M.set_tree(cfg, parent, rank)
    assert M.lib().medusa_tree_size(ctypes.byref(cfg), None, None, None) == -1, (parent, rank)
    assert M.workspace_bytes(cfg) == 0


def test_explicit_tree_sizes_and_limits():
    s = synth.SHAPES["7b-mini"]
    cfg = M.make_config(s, depth=2)
    cfg.topk[0], cfg.topk[1] = 2, 2
    M.set_tree(cfg, [-1, 0, 0, 1], [0, 0, 1, 0])  # a depth-1 leaf and a depth-2 leaf
    assert M.tree_size(cfg) == (4, 2, 1)
    cfg.tree_nodes = 513  # above 512
    assert M.lib().medusa_tree_size(ctypes.byref(cfg), None, None, None) == -2


def test_null_pointers_are_rejected_before_any_launch():
    cfg = M.make_config(synth.SHAPES["tiny-fp32"])
    L = M.lib()
    assert L.medusa_heads_topk(ctypes.byref(cfg), None, None, None, None, None, None, None, None) == -1
    assert L.medusa_tree_build(ctypes.byref(cfg), None, None, None, None) == -1
    assert L.medusa_tree_attn(ctypes.byref(cfg), None, None, None, None, None, None, None, None, None) == -1
    assert L.medusa_verify_accept(ctypes.byref(cfg), None, None, None, *([None] * 10)) == -1
    assert L.medusa_step(ctypes.byref(cfg), None, None, None) == -1
    assert L.medusa_get_device_error(None, None, None) == -1
    assert L.medusa_tree_attn_lens(ctypes.byref(cfg), *([None] * 10)) == -1
    assert L.medusa_kv_commit(ctypes.byref(cfg), *([None] * 9)) == -1
    assert L.medusa_next_inputs(ctypes.byref(cfg), *([None] * 8)) == -1
    # misaligned (not 16-byte) pointers
    assert L.medusa_heads_topk(ctypes.byref(cfg), 8, 16, 16, 16, 16, 16, 16, None) == -1


def test_status_strings():
    assert M.status_string(0) == "MEDUSA_OK"
    assert M.status_string(-4) == "MEDUSA_ERR_TIMEOUT"
    assert M.status_string(123) == "MEDUSA_ERR_UNKNOWN"


def test_noalloc_rejects_configs_beyond_its_scratch_on_the_host():
    """The fixed-scratch heads entry point checks the heads stage's own
    scratch against its 16 MiB before any launch.  Batch 32 with two lists
    of 16 entries needs 2 x 1024 x 4 x 32 x 16 x 4 B = 16 MiB of top-k
    candidates plus 10.5 MB of cut-tile partials; batch 64 (the CUDA-core heads) with 8 heads of width
    8192 needs 64 x 8 x 8192 x 4 B = 16.8 MB of fp32 activations.  Both are
    refused with MEDUSA_ERR_UNSUPPORTED and no device call is made."""
    fake = ctypes.c_void_p(4096)  # aligned, never dereferenced: the call stops on the host
    for over in (dict(batch=32, depth=2, topk=(ctypes.c_int32 * 8)(16, 16, 0, 0, 0, 0, 0, 0)),
                 dict(batch=64, hidden=8192, n_q_heads=64, n_kv_heads=64, n_heads=8)):
        cfg = M.make_config(synth.SHAPES["7b-mini"], **over)
        r = M.lib().medusa_heads_topk_noalloc(ctypes.byref(cfg), fake, fake, fake, fake, fake, fake, None)
        assert r == -2, (over, r)


def test_schedule_launch_counts():
    """The overlap schedule runs the attention unsplit (no combine launch).
    AUTO (148 SMs assumed without a device) takes the overlap order wherever
    it is supported (bf16, head dim 128, batch <= 32) and the serial order
    elsewhere (fp32, head dim 64)."""
    def n(name, **over):
        return M.step_launches(M.make_config(synth.SHAPES[name], **over))
    assert n("7b-bf16", schedule=M.SERIAL) == 8   # 6 stages + attention combine + verification merge
    assert n("7b-bf16", schedule=M.OVERLAP) == 7
    assert n("tiny-fp32") == 6  # two branches: layer, projection, merge + tree | attention, verification; acceptance
    for name in ("7b-bf16", "7b-sample", "7b-sparse64", "13b-bf16", "gqa128k-bf16", "33b-bf16", "b5-mini"):
        assert n(name) == n(name, schedule=M.OVERLAP), name
    for name in ("tiny-fp32", "33b-b32-mini", "deep-bf16"):  # fp32; bf16 with head dim 64
        assert n(name) == n(name, schedule=M.SERIAL), name


def test_vocabulary_shard_configs_on_the_host():
    """Shard ranges are validated before any launch: a range past the
    vocabulary or an offset without rows is MEDUSA_ERR_INVALID_ARG, fewer rows
    than the longest top-k list MEDUSA_ERR_UNSUPPORTED; a shard config is
    refused by the unsharded entry points and an unsharded one by the shard
    entry points; the record size follows the layout of the header (16 bytes
    of header, then lists, node states and, for typical acceptance, the
    candidates' scores, each section 16-byte aligned)."""
    fake = ctypes.c_void_p(4096)  # aligned, never dereferenced: every call below stops on the host
    s = synth.SHAPES["7b-mini"]
    bad = [(dict(vocab_begin=s.vocab - 10, vocab_rows=11), -1), (dict(vocab_begin=5, vocab_rows=0), -1),
           (dict(vocab_begin=0, vocab_rows=3), -2)]
    for over, code in bad:
        cfg = M.make_config(s, **over)
        assert M.lib().medusa_workspace_bytes(ctypes.byref(cfg)) == 0, over
        T = ctypes.c_int32()
        assert M.lib().medusa_tree_size(ctypes.byref(cfg), ctypes.byref(T), None, None) == code, over
    shard = M.make_config(s, vocab_begin=1000, vocab_rows=1001)
    io = M.StepIO()
    assert M.lib().medusa_step(ctypes.byref(shard), ctypes.byref(io), fake, None) == -1
    assert M.lib().medusa_heads_topk(ctypes.byref(shard), fake, fake, fake, fake, fake, fake, fake, None) == -1
    assert M.lib().medusa_heads_topk_noalloc(ctypes.byref(shard), fake, fake, fake, fake, fake, fake, None) == -1
    assert M.step_launches_raw(shard) == -1
    whole = M.make_config(s)
    assert M.shard_record_bytes(whole) == 0
    assert M.lib().medusa_shard_partial(ctypes.byref(whole), ctypes.byref(io), fake, fake, None) == -1
    assert M.lib().medusa_shard_finish(ctypes.byref(whole), ctypes.byref(io), fake, 2, fake, None) == -1
    assert M.lib().medusa_shard_finish(ctypes.byref(shard), ctypes.byref(io), fake, 0, fake, None) == -1
    B, K, kmax, T = s.batch, s.n_heads, max(s.topk), s.n_nodes
    up = lambda x: (x + 15) // 16 * 16
    lists = up(16 + B * K * kmax * 4)
    lists = up(lists + B * K * kmax * 4)
    assert M.shard_record_bytes(shard) == up(lists + B * T * 16)
    g = synth.SHAPES["gqa-mini"]
    tg = M.make_config(g, vocab_begin=0, vocab_rows=2000)
    B, K, kmax, T = g.batch, g.n_heads, max(g.topk), g.n_nodes
    lists = up(16 + B * K * kmax * 4)
    lists = up(lists + B * K * kmax * 4)
    assert M.shard_record_bytes(tg) == up(up(lists + B * T * 16) + B * T * kmax * 4)
