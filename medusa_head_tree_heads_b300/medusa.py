"""Thin ctypes binding of libmedusa.so (include/medusa.h).

Argument marshalling only: every function here converts torch tensors to
device pointers, passes the current CUDA stream, calls the C entry point of
the same name and raises on a non-zero status.  All arithmetic of the step
runs in the library's CUDA kernels; there is no other path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmedusa.so")

MAX_DEPTH = 8
F32, BF16 = 0, 1
GREEDY, TYPICAL, SAMPLE, TYPICAL_SAMPLE = 0, 1, 2, 3
AUTO, SERIAL, OVERLAP = 0, 1, 2  # medusa_schedule_t
STATUS = {0: "MEDUSA_OK", -1: "MEDUSA_ERR_INVALID_ARG", -2: "MEDUSA_ERR_UNSUPPORTED", -3: "MEDUSA_ERR_CUDA",
          -4: "MEDUSA_ERR_TIMEOUT", -5: "MEDUSA_ERR_DEVICE"}

# every symbol include/medusa.h declares
EXPORTS = ("medusa_workspace_bytes", "medusa_tree_size", "medusa_heads_topk", "medusa_tree_build",
           "medusa_tree_attn", "medusa_verify_accept", "medusa_step", "medusa_step_profiled",
           "medusa_step_launches", "medusa_get_device_error", "medusa_status_string",
           "medusa_heads_topk_noalloc", "medusa_check_bounded_wait", "medusa_tree_attn_lens", "medusa_kv_commit",
           "medusa_next_inputs", "medusa_shard_record_bytes", "medusa_shard_partial", "medusa_shard_finish")
STEP_KERNELS = ("head_layer", "head_proj_topk", "tree_build", "tree_attn", "verify_proj", "accept")


class MedusaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {code} ({STATUS.get(code, 'unknown')})")
        self.code = code


class Config(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("hidden", ctypes.c_int32), ("vocab", ctypes.c_int32),
                ("n_heads", ctypes.c_int32), ("depth", ctypes.c_int32), ("topk", ctypes.c_int32 * MAX_DEPTH),
                ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("kv_len", ctypes.c_int32), ("kv_capacity", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("accept_mode", ctypes.c_int32), ("temperature", ctypes.c_float), ("eps", ctypes.c_float),
                ("delta", ctypes.c_float), ("tree_nodes", ctypes.c_int32),
                ("tree_parent", ctypes.POINTER(ctypes.c_int32)), ("tree_rank", ctypes.POINTER(ctypes.c_int32)),
                ("sample_seed", ctypes.c_uint32 * 2), ("sample_step", ctypes.c_int32),
                ("schedule", ctypes.c_int32), ("vocab_begin", ctypes.c_int32), ("vocab_rows", ctypes.c_int32)]


class Tree(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("token", "parent", "depth", "rank", "mask", "paths", "pos")]


class StepIO(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "h", "W1", "b1", "W2", "lm_head", "root_token", "q", "k_tree", "v_tree", "k_cache", "v_cache",
        "topk_idx", "topk_val")] + [("tree", Tree)] + [(n, ctypes.c_void_p) for n in (
            "attn_out", "node_argmax", "node_maxlogit", "node_lse", "node_entropy", "accept_len", "acc_tokens",
            "acc_nodes", "bonus", "kv_lens")]


_lib = None


def lib() -> ctypes.CDLL:
    """Loads libmedusa.so; raises if it is missing (there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with python -m medusa_head_tree_heads_b300.build")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32p = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)
        cfgp = ctypes.POINTER(Config)
        L.medusa_workspace_bytes.argtypes = [cfgp]
        L.medusa_workspace_bytes.restype = ctypes.c_size_t
        L.medusa_tree_size.argtypes = [cfgp, i32p, i32p, i32p]
        L.medusa_heads_topk.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.medusa_tree_build.argtypes = [cfgp, vp, vp, ctypes.POINTER(Tree), vp]
        L.medusa_tree_attn.argtypes = [cfgp, vp, vp, vp, vp, vp, ctypes.POINTER(Tree), vp, vp, vp]
        L.medusa_verify_accept.argtypes = [cfgp, vp, vp, ctypes.POINTER(Tree)] + [vp] * 10
        L.medusa_step.argtypes = [cfgp, ctypes.POINTER(StepIO), vp, vp]
        L.medusa_step_profiled.argtypes = [cfgp, ctypes.POINTER(StepIO), vp, vp, ctypes.POINTER(vp), ctypes.c_int32]
        L.medusa_get_device_error.argtypes = [vp, i32p, vp]
        L.medusa_tree_attn_lens.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, ctypes.POINTER(Tree), vp, vp, vp]
        L.medusa_kv_commit.argtypes = [cfgp] + [vp] * 9
        L.medusa_next_inputs.argtypes = [cfgp] + [vp] * 8
        L.medusa_step_launches.argtypes = [cfgp]
        L.medusa_heads_topk_noalloc.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, vp]
        L.medusa_check_bounded_wait.argtypes = [vp, ctypes.c_int32, vp]
        L.medusa_shard_record_bytes.argtypes = [cfgp]
        L.medusa_shard_record_bytes.restype = ctypes.c_size_t
        L.medusa_shard_partial.argtypes = [cfgp, ctypes.POINTER(StepIO), vp, vp, vp]
        L.medusa_shard_finish.argtypes = [cfgp, ctypes.POINTER(StepIO), vp, ctypes.c_int32, vp, vp]
        L.medusa_status_string.argtypes = [ctypes.c_int]
        L.medusa_status_string.restype = ctypes.c_char_p
        for f in EXPORTS:
            if f not in ("medusa_workspace_bytes", "medusa_status_string", "medusa_shard_record_bytes"):
                getattr(L, f).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(fn: str, code: int) -> None:
    if code != 0:
        raise MedusaError(fn, code)


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def make_config(shape, **over) -> Config:
    """Config from any object with the workload fields (see synth.Shape)."""
    c = Config()
    c.batch, c.hidden, c.vocab, c.n_heads = shape.batch, shape.hidden, shape.vocab, shape.n_heads
    c.depth = len(shape.topk)
    for i, k in enumerate(shape.topk):
        c.topk[i] = k
    c.n_q_heads, c.n_kv_heads, c.head_dim = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    c.kv_len = shape.kv_len
    c.kv_capacity = shape.kv_capacity if shape.kv_capacity else shape.kv_len
    c.dtype = F32 if shape.dtype == "f32" else BF16
    c.accept_mode = {"greedy": GREEDY, "typical": TYPICAL, "sample": SAMPLE,
                     "typical-sample": TYPICAL_SAMPLE}[shape.accept]
    seed = getattr(shape, "sample_seed", (0, 0))
    c.sample_seed[0], c.sample_seed[1] = seed
    c.sample_step = getattr(shape, "sample_step", 0)
    c.schedule = getattr(shape, "schedule", AUTO)
    c.temperature, c.eps, c.delta = shape.temperature, shape.eps, shape.delta
    parent = getattr(shape, "tree_parent", None)
    if parent is not None:  # explicit tree: host arrays kept alive with the config
        rank = shape.tree_rank
        set_tree(c, parent, rank)
    for k, v in over.items():
        setattr(c, k, v)
    return c


def set_tree(c: Config, parent, rank) -> None:
    """Gives the config an explicit tree (host arrays owned by the config)."""
    n = len(parent)
    pa, ra = (ctypes.c_int32 * n)(*parent), (ctypes.c_int32 * n)(*rank)
    c._tree_arrays = (pa, ra)
    c.tree_nodes = n
    c.tree_parent = ctypes.cast(pa, ctypes.POINTER(ctypes.c_int32))
    c.tree_rank = ctypes.cast(ra, ctypes.POINTER(ctypes.c_int32))


def workspace_bytes(cfg: Config) -> int:
    return int(lib().medusa_workspace_bytes(ctypes.byref(cfg)))


def tree_size(cfg: Config):
    T, NL, W = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check("medusa_tree_size", lib().medusa_tree_size(ctypes.byref(cfg), ctypes.byref(T), ctypes.byref(NL),
                                                      ctypes.byref(W)))
    return T.value, NL.value, W.value


def alloc_workspace(cfg: Config, device="cuda") -> torch.Tensor:
    n = workspace_bytes(cfg)
    if n == 0:
        raise MedusaError("medusa_workspace_bytes", -1)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def alloc_tree(cfg: Config, device="cuda") -> Dict[str, torch.Tensor]:
    T, NL, W = tree_size(cfg)
    i32 = dict(dtype=torch.int32, device=device)
    return {"token": torch.empty(cfg.batch, T, **i32), "parent": torch.empty(T, **i32),
            "depth": torch.empty(T, **i32), "rank": torch.empty(T, **i32),
            "mask": torch.empty(T, W, **i32), "paths": torch.empty(NL, cfg.depth + 1, **i32),
            "pos": torch.empty(T, **i32)}


def _tree_struct(t: Dict[str, torch.Tensor]) -> Tree:
    return Tree(*[t[n].data_ptr() for n in ("token", "parent", "depth", "rank", "mask", "paths", "pos")])


def medusa_heads_topk(cfg: Config, h, W1, b1, W2, topk_idx, topk_val, ws, stream=None) -> None:
    _check("medusa_heads_topk", lib().medusa_heads_topk(ctypes.byref(cfg), _p(h), _p(W1), _p(b1), _p(W2),
                                                        _p(topk_idx), _p(topk_val), _p(ws), _stream(stream)))


def medusa_heads_topk_noalloc(cfg: Config, h, W1, b1, W2, topk_idx, topk_val, stream=None) -> None:
    """medusa_heads_topk for callers that cannot allocate device memory: no
    workspace argument; the library's fixed device scratch array is used."""
    _check("medusa_heads_topk_noalloc", lib().medusa_heads_topk_noalloc(
        ctypes.byref(cfg), _p(h), _p(W1), _p(b1), _p(W2), _p(topk_idx), _p(topk_val), _stream(stream)))


def medusa_tree_build(cfg: Config, topk_idx, root_token, tree: Dict[str, torch.Tensor], stream=None) -> None:
    ts = _tree_struct(tree)
    _check("medusa_tree_build", lib().medusa_tree_build(ctypes.byref(cfg), _p(topk_idx), _p(root_token),
                                                        ctypes.byref(ts), _stream(stream)))


def medusa_tree_attn(cfg: Config, q, k_tree, v_tree, k_cache, v_cache, tree, attn_out, ws, stream=None) -> None:
    ts = _tree_struct(tree)
    _check("medusa_tree_attn", lib().medusa_tree_attn(ctypes.byref(cfg), _p(q), _p(k_tree), _p(v_tree),
                                                      _p(k_cache), _p(v_cache), ctypes.byref(ts), _p(attn_out),
                                                      _p(ws), _stream(stream)))


def medusa_verify_accept(cfg: Config, attn_out, lm_head, tree, out: Dict[str, torch.Tensor], ws,
                         stream=None) -> None:
    ts = _tree_struct(tree)
    _check("medusa_verify_accept", lib().medusa_verify_accept(
        ctypes.byref(cfg), _p(attn_out), _p(lm_head), ctypes.byref(ts), _p(out["node_argmax"]),
        _p(out["node_maxlogit"]), _p(out.get("node_lse")), _p(out.get("node_entropy")), _p(out["accept_len"]),
        _p(out["acc_tokens"]), _p(out["acc_nodes"]), _p(out["bonus"]), _p(ws), _stream(stream)))


def alloc_outputs(cfg: Config, device="cuda") -> Dict[str, torch.Tensor]:
    """Every output tensor of one step, in the layouts of include/medusa.h."""
    T, NL, W = tree_size(cfg)
    B, D, K = cfg.batch, cfg.depth, cfg.n_heads
    kmax = max([cfg.topk[i] for i in range(D)] + [1])
    dt = torch.float32 if cfg.dtype == F32 else torch.bfloat16
    i32 = dict(dtype=torch.int32, device=device)
    f32 = dict(dtype=torch.float32, device=device)
    return {"topk_idx": torch.empty(B, K, kmax, **i32), "topk_val": torch.empty(B, K, kmax, **f32),
            "tree": alloc_tree(cfg, device), "attn_out": torch.empty(B, T, cfg.hidden, dtype=dt, device=device),
            "node_argmax": torch.empty(B, T, **i32), "node_maxlogit": torch.empty(B, T, **f32),
            "node_lse": torch.empty(B, T, **f32), "node_entropy": torch.empty(B, T, **f32),
            "accept_len": torch.empty(B, **i32), "acc_tokens": torch.empty(B, max(D, 1), **i32),
            "acc_nodes": torch.empty(B, D + 1, **i32), "bonus": torch.empty(B, **i32)}


def step_io(inputs: Dict[str, torch.Tensor], out: Dict[str, torch.Tensor], kv_lens=None) -> StepIO:
    """kv_lens: optional int32 device tensor [B] of per-sequence cache lengths."""
    io = StepIO()
    io.kv_lens = kv_lens.data_ptr() if kv_lens is not None else None
    for n in ("h", "W1", "b1", "W2", "lm_head", "root_token", "q", "k_tree", "v_tree", "k_cache", "v_cache"):
        setattr(io, n, inputs[n].data_ptr())
    for n in ("topk_idx", "topk_val", "attn_out", "node_argmax", "node_maxlogit", "node_lse", "node_entropy",
              "accept_len", "acc_tokens", "acc_nodes", "bonus"):
        setattr(io, n, out[n].data_ptr())
    io.tree = _tree_struct(out["tree"])
    return io


def medusa_tree_attn_lens(cfg: Config, q, k_tree, v_tree, k_cache, v_cache, kv_lens, tree, attn_out, ws,
                          stream=None) -> None:
    ts = _tree_struct(tree)
    _check("medusa_tree_attn_lens", lib().medusa_tree_attn_lens(
        ctypes.byref(cfg), _p(q), _p(k_tree), _p(v_tree), _p(k_cache), _p(v_cache), _p(kv_lens), ctypes.byref(ts),
        _p(attn_out), _p(ws), _stream(stream)))


def medusa_kv_commit(cfg: Config, acc_nodes, accept_len, k_tree, v_tree, k_cache, v_cache, kv_lens, ws,
                     stream=None) -> None:
    _check("medusa_kv_commit", lib().medusa_kv_commit(
        ctypes.byref(cfg), _p(acc_nodes), _p(accept_len), _p(k_tree), _p(v_tree), _p(k_cache), _p(v_cache),
        _p(kv_lens), _p(ws), _stream(stream)))


def medusa_next_inputs(cfg: Config, attn_out, acc_nodes, accept_len, bonus, h_next, root_next, ws,
                       stream=None) -> None:
    _check("medusa_next_inputs", lib().medusa_next_inputs(
        ctypes.byref(cfg), _p(attn_out), _p(acc_nodes), _p(accept_len), _p(bonus), _p(h_next), _p(root_next),
        _p(ws), _stream(stream)))


def medusa_step(cfg: Config, io: StepIO, ws, stream=None) -> None:
    _check("medusa_step", lib().medusa_step(ctypes.byref(cfg), ctypes.byref(io), _p(ws), _stream(stream)))


def medusa_step_profiled(cfg: Config, io: StepIO, ws, events, stream=None) -> None:
    """events: 2 * len(STEP_KERNELS) torch.cuda.Event(enable_timing=True);
    events[2k] / events[2k+1] bracket kernel k."""
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check("medusa_step_profiled", lib().medusa_step_profiled(ctypes.byref(cfg), ctypes.byref(io), _p(ws),
                                                              _stream(stream), arr, len(events)))


def shard_record_bytes(cfg: Config) -> int:
    """Bytes of one vocabulary shard's exchange record (0 if the config names no shard)."""
    return int(lib().medusa_shard_record_bytes(ctypes.byref(cfg)))


def medusa_shard_partial(cfg: Config, io: StepIO, record, ws, stream=None) -> None:
    _check("medusa_shard_partial", lib().medusa_shard_partial(ctypes.byref(cfg), ctypes.byref(io), _p(record),
                                                              _p(ws), _stream(stream)))


def medusa_shard_finish(cfg: Config, io: StepIO, records, n_shards: int, ws, stream=None) -> None:
    _check("medusa_shard_finish", lib().medusa_shard_finish(ctypes.byref(cfg), ctypes.byref(io), _p(records),
                                                            n_shards, _p(ws), _stream(stream)))


def medusa_get_device_error(ws, stream=None) -> int:
    code = ctypes.c_int32()
    _check("medusa_get_device_error", lib().medusa_get_device_error(_p(ws), ctypes.byref(code), _stream(stream)))
    return code.value


def medusa_check_bounded_wait(ws, budget_us: int, stream=None) -> None:
    _check("medusa_check_bounded_wait", lib().medusa_check_bounded_wait(_p(ws), budget_us, _stream(stream)))


def step_launches_raw(cfg: Config) -> int:
    """medusa_step_launches as returned (a negative status on a bad config)."""
    return int(lib().medusa_step_launches(ctypes.byref(cfg)))


def step_launches(cfg: Config) -> int:
    n = lib().medusa_step_launches(ctypes.byref(cfg))
    if n < 0:
        raise MedusaError("medusa_step_launches", n)
    return n


def status_string(code: int) -> str:
    return lib().medusa_status_string(code).decode()
