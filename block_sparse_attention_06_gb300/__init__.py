"""MiniMax Sparse Attention (MSA) hot path for NVIDIA GB300 (sm_103a).

A thin ctypes binding over libmsa.so (C ABI in include/msa.h).  Every function
here only marshals arguments: it checks dtypes, shapes and devices, allocates
outputs with torch when the caller passes none, and calls the C entry point of
the same name on torch's current CUDA stream.  All arithmetic runs in the CUDA
kernels; there is no CPU path.  Importing this package without the built
library raises immediately.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass
from typing import Optional, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmsa.so")

MSA_PHASE_DECODE = 0
MSA_PHASE_PREFILL = 1
MSA_PHASE_DECODE_MULTI = 2
MSA_OP_INVERT = 0
MSA_OP_DECODE = 1
MSA_OP_PREFILL = 2
MSA_OP_SELECT_PREFILL = 3
MSA_OP_SELECT_INVERT_PREFILL = 4

STATUS = {0: "MSA_OK", 1: "MSA_ERR_INVALID_ARG", 2: "MSA_ERR_UNSUPPORTED", 3: "MSA_ERR_CUDA",
          4: "MSA_ERR_DEVICE_BOUNDS", 5: "MSA_ERR_TIMEOUT", 6: "MSA_ERR_WORKSPACE",
          7: "MSA_ERR_DEVICE_UNSUPPORTED"}


class MsaError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        super().__init__(f"{where}: {STATUS.get(status, status)}: {detail}")
        self.status = status


class msa_dims_t(ctypes.Structure):
    _fields_ = [("Hq", ctypes.c_int32), ("G", ctypes.c_int32), ("D", ctypes.c_int32),
                ("Di", ctypes.c_int32), ("page_size", ctypes.c_int32), ("topk", ctypes.c_int32),
                ("max_blocks", ctypes.c_int32), ("sm_scale", ctypes.c_float)]


@dataclass(frozen=True)
class Dims:
    Hq: int
    G: int
    D: int
    Di: int
    topk: int
    max_blocks: int
    sm_scale: Optional[float] = None
    page_size: int = 128

    def c(self) -> msa_dims_t:
        sc = self.sm_scale if self.sm_scale is not None else 1.0 / math.sqrt(self.D)
        return msa_dims_t(self.Hq, self.G, self.D, self.Di, self.page_size, self.topk, self.max_blocks, sc)


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmsa.so is not built ({LIB_PATH}); run __graft_entry__.build() "
                          "or python -m block_sparse_attention_06_gb300._build")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, S, D = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.POINTER(msa_dims_t)
    sigs = {
        "msa_index_score": [P, P, P, P, P, I, I, I, D, I, P, P, P],
        "msa_topk_blocks": [P, P, I, D, P, P, P],
        "msa_build_page_table": [P, P, P, I, I, D, P, P, P, P],
        "msa_invert_selection": [P, P, I, I, D, P, P, P, P, S, P, P],
        "msa_sparse_attn_prefill": [P, P, P, P, P, P, P, P, I, I, I, D, P, P, P, S, P, P],
        "msa_lse_merge": [P, P, P, P, I, D, P, P, P, P],
        "msa_sparse_attn_decode": [P, P, P, P, P, I, I, D, P, P, P, S, P, P],
        "msa_decode_step": [P, P, P, P, P, P, P, I, I, D, P, P, P, P, P, P, P, S, P, P],
        "msa_offload_gather": [P, P, I, P, I, D, P, P, P, P, P],
        "msa_stage_from_host": [P, P, S, P],
        "msa_select_prefill": [P, P, P, P, P, I, I, I, D, P, P, S, P, P],
        "msa_check": [P, P],
    }
    for name, argt in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = argt
        fn.restype = ctypes.c_int
    lib.msa_workspace_bytes.argtypes = [I, I, I, D]
    lib.msa_workspace_bytes.restype = ctypes.c_size_t
    lib.msa_last_error.restype = ctypes.c_char_p
    lib.msa_last_error.argtypes = []
    lib.msa_status_str.restype = ctypes.c_char_p
    lib.msa_status_str.argtypes = [ctypes.c_int]
    lib.msa_version.restype = ctypes.c_int32
    lib.msa_version.argtypes = []
    return lib


_lib = _load()


def library() -> ctypes.CDLL:
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _call(name: str, *args):
    rc = getattr(_lib, name)(*args)
    if rc != 0:
        raise MsaError(rc, name, _lib.msa_last_error().decode(errors="replace"))


def _req_result(t: torch.Tensor, dtype, name: str, shape=None):
    """A decode result buffer: a CUDA tensor, or a page-locked CPU tensor that the attention
    kernel writes directly over the host link."""
    if isinstance(t, torch.Tensor) and not t.is_cuda:
        if not t.is_pinned():
            raise ValueError(f"{name} must be a CUDA tensor or page-locked (pinned) host memory")
        if t.dtype != dtype or not t.is_contiguous() or (shape is not None and tuple(t.shape) != tuple(shape)):
            raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {shape}")
        return t
    return _req(t, dtype, name, shape)


def _req(t: torch.Tensor, dtype, name: str, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t


def new_err_word(device) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


def msa_check(err_word: torch.Tensor) -> None:
    """Synchronise the current stream, raise MsaError if a kernel flagged an error, clear the word."""
    _req(err_word, torch.int32, "err_word")
    _call("msa_check", _ptr(err_word), _stream(err_word.device))


def msa_selftest_timeout(err_word: torch.Tensor) -> None:
    """Queue the device self-test of the bounded-wait timeout: a wait that nothing
    completes gives up after its limit (2 s) and raises MSA_FLAG_TIMEOUT in err_word,
    which the next msa_check reports as MSA_ERR_TIMEOUT."""
    _req(err_word, torch.int32, "err_word")
    _call("msa_selftest_timeout", _ptr(err_word), _stream(err_word.device))


def msa_workspace_bytes(op: int, n_rows: int, n_req: int, dims: Dims) -> int:
    d = dims.c()
    return int(_lib.msa_workspace_bytes(op, n_rows, n_req, ctypes.byref(d)))


def msa_index_score(q_idx, kidx_cache, block_table, q_req, q_pos, dims: Dims, phase: int,
                    scores=None, err_word=None):
    n_rows = q_idx.shape[0]
    _req(q_idx, torch.bfloat16, "q_idx", (n_rows, dims.G, dims.Di))
    _req(kidx_cache, torch.bfloat16, "kidx_cache")
    if kidx_cache.dim() != 4 or tuple(kidx_cache.shape[1:]) != (dims.page_size, dims.G, dims.Di):
        raise ValueError("kidx_cache must be [n_pages][128][G][Di]")
    _req(block_table, torch.int32, "block_table")
    if block_table.dim() != 2 or block_table.shape[1] != dims.max_blocks:
        raise ValueError("block_table must be [n_req][max_blocks]")
    _req(q_req, torch.int32, "q_req", (n_rows,))
    _req(q_pos, torch.int32, "q_pos", (n_rows,))
    dev = q_idx.device
    if scores is None:
        scores = torch.empty((n_rows, dims.G, dims.max_blocks), dtype=torch.float32, device=dev)
    _req(scores, torch.float32, "scores", (n_rows, dims.G, dims.max_blocks))
    err_word = new_err_word(dev) if err_word is None else err_word
    d = dims.c()
    _call("msa_index_score", _ptr(q_idx), _ptr(kidx_cache), _ptr(block_table), _ptr(q_req), _ptr(q_pos),
          n_rows, block_table.shape[0], kidx_cache.shape[0], ctypes.byref(d), phase, _ptr(scores),
          _ptr(err_word), _stream(dev))
    return scores


def msa_select_prefill(q_idx, kidx_cache, block_table, q_req, q_pos, dims: Dims, sel=None, workspace=None,
                       err_word=None):
    """Prefill scoring and top-k in one pass (the selection of msa_index_score +
    msa_topk_blocks, without the scores); topk <= 16."""
    n_rows = q_idx.shape[0]
    _req(q_idx, torch.bfloat16, "q_idx", (n_rows, dims.G, dims.Di))
    _req(kidx_cache, torch.bfloat16, "kidx_cache")
    if kidx_cache.dim() != 4 or tuple(kidx_cache.shape[1:]) != (dims.page_size, dims.G, dims.Di):
        raise ValueError("kidx_cache must be [n_pages][128][G][Di]")
    _req(block_table, torch.int32, "block_table")
    if block_table.dim() != 2 or block_table.shape[1] != dims.max_blocks:
        raise ValueError("block_table must be [n_req][max_blocks]")
    _req(q_req, torch.int32, "q_req", (n_rows,))
    _req(q_pos, torch.int32, "q_pos", (n_rows,))
    dev = q_idx.device
    n_req = block_table.shape[0]
    if sel is None:
        sel = torch.empty((n_rows, dims.G, dims.topk), dtype=torch.int32, device=dev)
    _req(sel, torch.int32, "sel", (n_rows, dims.G, dims.topk))
    need = msa_workspace_bytes(MSA_OP_SELECT_PREFILL, n_rows, n_req, dims)
    if workspace is None:
        workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=dev)
    _req(workspace, torch.uint8, "workspace")
    err_word = new_err_word(dev) if err_word is None else err_word
    d = dims.c()
    _call("msa_select_prefill", _ptr(q_idx), _ptr(kidx_cache), _ptr(block_table), _ptr(q_req), _ptr(q_pos), n_rows,
          n_req, kidx_cache.shape[0], ctypes.byref(d), _ptr(sel), _ptr(workspace), workspace.numel(), _ptr(err_word),
          _stream(dev))
    return sel


def msa_topk_blocks(scores, q_pos, dims: Dims, sel=None, err_word=None):
    n_rows = scores.shape[0]
    _req(scores, torch.float32, "scores", (n_rows, dims.G, dims.max_blocks))
    _req(q_pos, torch.int32, "q_pos", (n_rows,))
    dev = scores.device
    if sel is None:
        sel = torch.empty((n_rows, dims.G, dims.topk), dtype=torch.int32, device=dev)
    _req(sel, torch.int32, "sel", (n_rows, dims.G, dims.topk))
    err_word = new_err_word(dev) if err_word is None else err_word
    d = dims.c()
    _call("msa_topk_blocks", _ptr(scores), _ptr(q_pos), n_rows, ctypes.byref(d), _ptr(sel), _ptr(err_word),
          _stream(dev))
    return sel


def msa_build_page_table(sel, block_table, seq_lens, n_pages: int, dims: Dims, page_table=None, row_len=None,
                         err_word=None):
    B = sel.shape[0]
    _req(sel, torch.int32, "sel", (B, dims.G, dims.topk))
    _req(block_table, torch.int32, "block_table", (B, dims.max_blocks))
    _req(seq_lens, torch.int32, "seq_lens", (B,))
    dev = sel.device
    if page_table is None:
        page_table = torch.empty((B * dims.G, dims.topk), dtype=torch.int32, device=dev)
    if row_len is None:
        row_len = torch.empty((B * dims.G,), dtype=torch.int32, device=dev)
    _req(page_table, torch.int32, "page_table", (B * dims.G, dims.topk))
    _req(row_len, torch.int32, "row_len", (B * dims.G,))
    err_word = new_err_word(dev) if err_word is None else err_word
    d = dims.c()
    _call("msa_build_page_table", _ptr(sel), _ptr(block_table), _ptr(seq_lens), B, n_pages, ctypes.byref(d),
          _ptr(page_table), _ptr(row_len), _ptr(err_word), _stream(dev))
    return page_table, row_len


def msa_select_invert_prefill(q_idx, kidx_cache, block_table, q_req, q_pos, dims: Dims, sel=None, blk_off=None,
                              blk_ent=None, ent_pos=None, workspace=None, err_word=None):
    """msa_select_prefill then msa_invert_selection in one call, the inversion's
    marking pass done by the list merge -> (sel, blk_off, blk_ent, ent_pos); the
    requests are the rows of block_table; topk <= 16."""
    n_rows = q_idx.shape[0]
    _req(q_idx, torch.bfloat16, "q_idx", (n_rows, dims.G, dims.Di))
    _req(kidx_cache, torch.bfloat16, "kidx_cache")
    if kidx_cache.dim() != 4 or tuple(kidx_cache.shape[1:]) != (dims.page_size, dims.G, dims.Di):
        raise ValueError("kidx_cache must be [n_pages][128][G][Di]")
    _req(block_table, torch.int32, "block_table")
    if block_table.dim() != 2 or block_table.shape[1] != dims.max_blocks:
        raise ValueError("block_table must be [n_req][max_blocks]")
    _req(q_req, torch.int32, "q_req", (n_rows,))
    _req(q_pos, torch.int32, "q_pos", (n_rows,))
    dev = q_idx.device
    n_req = block_table.shape[0]
    n_keys = dims.G * n_req * dims.max_blocks
    if sel is None:
        sel = torch.empty((n_rows, dims.G, dims.topk), dtype=torch.int32, device=dev)
    if blk_off is None:
        blk_off = torch.empty((n_keys + 1,), dtype=torch.int32, device=dev)
    if blk_ent is None:
        blk_ent = torch.empty((max(1, n_rows * dims.G * dims.topk),), dtype=torch.int32, device=dev)
    if ent_pos is None:
        ent_pos = torch.empty((n_rows, dims.G, dims.topk), dtype=torch.int32, device=dev)
    _req(sel, torch.int32, "sel", (n_rows, dims.G, dims.topk))
    _req(blk_off, torch.int32, "blk_off", (n_keys + 1,))
    _req(blk_ent, torch.int32, "blk_ent")
    if blk_ent.numel() < n_rows * dims.G * dims.topk:
        raise ValueError("blk_ent too small")
    _req(ent_pos, torch.int32, "ent_pos", (n_rows, dims.G, dims.topk))
    need = msa_workspace_bytes(MSA_OP_SELECT_INVERT_PREFILL, n_rows, n_req, dims)
    if workspace is None:
        workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=dev)
    _req(workspace, torch.uint8, "workspace")
    err_word = new_err_word(dev) if err_word is None else err_word
    d = dims.c()
    _call("msa_select_invert_prefill", _ptr(q_idx), _ptr(kidx_cache), _ptr(block_table), _ptr(q_req), _ptr(q_pos),
          n_rows, n_req, kidx_cache.shape[0], ctypes.byref(d), _ptr(sel), _ptr(blk_off), _ptr(blk_ent),
          _ptr(ent_pos), _ptr(workspace), workspace.numel(), _ptr(err_word), _stream(dev))
    return sel, blk_off, blk_ent, ent_pos


def msa_invert_selection(sel, q_req, n_req: int, dims: Dims, blk_off=None, blk_ent=None, ent_pos=None,
                         workspace=None, err_word=None):
    """-> (blk_off, blk_ent, ent_pos): the {block -> queries} CSR and each selected
    (row, group, slot)'s position in it."""
    n_rows = sel.shape[0]
    _req(sel, torch.int32, "sel", (n_rows, dims.G, dims.topk))
    _req(q_req, torch.int32, "q_req", (n_rows,))
    dev = sel.device
    n_keys = dims.G * n_req * dims.max_blocks
    if blk_off is None:
        blk_off = torch.empty((n_keys + 1,), dtype=torch.int32, device=dev)
    if blk_ent is None:
        blk_ent = torch.empty((max(1, n_rows * dims.G * dims.topk),), dtype=torch.int32, device=dev)
    _req(blk_off, torch.int32, "blk_off", (n_keys + 1,))
    _req(blk_ent, torch.int32, "blk_ent")
    if blk_ent.numel() < n_rows * dims.G * dims.topk:
        raise ValueError("blk_ent too small")
    if ent_pos is None:
        ent_pos = torch.empty((n_rows, dims.G, dims.topk), dtype=torch.int32, device=dev)
    _req(ent_pos, torch.int32, "ent_pos", (n_rows, dims.G, dims.topk))
    need = msa_workspace_bytes(MSA_OP_INVERT, n_rows, n_req, dims)
    if workspace is None:
        workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=dev)
    _req(workspace, torch.uint8, "workspace")
    err_word = new_err_word(dev) if err_word is None else err_word
    d = dims.c()
    _call("msa_invert_selection", _ptr(sel), _ptr(q_req), n_rows, n_req, ctypes.byref(d), _ptr(blk_off),
          _ptr(blk_ent), _ptr(ent_pos), _ptr(workspace), workspace.numel(), _ptr(err_word), _stream(dev))
    return blk_off, blk_ent, ent_pos


def partials_shape(n_ent: int, hpg: int, D: int):
    """Shape of the prefill partials buffer: per entry, D // 8 column chunks x hpg heads x 8 bf16
    (the layout msa.h documents)."""
    return (n_ent, D // 8, hpg, 8)


def partials_entry_major(o_part, n_ent: int, hpg: int, D: int):
    """The partials rearranged as [n_ent][hpg][D] (a permute; for inspection and tests)."""
    return o_part[:n_ent].permute(0, 2, 1, 3).reshape(n_ent, hpg, D)


def partials_from_entry_major(o_ent, hpg: int, D: int):
    """[n_ent][hpg][D] partials rearranged into the prefill partials layout (the inverse of
    partials_entry_major)."""
    n_ent = o_ent.shape[0]
    return o_ent.reshape(n_ent, hpg, D // 8, 8).permute(0, 2, 1, 3).contiguous()


def msa_sparse_attn_prefill(q, k_cache, v_cache, block_table, q_req, q_pos, blk_off, blk_ent, dims: Dims,
                            o_part=None, lse_part=None, workspace=None, err_word=None):
    n_rows = q.shape[0]
    _req(q, torch.bfloat16, "q", (n_rows, dims.Hq, dims.D))
    _req(k_cache, torch.bfloat16, "k_cache")
    _req(v_cache, torch.bfloat16, "v_cache", tuple(k_cache.shape))
    if k_cache.dim() != 4 or tuple(k_cache.shape[1:]) != (dims.page_size, dims.G, dims.D):
        raise ValueError("k_cache must be [n_pages][128][G][D]")
    _req(block_table, torch.int32, "block_table")
    n_req = block_table.shape[0]
    _req(q_req, torch.int32, "q_req", (n_rows,))
    _req(q_pos, torch.int32, "q_pos", (n_rows,))
    _req(blk_off, torch.int32, "blk_off", (dims.G * n_req * dims.max_blocks + 1,))
    _req(blk_ent, torch.int32, "blk_ent")
    dev = q.device
    n_ent, hpg = n_rows * dims.G * dims.topk, dims.Hq // dims.G
    if o_part is None:
        o_part = torch.empty(partials_shape(n_ent, hpg, dims.D), dtype=torch.bfloat16, device=dev)
    if lse_part is None:
        lse_part = torch.empty((n_ent, hpg), dtype=torch.float32, device=dev)
    _req(o_part, torch.bfloat16, "o_part", partials_shape(n_ent, hpg, dims.D))
    _req(lse_part, torch.float32, "lse_part", (n_ent, hpg))
    need = msa_workspace_bytes(MSA_OP_PREFILL, n_rows, n_req, dims)
    if workspace is None:
        workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=dev)
    _req(workspace, torch.uint8, "workspace")
    err_word = new_err_word(dev) if err_word is None else err_word
    d = dims.c()
    _call("msa_sparse_attn_prefill", _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(q_req),
          _ptr(q_pos), _ptr(blk_off), _ptr(blk_ent), n_rows, n_req, k_cache.shape[0], ctypes.byref(d),
          _ptr(o_part), _ptr(lse_part), _ptr(workspace), workspace.numel(), _ptr(err_word), _stream(dev))
    return o_part, lse_part


def msa_lse_merge(o_part, lse_part, sel, ent_pos, dims: Dims, out=None, lse=None, err_word=None):
    n_rows = sel.shape[0]
    n_ent, hpg = n_rows * dims.G * dims.topk, dims.Hq // dims.G
    _req(o_part, torch.bfloat16, "o_part", partials_shape(n_ent, hpg, dims.D))
    _req(lse_part, torch.float32, "lse_part", (n_ent, hpg))
    _req(sel, torch.int32, "sel", (n_rows, dims.G, dims.topk))
    _req(ent_pos, torch.int32, "ent_pos", (n_rows, dims.G, dims.topk))
    dev = o_part.device
    if out is None:
        out = torch.empty((n_rows, dims.Hq, dims.D), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((n_rows, dims.Hq), dtype=torch.float32, device=dev)
    _req(out, torch.bfloat16, "out", (n_rows, dims.Hq, dims.D))
    _req(lse, torch.float32, "lse", (n_rows, dims.Hq))
    err_word = new_err_word(dev) if err_word is None else err_word
    d = dims.c()
    _call("msa_lse_merge", _ptr(o_part), _ptr(lse_part), _ptr(sel), _ptr(ent_pos), n_rows, ctypes.byref(d),
          _ptr(out), _ptr(lse), _ptr(err_word), _stream(dev))
    return out, lse


def msa_sparse_attn_decode(q, k_cache, v_cache, page_table, row_len, dims: Dims, out=None, lse=None,
                           workspace=None, err_word=None):
    B = q.shape[0]
    _req(q, torch.bfloat16, "q", (B, dims.Hq, dims.D))
    _req(k_cache, torch.bfloat16, "k_cache")
    _req(v_cache, torch.bfloat16, "v_cache", tuple(k_cache.shape))
    if k_cache.dim() != 4 or tuple(k_cache.shape[1:]) != (dims.page_size, dims.G, dims.D):
        raise ValueError("k_cache must be [n_pages][128][G][D]")
    _req(page_table, torch.int32, "page_table", (B * dims.G, dims.topk))
    _req(row_len, torch.int32, "row_len", (B * dims.G,))
    dev = q.device
    if out is None:
        out = torch.empty((B, dims.Hq, dims.D), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, dims.Hq), dtype=torch.float32, device=dev)
    _req_result(out, torch.bfloat16, "out", (B, dims.Hq, dims.D))
    _req_result(lse, torch.float32, "lse", (B, dims.Hq))
    need = msa_workspace_bytes(MSA_OP_DECODE, B, 0, dims)
    if workspace is None:
        workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=dev)
    _req(workspace, torch.uint8, "workspace")
    err_word = new_err_word(dev) if err_word is None else err_word
    d = dims.c()
    _call("msa_sparse_attn_decode", _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table), _ptr(row_len), B,
          k_cache.shape[0], ctypes.byref(d), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
          _ptr(err_word), _stream(dev))
    return out, lse


def msa_offload_gather(host_k_cache, host_v_cache, page_table, dims: Dims, pool_k=None, pool_v=None,
                       pool_page_table=None, err_word=None):
    """Gather the selected group slices of host-resident K/V pages into a device pool;
    returns (pool_k, pool_v, pool_page_table) for msa_sparse_attn_decode."""
    for t, name in ((host_k_cache, "host_k_cache"), (host_v_cache, "host_v_cache")):
        if not isinstance(t, torch.Tensor) or t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous bf16 CPU tensor")
        if not t.is_pinned():
            raise ValueError(f"{name} must be page-locked (pin_memory)")
        if t.dim() != 4 or tuple(t.shape[1:]) != (dims.page_size, dims.G, dims.D):
            raise ValueError(f"{name} must be [n_pages][128][G][D]")
    if tuple(host_v_cache.shape) != tuple(host_k_cache.shape):
        raise ValueError("host_v_cache must match host_k_cache")
    rows = page_table.shape[0]
    _req(page_table, torch.int32, "page_table", (rows, dims.topk))
    if rows % dims.G:
        raise ValueError("page_table rows must be B*G")
    B = rows // dims.G
    dev = page_table.device
    shape = (B * dims.topk, dims.page_size, dims.G, dims.D)
    pool_k = torch.empty(shape, dtype=torch.bfloat16, device=dev) if pool_k is None else pool_k
    pool_v = torch.empty(shape, dtype=torch.bfloat16, device=dev) if pool_v is None else pool_v
    _req(pool_k, torch.bfloat16, "pool_k", shape)
    _req(pool_v, torch.bfloat16, "pool_v", shape)
    if pool_page_table is None:
        pool_page_table = torch.empty_like(page_table)
    _req(pool_page_table, torch.int32, "pool_page_table", tuple(page_table.shape))
    err_word = new_err_word(dev) if err_word is None else err_word
    d = dims.c()
    _call("msa_offload_gather", _ptr(host_k_cache), _ptr(host_v_cache), host_k_cache.shape[0], _ptr(page_table), B,
          ctypes.byref(d), _ptr(pool_k), _ptr(pool_v), _ptr(pool_page_table), _ptr(err_word), _stream(dev))
    return pool_k, pool_v, pool_page_table


def msa_decode_step(q, q_idx, k_cache, v_cache, kidx_cache, block_table, seq_lens, dims: Dims, scores=None,
                    sel=None, page_table=None, row_len=None, out=None, lse=None, workspace=None, err_word=None):
    """One whole decode step (index scan, top-k, page tables, sparse attention) in one
    call; returns (out, lse, sel, page_table, row_len, scores)."""
    B = q.shape[0]
    _req(q, torch.bfloat16, "q", (B, dims.Hq, dims.D))
    _req(q_idx, torch.bfloat16, "q_idx", (B, dims.G, dims.Di))
    _req(k_cache, torch.bfloat16, "k_cache")
    _req(v_cache, torch.bfloat16, "v_cache", tuple(k_cache.shape))
    if k_cache.dim() != 4 or tuple(k_cache.shape[1:]) != (dims.page_size, dims.G, dims.D):
        raise ValueError("k_cache must be [n_pages][128][G][D]")
    _req(kidx_cache, torch.bfloat16, "kidx_cache", (k_cache.shape[0], dims.page_size, dims.G, dims.Di))
    _req(block_table, torch.int32, "block_table", (B, dims.max_blocks))
    _req(seq_lens, torch.int32, "seq_lens", (B,))
    dev = q.device
    f = dict(device=dev)
    scores = torch.empty((B, dims.G, dims.max_blocks), dtype=torch.float32, **f) if scores is None else scores
    sel = torch.empty((B, dims.G, dims.topk), dtype=torch.int32, **f) if sel is None else sel
    if page_table is None:
        page_table = torch.empty((B * dims.G, dims.topk), dtype=torch.int32, **f)
    row_len = torch.empty((B * dims.G,), dtype=torch.int32, **f) if row_len is None else row_len
    out = torch.empty((B, dims.Hq, dims.D), dtype=torch.bfloat16, **f) if out is None else out
    lse = torch.empty((B, dims.Hq), dtype=torch.float32, **f) if lse is None else lse
    _req(scores, torch.float32, "scores", (B, dims.G, dims.max_blocks))
    _req(sel, torch.int32, "sel", (B, dims.G, dims.topk))
    _req(page_table, torch.int32, "page_table", (B * dims.G, dims.topk))
    _req(row_len, torch.int32, "row_len", (B * dims.G,))
    _req_result(out, torch.bfloat16, "out", (B, dims.Hq, dims.D))
    _req_result(lse, torch.float32, "lse", (B, dims.Hq))
    need = msa_workspace_bytes(MSA_OP_DECODE, B, 0, dims)
    if workspace is None:
        workspace = torch.empty((max(need, 1),), dtype=torch.uint8, **f)
    _req(workspace, torch.uint8, "workspace")
    err_word = new_err_word(dev) if err_word is None else err_word
    d = dims.c()
    _call("msa_decode_step", _ptr(q), _ptr(q_idx), _ptr(k_cache), _ptr(v_cache), _ptr(kidx_cache), _ptr(block_table),
          _ptr(seq_lens), B, k_cache.shape[0], ctypes.byref(d), _ptr(scores), _ptr(sel), _ptr(page_table),
          _ptr(row_len), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(), _ptr(err_word), _stream(dev))
    return out, lse, sel, page_table, row_len, scores


# ------------------------------------------------------------------ whole-path helpers

def dims_of(case) -> Dims:
    """Dims of a workload from the seeded generator (msa_inputs.Case)."""
    d = case.dims
    return Dims(d.Hq, d.G, d.D, d.Di, d.topk, case.max_blocks, d.sm_scale, d.page)


class DecodeStep:
    """One MSA decode step with preallocated buffers: index scoring -> top-k ->
    page table -> paged sparse attention.  Buffers are reused across calls so the
    step can be replayed (and captured in a CUDA graph).

    Calling the object runs the fused entry point msa_decode_step (three kernels);
    composed() runs the same step through the four separate entry points."""

    def __init__(self, dims: Dims, B: int, n_req: int, n_pages: int, device):
        self.dims, self.B, self.n_req, self.n_pages = dims, B, n_req, n_pages
        f = dict(device=device)
        self.scores = torch.empty((B, dims.G, dims.max_blocks), dtype=torch.float32, **f)
        self.sel = torch.empty((B, dims.G, dims.topk), dtype=torch.int32, **f)
        self.page_table = torch.empty((B * dims.G, dims.topk), dtype=torch.int32, **f)
        self.row_len = torch.empty((B * dims.G,), dtype=torch.int32, **f)
        # out and lse share one device buffer, so a step's results come back in one copy
        self._out_buf, (self.out, self.lse) = _packed(
            [((B, dims.Hq, dims.D), torch.bfloat16), ((B, dims.Hq), torch.float32)], device)
        self.workspace = torch.empty((max(1, msa_workspace_bytes(MSA_OP_DECODE, B, 0, dims)),),
                                     dtype=torch.uint8, **f)
        self.err = new_err_word(device)
        self.q_req = torch.arange(B, dtype=torch.int32, **f)
        self.kernel_launches = 3   # index scan, selection (top-k + page table), attention with merge

    def scores_only(self, q_idx, kidx_cache, block_table, q_pos):
        return msa_index_score(q_idx, kidx_cache, block_table, self.q_req, q_pos, self.dims, MSA_PHASE_DECODE,
                               scores=self.scores, err_word=self.err)

    def rest(self, q, k_cache, v_cache, block_table, q_pos, seq_lens):
        msa_topk_blocks(self.scores, q_pos, self.dims, sel=self.sel, err_word=self.err)
        msa_build_page_table(self.sel, block_table, seq_lens, self.n_pages, self.dims, self.page_table,
                             self.row_len, err_word=self.err)
        return msa_sparse_attn_decode(q, k_cache, v_cache, self.page_table, self.row_len, self.dims, self.out,
                                      self.lse, self.workspace, err_word=self.err)

    def composed(self, q, q_idx, k_cache, v_cache, kidx_cache, block_table, seq_lens, q_pos):
        self.scores_only(q_idx, kidx_cache, block_table, q_pos)
        return self.rest(q, k_cache, v_cache, block_table, q_pos, seq_lens)

    def offloaded(self, q, q_idx, host_k_cache, host_v_cache, kidx_cache, block_table, seq_lens, q_pos):
        """The step with K/V in page-locked host memory and the k-index on the GPU: scan,
        top-k and page tables on the GPU, then only the selected pages are gathered into a
        device pool (msa_offload_gather) and attended there."""
        self.scores_only(q_idx, kidx_cache, block_table, q_pos)
        msa_topk_blocks(self.scores, q_pos, self.dims, sel=self.sel, err_word=self.err)
        msa_build_page_table(self.sel, block_table, seq_lens, self.n_pages, self.dims, self.page_table,
                             self.row_len, err_word=self.err)
        if getattr(self, "_pool", None) is None:
            self._pool = (None, None, None)
        pk, pv, ppt = msa_offload_gather(host_k_cache, host_v_cache, self.page_table, self.dims, *self._pool,
                                         err_word=self.err)
        self._pool = (pk, pv, ppt)
        return msa_sparse_attn_decode(q, pk, pv, ppt, self.row_len, self.dims, self.out, self.lse, self.workspace,
                                      err_word=self.err)

    def __call__(self, q, q_idx, k_cache, v_cache, kidx_cache, block_table, seq_lens, q_pos=None, out=None,
                 lse=None):
        """The step through msa_decode_step; out and lse default to the step's device buffers
        and may be page-locked host views (host_results()), which the step then writes directly."""
        out = self.out if out is None else out
        lse = self.lse if lse is None else lse
        msa_decode_step(q, q_idx, k_cache, v_cache, kidx_cache, block_table, seq_lens, self.dims, self.scores,
                        self.sel, self.page_table, self.row_len, out, lse, self.workspace, self.err)
        return out, lse

    def capture(self, q, q_idx, k_cache, v_cache, kidx_cache, block_table, seq_lens, inputs=None,
                host_results=None):
        """Record one whole step on these tensors into a CUDA graph and keep it for replay():
        a serving engine replays the decode step instead of launching its kernels one by
        one.  With `inputs` (a DecodeInputs whose device views are the tensors passed here)
        the graph also holds that step's upload, and with `host_results` (the buffer from
        host_results()) the attention kernel writes out and lse straight into that
        page-locked buffer, so they need no copy of their own.  The tensors are baked into
        the graph: write new values into them, then replay().  One eager call runs first,
        so every kernel's attributes are set before capture."""
        args = (q, q_idx, k_cache, v_cache, kidx_cache, block_table, seq_lens)
        res = {}
        if host_results is not None:
            _, (h_out, h_lse) = self._host_views(host_results)
            res = dict(out=h_out, lse=h_lse)
        if inputs is not None:
            inputs.upload()
        self._graph_results = self(*args, **res)
        torch.cuda.synchronize(q.device)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            if inputs is not None:
                inputs.upload()
            self(*args, **res)
        self._graph = graph
        return graph

    def replay(self):
        """Replay the step recorded by capture() on the current stream; returns the (out,
        lse) it writes (the host views when it was captured with host_results)."""
        self._graph.replay()
        return self._graph_results

    def host_results(self):
        """Page-locked host buffer laid out like the device (out, lse) buffer, with its
        (out, lse) views: download() fills it from the device buffer, and a step given the
        views (or captured with the buffer) writes them directly."""
        buf = torch.empty(self._out_buf.shape, dtype=torch.uint8).pin_memory()
        return self._host_views(buf)

    def _host_views(self, buf):
        return buf, _views(buf, [(tuple(self.out.shape), self.out.dtype), (tuple(self.lse.shape), self.lse.dtype)])

    def download(self, host_buf):
        """Queue one device-to-host copy of out and lse into host_buf (from host_results)."""
        host_buf.copy_(self._out_buf, non_blocking=True)


def _layout(specs):
    """Byte offsets of tensors packed back to back, each on a 256-byte boundary."""
    offs, n = [], 0
    for shape, dtype in specs:
        offs.append(n)
        nbytes = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
        n += (nbytes + 255) // 256 * 256
    return offs, max(n, 1)


def _views(buf, specs):
    offs, _ = _layout(specs)
    out = []
    for (shape, dtype), o in zip(specs, offs):
        nbytes = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
        out.append(buf[o:o + nbytes].view(dtype).view(shape))
    return out


def _packed(specs, device):
    _, n = _layout(specs)
    buf = torch.empty((n,), dtype=torch.uint8, device=device)
    return buf, _views(buf, specs)


def msa_stage_from_host(host: torch.Tensor, dev: torch.Tensor) -> torch.Tensor:
    """Copy the bytes of a page-locked host tensor into a device tensor of the same byte
    size with the staging kernel of msa_stage_from_host (16-byte loads reading the host
    buffer in place), queued on the current stream."""
    if host.is_cuda or not host.is_pinned():
        raise ValueError("host must be a page-locked CPU tensor")
    if not host.is_contiguous():
        raise ValueError("host must be contiguous")
    _req(dev, dev.dtype, "dev")
    n = host.numel() * host.element_size()
    if dev.numel() * dev.element_size() != n:
        raise ValueError(f"dev holds {dev.numel() * dev.element_size()} bytes, host {n}")
    _call("msa_stage_from_host", _ptr(host), _ptr(dev), n, _stream(dev.device))
    return dev


class DecodeInputs:
    """The per-step inputs of a decode step for B requests -- q, q_idx, seq_lens,
    q_pos and block_table -- packed in one page-locked host buffer and one device
    buffer of the same layout, so a step's host-to-device traffic is one staging kernel
    (upload, msa_stage_from_host) instead of one copy per tensor.  Fill the host views
    (h_q, ...), call upload(), then pass the device views (q, ...) to DecodeStep."""

    def __init__(self, dims: Dims, B: int, device):
        specs = [((B, dims.Hq, dims.D), torch.bfloat16), ((B, dims.G, dims.Di), torch.bfloat16),
                 ((B,), torch.int32), ((B,), torch.int32), ((B, dims.max_blocks), torch.int32)]
        _, n = _layout(specs)
        self.host = torch.empty((n,), dtype=torch.uint8).pin_memory()
        self.h_q, self.h_q_idx, self.h_seq_lens, self.h_q_pos, self.h_block_table = _views(self.host, specs)
        self.dev, (self.q, self.q_idx, self.seq_lens, self.q_pos, self.block_table) = _packed(specs, device)

    @property
    def nbytes(self) -> int:
        return self.host.numel()

    def upload(self):
        """Queue the host-to-device copy of all inputs on the current stream: one staging
        kernel reads the page-locked buffer over the host link (a copy-engine transfer of
        these few hundred KB costs about 10 us more per step on a Grace-Blackwell node)."""
        msa_stage_from_host(self.host, self.dev)


class PrefillStep:
    """One MSA prefill chunk: tensor-core index scoring -> top-k -> {q,blk}->{blk,q}
    inversion -> KV-block-major sparse attention -> LSE merge.

    With fuse_topk (the default where topk <= 16 and max_blocks <= 8704) scoring,
    top-k and the inversion run as msa_select_invert_prefill and no scores are kept;
    otherwise msa_index_score writes `scores`, msa_topk_blocks selects from them and
    msa_invert_selection inverts."""

    def __init__(self, dims: Dims, n_rows: int, n_req: int, device, fuse_topk=None):
        self.dims, self.n_rows, self.n_req = dims, n_rows, n_req
        f = dict(device=device)
        n_chunks = (dims.max_blocks + 127) // 128
        if fuse_topk is None:
            fuse_topk = dims.topk <= 16 and n_chunks * 15 <= 1024
        self.fuse_topk = bool(fuse_topk)
        if self.fuse_topk:
            self.scores = None
            self.sel_ws = torch.empty(
                (max(1, msa_workspace_bytes(MSA_OP_SELECT_INVERT_PREFILL, n_rows, n_req, dims)),),
                dtype=torch.uint8, **f)
        else:
            self.scores = torch.empty((n_rows, dims.G, dims.max_blocks), dtype=torch.float32, **f)
        self.sel = torch.empty((n_rows, dims.G, dims.topk), dtype=torch.int32, **f)
        n_keys = dims.G * n_req * dims.max_blocks
        self.blk_off = torch.empty((n_keys + 1,), dtype=torch.int32, **f)
        self.blk_ent = torch.empty((max(1, n_rows * dims.G * dims.topk),), dtype=torch.int32, **f)
        self.ent_pos = torch.empty((n_rows, dims.G, dims.topk), dtype=torch.int32, **f)
        self.inv_ws = None if self.fuse_topk else torch.empty(
            (max(1, msa_workspace_bytes(MSA_OP_INVERT, n_rows, n_req, dims)),), dtype=torch.uint8, **f)
        self.attn_ws = torch.empty((max(1, msa_workspace_bytes(MSA_OP_PREFILL, n_rows, n_req, dims)),),
                                   dtype=torch.uint8, **f)
        n_ent, hpg = n_rows * dims.G * dims.topk, dims.Hq // dims.G
        self.o_part = torch.empty(partials_shape(n_ent, hpg, dims.D), dtype=torch.bfloat16, **f)
        self.lse_part = torch.empty((n_ent, hpg), dtype=torch.float32, **f)
        self.out = torch.empty((n_rows, dims.Hq, dims.D), dtype=torch.bfloat16, **f)
        self.lse = torch.empty((n_rows, dims.Hq), dtype=torch.float32, **f)
        self.err = new_err_word(device)
        # fused: scoring, list merge (+ the inversion's marks), 3 inversion kernels, plan, attention, merge;
        # otherwise scoring, top-k and 4 inversion kernels
        self.kernel_launches = 8 if self.fuse_topk else 9

    def select(self, q_idx, kidx_cache, block_table, q_req, q_pos):
        if self.fuse_topk:
            msa_select_invert_prefill(q_idx, kidx_cache, block_table, q_req, q_pos, self.dims, self.sel,
                                      self.blk_off, self.blk_ent, self.ent_pos, self.sel_ws, err_word=self.err)
            return
        msa_index_score(q_idx, kidx_cache, block_table, q_req, q_pos, self.dims, MSA_PHASE_PREFILL,
                        scores=self.scores, err_word=self.err)
        msa_topk_blocks(self.scores, q_pos, self.dims, sel=self.sel, err_word=self.err)
        msa_invert_selection(self.sel, q_req, self.n_req, self.dims, self.blk_off, self.blk_ent, self.ent_pos,
                             self.inv_ws, err_word=self.err)

    def attend(self, q, k_cache, v_cache, block_table, q_req, q_pos):
        msa_sparse_attn_prefill(q, k_cache, v_cache, block_table, q_req, q_pos, self.blk_off, self.blk_ent,
                                self.dims, self.o_part, self.lse_part, self.attn_ws, err_word=self.err)
        return msa_lse_merge(self.o_part, self.lse_part, self.sel, self.ent_pos, self.dims, self.out, self.lse,
                             err_word=self.err)

    def partials_by_slot(self):
        """The partials rearranged as [rows][topk][Hq][D] / [rows][topk][Hq] (host copies;
        slots with sel < 0 hold zeros / -inf).  For inspection and tests."""
        sel, pos = self.sel.cpu(), self.ent_pos.cpu()
        n_rows, G, k = sel.shape
        hpg = self.dims.Hq // G
        op = partials_entry_major(self.o_part.cpu(), n_rows * G * k, hpg, self.dims.D)
        lp = self.lse_part.cpu()
        valid = sel >= 0
        p = torch.where(valid, pos, torch.zeros_like(pos)).long()
        o = op[p]                                  # [rows][G][k][hpg][D]
        lse = lp[p]                                # [rows][G][k][hpg]
        o = torch.where(valid[..., None, None], o, torch.zeros_like(o))
        lse = torch.where(valid[..., None], lse, torch.full_like(lse, float("-inf")))
        o = o.permute(0, 2, 1, 3, 4).reshape(n_rows, k, G * hpg, -1)
        lse = lse.permute(0, 2, 1, 3).reshape(n_rows, k, G * hpg)
        return o, lse

    def __call__(self, q, q_idx, k_cache, v_cache, kidx_cache, block_table, q_req, q_pos):
        self.select(q_idx, kidx_cache, block_table, q_req, q_pos)
        return self.attend(q, k_cache, v_cache, block_table, q_req, q_pos)


class MixedStep:
    """One step of a chunked-prefill engine over ONE shared page pool: a batch of decode
    requests (one new token each) and a prefill chunk of one or more requests.  Decode
    rows take the decode path (index scan, top-k + page tables, paged attention:
    msa_decode_step); chunk rows take the block-major path (tensor-core scoring with the
    top-k fused, inversion, block-major attention, LSE merge: PrefillStep).  The two
    halves share the K, V and k-index caches and read disjoint block-table rows.

    With overlap=True the decode half runs on a side stream that forks from the caller's
    current stream and joins it again before the call returns, so the HBM-bound decode
    scan can run beside the prefill kernels where SM resources allow; otherwise both run
    in order on the current stream.  Either way every result is produced by the same
    kernels as the separate steps, so the outputs are bit-identical to them."""

    def __init__(self, dims: Dims, n_decode: int, n_prefill_rows: int, n_prefill_req: int, n_pages: int, device,
                 overlap: bool = True):
        self.decode = DecodeStep(dims, n_decode, n_decode, n_pages, device)
        self.prefill = PrefillStep(dims, n_prefill_rows, n_prefill_req, device)
        self.overlap = bool(overlap)
        self.device = torch.device(device)
        self._side = torch.cuda.Stream(device=self.device) if self.overlap else None
        self.kernel_launches = self.decode.kernel_launches + self.prefill.kernel_launches

    @property
    def err_words(self):
        return (self.decode.err, self.prefill.err)

    def __call__(self, k_cache, v_cache, kidx_cache, dec_q, dec_q_idx, dec_block_table, dec_seq_lens, pre_q,
                 pre_q_idx, pre_block_table, pre_q_req, pre_q_pos):
        """-> (decode out, decode lse, prefill out, prefill lse)"""
        if not self.overlap:
            self.decode(dec_q, dec_q_idx, k_cache, v_cache, kidx_cache, dec_block_table, dec_seq_lens)
            self.prefill(pre_q, pre_q_idx, k_cache, v_cache, kidx_cache, pre_block_table, pre_q_req, pre_q_pos)
            return self.decode.out, self.decode.lse, self.prefill.out, self.prefill.lse
        main = torch.cuda.current_stream(self.device)
        self._side.wait_stream(main)                 # inputs written on the caller's stream are visible
        with torch.cuda.stream(self._side):
            self.decode(dec_q, dec_q_idx, k_cache, v_cache, kidx_cache, dec_block_table, dec_seq_lens)
        self.prefill(pre_q, pre_q_idx, k_cache, v_cache, kidx_cache, pre_block_table, pre_q_req, pre_q_pos)
        main.wait_stream(self._side)                 # the decode results are complete on the caller's stream
        return self.decode.out, self.decode.lse, self.prefill.out, self.prefill.lse
