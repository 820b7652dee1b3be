"""MSA oracle -- TEST INFRASTRUCTURE ONLY.

A plain fp64 CPU restatement of MiniMax Sparse Attention (see msa_oracle.c for
the cited passages and the readings taken where the pages are silent).  Only the
test suite, the package smoke check and the benchmark's CPU-baseline leg may
import this module; the CUDA library never does, and the two share no code.

Every function takes torch CPU tensors (bf16 inputs are passed as their raw
16-bit patterns) and returns float64 / int32 torch tensors.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "msa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libmsa_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (strict IEEE double: no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
                               "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # MSA_ORACLE_LIB points the pins at a deliberately broken copy of the
            # oracle (the mutation test); unset, the oracle is built from source here.
            lib = ctypes.CDLL(os.environ.get("MSA_ORACLE_LIB") or build())
            P = ctypes.c_void_p
            I = ctypes.c_int32
            Dd = ctypes.c_double
            sigs = {
                "oracle_block_scores": [P, P, P, I, P, P, I, I, I, I, I, I, I, P],
                "oracle_topk": [P, P, I, I, I, I, I, P],
                "oracle_page_table": [P, P, I, P, I, I, I, I, P, P],
                "oracle_invert": [P, P, I, I, I, I, I, P, P],
                "oracle_attention": [P, P, P, P, I, P, P, P, I, I, I, I, I, I, I, I, Dd, P, P],
                "oracle_block_partials": [P, P, P, P, I, P, P, P, I, I, I, I, I, I, I, I, Dd, P, P],
                "oracle_lse_merge": [P, P, I, I, I, I, P, P],
                "oracle_paged_attention": [P, P, P, P, P, I, I, I, I, I, I, I, Dd, P, P],
            }
            for name, argt in sigs.items():
                fn = getattr(lib, name)
                fn.argtypes = argt
                fn.restype = ctypes.c_int
            _lib = lib
    return _lib


def _u16(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype in (torch.int16, torch.uint16):
        return t.numpy().view(np.uint16)
    raise TypeError(f"expected bf16 tensor, got {t.dtype}")


def _i32(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu().contiguous().to(torch.int32).numpy()
    return np.ascontiguousarray(np.asarray(t, dtype=np.int32))


def _f64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu().contiguous().to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(t, dtype=np.float64))


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, name: str):
    if rc != 0:
        raise ValueError(f"{name}: index out of range (code {rc})")


def block_scores(q_idx, kidx_cache, block_table, q_req, q_pos, max_blocks: int) -> torch.Tensor:
    """[rows][G][max_blocks] float64; -inf for non-candidate blocks."""
    lib = _load()
    qi, kc = _u16(q_idx), _u16(kidx_cache)
    bt, qr, qp = _i32(block_table), _i32(q_req), _i32(q_pos)
    n_rows, G, Di = q_idx.shape
    n_pages, page = kidx_cache.shape[0], kidx_cache.shape[1]
    out = np.empty((n_rows, G, max_blocks), dtype=np.float64)
    rc = lib.oracle_block_scores(_p(qi), _p(kc), _p(bt), bt.shape[1], _p(qr), _p(qp), n_rows,
                                 bt.shape[0], G, Di, page, n_pages, max_blocks, _p(out))
    _check(rc, "block_scores")
    return torch.from_numpy(out)


def topk(scores, q_pos, topk_: int, page: int = 128) -> torch.Tensor:
    """[rows][G][topk] int32: own block forced, others by (score desc, id asc), ascending, -1 pad."""
    lib = _load()
    s, qp = _f64(scores), _i32(q_pos)
    n_rows, G, max_blocks = s.shape
    sel = np.empty((n_rows, G, topk_), dtype=np.int32)
    _check(lib.oracle_topk(_p(s), _p(qp), n_rows, G, page, max_blocks, topk_, _p(sel)), "topk")
    return torch.from_numpy(sel)


def page_table(sel, block_table, seq_lens, page: int = 128):
    """Decode rows r = b*G + g -> (pt [B*G][topk], row_len [B*G])."""
    lib = _load()
    sl, bt, ln = _i32(sel), _i32(block_table), _i32(seq_lens)
    B, G, k = sl.shape
    pt = np.empty((B * G, k), dtype=np.int32)
    rl = np.empty((B * G,), dtype=np.int32)
    _check(lib.oracle_page_table(_p(sl), _p(bt), bt.shape[1], _p(ln), B, G, k, page, _p(pt), _p(rl)),
           "page_table")
    return torch.from_numpy(pt), torch.from_numpy(rl)


def invert(sel, q_req, n_req: int, max_blocks: int):
    """CSR over keys (g*n_req + req)*max_blocks + block -> (blk_off, blk_ent)."""
    lib = _load()
    sl, qr = _i32(sel), _i32(q_req)
    n_rows, G, k = sl.shape
    n_keys = G * n_req * max_blocks
    off = np.empty((n_keys + 1,), dtype=np.int32)
    ent = np.empty((max(1, int((sl >= 0).sum())),), dtype=np.int32)
    _check(lib.oracle_invert(_p(sl), _p(qr), n_rows, n_req, G, k, max_blocks, _p(off), _p(ent)),
           "invert")
    return torch.from_numpy(off), torch.from_numpy(ent[:int(off[-1])])


def attention(q, k_cache, v_cache, block_table, q_req, q_pos, sel, sm_scale: float):
    """Exact attention over the selected blocks -> (out [rows][Hq][D] f64, lse [rows][Hq] f64)."""
    lib = _load()
    qq, kc, vc = _u16(q), _u16(k_cache), _u16(v_cache)
    bt, qr, qp, sl = _i32(block_table), _i32(q_req), _i32(q_pos), _i32(sel)
    n_rows, Hq, D = q.shape
    n_pages, page, G, _ = k_cache.shape
    k = sl.shape[2]
    out = np.empty((n_rows, Hq, D), dtype=np.float64)
    lse = np.empty((n_rows, Hq), dtype=np.float64)
    rc = lib.oracle_attention(_p(qq), _p(kc), _p(vc), _p(bt), bt.shape[1], _p(qr), _p(qp), _p(sl),
                              n_rows, bt.shape[0], Hq, G, D, page, n_pages, k, float(sm_scale),
                              _p(out), _p(lse))
    _check(rc, "attention")
    return torch.from_numpy(out), torch.from_numpy(lse)


def block_partials(q, k_cache, v_cache, block_table, q_req, q_pos, sel, sm_scale: float):
    """Per-slot normalised partials -> (o_part [rows][topk][Hq][D], lse_part [rows][topk][Hq])."""
    lib = _load()
    qq, kc, vc = _u16(q), _u16(k_cache), _u16(v_cache)
    bt, qr, qp, sl = _i32(block_table), _i32(q_req), _i32(q_pos), _i32(sel)
    n_rows, Hq, D = q.shape
    n_pages, page, G, _ = k_cache.shape
    k = sl.shape[2]
    op = np.empty((n_rows, k, Hq, D), dtype=np.float64)
    lp = np.empty((n_rows, k, Hq), dtype=np.float64)
    rc = lib.oracle_block_partials(_p(qq), _p(kc), _p(vc), _p(bt), bt.shape[1], _p(qr), _p(qp),
                                   _p(sl), n_rows, bt.shape[0], Hq, G, D, page, n_pages, k,
                                   float(sm_scale), _p(op), _p(lp))
    _check(rc, "block_partials")
    return torch.from_numpy(op), torch.from_numpy(lp)


def lse_merge(o_part, lse_part):
    """Merge [rows][topk][Hq][D] partials -> (out [rows][Hq][D], lse [rows][Hq])."""
    lib = _load()
    op, lp = _f64(o_part), _f64(lse_part)
    n_rows, k, Hq, D = op.shape
    out = np.empty((n_rows, Hq, D), dtype=np.float64)
    lse = np.empty((n_rows, Hq), dtype=np.float64)
    _check(lib.oracle_lse_merge(_p(op), _p(lp), n_rows, Hq, D, k, _p(out), _p(lse)), "lse_merge")
    return torch.from_numpy(out), torch.from_numpy(lse)


def paged_attention(q, k_cache, v_cache, pt, row_len, sm_scale: float):
    """Attention over decode page tables -> (out [B][Hq][D], lse [B][Hq])."""
    lib = _load()
    qq, kc, vc = _u16(q), _u16(k_cache), _u16(v_cache)
    p, rl = _i32(pt), _i32(row_len)
    B, Hq, D = q.shape
    n_pages, page, G, _ = k_cache.shape
    k = p.shape[1]
    out = np.empty((B, Hq, D), dtype=np.float64)
    lse = np.empty((B, Hq), dtype=np.float64)
    rc = lib.oracle_paged_attention(_p(qq), _p(kc), _p(vc), _p(p), _p(rl), B, Hq, G, D, page,
                                    n_pages, k, float(sm_scale), _p(out), _p(lse))
    _check(rc, "paged_attention")
    return torch.from_numpy(out), torch.from_numpy(lse)


def decode(case, rows=None):
    """Whole decode path for a decode case: scores -> top-k -> page table -> paged attention.
    `rows` optionally restricts to a subset of requests (the page pool is shared)."""
    c = case
    idx = torch.arange(c.n_rows) if rows is None else torch.as_tensor(rows)
    qi, qq = c.q_idx.cpu()[idx], c.q.cpu()[idx]
    qr, qp = c.q_req.cpu()[idx], c.q_pos.cpu()[idx]
    bt = c.block_table.cpu()[qr.long()]
    local_req = torch.arange(len(idx), dtype=torch.int32)
    sc = block_scores(qi, c.kidx_cache.cpu(), bt, local_req, qp, c.max_blocks)
    sel = topk(sc, qp, c.dims.topk, c.dims.page)
    pt, rl = page_table(sel, bt, qp + 1, c.dims.page)
    out, lse = paged_attention(qq, c.k_cache.cpu(), c.v_cache.cpu(), pt, rl, c.dims.sm_scale)
    return dict(scores=sc, sel=sel, pt=pt, row_len=rl, out=out, lse=lse)
