"""Helpers for the CUDA-vs-oracle parity tests.

Tolerances (fixed for the MSA hot path):
  block scores   |gpu - oracle| <= 2e-3 * (|oracle| + 1)
  selection      top-k on the oracle's fp32-rounded scores: bit-exact;
                 end to end: identical wherever the oracle's gap between the last
                 kept and the first dropped candidate exceeds 1e-2
  lse            |gpu - oracle| <= 1e-3
  bf16 output    max |gpu - oracle| <= 1.5e-2 and mean |gpu - oracle| <= 2e-3
"""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np
import torch

import oracle

SCORE_RTOL = 2e-3
GAP = 1e-2
LSE_ATOL = 1e-3
OUT_MAX = 1.5e-2
OUT_MEAN = 2e-3


def assert_scores(gpu: torch.Tensor, ref: torch.Tensor, q_pos: torch.Tensor, page: int = 128):
    g = gpu.detach().cpu().double()
    r = ref.detach().cpu().double()
    n_cand = (q_pos.cpu().long() // page + 1)
    mb = r.shape[-1]
    cand = torch.arange(mb)[None, None, :] < n_cand[:, None, None]
    assert torch.all(torch.isneginf(g[~cand.expand_as(g)])), "non-candidate blocks must be -inf"
    diff = (g - r).abs()[cand.expand_as(g)]
    tol = (SCORE_RTOL * (r.abs() + 1.0))[cand.expand_as(g)]
    bad = diff > tol
    assert not bool(bad.any()), f"{int(bad.sum())} scores outside 2e-3*(|s|+1); worst {float((diff - tol).max()):.3e}"


def selection_gap(scores: torch.Tensor, q_pos: torch.Tensor, topk: int, page: int = 128) -> torch.Tensor:
    """Per (row, group): score of the last kept non-own candidate minus the best dropped one
    (+inf when every candidate is kept)."""
    s = scores.detach().cpu().double().numpy()
    pos = q_pos.cpu().numpy()
    R, G, _ = s.shape
    gap = np.full((R, G), np.inf)
    for r in range(R):
        own = int(pos[r]) // page
        k_eff = min(topk, own + 1)
        if own + 1 <= topk:
            continue
        for g in range(G):
            v = np.sort(s[r, g, :own])[::-1]
            gap[r, g] = v[k_eff - 2] - v[k_eff - 1] if k_eff >= 2 else np.inf
    return torch.from_numpy(gap)


def assert_selection_where_unambiguous(gpu_sel, ref_sel, gap):
    ok = gap > GAP
    g, r = gpu_sel.cpu(), ref_sel.cpu()
    diff = (g != r).any(dim=-1) & ok
    assert not bool(diff.any()), f"{int(diff.sum())} unambiguous (row, group) selections differ"
    return ok


def assert_selection_valid(gpu_sel, ref_scores, q_pos, topk: int, page: int = 128):
    """Every (row, group) selection -- near ties included -- is *a* correct top-k of the
    oracle's scores within the score tolerance:

      * k_eff = min(topk, own + 1) ids, strictly ascending, then -1 padding;
      * every id is a candidate (0 .. own) and the last one is the own block;
      * no dropped candidate beats a kept one by more than the two scores' tolerances:
        min over kept non-own j of (s_j + tol_j) >= max over dropped i of (s_i - tol_i),
        tol = 2e-3 * (|s| + 1) (the GPU scores are within that of the oracle's, so any
        order the GPU can see between two blocks is one the oracle's values allow).
    """
    sel = gpu_sel.detach().cpu().numpy().astype(np.int64)
    s = ref_scores.detach().cpu().double().numpy()
    pos = q_pos.detach().cpu().numpy().astype(np.int64)
    R, G, k = sel.shape
    assert k == topk
    own = pos // page
    k_eff = np.minimum(topk, own + 1)
    slot = np.arange(k)[None, None, :]
    filled = np.broadcast_to(slot < k_eff[:, None, None], sel.shape)
    assert np.all(sel[~filled] == -1), "padding slots past k_eff must be -1"
    assert np.all(sel[filled] >= 0), "the first k_eff slots must hold block ids"
    assert np.all(sel <= own[:, None, None]), "a selected block lies past the row's own block"
    asc = np.diff(sel, axis=-1) > 0
    need_asc = filled[..., 1:]
    assert np.all(asc[need_asc]), "selected ids must be strictly ascending"
    last = np.take_along_axis(sel, (k_eff - 1)[:, None, None].repeat(G, axis=1), axis=-1)[..., 0]
    assert np.all(last == own[:, None]), "the own block must be selected (the last id)"
    tol = SCORE_RTOL * (np.abs(s) + 1.0)
    worst = 0.0
    for r in range(R):
        o = int(own[r])
        if o + 1 <= topk or topk == 1:   # every candidate kept, or only the own block: nothing to rank
            continue
        for g in range(G):
            kept = np.zeros(o, dtype=bool)
            ids = sel[r, g, :k_eff[r]]
            kept[ids[ids < o]] = True
            lo = np.min(s[r, g, :o][kept] + tol[r, g, :o][kept])
            hi = np.max(s[r, g, :o][~kept] - tol[r, g, :o][~kept])
            worst = max(worst, hi - lo)
    assert worst <= 0.0, f"a dropped block outranks a kept one by {worst:.3e} beyond the score tolerance"


def assert_topk_of_own_scores(gpu_sel, gpu_scores, q_pos, topk: int):
    """The GPU's selection is bit-exactly the oracle's top-k rule applied to the GPU's own
    fp32 scores: near ties are then resolved exactly as the rule says (ties to the lower
    block id), with nothing left to tolerance."""
    want = oracle.topk(gpu_scores.detach().cpu().double(), q_pos.detach().cpu(), topk)
    got = gpu_sel.detach().cpu()
    bad = (got != want).any(dim=-1)
    assert not bool(bad.any()), f"{int(bad.sum())} (row, group) selections differ from top-k of the GPU's scores"


def assert_out(gpu_out, ref_out, what="out"):
    g = gpu_out.detach().cpu().double()
    r = ref_out.detach().cpu().double()
    d = (g - r).abs()
    assert float(d.max()) <= OUT_MAX, f"{what}: max abs err {float(d.max()):.3e} > {OUT_MAX}"
    assert float(d.mean()) <= OUT_MEAN, f"{what}: mean abs err {float(d.mean()):.3e} > {OUT_MEAN}"


def assert_lse(gpu_lse, ref_lse, what="lse"):
    g = gpu_lse.detach().cpu().double()
    r = ref_lse.detach().cpu().double()
    both_inf = torch.isneginf(g) & torch.isneginf(r)
    d = (g - r).abs()
    d[both_inf] = 0
    assert float(d.max()) <= LSE_ATOL, f"{what}: max abs err {float(d.max()):.3e} > {LSE_ATOL}"


def assert_ent_pos(sel, ent_pos, ent):
    """ent_pos is the inverse of the CSR entry list: the entry at position
    ent_pos[q][g][s] is (q, slot s) for every selected (q, g, s), and every CSR
    position is claimed once."""
    sel, pos = sel.cpu(), ent_pos.cpu()
    n_rows, G, k = sel.shape
    valid = sel >= 0
    p = pos[valid].long()
    assert int(p.numel()) == int(ent.numel())
    assert bool((p >= 0).all()) and bool((p < ent.numel()).all())
    q = torch.arange(n_rows)[:, None, None].expand(n_rows, G, k)[valid]
    s = torch.arange(k)[None, None, :].expand(n_rows, G, k)[valid]
    assert torch.equal(ent[p].long(), (q * k + s).long())
    assert int(torch.unique(p).numel()) == int(p.numel())


def compact_pages(block_table: torch.Tensor, sel: torch.Tensor, q_req: torch.Tensor):
    """Pages a selection touches, and a block table remapped onto a compact pool
    holding only those pages (unselected blocks map to page 0)."""
    bt = block_table.cpu()
    s = sel.cpu()
    req = q_req.cpu().long()
    used = {}
    new_bt = torch.zeros_like(bt)
    for r in range(s.shape[0]):
        for j in s[r].flatten().tolist():
            if j < 0:
                continue
            p = int(bt[req[r], j])
            if p not in used:
                used[p] = len(used)
            new_bt[req[r], j] = used[p]
    pages = torch.tensor(sorted(used, key=used.get), dtype=torch.long)
    return pages, new_bt


def oracle_decode_rows(case, rows):
    """Oracle decode (scores, selection, page table, output) for a subset of requests,
    pulling only the caches it needs from the device."""
    idx = torch.as_tensor(rows, dtype=torch.long)
    q_pos = case.q_pos.cpu()[idx]
    q_req = case.q_req.cpu()[idx]
    bt = case.block_table.cpu()[q_req.long()]
    local = torch.arange(len(idx), dtype=torch.int32)
    # k-index: only the pages of these requests
    need = sorted({int(p) for p in bt.flatten().tolist() if p >= 0})
    remap = {p: i for i, p in enumerate(need)}
    kidx = case.kidx_cache[torch.tensor(need, device=case.kidx_cache.device)].cpu()
    bt_k = bt.clone()
    for a in range(bt.shape[0]):
        for b in range(bt.shape[1]):
            if int(bt[a, b]) >= 0:
                bt_k[a, b] = remap[int(bt[a, b])]
    sc = oracle.block_scores(case.q_idx.cpu()[idx], kidx, bt_k, local, q_pos, case.max_blocks)
    sel = oracle.topk(sc, q_pos, case.dims.topk)
    pt, rl = oracle.page_table(sel, bt, q_pos + 1)
    return dict(scores=sc, sel=sel, pt=pt, row_len=rl)


def oracle_attention_on(case, rows, sel, block_table=None):
    """Oracle attention of query rows `rows` over selection `sel` (rows x G x k)."""
    idx = torch.as_tensor(rows, dtype=torch.long)
    q_req = case.q_req.cpu()[idx]
    bt = (case.block_table if block_table is None else block_table).cpu()[q_req.long()]
    local = torch.arange(len(idx), dtype=torch.int32)
    pages, bt_c = compact_pages(bt, sel, local)
    dev = case.k_cache.device
    kc = case.k_cache[pages.to(dev)].cpu()
    vc = case.v_cache[pages.to(dev)].cpu()
    return oracle.attention(case.q.cpu()[idx], kc, vc, bt_c, local, case.q_pos.cpu()[idx], sel.cpu(),
                            case.dims.sm_scale)


def in_row_chunks(fn, rows, *, threads=None, min_rows=8):
    """Run fn(chunk_of_rows) -> tuple of tensors over row chunks in threads (the C oracle
    releases the GIL) and concatenate the results along dim 0, in row order."""
    rows = list(rows)
    n = threads or min(16, os.cpu_count() or 1)
    if len(rows) < 2 * min_rows or n <= 1:
        return fn(rows)
    step = max(min_rows, (len(rows) + n - 1) // n)
    chunks = [rows[i:i + step] for i in range(0, len(rows), step)]
    with cf.ThreadPoolExecutor(max_workers=n) as ex:
        parts = list(ex.map(fn, chunks))
    if isinstance(parts[0], tuple):
        return tuple(torch.cat([p[i] for p in parts], dim=0) for i in range(len(parts[0])))
    return torch.cat(parts, dim=0)
