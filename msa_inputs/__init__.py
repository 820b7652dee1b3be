"""Seeded synthetic workloads for the MiniMax Sparse Attention (MSA) hot path.

This module is shared by the CPU oracle tests, the CUDA parity tests and the
benchmark.  It holds no arithmetic of the method itself: only random draws,
page placement in a shared pool, and the planted "needle" structure that makes
block selection non-trivial.  Everything is a pure function of the seed.

Layouts (one physical pool, pages of 128 tokens, token stride = groups * dim,
as in the strided paged-KV view of "将 MSA 与分页注意力集成" on the Together AI
page "Together AI 解析如何高效服务 MiniMax M3：1M token 上下文与多模态推理优化"):

    k_cache, v_cache : bf16 [n_pages][page][G][D]
    kidx_cache       : bf16 [n_pages][page][G][Di]   (same page ids as K/V)
    block_table      : int32 [n_req][max_blocks]     logical block -> page, -1 = none
    seq_lens         : int32 [n_req]                 tokens in the cache, incl. new ones
    q                : bf16 [rows][Hq][D]
    q_idx            : bf16 [rows][G][Di]
    q_req, q_pos     : int32 [rows]                  request and absolute position

Values are drawn in fp32 from N(0, 1) and rounded to bf16 (round-to-nearest-even,
torch's conversion).  A needle adds 3 * u to the fp32 index keys of every token of
one (block, group) before rounding, where u is a unit vector along the query-side
index direction of that group.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import torch

PAGE = 128

__all__ = [
    "PAGE", "Dims", "Case", "decode_case", "prefill_case", "tiny_case",
    "ragged_lengths", "named_case", "CONFIG_NAMES", "mixed_case",
]


@dataclass(frozen=True)
class Dims:
    Hq: int
    G: int
    D: int
    Di: int
    topk: int
    page: int = PAGE

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


@dataclass
class Case:
    """One synthetic workload: a paged cache plus query rows."""
    dims: Dims
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    kidx_cache: torch.Tensor
    block_table: torch.Tensor
    seq_lens: torch.Tensor
    q: torch.Tensor
    q_idx: torch.Tensor
    q_req: torch.Tensor
    q_pos: torch.Tensor
    max_blocks: int
    needles: List[Tuple[int, int, int]] = field(default_factory=list)  # (req, group, block)
    name: str = ""

    @property
    def n_pages(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def n_rows(self) -> int:
        return int(self.q.shape[0])

    @property
    def n_req(self) -> int:
        return int(self.block_table.shape[0])

    def to(self, device) -> "Case":
        out = Case(**{k: (v.to(device) if isinstance(v, torch.Tensor) else v)
                      for k, v in self.__dict__.items()})
        return out


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn_f32(shape, gen, device) -> torch.Tensor:
    return torch.randn(tuple(shape), generator=gen, device=device, dtype=torch.float32)


def _pool_bf16(n_pages: int, page: int, G: int, width: int, gen, device,
               shifts: Optional[dict] = None) -> torch.Tensor:
    """Draw a paged pool chunk by chunk; `shifts` maps page -> [(group, fp32 vector)]
    added to every token of that (page, group) before the bf16 rounding."""
    out = torch.empty((n_pages, page, G, width), dtype=torch.bfloat16, device=device)
    per_page = page * G * width
    step = max(1, (1 << 25) // per_page)
    for p0 in range(0, n_pages, step):
        n = min(step, n_pages - p0)
        x = _randn_f32((n, page, G, width), gen, device)
        if shifts:
            for p in range(p0, p0 + n):
                for (grp, vec) in shifts.get(p, ()):
                    x[p - p0, :, grp, :] += vec.to(device)
        out[p0:p0 + n] = x.to(torch.bfloat16)
    return out


def _place_pages(lens: Sequence[int], pool_pages: int, page: int, gen_cpu) -> Tuple[torch.Tensor, int]:
    n_blk = [(L + page - 1) // page for L in lens]
    total = sum(n_blk)
    if total > pool_pages:
        raise ValueError(f"pool of {pool_pages} pages cannot hold {total} blocks")
    max_blocks = max(n_blk)
    perm = torch.randperm(pool_pages, generator=gen_cpu)
    bt = torch.full((len(lens), max_blocks), -1, dtype=torch.int32)
    cur = 0
    for b, nb in enumerate(n_blk):
        bt[b, :nb] = perm[cur:cur + nb].to(torch.int32)
        cur += nb
    return bt, max_blocks


def _unit(v: torch.Tensor) -> torch.Tensor:
    n = torch.linalg.vector_norm(v)
    return v / n if float(n) > 0 else v


def _pick_needles(n_cand_excl_own: int, count: int, gen_cpu,
                  ranges: Optional[Sequence[Tuple[int, int, int]]] = None) -> List[int]:
    """Distinct block ids in [0, n_cand_excl_own).  `ranges` = [(lo, hi, count)] overrides
    the uniform draw (used for the 1M-token placement at the start, middle and end)."""
    if n_cand_excl_own <= 0:
        return []
    if ranges is None:
        count = min(count, n_cand_excl_own)
        return sorted(torch.randperm(n_cand_excl_own, generator=gen_cpu)[:count].tolist())
    picked: List[int] = []
    for lo, hi, c in ranges:
        hi = min(hi, n_cand_excl_own)
        lo = max(0, min(lo, hi))
        if hi <= lo:
            continue
        cand = torch.randperm(hi - lo, generator=gen_cpu)[:min(c, hi - lo)] + lo
        picked.extend(int(x) for x in cand.tolist())
    return sorted(set(picked))


def decode_case(lens: Sequence[int], Hq: int, G: int, D: int, Di: int, topk: int,
                pool_pages: int, needles_per_group: int, seed: int, device="cpu",
                needle_ranges_frac: Optional[Sequence[Tuple[float, float, int]]] = None,
                name: str = "") -> Case:
    """Decode batch: request b holds lens[b] cached tokens (incl. the new one); one
    query row per request at position lens[b] - 1.  Needles sit in blocks other than
    the query's own block, shifted along u = q_idx[b, g] / |q_idx[b, g]|."""
    page = PAGE
    dims = Dims(Hq, G, D, Di, topk, page)
    gc = _gen(seed, "cpu")
    bt, max_blocks = _place_pages(lens, pool_pages, page, gc)
    B = len(lens)
    gd = _gen(seed + 7919, device)
    q = _randn_f32((B, Hq, D), gd, device).to(torch.bfloat16)
    q_idx = _randn_f32((B, G, Di), gd, device).to(torch.bfloat16)
    shifts: dict = {}
    needles: List[Tuple[int, int, int]] = []
    qi_cpu = q_idx.float().cpu()
    for b, L in enumerate(lens):
        own = (L - 1) // page
        for g in range(G):
            if needle_ranges_frac is not None:
                nb = (L + page - 1) // page
                ranges = [(int(math.floor(lo * nb)), int(math.ceil(hi * nb)), c)
                          for (lo, hi, c) in needle_ranges_frac]
                blocks = _pick_needles(own, 0, gc, ranges)
            else:
                blocks = _pick_needles(own, needles_per_group, gc)
            u = _unit(qi_cpu[b, g])
            for j in blocks:
                p = int(bt[b, j])
                shifts.setdefault(p, []).append((g, 3.0 * u))
                needles.append((b, g, j))
    kidx = _pool_bf16(pool_pages, page, G, Di, gd, device, shifts)
    k_cache = _pool_bf16(pool_pages, page, G, D, gd, device)
    v_cache = _pool_bf16(pool_pages, page, G, D, gd, device)
    seq = torch.tensor(list(lens), dtype=torch.int32)
    return Case(dims, k_cache, v_cache, kidx, bt.to(device), seq.to(device), q, q_idx,
                torch.arange(B, dtype=torch.int32, device=device),
                (seq - 1).to(torch.int32).to(device), max_blocks, needles, name)


def prefill_case(prefix: int, chunk: int, Hq: int, G: int, D: int, Di: int, topk: int,
                 pool_pages: int, seed: int, device="cpu", span: int = 256,
                 span_sigma: float = 0.5, name: str = "") -> Case:
    """Chunked prefill of one request: `chunk` new query rows at positions
    prefix .. prefix+chunk-1 over a cache of prefix+chunk tokens (the chunk's own
    K/V/index keys already appended).  Query-side index vectors of rows in the same
    `span`-token window are drawn around a shared centre c ~ N(0, 1) per (window,
    group): q_idx = c + span_sigma * N(0, 1), so many rows pick the same blocks."""
    page = PAGE
    dims = Dims(Hq, G, D, Di, topk, page)
    L = prefix + chunk
    gc = _gen(seed, "cpu")
    bt, max_blocks = _place_pages([L], pool_pages, page, gc)
    gd = _gen(seed + 7919, device)
    q = _randn_f32((chunk, Hq, D), gd, device).to(torch.bfloat16)
    n_span = (chunk + span - 1) // span
    centres = _randn_f32((n_span, G, Di), gd, device)
    noise = _randn_f32((chunk, G, Di), gd, device)
    span_of_row = torch.arange(chunk, device=device) // span
    q_idx = (centres[span_of_row] + span_sigma * noise).to(torch.bfloat16)
    kidx = _pool_bf16(pool_pages, page, G, Di, gd, device)
    k_cache = _pool_bf16(pool_pages, page, G, D, gd, device)
    v_cache = _pool_bf16(pool_pages, page, G, D, gd, device)
    pos = torch.arange(prefix, L, dtype=torch.int32, device=device)
    return Case(dims, k_cache, v_cache, kidx, bt.to(device),
                torch.tensor([L], dtype=torch.int32, device=device), q, q_idx,
                torch.zeros(chunk, dtype=torch.int32, device=device), pos, max_blocks, [], name)


def multi_token_decode_case(lens: Sequence[int], T: int, Hq: int, G: int, D: int, Di: int, topk: int,
                            pool_pages: int, seed: int, device="cpu", name: str = "") -> Case:
    """Multi-token (speculative) decode: request b holds lens[b] cached tokens, the
    last T of them new; its T query rows sit at positions lens[b]-T .. lens[b]-1 and
    are consecutive rows, requests in order (rows grouped by request)."""
    assert T >= 1 and all(L >= T for L in lens)
    page = PAGE
    dims = Dims(Hq, G, D, Di, topk, page)
    gc = _gen(seed, "cpu")
    bt, max_blocks = _place_pages(list(lens), pool_pages, page, gc)
    gd = _gen(seed + 7919, device)
    n_rows = T * len(lens)
    q = _randn_f32((n_rows, Hq, D), gd, device).to(torch.bfloat16)
    q_idx = _randn_f32((n_rows, G, Di), gd, device).to(torch.bfloat16)
    kidx = _pool_bf16(pool_pages, page, G, Di, gd, device)
    k_cache = _pool_bf16(pool_pages, page, G, D, gd, device)
    v_cache = _pool_bf16(pool_pages, page, G, D, gd, device)
    q_req = torch.arange(len(lens), dtype=torch.int32, device=device).repeat_interleave(T)
    q_pos = torch.cat([torch.arange(L - T, L, dtype=torch.int32, device=device) for L in lens])
    return Case(dims, k_cache, v_cache, kidx, bt.to(device),
                torch.tensor(list(lens), dtype=torch.int32, device=device), q, q_idx, q_req, q_pos, max_blocks, [],
                name)


def ragged_prefill_case(prefixes: Sequence[int], chunks: Sequence[int], Hq: int, G: int, D: int,
                        Di: int, topk: int, pool_pages: int, seed: int, device="cpu", span: int = 256,
                        span_sigma: float = 0.5, name: str = "") -> Case:
    """One prefill chunk holding several requests, as a chunked-prefill engine
    batches them: request r contributes chunks[r] new rows at positions
    prefixes[r] .. prefixes[r]+chunks[r]-1 over a cache of prefixes[r]+chunks[r]
    tokens.  The rows are concatenated in request order, so 128-row tiles may
    straddle requests.  Per request, the query-side index vectors follow the same
    span structure as prefill_case."""
    assert len(prefixes) == len(chunks) and len(chunks) > 0
    page = PAGE
    dims = Dims(Hq, G, D, Di, topk, page)
    lens = [p + c for p, c in zip(prefixes, chunks)]
    gc = _gen(seed, "cpu")
    bt, max_blocks = _place_pages(lens, pool_pages, page, gc)
    gd = _gen(seed + 7919, device)
    n_rows = sum(chunks)
    q = _randn_f32((n_rows, Hq, D), gd, device).to(torch.bfloat16)
    parts_idx, parts_req, parts_pos = [], [], []
    for r, (p, c) in enumerate(zip(prefixes, chunks)):
        n_span = (c + span - 1) // span
        centres = _randn_f32((n_span, G, Di), gd, device)
        noise = _randn_f32((c, G, Di), gd, device)
        span_of_row = torch.arange(c, device=device) // span
        parts_idx.append(centres[span_of_row] + span_sigma * noise)
        parts_req.append(torch.full((c,), r, dtype=torch.int32, device=device))
        parts_pos.append(torch.arange(p, p + c, dtype=torch.int32, device=device))
    q_idx = torch.cat(parts_idx).to(torch.bfloat16)
    kidx = _pool_bf16(pool_pages, page, G, Di, gd, device)
    k_cache = _pool_bf16(pool_pages, page, G, D, gd, device)
    v_cache = _pool_bf16(pool_pages, page, G, D, gd, device)
    return Case(dims, k_cache, v_cache, kidx, bt.to(device),
                torch.tensor(lens, dtype=torch.int32, device=device), q, q_idx,
                torch.cat(parts_req), torch.cat(parts_pos), max_blocks, [], name)


def mixed_case(decode_lens: Sequence[int], prefixes: Sequence[int], chunks: Sequence[int], Hq: int, G: int,
               D: int, Di: int, topk: int, seed: int, device="cpu", pool_pages: Optional[int] = None,
               needles_per_group: int = 4, span: int = 256, span_sigma: float = 0.5,
               name: str = "") -> Tuple[Case, Case]:
    """One step of a chunked-prefill engine: a batch that mixes decode requests (one new
    token each) with a prefill chunk of one or more requests, over ONE shared page pool.

    Requests 0 .. Bd-1 are the decode requests (request b holds decode_lens[b] tokens, its
    query at position decode_lens[b] - 1, with needle blocks as in decode_case); requests
    Bd .. Bd+Bp-1 are the prefill requests (request Bd + r appends chunks[r] rows at
    positions prefixes[r] .. prefixes[r]+chunks[r]-1, with the span structure of
    prefill_case for its query-side index vectors).  Returns (decode Case, prefill Case):
    they share the cache tensors; the decode case's block table is rows 0 .. Bd-1 of the
    joint table and the prefill case's rows Bd .., both views of one tensor, so q_req of a
    prefill row counts from 0 within the prefill case."""
    page = PAGE
    dims = Dims(Hq, G, D, Di, topk, page)
    Bd, Bp = len(decode_lens), len(chunks)
    assert Bd > 0 and Bp > 0 and len(prefixes) == Bp
    pre_lens = [p + c for p, c in zip(prefixes, chunks)]
    lens = list(decode_lens) + pre_lens
    if pool_pages is None:
        pool_pages = int(math.ceil(1.1 * sum((L + page - 1) // page for L in lens))) + 8
    gc = _gen(seed, "cpu")
    bt, max_blocks = _place_pages(lens, pool_pages, page, gc)
    gd = _gen(seed + 7919, device)
    # decode rows
    q_d = _randn_f32((Bd, Hq, D), gd, device).to(torch.bfloat16)
    qi_d = _randn_f32((Bd, G, Di), gd, device).to(torch.bfloat16)
    shifts: dict = {}
    needles: List[Tuple[int, int, int]] = []
    qi_cpu = qi_d.float().cpu()
    for b, L in enumerate(decode_lens):
        own = (L - 1) // page
        for g in range(G):
            u = _unit(qi_cpu[b, g])
            for j in _pick_needles(own, needles_per_group, gc):
                shifts.setdefault(int(bt[b, j]), []).append((g, 3.0 * u))
                needles.append((b, g, j))
    # prefill rows
    n_rows = sum(chunks)
    q_p = _randn_f32((n_rows, Hq, D), gd, device).to(torch.bfloat16)
    parts_idx, parts_req, parts_pos = [], [], []
    for r, (p0, c) in enumerate(zip(prefixes, chunks)):
        n_span = (c + span - 1) // span
        centres = _randn_f32((n_span, G, Di), gd, device)
        noise = _randn_f32((c, G, Di), gd, device)
        span_of_row = torch.arange(c, device=device) // span
        parts_idx.append(centres[span_of_row] + span_sigma * noise)
        parts_req.append(torch.full((c,), r, dtype=torch.int32, device=device))
        parts_pos.append(torch.arange(p0, p0 + c, dtype=torch.int32, device=device))
    kidx = _pool_bf16(pool_pages, page, G, Di, gd, device, shifts)
    k_cache = _pool_bf16(pool_pages, page, G, D, gd, device)
    v_cache = _pool_bf16(pool_pages, page, G, D, gd, device)
    btd = bt.to(device)
    seq = torch.tensor(lens, dtype=torch.int32, device=device)
    dec = Case(dims, k_cache, v_cache, kidx, btd[:Bd], seq[:Bd], q_d, qi_d,
               torch.arange(Bd, dtype=torch.int32, device=device), (seq[:Bd] - 1).to(torch.int32), max_blocks,
               needles, name + "-decode")
    pre = Case(dims, k_cache, v_cache, kidx, btd[Bd:], seq[Bd:], q_p, torch.cat(parts_idx).to(torch.bfloat16),
               torch.cat(parts_req), torch.cat(parts_pos), max_blocks, [], name + "-prefill")
    return dec, pre


def tiny_case(seed: int = 1000, device="cpu", L: int = 2048, n_decode: int = 16,
              Hq: int = 8, G: int = 2, D: int = 64, Di: int = 32, topk: int = 4,
              pool_pages: int = 32, needles_per_group: int = 2) -> Tuple[Case, Case]:
    """Small prefill + decode pair over ONE cache.

    The cache holds L + n_decode tokens.  The prefill case has rows at positions
    0 .. L-1 (causal).  The decode case has n_decode rows, one per decode step, at
    positions L .. L+n_decode-1; all rows share request 0's pages, and row i sees
    seq_len L+i+1 (equivalent to appending one token per step, since a row never
    attends past its own position).  Needles: `needles_per_group` blocks per group,
    shifted along u_g = unit(mean over the prefill rows of q_idx[:, g])."""
    page = PAGE
    dims = Dims(Hq, G, D, Di, topk, page)
    total = L + n_decode
    gc = _gen(seed, "cpu")
    bt, max_blocks = _place_pages([total], pool_pages, page, gc)
    gd = _gen(seed + 7919, device)
    q = _randn_f32((total, Hq, D), gd, device).to(torch.bfloat16)
    q_idx = _randn_f32((total, G, Di), gd, device).to(torch.bfloat16)
    qi_cpu = q_idx[:L].float().cpu()
    shifts: dict = {}
    needles: List[Tuple[int, int, int]] = []
    n_full = L // page
    for g in range(G):
        u = _unit(qi_cpu[:, g, :].mean(dim=0))
        for j in _pick_needles(max(n_full - 1, 0), needles_per_group, gc):
            shifts.setdefault(int(bt[0, j]), []).append((g, 3.0 * u))
            needles.append((0, g, j))
    kidx = _pool_bf16(pool_pages, page, G, Di, gd, device, shifts)
    k_cache = _pool_bf16(pool_pages, page, G, D, gd, device)
    v_cache = _pool_bf16(pool_pages, page, G, D, gd, device)
    btd = bt.to(device)
    pre = Case(dims, k_cache, v_cache, kidx, btd,
               torch.tensor([total], dtype=torch.int32, device=device),
               q[:L].contiguous(), q_idx[:L].contiguous(),
               torch.zeros(L, dtype=torch.int32, device=device),
               torch.arange(L, dtype=torch.int32, device=device), max_blocks, needles, "tiny-prefill")
    dec_bt = btd.expand(n_decode, -1).contiguous()
    lens = torch.arange(L + 1, L + n_decode + 1, dtype=torch.int32, device=device)
    dec = Case(dims, k_cache, v_cache, kidx, dec_bt, lens,
               q[L:].contiguous(), q_idx[L:].contiguous(),
               torch.arange(n_decode, dtype=torch.int32, device=device),
               (lens - 1).to(torch.int32), max_blocks, needles, "tiny-decode")
    return pre, dec


def ragged_lengths(B: int, seed: int, lo: int = 4096, hi: int = 131072) -> List[int]:
    """Per-request context lengths drawn log-uniform in [lo, hi] (seeded)."""
    g = _gen(seed, "cpu")
    u = torch.rand(B, generator=g, dtype=torch.float64)
    return [int(round(math.exp(math.log(lo) + float(x) * (math.log(hi) - math.log(lo))))) for x in u]


CONFIG_NAMES = ("tiny", "decode60k", "prefill68k", "ragged1", "ragged8", "ragged32",
                "ragged64", "decode1m", "mixed")


def named_case(name: str, device="cpu"):
    """The five named workloads (seed 1000 + workload number).  "tiny" returns a
    (prefill, decode) pair; the others return one Case."""
    H = dict(Hq=64, G=8, D=128, Di=64, topk=16)
    if name == "tiny":
        return tiny_case(seed=1000, device=device)
    if name == "decode60k":
        return decode_case([60000] * 8, pool_pages=4096, needles_per_group=4,
                           seed=1001, device=device, name=name, **H)
    if name == "prefill68k":
        return prefill_case(60000, 8192, pool_pages=4096, seed=1002, device=device,
                            name=name, **H)
    if name.startswith("ragged"):
        B = int(name[len("ragged"):])
        lens = ragged_lengths(B, seed=1003 + B)
        pool = int(math.ceil(1.25 * sum((L + PAGE - 1) // PAGE for L in lens)))
        return decode_case(lens, pool_pages=pool, needles_per_group=4, seed=1003,
                           device=device, name=name, **H)
    if name == "mixed":
        # decode60k's batch and prefill68k's chunk in one step over one pool
        return mixed_case([60000] * 8, [60000], [8192], seed=1005, device=device, name=name, **H)
    if name == "decode1m":
        ranges = [(0.0, 0.05, 3), (0.475, 0.525, 3), (0.95, 1.0, 2)]
        return decode_case([1 << 20] * 2, pool_pages=16640, needles_per_group=8,
                           seed=1004, device=device, needle_ranges_frac=ranges,
                           name=name, **H)
    raise KeyError(name)
