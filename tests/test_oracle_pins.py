"""Pins of the fp64 oracle to things other than itself (no GPU needed).

Each check is chosen so that a plausible slip in the oracle -- a dropped causal
mask, a wrong tie-break, a wrong head->group map, a transposed operand, a wrong
log base in the merge, an unstable inversion -- fails at least one of them:

* a hand-worked fixture with closed-form values (tests/golden/worked_example.json);
* brute force through a different route (numpy einsum + reshape + max);
* library routines on special cases (torch SDPA in fp64, Python's sorted());
* closed forms (planted index keys, merge of equal partials);
* invariants fixed by the method (LSE merge == one-pass softmax, block visit
  order, decode row == prefill row, causality, inversion round trip).
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import msa_inputs as mi
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example.json")


def _ev(x):
    if isinstance(x, str):
        return float(eval(x, {"__builtins__": {}}, {"e": math.e, "log": math.log, "inf": math.inf}))
    return float(x)


def _bf16(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16)


@pytest.fixture(scope="module")
def golden():
    with open(GOLDEN) as f:
        g = json.load(f)
    d = g["dims"]
    page, G = d["page"], d["G"]
    bt = torch.tensor(g["block_table"], dtype=torch.int32)
    tok = g["tokens_by_position"]
    n_pages = 3

    def paged(vals):
        width = len(vals[0])
        pool = torch.zeros(n_pages, page, G, width)
        for pos, v in enumerate(vals):
            pool[bt[0, pos // page], pos % page, 0] = torch.tensor(v, dtype=torch.float32)
        return pool.to(torch.bfloat16)

    rows = g["rows"]
    n = len(rows["q_pos"])
    case = dict(
        kidx=paged(tok["k_idx"]), k=paged(tok["k"]), v=paged(tok["v"]), bt=bt,
        q_idx=_bf16([[r] for r in rows["q_idx"]]),
        q=_bf16([rows["q_heads"]] * n),
        q_pos=torch.tensor(rows["q_pos"], dtype=torch.int32),
        q_req=torch.zeros(n, dtype=torch.int32),
        max_blocks=3, topk=d["topk"], sm_scale=d["sm_scale"], page=page,
    )
    return g, case


def test_golden_scores_and_selection(golden):
    g, c = golden
    sc = oracle.block_scores(c["q_idx"], c["kidx"], c["bt"], c["q_req"], c["q_pos"], c["max_blocks"])
    want = torch.tensor([[_ev(v) if v != "-inf" else -math.inf for v in row]
                         for row in g["expected"]["scores"]], dtype=torch.float64)
    assert torch.equal(sc[:, 0, :], want)
    sel = oracle.topk(sc, c["q_pos"], c["topk"], c["page"])
    assert sel[:, 0, :].tolist() == g["expected"]["sel"]


def test_golden_attention_partials_merge(golden):
    g, c = golden
    sel = torch.tensor(g["expected"]["sel"], dtype=torch.int32)[:, None, :]
    out, lse = oracle.attention(c["q"], c["k"], c["v"], c["bt"], c["q_req"], c["q_pos"], sel, c["sm_scale"])
    want_o = torch.tensor([[[_ev(x) for x in h] for h in r] for r in g["expected"]["out"]], dtype=torch.float64)
    want_l = torch.tensor([[_ev(x) for x in r] for r in g["expected"]["lse"]], dtype=torch.float64)
    torch.testing.assert_close(out, want_o, rtol=0, atol=1e-13)
    torch.testing.assert_close(lse, want_l, rtol=0, atol=1e-13)
    op, lp = oracle.block_partials(c["q"], c["k"], c["v"], c["bt"], c["q_req"], c["q_pos"], sel, c["sm_scale"])
    pa = g["expected"]["partials_row_A_head_0"]
    for slot, key in ((0, "slot0_block0"), (1, "slot1_block2")):
        assert abs(float(lp[0, slot, 0]) - _ev(pa[key]["lse"])) < 1e-13
        for d in range(2):
            assert abs(float(op[0, slot, 0, d]) - _ev(pa[key]["o"][d])) < 1e-13
    # row D has an empty slot: lse -inf, zero output
    assert lp[3, 1, 0] == -math.inf and torch.all(op[3, 1] == 0)
    mo, ml = oracle.lse_merge(op, lp)
    torch.testing.assert_close(mo, want_o, rtol=0, atol=1e-13)
    torch.testing.assert_close(ml, want_l, rtol=0, atol=1e-13)


def test_golden_inversion_and_page_table(golden):
    g, c = golden
    sel = torch.tensor(g["expected"]["sel"], dtype=torch.int32)[:, None, :]
    off, ent = oracle.invert(sel, c["q_req"], 1, c["max_blocks"])
    assert off.tolist() == g["expected"]["blk_off"]
    assert ent.tolist() == g["expected"]["blk_ent"]
    dec = g["expected"]["decode"]
    idx = [g["rows"]["names"].index(n) for n in dec["rows_as_requests"]]
    dsel = sel[idx]
    bt = c["bt"].expand(len(idx), -1).contiguous()
    pt, rl = oracle.page_table(dsel, bt, torch.tensor(dec["seq_lens"], dtype=torch.int32), c["page"])
    assert pt.tolist() == dec["page_table"]
    assert rl.tolist() == dec["row_len"]
    # attention through the page table equals attention over the selected tokens
    q = c["q"][idx]
    po, pl = oracle.paged_attention(q, c["k"], c["v"], pt, rl, c["sm_scale"])
    want_o = torch.tensor([[[_ev(x) for x in h] for h in g["expected"]["out"][i]] for i in idx], dtype=torch.float64)
    torch.testing.assert_close(po, want_o, rtol=0, atol=1e-13)


# ---------------------------------------------------------------- small random paged caches

def _small_cache(seed, lens, page, G, Hq, D, Di, extra_pages=3):
    gen = torch.Generator().manual_seed(seed)
    nb = [(L + page - 1) // page for L in lens]
    n_pages = sum(nb) + extra_pages
    perm = torch.randperm(n_pages, generator=gen)
    mb = max(nb)
    bt = torch.full((len(lens), mb), -1, dtype=torch.int32)
    cur = 0
    for b, n in enumerate(nb):
        bt[b, :n] = perm[cur:cur + n].to(torch.int32)
        cur += n
    rnd = lambda *s: torch.randn(*s, generator=gen).to(torch.bfloat16)
    return dict(bt=bt, mb=mb, n_pages=n_pages,
                kidx=rnd(n_pages, page, G, Di), k=rnd(n_pages, page, G, D), v=rnd(n_pages, page, G, D),
                gen=gen, rnd=rnd)


def _brute_scores(q_idx, kidx, bt, q_req, q_pos, mb):
    """All token dots via einsum over the gathered logical sequence, then mask + block max."""
    n_rows, G, Di = q_idx.shape
    page = kidx.shape[1]
    out = np.full((n_rows, G, mb), -np.inf)
    for r in range(n_rows):
        pages = bt[int(q_req[r])]
        nb = int(q_pos[r]) // page + 1
        seq = kidx[pages[:nb].long()].double().reshape(nb * page, G, Di).numpy()
        dots = np.einsum("tgd,gd->gt", seq, q_idx[r].double().numpy())
        dots[:, int(q_pos[r]) + 1:] = -np.inf
        out[r, :, :nb] = dots.reshape(G, nb, page).max(axis=2)
    return torch.from_numpy(out)


@pytest.mark.parametrize("page", [1, 4, 16, 128])
def test_scores_match_brute_force(page):
    lens = [3 * page + 1, page, 5 * page - 1, 2]
    G, Di = 3, 8
    c = _small_cache(7 + page, lens, page, G, 6, 4, Di)
    rows_req, rows_pos = [], []
    for b, L in enumerate(lens):
        for p in sorted({0, L // 2, L - 1}):
            rows_req.append(b)
            rows_pos.append(p)
    q_req = torch.tensor(rows_req, dtype=torch.int32)
    q_pos = torch.tensor(rows_pos, dtype=torch.int32)
    q_idx = c["rnd"](len(rows_req), G, Di)
    got = oracle.block_scores(q_idx, c["kidx"], c["bt"], q_req, q_pos, c["mb"])
    want = _brute_scores(q_idx, c["kidx"], c["bt"], q_req, q_pos, c["mb"])
    torch.testing.assert_close(got, want, rtol=1e-14, atol=1e-14)


def test_scores_planted_closed_form():
    """Index keys planted as integer multiples of the query index: score = max_t c_t * |q|^2."""
    page, G, Di = 128, 2, 32
    q_idx = torch.zeros(1, G, Di)
    q_idx[0, 0, :4] = torch.tensor([1.0, -2.0, 0.5, 3.0])   # |q|^2 = 14.25
    q_idx[0, 1, 5] = 2.0                                    # |q|^2 = 4
    kidx = torch.zeros(2, page, G, Di)
    coef = torch.linspace(-3, 4, page).round()               # integers -3..4
    for t in range(page):
        kidx[1, t, 0] = coef[t] * q_idx[0, 0]
        kidx[1, t, 1] = -coef[t] * q_idx[0, 1]
    bt = torch.tensor([[1]], dtype=torch.int32)
    p = 100                                                  # tokens 0..100 visible
    sc = oracle.block_scores(q_idx.to(torch.bfloat16), kidx.to(torch.bfloat16), bt,
                             torch.tensor([0], dtype=torch.int32), torch.tensor([p], dtype=torch.int32), 1)
    assert float(sc[0, 0, 0]) == float(coef[:p + 1].max()) * 14.25
    assert float(sc[0, 1, 0]) == float((-coef[:p + 1]).max()) * 4.0


def test_topk_matches_sorted_with_ties():
    gen = torch.Generator().manual_seed(3)
    n_rows, G, mb, k = 40, 3, 37, 6
    vals = torch.tensor([-1.5, -0.0, 0.0, 0.25, 2.0, 2.0, 7.0], dtype=torch.float64)
    scores = vals[torch.randint(0, len(vals), (n_rows, G, mb), generator=gen)]
    q_pos = torch.randint(0, mb * 128, (n_rows,), generator=gen, dtype=torch.int32)
    q_pos[:4] = torch.tensor([0, 127, 128, 5 * 128 + 3])
    sel = oracle.topk(scores, q_pos, k)
    for r in range(n_rows):
        own = int(q_pos[r]) // 128
        k_eff = min(k, own + 1)
        for g in range(G):
            s = scores[r, g]
            others = sorted(range(own), key=lambda j: (-float(s[j]), j))[:k_eff - 1]
            want = sorted(others + [own]) + [-1] * (k - k_eff)
            assert sel[r, g].tolist() == want, (r, g)


def _sdpa_reference(q, k_seq, v_seq, allowed, sm_scale):
    """torch SDPA in fp64 per head; q [Hq][D], k_seq/v_seq [T][Hq][D], allowed [Hq][T]."""
    qq = q.double()[:, None, :]                            # [Hq, 1, D]
    kk = k_seq.double().permute(1, 0, 2)                   # [Hq, T, D]
    vv = v_seq.double().permute(1, 0, 2)
    o = F.scaled_dot_product_attention(qq[None], kk[None], vv[None], attn_mask=allowed[None, :, None, :],
                                       scale=sm_scale)[0, :, 0, :]
    logits = (qq @ kk.transpose(1, 2))[:, 0, :] * sm_scale
    logits = logits.masked_fill(~allowed, -math.inf)
    return o, torch.logsumexp(logits, dim=-1)


def _gather_seq(cache, bt_row, n_tok, page):
    nb = (n_tok + page - 1) // page
    return cache[bt_row[:nb].long()].reshape(nb * page, cache.shape[2], cache.shape[3])[:n_tok]


@pytest.mark.parametrize("dense", [True, False])
def test_attention_matches_sdpa(dense):
    """k >= n_cand reduces MSA to dense causal GQA attention; with a smaller k the
    result equals SDPA under the mask 'token's block is selected for the head's group'."""
    pre, _ = mi.tiny_case(seed=11, L=700, n_decode=1, pool_pages=12, Hq=8, G=2, D=64, Di=32)
    rows = torch.tensor([0, 1, 127, 128, 300, 511, 512, 699])
    q, q_pos, q_req = pre.q[rows], pre.q_pos[rows], pre.q_req[rows]
    n_blocks = pre.max_blocks
    if dense:
        k = n_blocks + 2
        sel = torch.full((len(rows), 2, k), -1, dtype=torch.int32)
        for i, p in enumerate(q_pos.tolist()):
            sel[i, :, :p // 128 + 1] = torch.arange(p // 128 + 1, dtype=torch.int32)
    else:
        sc = oracle.block_scores(pre.q_idx[rows], pre.kidx_cache, pre.block_table, q_req, q_pos, n_blocks)
        sel = oracle.topk(sc, q_pos, 2)
    out, lse = oracle.attention(q, pre.k_cache, pre.v_cache, pre.block_table, q_req, q_pos, sel,
                                pre.dims.sm_scale)
    Hq, G = 8, 2
    for i, p in enumerate(q_pos.tolist()):
        T = p + 1
        kseq = _gather_seq(pre.k_cache, pre.block_table[0], T, 128).repeat_interleave(Hq // G, dim=1)
        vseq = _gather_seq(pre.v_cache, pre.block_table[0], T, 128).repeat_interleave(Hq // G, dim=1)
        blk = torch.arange(T) // 128
        allowed = torch.zeros(Hq, T, dtype=torch.bool)
        for h in range(Hq):
            chosen = [j for j in sel[i, h // (Hq // G)].tolist() if j >= 0]
            allowed[h] = torch.isin(blk, torch.tensor(chosen))
        o_ref, l_ref = _sdpa_reference(q[i], kseq, vseq, allowed, pre.dims.sm_scale)
        torch.testing.assert_close(out[i], o_ref, rtol=0, atol=1e-12)
        torch.testing.assert_close(lse[i], l_ref, rtol=0, atol=1e-12)


def test_merge_equals_one_pass_and_order_invariant():
    pre, _ = mi.tiny_case(seed=5, L=1000, n_decode=1, pool_pages=12)
    rows = torch.arange(0, 1000, 37)
    q_pos, q_req = pre.q_pos[rows], pre.q_req[rows]
    sc = oracle.block_scores(pre.q_idx[rows], pre.kidx_cache, pre.block_table, q_req, q_pos, pre.max_blocks)
    sel = oracle.topk(sc, q_pos, 4)
    args = (pre.q[rows], pre.k_cache, pre.v_cache, pre.block_table, q_req, q_pos)
    out, lse = oracle.attention(*args, sel, pre.dims.sm_scale)
    op, lp = oracle.block_partials(*args, sel, pre.dims.sm_scale)
    mo, ml = oracle.lse_merge(op, lp)
    torch.testing.assert_close(mo, out, rtol=0, atol=1e-12)
    torch.testing.assert_close(ml, lse, rtol=0, atol=1e-12)
    # visit blocks in a different order: reversed slots give the same result
    mo2, ml2 = oracle.lse_merge(op.flip(1), lp.flip(1))
    torch.testing.assert_close(mo2, out, rtol=0, atol=1e-12)
    torch.testing.assert_close(ml2, lse, rtol=0, atol=1e-12)


def test_merge_closed_forms():
    o = torch.randn(1, 2, 1, 5, dtype=torch.float64)
    o[0, 1] = o[0, 0]
    lse = torch.tensor([[[0.75], [0.75]]], dtype=torch.float64)
    mo, ml = oracle.lse_merge(o, lse)
    assert abs(float(ml[0, 0]) - (0.75 + math.log(2.0))) < 1e-14
    torch.testing.assert_close(mo[0, 0], o[0, 0, 0], rtol=0, atol=1e-14)
    # weights exp(lse_s - lse): lse 0 and log 3 -> 1/4, 3/4
    o2 = torch.zeros(1, 3, 1, 2, dtype=torch.float64)
    o2[0, 0, 0] = torch.tensor([4.0, 0.0])
    o2[0, 1, 0] = torch.tensor([0.0, 8.0])
    lse2 = torch.tensor([[[0.0], [math.log(3.0)], [-math.inf]]], dtype=torch.float64)
    mo, ml = oracle.lse_merge(o2, lse2)
    torch.testing.assert_close(mo[0, 0], torch.tensor([1.0, 6.0], dtype=torch.float64), rtol=0, atol=1e-14)
    assert abs(float(ml[0, 0]) - math.log(4.0)) < 1e-14


def test_invert_round_trip_and_order():
    gen = torch.Generator().manual_seed(9)
    n_rows, G, k, n_req, mb = 300, 3, 5, 2, 20
    q_req = torch.randint(0, n_req, (n_rows,), generator=gen, dtype=torch.int32)
    sel = torch.full((n_rows, G, k), -1, dtype=torch.int32)
    for q in range(n_rows):
        for g in range(G):
            m = int(torch.randint(1, k + 1, (1,), generator=gen))
            sel[q, g, :m] = torch.randperm(mb, generator=gen)[:m].sort().values.to(torch.int32)
    off, ent = oracle.invert(sel, q_req, n_req, mb)
    assert int(off[-1]) == int((sel >= 0).sum()) and torch.all(off[1:] >= off[:-1])
    back = torch.full_like(sel, -1)
    for key in range(G * n_req * mb):
        g, rest = divmod(key, n_req * mb)
        req, j = divmod(rest, mb)
        qs = []
        for e in ent[off[key]:off[key + 1]].tolist():
            q, s = divmod(e, k)
            assert int(q_req[q]) == req
            back[q, g, s] = j
            qs.append(q)
        assert qs == sorted(qs) and len(set(qs)) == len(qs)
    assert torch.equal(back, sel)


def test_page_table_closed_form_and_paged_equals_selected():
    dec = mi.decode_case([300, 129, 128, 1000, 1], Hq=8, G=2, D=64, Di=32, topk=3, pool_pages=20,
                         needles_per_group=1, seed=21)
    r = oracle.decode(dec)
    pt, rl, sel = r["pt"], r["row_len"], r["sel"]
    for b, L in enumerate(dec.seq_lens.tolist()):
        own = (L - 1) // 128
        k_eff = min(3, own + 1)
        for g in range(2):
            row = b * 2 + g
            assert int(rl[row]) == (k_eff - 1) * 128 + (L - own * 128)
            for s in range(3):
                j = int(sel[b, g, s])
                assert int(pt[row, s]) == (int(dec.block_table[b, j]) if j >= 0 else -1)
    out, lse = oracle.attention(dec.q, dec.k_cache, dec.v_cache, dec.block_table, dec.q_req, dec.q_pos, sel,
                                dec.dims.sm_scale)
    torch.testing.assert_close(r["out"], out, rtol=0, atol=1e-12)
    torch.testing.assert_close(r["lse"], lse, rtol=0, atol=1e-12)


def test_decode_row_equals_prefill_row():
    pre, dec = mi.tiny_case(seed=1000)
    r = oracle.decode(dec)
    # the same rows treated as prefill rows (scores/top-k/attention at their positions)
    sc = oracle.block_scores(dec.q_idx, dec.kidx_cache, dec.block_table, dec.q_req, dec.q_pos, dec.max_blocks)
    sel = oracle.topk(sc, dec.q_pos, dec.dims.topk)
    assert torch.equal(sel, r["sel"])
    out, lse = oracle.attention(dec.q, dec.k_cache, dec.v_cache, dec.block_table, dec.q_req, dec.q_pos, sel,
                                dec.dims.sm_scale)
    torch.testing.assert_close(r["out"], out, rtol=0, atol=1e-12)
    torch.testing.assert_close(r["lse"], lse, rtol=0, atol=1e-12)


def test_causal_tokens_beyond_position_are_ignored():
    dec = mi.decode_case([200, 390], Hq=4, G=2, D=64, Di=32, topk=2, pool_pages=8, needles_per_group=1, seed=4)
    base = oracle.decode(dec)
    # overwrite every token slot past each request's length (inside its last page) with large values
    for b, L in enumerate(dec.seq_lens.tolist()):
        pg = int(dec.block_table[b, (L - 1) // 128])
        t0 = L % 128
        if t0:
            dec.kidx_cache[pg, t0:] = 50.0
            dec.k_cache[pg, t0:] = 50.0
            dec.v_cache[pg, t0:] = -50.0
    again = oracle.decode(dec)
    for key in ("scores", "sel", "out", "lse"):
        assert torch.equal(base[key], again[key]), key
