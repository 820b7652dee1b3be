"""Prefill path on the GPU against the fp64 oracle: tensor-core index scoring,
top-k, {q,blk}->{blk,q} inversion, KV-block-major attention partials and the
Log-Sum-Exp merge -- through the C ABI, on seeded workloads."""
import pytest
import torch

import msa_inputs as mi
import oracle
from tests import _parity as P

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def msa():
    import block_sparse_attention_06_gb300 as m
    return m


def _run(m, case, fuse_topk=False):
    dims = m.dims_of(case)
    step = m.PrefillStep(dims, case.n_rows, case.n_req, DEV, fuse_topk=fuse_topk)
    step(case.q, case.q_idx, case.k_cache, case.v_cache, case.kidx_cache, case.block_table, case.q_req, case.q_pos)
    m.msa_check(step.err)
    torch.cuda.synchronize()
    return step


def _check_prefill(m, case, rows=None, check_partials=True):
    step = _run(m, case)
    n = case.n_rows
    rows = list(range(n)) if rows is None else rows
    idx = torch.as_tensor(rows)
    q_pos, q_req = case.q_pos.cpu()[idx], case.q_req.cpu()[idx]
    bt = case.block_table.cpu()
    local_bt = bt[q_req.long()]
    kidx = case.kidx_cache.cpu()
    q_idx = case.q_idx.cpu()

    def scores_of(chunk):   # chunk: positions into `rows`
        ci = torch.as_tensor(chunk)
        return oracle.block_scores(q_idx[idx[ci]], kidx, local_bt[ci], torch.arange(len(chunk), dtype=torch.int32),
                                   q_pos[ci], case.max_blocks)

    ref_sc = P.in_row_chunks(scores_of, range(len(rows)))
    P.assert_scores(step.scores.cpu()[idx], ref_sc, q_pos)
    ref_sel = oracle.topk(ref_sc, q_pos, case.dims.topk)
    gap = P.selection_gap(ref_sc, q_pos, case.dims.topk)
    gsel = step.sel.cpu()[idx]
    P.assert_selection_where_unambiguous(gsel, ref_sel, gap)
    # near ties too: a valid top-k of the oracle's scores, and exactly the top-k of the GPU's own scores
    P.assert_selection_valid(gsel, ref_sc, q_pos, case.dims.topk)
    P.assert_topk_of_own_scores(gsel, step.scores.cpu()[idx], q_pos, case.dims.topk)
    # inversion of the GPU's full selection is bit-exact, and ent_pos is its inverse
    off, ent = oracle.invert(step.sel.cpu(), case.q_req.cpu(), case.n_req, case.max_blocks)
    assert torch.equal(step.blk_off.cpu(), off)
    assert torch.equal(step.blk_ent.cpu()[:int(off[-1])], ent)
    P.assert_ent_pos(step.sel.cpu(), step.ent_pos.cpu(), ent)
    # per-block partials (valid slots) and the merged output on the GPU's selection
    if check_partials:
        kc, vc, qc = case.k_cache.cpu(), case.v_cache.cpu(), case.q.cpu()

        def partials_of(chunk):
            ci = torch.as_tensor(chunk)
            return oracle.block_partials(qc[idx[ci]], kc, vc, local_bt[ci], torch.arange(len(chunk), dtype=torch.int32),
                                         q_pos[ci], gsel[ci], case.dims.sm_scale)

        op, lp = P.in_row_chunks(partials_of, range(len(rows)))
        hpg = case.dims.Hq // case.dims.G
        valid = (gsel >= 0).repeat_interleave(hpg, dim=1).transpose(1, 2)   # [rows][topk][Hq]
        o_by_slot, l_by_slot = step.partials_by_slot()
        P.assert_lse(l_by_slot[idx][valid], lp[valid], "lse_part")
        P.assert_out(o_by_slot[idx][valid], op[valid], "o_part")
    o_ref, l_ref = P.in_row_chunks(
        lambda ch: P.oracle_attention_on(case, [rows[i] for i in ch], gsel[torch.as_tensor(ch)]), range(len(rows)))
    P.assert_out(step.out.cpu()[idx], o_ref)
    P.assert_lse(step.lse.cpu()[idx], l_ref)
    return step


def test_tiny_prefill(msa):
    """2048 causal rows, Hq=8, G=2, D=64, Di=32, k=4 (16 blocks, 16 row tiles)."""
    pre, _ = mi.tiny_case(seed=1000, device=DEV)
    _check_prefill(msa, pre)


@pytest.mark.parametrize("prefix,chunk", [(1000, 300), (0, 257), (127, 1)])
def test_small_prefill_ragged(msa, prefix, chunk):
    case = mi.prefill_case(prefix, chunk, Hq=16, G=2, D=128, Di=64, topk=6, pool_pages=40, seed=12, device=DEV)
    _check_prefill(msa, case)


@pytest.mark.parametrize("prefixes,chunks,hq,g,d,di", [
    ([300, 0, 1000], [100, 257, 129], 16, 2, 128, 64),     # 128-row tiles straddle two requests
    ([0, 5000, 64, 130], [1, 300, 63, 200], 8, 2, 64, 32),  # a one-row request, several per tile
    ([2000, 2000], [384, 128], 32, 8, 128, 64),             # tile-aligned requests
])
def test_prefill_ragged_multi_request(msa, prefixes, chunks, hq, g, d, di):
    """One chunk holding several requests back to back (chunked prefill of a batch): every
    step of the prefill path against the oracle on all rows."""
    case = mi.ragged_prefill_case(prefixes, chunks, Hq=hq, G=g, D=d, Di=di, topk=6, pool_pages=120,
                                  seed=21, device=DEV)
    _check_prefill(msa, case)


@pytest.mark.parametrize("hq,g,d,di", [(32, 8, 128, 64), (16, 4, 64, 32), (8, 2, 128, 32)])
def test_prefill_shape_variants(msa, hq, g, d, di):
    case = mi.prefill_case(2100, 400, Hq=hq, G=g, D=d, Di=di, topk=8, pool_pages=40, seed=13, device=DEV)
    _check_prefill(msa, case)


@pytest.mark.parametrize("topk", [1, 32])
def test_prefill_topk_limits(msa, topk):
    """topk = 1 (each row attends its own block only) and topk = 32 (the largest
    supported, past the fused selection's limit of 16): 300 rows from position 3,900,
    so early rows have fewer than 32 candidates and later ones more."""
    case = mi.prefill_case(3900, 300, Hq=16, G=2, D=128, Di=64, topk=topk, pool_pages=60, seed=14, device=DEV)
    _check_prefill(msa, case)
    fused = _run(msa, case, fuse_topk=None)   # the default path PrefillStep picks for this topk
    unfused = _run(msa, case, fuse_topk=False)
    assert fused.fuse_topk == (topk <= 16)
    assert torch.equal(fused.out, unfused.out) and torch.equal(fused.lse, unfused.lse)


def test_prefill_large_score_spread(msa):
    """Peaky attention: keys of tokens 70 and 100 of every page scaled by -30 and 40, so a
    row's scores inside one block spread over hundreds of units and one token takes nearly
    all the weight (exp2 of very negative arguments, masked and unmasked chunks alike).  V is
    scaled by 1/4: the output is then close to a single V row, and a row of N(0,1) values
    rounded to bf16 twice (partial, merged output) can miss by 2^-8 of its magnitude, so the
    smaller V keeps that rounding inside the absolute tolerance the test applies."""
    case = mi.prefill_case(1000, 300, Hq=16, G=2, D=128, Di=64, topk=6, pool_pages=40, seed=12, device=DEV)
    case.k_cache[:, 100] = (case.k_cache[:, 100].float() * 40).to(torch.bfloat16)
    case.k_cache[:, 70] = (case.k_cache[:, 70].float() * -30).to(torch.bfloat16)
    case.v_cache.mul_(0.25)
    step = _check_prefill(msa, case)
    # the spread is there: some row's score on token 100 lies more than 64 (log2 units) above zero
    q = case.q.float().cpu()
    k100 = case.k_cache[:, 100].float().cpu()                    # [pages][G][D]
    hpg = case.dims.Hq // case.dims.G
    s100 = torch.einsum("rgd,pgd->rgp", q.view(q.shape[0], case.dims.G, hpg, -1)[:, :, 0], k100)
    assert float(s100.max()) * case.dims.sm_scale * 1.4427 > 64 + 10


def test_prefill68k_sampled(msa):
    """8192-row chunk on a 60,000-token prefix, full launch; oracle on sampled rows: the
    first and last row of every 128-row tile (the chunk starts at position 60,000, in the
    middle of block 468, so tile edges and block edges differ), the rows around every
    block edge inside the chunk, and a stride-37 sample through the whole chunk (471
    rows) -- scores, selection, per-block partials, merged output and lse on each."""
    case = mi.named_case("prefill68k", device=DEV)
    n = case.n_rows
    first = int(case.q_pos[0])
    rows = {0, n - 1}
    for t in range(0, n, 128):                      # 128-row tile edges
        rows.update((t, min(n - 1, t + 127)))
    for p in range((first // 128 + 1) * 128, first + n, 128):   # block edges: last row of a block, first of the next
        rows.update((p - first - 1, p - first))
    rows.update(range(5, n, 37))                    # stride sample (every row position class alike)
    rows = sorted(rows)
    assert 400 <= len(rows) <= 520
    _check_prefill(msa, case, rows, check_partials=True)


def _fused_cases():
    yield "tiny", lambda: mi.tiny_case(seed=1000, device=DEV)[0]
    yield "ragged", lambda: mi.prefill_case(1000, 300, Hq=16, G=2, D=128, Di=64, topk=6, pool_pages=40, seed=12,
                                            device=DEV)
    yield "one_row", lambda: mi.prefill_case(127, 1, Hq=16, G=2, D=128, Di=64, topk=6, pool_pages=40, seed=12,
                                             device=DEV)
    yield "multi_request", lambda: mi.ragged_prefill_case([0, 5000, 64, 130], [1, 300, 63, 200], Hq=8, G=2, D=64,
                                                          Di=32, topk=6, pool_pages=120, seed=21, device=DEV)
    yield "g8_k16", lambda: mi.prefill_case(2100, 400, Hq=32, G=8, D=128, Di=64, topk=16, pool_pages=40, seed=13,
                                            device=DEV)
    yield "prefill68k", lambda: mi.named_case("prefill68k", device=DEV)
    # rows of 7 and 8 chunk lists (the per-thread k-way merge at its widest) and of 9 (the warp merge)
    yield "chunks7", lambda: mi.prefill_case(110000, 300, Hq=16, G=2, D=64, Di=32, topk=16, pool_pages=900, seed=31,
                                             device=DEV)
    yield "chunks8", lambda: mi.prefill_case(126000, 300, Hq=16, G=2, D=64, Di=32, topk=16, pool_pages=1000,
                                             seed=32, device=DEV)
    yield "chunks9", lambda: mi.prefill_case(140000, 300, Hq=16, G=2, D=64, Di=32, topk=16, pool_pages=1100,
                                             seed=33, device=DEV)


@pytest.mark.parametrize("name,make", list(_fused_cases()), ids=[n for n, _ in _fused_cases()])
def test_fused_select_equals_score_then_topk(msa, name, make):
    """msa_select_invert_prefill (top-k fused into scoring, the inversion's marks into
    the list merge) selects and inverts exactly what msa_index_score + msa_topk_blocks +
    msa_invert_selection do, so the whole prefill step gives identical bits."""
    case = make()
    unfused = _run(msa, case, fuse_topk=False)
    fused = _run(msa, case, fuse_topk=True)
    assert fused.fuse_topk and fused.scores is None
    assert torch.equal(fused.sel, unfused.sel)
    n_ent = int(unfused.blk_off[-1])        # entries past the CSR's end are scratch
    assert torch.equal(fused.blk_off, unfused.blk_off)
    assert torch.equal(fused.blk_ent[:n_ent], unfused.blk_ent[:n_ent])
    assert torch.equal(fused.ent_pos, unfused.ent_pos)
    assert torch.equal(fused.out, unfused.out)
    assert torch.equal(fused.lse, unfused.lse)
    # msa_select_prefill alone (no inversion) selects the same
    d = msa.dims_of(case)
    sel = msa.msa_select_prefill(case.q_idx, case.kidx_cache, case.block_table, case.q_req, case.q_pos, d)
    assert torch.equal(sel, unfused.sel)


def test_topk_bit_exact_on_oracle_scores(msa):
    """The top-k kernel on the oracle's scores, with ties and signed zeros planted."""
    gen = torch.Generator().manual_seed(4)
    n_rows, G, mb, k = 300, 8, 600, 16
    vals = torch.tensor([-3.0, -0.0, 0.0, 0.5, 1.25, 1.25, 7.0], dtype=torch.float64)
    scores = vals[torch.randint(0, len(vals), (n_rows, G, mb), generator=gen)]
    scores += torch.randn(n_rows, G, mb, generator=gen, dtype=torch.float64).round() * 0.5
    q_pos = torch.randint(0, mb * 128, (n_rows,), generator=gen, dtype=torch.int32)
    q_pos[:5] = torch.tensor([0, 127, 128, 16 * 128, 599 * 128 + 5], dtype=torch.int32)
    sc32 = scores.float()
    dims = msa.Dims(64, G, 128, 64, k, mb)
    got = msa.msa_topk_blocks(sc32.to(DEV), q_pos.to(DEV), dims)
    want = oracle.topk(sc32.double(), q_pos, k)
    assert torch.equal(got.cpu(), want)


@pytest.mark.parametrize("mb", [1500, 8192, 16384])
def test_topk_long_candidate_lists(msa, mb):
    gen = torch.Generator().manual_seed(mb)
    n_rows, G, k = 4, 8, 16
    scores = torch.randn(n_rows, G, mb, generator=gen).round(decimals=1)   # many ties
    q_pos = torch.tensor([mb * 128 - 1, 5000, 129, (mb // 2) * 128 + 7], dtype=torch.int32)
    dims = msa.Dims(64, G, 128, 64, k, mb)
    got = msa.msa_topk_blocks(scores.to(DEV), q_pos.to(DEV), dims)
    assert torch.equal(got.cpu(), oracle.topk(scores.double(), q_pos, k))


def test_invert_bit_exact_multi_request(msa):
    gen = torch.Generator().manual_seed(8)
    n_rows, G, k, n_req, mb = 1000, 4, 7, 3, 50
    q_req = torch.randint(0, n_req, (n_rows,), generator=gen, dtype=torch.int32)
    sel = torch.full((n_rows, G, k), -1, dtype=torch.int32)
    for q in range(n_rows):
        for g in range(G):
            c = int(torch.randint(1, k + 1, (1,), generator=gen))
            sel[q, g, :c] = torch.randperm(mb, generator=gen)[:c].sort().values.to(torch.int32)
    dims = msa.Dims(16, G, 128, 64, k, mb)
    off, ent, pos = msa.msa_invert_selection(sel.to(DEV), q_req.to(DEV), n_req, dims)
    roff, rent = oracle.invert(sel, q_req, n_req, mb)
    assert torch.equal(off.cpu(), roff)
    assert torch.equal(ent.cpu()[:int(roff[-1])], rent)
    P.assert_ent_pos(sel, pos.cpu(), rent)


def test_lse_merge_matches_oracle(msa):
    """The merge on partials stored in an arbitrary entry order (ent_pos a random
    permutation), against the oracle's merge of the same partials by slot."""
    gen = torch.Generator().manual_seed(2)
    n_rows, G, Hq, D, k = 64, 4, 32, 128, 9
    hpg = Hq // G
    sel = torch.randint(-1, 20, (n_rows, G, k), generator=gen, dtype=torch.int32)
    o = torch.randn(n_rows, k, Hq, D, generator=gen).to(torch.bfloat16)
    lse = torch.randn(n_rows, k, Hq, generator=gen) * 3
    n_ent = n_rows * G * k
    ent_pos = torch.randperm(n_ent, generator=gen).to(torch.int32).reshape(n_rows, G, k)
    o_ent = torch.zeros(n_ent, hpg, D, dtype=torch.bfloat16)
    l_ent = torch.zeros(n_ent, hpg)
    o_g = o.reshape(n_rows, k, G, hpg, D).permute(0, 2, 1, 3, 4)      # [rows][G][k][hpg][D]
    l_g = lse.reshape(n_rows, k, G, hpg).permute(0, 2, 1, 3)
    o_ent[ent_pos.long().flatten()] = o_g.reshape(-1, hpg, D)
    l_ent[ent_pos.long().flatten()] = l_g.reshape(-1, hpg)
    dims = msa.Dims(Hq, G, D, 64, k, 20)
    o_lay = msa.partials_from_entry_major(o_ent, hpg, D)   # the kernel's partials layout
    out, l = msa.msa_lse_merge(o_lay.to(DEV), l_ent.to(DEV), sel.to(DEV), ent_pos.to(DEV), dims)
    valid = (sel >= 0).repeat_interleave(Hq // G, dim=1).transpose(1, 2)
    lse_m = torch.where(valid, lse.double(), torch.tensor(float("-inf"), dtype=torch.float64))
    ro, rl = oracle.lse_merge(o.double() * valid[..., None], lse_m)
    P.assert_out(out.cpu(), ro)
    P.assert_lse(l.cpu(), rl)
