"""Mixed batches: decode requests and a prefill chunk in one step over one page pool
(chunked-prefill engines co-schedule both kinds of row; the NVIDIA page's SGLang section
runs with --chunked-prefill-size 8192).  Decode rows take the decode path, chunk rows the
block-major prefill path.  Both halves are checked against the fp64 oracle, and the mixed
step -- serial or with the decode half on a side stream -- gives the same bits as the two
steps run separately."""
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


def _mixed_args(dec, pre):
    return (dec.k_cache, dec.v_cache, dec.kidx_cache, dec.q, dec.q_idx, dec.block_table, dec.seq_lens, pre.q,
            pre.q_idx, pre.block_table, pre.q_req, pre.q_pos)


def _check_decode_half(dec, out, lse, sel, scores):
    rows = list(range(dec.n_rows))
    ref = P.oracle_decode_rows(dec, rows)
    q_pos = dec.q_pos.cpu()
    P.assert_scores(scores.cpu(), ref["scores"], q_pos)
    P.assert_selection_valid(sel.cpu(), ref["scores"], q_pos, dec.dims.topk)
    P.assert_topk_of_own_scores(sel.cpu(), scores.cpu(), q_pos, dec.dims.topk)
    o_ref, l_ref = P.oracle_attention_on(dec, rows, sel.cpu())
    P.assert_out(out.cpu(), o_ref, "decode half out")
    P.assert_lse(lse.cpu(), l_ref, "decode half lse")


def _check_prefill_half(pre, out, lse, sel):
    rows = list(range(pre.n_rows))
    q_pos, q_req = pre.q_pos.cpu(), pre.q_req.cpu()
    bt = pre.block_table.cpu()[q_req.long()]
    sc = oracle.block_scores(pre.q_idx.cpu(), pre.kidx_cache.cpu(), bt, torch.arange(pre.n_rows, dtype=torch.int32),
                             q_pos, pre.max_blocks)
    gsel = sel.cpu()
    P.assert_selection_where_unambiguous(gsel, oracle.topk(sc, q_pos, pre.dims.topk),
                                         P.selection_gap(sc, q_pos, pre.dims.topk))
    P.assert_selection_valid(gsel, sc, q_pos, pre.dims.topk)
    o_ref, l_ref = P.in_row_chunks(
        lambda ch: P.oracle_attention_on(pre, [rows[i] for i in ch], gsel[torch.as_tensor(ch)]), range(len(rows)))
    P.assert_out(out.cpu(), o_ref, "prefill half out")
    P.assert_lse(lse.cpu(), l_ref, "prefill half lse")


@pytest.mark.parametrize("dec_lens,prefixes,chunks,hq,g,d,di,topk", [
    ([129, 2500, 7000, 1], [1000, 0], [300, 257], 16, 2, 128, 64, 6),      # ragged decode rows, two prefill requests
    ([60000, 3000, 640], [5000], [1024], 64, 8, 128, 64, 16),              # the agentic shape, smaller
    ([700, 701], [127, 64, 2000], [1, 63, 200], 8, 2, 64, 32, 4),          # one-row and partial-tile chunks
])
def test_mixed_step_matches_oracle_and_separate_steps(msa, dec_lens, prefixes, chunks, hq, g, d, di, topk):
    dec, pre = mi.mixed_case(dec_lens, prefixes, chunks, Hq=hq, G=g, D=d, Di=di, topk=topk, seed=61, device=DEV)
    dims = msa.dims_of(dec)
    assert msa.dims_of(pre) == dims
    # the two halves run alone
    ds = msa.DecodeStep(dims, dec.n_rows, dec.n_req, dec.n_pages, DEV)
    ds(dec.q, dec.q_idx, dec.k_cache, dec.v_cache, dec.kidx_cache, dec.block_table, dec.seq_lens)
    msa.msa_check(ds.err)
    ps = msa.PrefillStep(dims, pre.n_rows, pre.n_req, DEV)
    ps(pre.q, pre.q_idx, pre.k_cache, pre.v_cache, pre.kidx_cache, pre.block_table, pre.q_req, pre.q_pos)
    msa.msa_check(ps.err)
    for overlap in (False, True):
        ms = msa.MixedStep(dims, dec.n_rows, pre.n_rows, pre.n_req, dec.n_pages, DEV, overlap=overlap)
        for _ in range(2):   # the second call reuses every buffer
            d_out, d_lse, p_out, p_lse = ms(*_mixed_args(dec, pre))
            for e in ms.err_words:
                msa.msa_check(e)
            torch.cuda.synchronize()
            assert torch.equal(d_out, ds.out) and torch.equal(d_lse, ds.lse), f"decode half (overlap={overlap})"
            assert torch.equal(p_out, ps.out) and torch.equal(p_lse, ps.lse), f"prefill half (overlap={overlap})"
            assert torch.equal(ms.decode.sel, ds.sel) and torch.equal(ms.prefill.sel, ps.sel)
    _check_decode_half(dec, ms.decode.out, ms.decode.lse, ms.decode.sel, ms.decode.scores)
    _check_prefill_half(pre, ms.prefill.out, ms.prefill.lse, ms.prefill.sel)
