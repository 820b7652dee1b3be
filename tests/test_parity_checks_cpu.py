"""The selection checks of the parity suite, exercised on the CPU with the oracle's own
scores: a correct top-k passes, and each planted mistake (own block dropped, ids out of
order, wrong padding, a clearly worse block kept, a near tie broken the wrong way) is
caught by the check meant for it."""
import pytest
import torch

import msa_inputs as mi
import oracle
from tests import _parity as P


@pytest.fixture(scope="module")
def scored():
    pre, _ = mi.tiny_case(seed=1000)
    rows = torch.arange(0, pre.n_rows, 7)            # rows from every block, candidates 1 .. 16
    q_pos = pre.q_pos[rows]
    local = torch.arange(len(rows), dtype=torch.int32)
    bt = pre.block_table[pre.q_req[rows].long()]
    sc = oracle.block_scores(pre.q_idx[rows], pre.kidx_cache, bt, local, q_pos, pre.max_blocks)
    sel = oracle.topk(sc, q_pos, pre.dims.topk)
    return sc, sel, q_pos, pre.dims.topk


def _ranked_row(sc, sel, q_pos, topk):
    """A (row, group) with more candidates than topk and a clear gap between its worst kept
    and best dropped non-own block."""
    for r in range(sel.shape[0]):
        own = int(q_pos[r]) // 128
        if own + 1 <= topk:
            continue
        for g in range(sel.shape[1]):
            kept = [j for j in sel[r, g].tolist() if 0 <= j < own]
            dropped = [j for j in range(own) if j not in kept]
            lo = min(kept, key=lambda j: float(sc[r, g, j]))
            worst_drop = min(dropped, key=lambda j: float(sc[r, g, j]))
            if float(sc[r, g, lo]) - float(sc[r, g, worst_drop]) > 0.5:
                return r, g, lo, worst_drop
    raise AssertionError("no ranked row in the fixture")


def test_correct_selection_passes(scored):
    sc, sel, q_pos, k = scored
    P.assert_selection_valid(sel, sc, q_pos, k)
    P.assert_topk_of_own_scores(sel, sc.float(), q_pos, k)


def test_dropped_own_block_is_caught(scored):
    sc, sel, q_pos, k = scored
    bad = sel.clone()
    r = int(torch.nonzero(q_pos >= 128 * k)[0])
    own = int(q_pos[r]) // 128
    candidates = [j for j in range(own) if j not in bad[r, 0].tolist()]
    bad[r, 0, k - 1] = candidates[0]
    bad[r, 0] = bad[r, 0].sort().values
    with pytest.raises(AssertionError):
        P.assert_selection_valid(bad, sc, q_pos, k)


def test_unsorted_ids_are_caught(scored):
    sc, sel, q_pos, k = scored
    bad = sel.clone()
    r = int(torch.nonzero(q_pos >= 128 * k)[0])
    bad[r, 1, 0], bad[r, 1, 1] = sel[r, 1, 1], sel[r, 1, 0]
    with pytest.raises(AssertionError):
        P.assert_selection_valid(bad, sc, q_pos, k)


def test_wrong_padding_is_caught(scored):
    sc, sel, q_pos, k = scored
    bad = sel.clone()
    r = int(torch.nonzero(q_pos < 128)[0])            # one candidate: slots 1.. are padding
    bad[r, 0, 1] = 0
    with pytest.raises(AssertionError):
        P.assert_selection_valid(bad, sc, q_pos, k)


def test_clearly_worse_block_is_caught(scored):
    sc, sel, q_pos, k = scored
    r, g, kept, dropped = _ranked_row(sc, sel, q_pos, k)
    bad = sel.clone()
    ids = [dropped if j == kept else j for j in bad[r, g].tolist()]
    bad[r, g] = torch.tensor(sorted(ids), dtype=torch.int32)
    with pytest.raises(AssertionError, match="outranks"):
        P.assert_selection_valid(bad, sc, q_pos, k)
    with pytest.raises(AssertionError):
        P.assert_topk_of_own_scores(bad, sc.float(), q_pos, k)


def test_near_tie_is_valid_but_not_the_exact_rule(scored):
    """Two blocks tied in score: either may be kept by a valid top-k, but the rule keeps
    the lower id, and the exact check on the scores themselves says so."""
    sc, sel, q_pos, k = scored
    r, g, kept, dropped = _ranked_row(sc, sel, q_pos, k)
    tied = sc.clone()
    lo, hi = min(kept, dropped), max(kept, dropped)
    tied[r, g, dropped] = tied[r, g, kept]              # an exact tie between a kept and a dropped block
    want = oracle.topk(tied, q_pos, k)
    assert lo in want[r, g].tolist() and hi not in want[r, g].tolist()
    swapped = want.clone()
    ids = [hi if j == lo else j for j in swapped[r, g].tolist()]
    swapped[r, g] = torch.tensor(sorted(ids), dtype=torch.int32)
    P.assert_selection_valid(swapped, tied, q_pos, k)   # within tolerance: a valid top-k
    with pytest.raises(AssertionError):
        P.assert_topk_of_own_scores(swapped, tied.float(), q_pos, k)
    P.assert_topk_of_own_scores(want, tied.float(), q_pos, k)
