"""Multi-token (speculative) decode index scoring on the GPU: several query rows per
request share one read of each candidate page (MSA_PHASE_DECODE_MULTI, keys as the
M side of bf16 tensor-core MMAs).  Checked against the fp64 oracle and against the
single-row decode scan on the same rows."""
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


def _oracle_scores(case):
    local = torch.arange(case.n_rows, dtype=torch.int32)
    bt = case.block_table.cpu()[case.q_req.cpu().long()]
    return oracle.block_scores(case.q_idx.cpu(), case.kidx_cache.cpu(), bt, local, case.q_pos.cpu(), case.max_blocks)


@pytest.mark.parametrize("lens,T,hq,g,d,di", [
    ([3000, 129, 20000], 4, 64, 8, 128, 64),      # rows straddle the block edge at 128 (L = 129)
    ([60000, 60000], 8, 64, 8, 128, 64),
    ([2049, 777], 16, 32, 16, 128, 64),           # two n-tiles, G = 16 (two groups per warp)
    ([1000, 5000, 300], 3, 8, 2, 64, 32),         # Di = 32, six idle warps
    ([128, 256], 1, 64, 8, 128, 64),              # one row per request: the single-row semantics
])
def test_multi_token_scores_match_oracle(msa, lens, T, hq, g, d, di):
    case = mi.multi_token_decode_case(lens, T, Hq=hq, G=g, D=d, Di=di, topk=8, pool_pages=1200, seed=31, device=DEV)
    dims = msa.dims_of(case)
    err = msa.new_err_word(DEV)
    got = msa.msa_index_score(case.q_idx, case.kidx_cache, case.block_table, case.q_req, case.q_pos, dims,
                              msa.MSA_PHASE_DECODE_MULTI, err_word=err)
    msa.msa_check(err)
    P.assert_scores(got, _oracle_scores(case), case.q_pos.cpu())
    # the single-row scan on the same rows agrees within the fp32 accumulation-order difference
    one = msa.msa_index_score(case.q_idx, case.kidx_cache, case.block_table, case.q_req, case.q_pos, dims,
                              msa.MSA_PHASE_DECODE, err_word=err)
    msa.msa_check(err)
    fin = torch.isfinite(one)
    assert torch.equal(fin, torch.isfinite(got))
    assert torch.allclose(got[fin], one[fin], rtol=1e-5, atol=1e-4)


def test_multi_token_rejects_ungrouped_rows(msa):
    """Rows not grouped by request raise MSA_FLAG_UNSUPPORTED (read by msa_check)."""
    case = mi.multi_token_decode_case([3000, 3000], 2, Hq=64, G=8, D=128, Di=64, topk=8, pool_pages=64, seed=32,
                                      device=DEV)
    dims = msa.dims_of(case)
    q_req = torch.tensor([0, 1, 0, 1], dtype=torch.int32, device=DEV)
    err = msa.new_err_word(DEV)
    msa.msa_index_score(case.q_idx, case.kidx_cache, case.block_table, q_req, case.q_pos, dims,
                        msa.MSA_PHASE_DECODE_MULTI, err_word=err)
    with pytest.raises(msa.MsaError, match="UNSUPPORTED"):
        msa.msa_check(err)


def test_multi_token_rejects_more_than_16_rows(msa):
    case = mi.multi_token_decode_case([3000], 17, Hq=64, G=8, D=128, Di=64, topk=8, pool_pages=64, seed=33,
                                      device=DEV)
    dims = msa.dims_of(case)
    err = msa.new_err_word(DEV)
    msa.msa_index_score(case.q_idx, case.kidx_cache, case.block_table, case.q_req, case.q_pos, dims,
                        msa.MSA_PHASE_DECODE_MULTI, err_word=err)
    with pytest.raises(msa.MsaError, match="UNSUPPORTED"):
        msa.msa_check(err)
