"""K/V offload with the k-index kept on the GPU: the decode step reads K/V from
page-locked host memory, gathering only the selected pages into a device pool
(msa_offload_gather).  The result must equal the all-on-device step bit for bit:
the same attention kernel runs on the same page contents, only the page ids differ.
It is also checked against the fp64 oracle, which reads K/V from the same host
copies the offloaded step gathers from."""
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


@pytest.mark.parametrize("lens,hq,g,d,di,topk", [
    ([3000, 60000, 129, 1], 64, 8, 128, 64, 16),     # a one-token request selects only its own page
    ([5000, 777], 16, 4, 64, 32, 6),
])
def test_offloaded_decode_equals_device_decode(msa, lens, hq, g, d, di, topk):
    case = mi.decode_case(lens, Hq=hq, G=g, D=d, Di=di, topk=topk, pool_pages=600, needles_per_group=3, seed=51,
                          device=DEV)
    dims = msa.dims_of(case)
    ref = msa.DecodeStep(dims, case.n_rows, case.n_req, case.n_pages, DEV)
    out_ref, lse_ref = ref.composed(case.q, case.q_idx, case.k_cache, case.v_cache, case.kidx_cache,
                                    case.block_table, case.seq_lens, case.q_pos)
    msa.msa_check(ref.err)
    host_k = case.k_cache.cpu().pin_memory()
    host_v = case.v_cache.cpu().pin_memory()
    off = msa.DecodeStep(dims, case.n_rows, case.n_req, case.n_pages, DEV)
    for _ in range(2):   # the pool is reused by the second step
        out, lse = off.offloaded(case.q, case.q_idx, host_k, host_v, case.kidx_cache, case.block_table,
                                 case.seq_lens, case.q_pos)
        msa.msa_check(off.err)
        torch.cuda.synchronize()
        assert torch.equal(off.page_table, ref.page_table)
        pk, pv, ppt = off._pool
        assert torch.equal(ppt < 0, ref.page_table < 0)
        assert torch.equal(out, out_ref)
        assert torch.equal(lse, lse_ref)
    # against the oracle: scores and selection of the GPU-resident k-index, then attention over the
    # GPU's selection with K/V taken from the host copies
    rows = list(range(case.n_rows))
    oref = P.oracle_decode_rows(case, rows)
    q_pos = case.q_pos.cpu()
    P.assert_scores(off.scores.cpu(), oref["scores"], q_pos)
    P.assert_selection_valid(off.sel.cpu(), oref["scores"], q_pos, topk)
    P.assert_topk_of_own_scores(off.sel.cpu(), off.scores.cpu(), q_pos, topk)
    pages, bt_c = P.compact_pages(case.block_table.cpu(), off.sel.cpu(), case.q_req.cpu())
    o_ref, l_ref = oracle.attention(case.q.cpu(), host_k[pages], host_v[pages], bt_c, case.q_req.cpu(), q_pos,
                                    off.sel.cpu(), dims.sm_scale)
    P.assert_out(out, o_ref, "offloaded out")
    P.assert_lse(lse, l_ref, "offloaded lse")
    # the pool holds exactly the selected group slices
    pt = ref.page_table.cpu()
    for r in (0, case.n_rows * g - 1):
        b, gg = divmod(r, g)
        for s in range(topk):
            if pt[r, s] >= 0:
                assert torch.equal(pk[b * topk + s, :, gg].cpu(), host_k[pt[r, s], :, gg])
                assert torch.equal(pv[b * topk + s, :, gg].cpu(), host_v[pt[r, s], :, gg])


def test_offload_rejects_unpinned_host_cache(msa):
    case = mi.decode_case([3000], Hq=64, G=8, D=128, Di=64, topk=8, pool_pages=64, needles_per_group=1, seed=52,
                          device=DEV)
    dims = msa.dims_of(case)
    pt = torch.full((8, 8), -1, dtype=torch.int32, device=DEV)
    with pytest.raises(ValueError, match="page-locked"):
        msa.msa_offload_gather(case.k_cache.cpu(), case.v_cache.cpu(), pt, dims)
    # the C entry point itself refuses pageable memory, also where the GPU could address it
    import ctypes
    k, v = case.k_cache.cpu(), case.v_cache.cpu()
    scratch, err = torch.empty(16, dtype=torch.uint8, device=DEV), msa.new_err_word(DEV)
    d, P = dims.c(), lambda t: ctypes.c_void_p(t.data_ptr())
    rc = msa.library().msa_offload_gather(P(k), P(v), k.shape[0], P(pt), 1, ctypes.byref(d), P(scratch), P(scratch),
                                          P(pt), P(err), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 1   # MSA_ERR_INVALID_ARG
