"""Decode path on the GPU against the fp64 oracle: index scoring, top-k, page
tables, paged sparse attention -- through the C ABI, on seeded workloads."""
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


def _run_decode(m, case):
    """The fused entry point msa_decode_step, and the same step through the four
    separate entry points; both must give identical bits (same kernels for the
    scan and attention, the same exact top-k rule)."""
    dims = m.dims_of(case)
    step = m.DecodeStep(dims, case.n_rows, case.n_req, case.n_pages, DEV)
    args = (case.q, case.q_idx, case.k_cache, case.v_cache, case.kidx_cache, case.block_table, case.seq_lens,
            case.q_pos)
    step(*args)
    m.msa_check(step.err)
    comp = m.DecodeStep(dims, case.n_rows, case.n_req, case.n_pages, DEV)
    comp.composed(*args)
    m.msa_check(comp.err)
    torch.cuda.synchronize()
    for name in ("scores", "sel", "page_table", "row_len", "out", "lse"):
        a, b = getattr(step, name), getattr(comp, name)
        assert torch.equal(a, b) or (name == "scores" and torch.equal(a.isneginf(), b.isneginf())
                                     and torch.equal(a[~a.isneginf()], b[~b.isneginf()])), name
    return step


def _check_decode(m, case, rows=None):
    step = _run_decode(m, case)
    rows = list(range(case.n_rows)) if rows is None else rows
    ref = P.oracle_decode_rows(case, rows)
    idx = torch.as_tensor(rows)
    q_pos = case.q_pos.cpu()[idx]
    P.assert_scores(step.scores.cpu()[idx], ref["scores"], q_pos)
    # top-k kernel on the oracle's scores (rounded to fp32) is bit-exact
    sc32 = ref["scores"].float()
    sel_on_ref = m.msa_topk_blocks(sc32.to(DEV), q_pos.to(DEV), m.dims_of(case))
    ref_sel32 = oracle.topk(sc32.double(), q_pos, case.dims.topk)
    assert torch.equal(sel_on_ref.cpu(), ref_sel32)
    # end to end: selection agrees where unambiguous
    gap = P.selection_gap(ref["scores"], q_pos, case.dims.topk)
    gsel = step.sel.cpu()[idx]
    P.assert_selection_where_unambiguous(gsel, ref["sel"], gap)
    # near ties too: a valid top-k of the oracle's scores, and exactly the top-k of the GPU's own scores
    P.assert_selection_valid(gsel, ref["scores"], q_pos, case.dims.topk)
    P.assert_topk_of_own_scores(gsel, step.scores.cpu()[idx], q_pos, case.dims.topk)
    # page table + row lengths bit-exact for the GPU's own selection
    pt, rl = oracle.page_table(gsel, case.block_table.cpu()[case.q_req.cpu()[idx].long()], q_pos + 1)
    G = case.dims.G
    grow = torch.cat([torch.arange(r * G, (r + 1) * G) for r in rows])
    assert torch.equal(step.page_table.cpu()[grow], pt)
    assert torch.equal(step.row_len.cpu()[grow], rl)
    # attention against the oracle on the GPU's selection
    o_ref, l_ref = P.oracle_attention_on(case, rows, gsel)
    P.assert_out(step.out.cpu()[idx], o_ref)
    P.assert_lse(step.lse.cpu()[idx], l_ref)
    return step, ref


def test_tiny_decode_steps(msa):
    """16 decode steps after a 2048-token prefix (Hq=8, G=2, D=64, Di=32, k=4)."""
    _, dec = mi.tiny_case(seed=1000, device=DEV)
    _check_decode(msa, dec)


@pytest.mark.parametrize("lens", [[1, 127, 128, 129, 300, 2049], [5000, 17, 128 * 16 + 5]])
def test_ragged_small_decode(msa, lens):
    case = mi.decode_case(lens, Hq=64, G=8, D=128, Di=64, topk=16, pool_pages=200, needles_per_group=4,
                          seed=77, device=DEV)
    _check_decode(msa, case)


@pytest.mark.parametrize("hq,g,d,di", [(16, 4, 64, 32), (16, 2, 128, 64), (32, 8, 64, 64)])
def test_decode_shape_variants(msa, hq, g, d, di):
    case = mi.decode_case([700, 1500, 3000], Hq=hq, G=g, D=d, Di=di, topk=5, pool_pages=60, needles_per_group=2,
                          seed=5, device=DEV)
    _check_decode(msa, case)


@pytest.mark.parametrize("topk", [1, 32])
def test_decode_topk_limits(msa, topk):
    """topk = 1 (the own block alone) and topk = 32 (the largest supported): rows with
    fewer candidates than topk, exactly topk, and many more."""
    case = mi.decode_case([100, 129, 32 * 128, 32 * 128 + 1, 20000], Hq=16, G=2, D=128, Di=64, topk=topk,
                          pool_pages=300, needles_per_group=2, seed=17, device=DEV)
    _check_decode(msa, case)


def test_decode60k_full(msa):
    case = mi.named_case("decode60k", device=DEV)
    _check_decode(msa, case)


@pytest.mark.parametrize("name,rows", [("ragged1", [0]), ("ragged8", None), ("ragged32", [0, 7, 19, 31]),
                                       ("ragged64", [1, 10, 33, 63])])
def test_ragged_sweep(msa, name, rows):
    case = mi.named_case(name, device=DEV)
    _check_decode(msa, case, rows)


def test_decode1m(msa):
    case = mi.named_case("decode1m", device=DEV)
    step, ref = _check_decode(msa, case)
    # the planted needles are found: every needle block is selected for its (request, group)
    sel = step.sel.cpu()
    hit = sum(int(j in sel[b, g].tolist()) for (b, g, j) in case.needles)
    assert hit >= int(0.9 * len(case.needles))


@pytest.mark.parametrize("blocks", [150, 901, 1800, 3001, 10000])
def test_decode_selection_tiers(msa, blocks):
    """The decode selection kernel's launch shapes by context length: a CTA per (request,
    group) row of 256 or 1,024 threads with one candidate each (up to 256 / 1,024 blocks),
    then 512 threads holding 4, 8 or 32 candidates each; a short request shares every
    batch."""
    lens = [blocks * 128 - 37, 3000]
    case = mi.decode_case(lens, Hq=8, G=2, D=64, Di=32, topk=16, pool_pages=blocks + 40, needles_per_group=3,
                          seed=600 + blocks, device=DEV)
    assert case.max_blocks == blocks
    _check_decode(msa, case)


def test_out_of_range_page_is_flagged(msa):
    case = mi.decode_case([600, 900], Hq=16, G=2, D=128, Di=64, topk=4, pool_pages=20, needles_per_group=1,
                          seed=3, device=DEV)
    bad_bt = case.block_table.clone()
    bad_bt[1, 2] = case.n_pages + 5
    dims = msa.dims_of(case)
    step = msa.DecodeStep(dims, case.n_rows, case.n_req, case.n_pages, DEV)
    step(case.q, case.q_idx, case.k_cache, case.v_cache, case.kidx_cache, bad_bt, case.seq_lens, case.q_pos)
    with pytest.raises(msa.MsaError) as ei:
        msa.msa_check(step.err)
    assert ei.value.status == 4
    # the error word was cleared: a clean call passes
    step(case.q, case.q_idx, case.k_cache, case.v_cache, case.kidx_cache, case.block_table, case.seq_lens,
         case.q_pos)
    msa.msa_check(step.err)


def test_packed_inputs_and_results(msa):
    """DecodeInputs (one staging kernel for all step inputs), DecodeStep.download (one copy
    of out and lse) and a step writing out and lse into page-locked host memory give the
    same bits as the step on separate device tensors."""
    case = mi.decode_case([700, 3000, 129], Hq=64, G=8, D=128, Di=64, topk=16, pool_pages=80, needles_per_group=2,
                          seed=11, device=DEV)
    dims = msa.dims_of(case)
    step = msa.DecodeStep(dims, case.n_rows, case.n_req, case.n_pages, DEV)
    out, lse = step(case.q, case.q_idx, case.k_cache, case.v_cache, case.kidx_cache, case.block_table,
                    case.seq_lens, case.q_pos)
    msa.msa_check(step.err)
    ref_out, ref_lse = out.cpu(), lse.cpu()
    inputs = msa.DecodeInputs(dims, case.n_rows, DEV)
    for n in ("q", "q_idx", "q_pos", "seq_lens", "block_table"):
        getattr(inputs, "h_" + n).copy_(getattr(case, n).cpu())
    host_res, (h_out, h_lse) = step.host_results()
    step.out.zero_()
    inputs.upload()
    step(inputs.q, inputs.q_idx, case.k_cache, case.v_cache, case.kidx_cache, inputs.block_table, inputs.seq_lens,
         inputs.q_pos)
    step.download(host_res)
    torch.cuda.synchronize()
    msa.msa_check(step.err)
    assert torch.equal(h_out, ref_out) and torch.equal(h_lse, ref_lse)
    # the step writing out and lse straight into page-locked host memory gives the same bits
    _, (z_out, z_lse) = step.host_results()
    step(inputs.q, inputs.q_idx, case.k_cache, case.v_cache, case.kidx_cache, inputs.block_table, inputs.seq_lens,
         inputs.q_pos, out=z_out, lse=z_lse)
    torch.cuda.synchronize()
    msa.msa_check(step.err)
    assert torch.equal(z_out, ref_out) and torch.equal(z_lse, ref_lse)
    with pytest.raises(ValueError):   # pageable host memory is refused
        step(inputs.q, inputs.q_idx, case.k_cache, case.v_cache, case.kidx_cache, inputs.block_table,
             inputs.seq_lens, inputs.q_pos, out=torch.empty_like(z_out), lse=z_lse)


def test_stage_from_host(msa):
    """msa_stage_from_host copies page-locked host bytes into device memory exactly (a size
    that ends inside a CTA's share too), and refuses, on the host, a source that is not
    page-locked host memory or a size that is not a multiple of 16 bytes."""
    import ctypes
    gen = torch.Generator().manual_seed(5)
    for n in (16, 4096 * 16 + 48, 155 * 1024):
        host = torch.randint(0, 256, (n,), generator=gen, dtype=torch.uint8).pin_memory()
        dev = torch.zeros(n, dtype=torch.uint8, device=DEV)
        msa.msa_stage_from_host(host, dev)
        torch.cuda.synchronize()
        assert torch.equal(dev.cpu(), host)
    lib, dev = msa.library(), torch.zeros(64, dtype=torch.uint8, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    pageable = torch.zeros(64, dtype=torch.uint8)
    pinned = torch.zeros(64, dtype=torch.uint8).pin_memory()
    for src, nbytes in ((pageable, 64), (dev, 64), (pinned, 40)):
        rc = lib.msa_stage_from_host(ctypes.c_void_p(src.data_ptr()), ctypes.c_void_p(dev.data_ptr()), nbytes, stream)
        assert rc == 1, (src.device, nbytes, rc)   # MSA_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        msa.msa_stage_from_host(pageable, dev)


def test_bounded_wait_timeout_is_reported_and_the_context_stays_usable(msa):
    """The device error path shared by every bounded wait: a wait that nothing completes
    (msa_selftest_timeout) gives up after its limit, the host reads MSA_ERR_TIMEOUT, the
    word is cleared, and the next decode step on the same stream runs clean."""
    err = msa.new_err_word(DEV)
    msa.msa_selftest_timeout(err)
    with pytest.raises(msa.MsaError) as ei:
        msa.msa_check(err)
    assert ei.value.status == 5 and "TIMEOUT" in str(ei.value)
    _, dec = mi.tiny_case(seed=1000, device=DEV)
    _check_decode(msa, dec)


def test_decode_step_graph_replay(msa):
    """DecodeStep.capture() records the whole step (and, with DecodeInputs and a host
    result buffer, its upload and its results written into host memory) into a CUDA
    graph; replay() gives the same bits as the eager step, and new inputs written into
    the captured tensors are picked up by the next replay."""
    case = mi.decode_case([700, 3000, 129, 60000], Hq=64, G=8, D=128, Di=64, topk=16, pool_pages=600,
                          needles_per_group=2, seed=19, device=DEV)
    dims = msa.dims_of(case)
    eager = msa.DecodeStep(dims, case.n_rows, case.n_req, case.n_pages, DEV)
    inputs = msa.DecodeInputs(dims, case.n_rows, DEV)
    for n in ("q", "q_idx", "q_pos", "seq_lens", "block_table"):
        getattr(inputs, "h_" + n).copy_(getattr(case, n).cpu())
    step = msa.DecodeStep(dims, case.n_rows, case.n_req, case.n_pages, DEV)
    host_res, (h_out, h_lse) = step.host_results()
    step.capture(inputs.q, inputs.q_idx, case.k_cache, case.v_cache, case.kidx_cache, inputs.block_table,
                 inputs.seq_lens, inputs=inputs, host_results=host_res)
    gen = torch.Generator().manual_seed(3)
    for it in range(3):
        if it > 0:   # new queries for the next step, written into the pinned inputs the graph uploads
            inputs.h_q.copy_(torch.randn(inputs.h_q.shape, generator=gen).to(torch.bfloat16))
            inputs.h_q_idx.copy_(torch.randn(inputs.h_q_idx.shape, generator=gen).to(torch.bfloat16))
        step.replay()
        torch.cuda.synchronize()
        msa.msa_check(step.err)
        eager(inputs.h_q.to(DEV), inputs.h_q_idx.to(DEV), case.k_cache, case.v_cache, case.kidx_cache,
              case.block_table, case.seq_lens)
        msa.msa_check(eager.err)
        torch.cuda.synchronize()
        for name in ("sel", "page_table", "row_len"):
            assert torch.equal(getattr(step, name), getattr(eager, name)), (it, name)
        # the captured step writes out and lse into the page-locked host buffer
        assert torch.equal(h_out, eager.out.cpu()) and torch.equal(h_lse, eager.lse.cpu()), it
