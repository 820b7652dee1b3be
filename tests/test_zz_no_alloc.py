"""msa_sparse_attn_decode_noalloc: decode attention for callers that cannot allocate.

Some callers cannot call cudaMalloc at all: for instance a serving engine that has
reserved nearly all HBM for its paged KV pool and routes every allocation through
its own allocator, or a plugin host that forbids libraries from using the CUDA
allocator.  For them the library offers a decode entry point whose split-by-page
scratch is a fixed 16 MiB device array inside the library instead of a
caller-provided workspace.

This test calls that entry point through the C ABI twice in a row, with
different queries each time, and checks both results against the workspace entry
point msa_sparse_attn_decode within the decode parity tolerances.  It sits in a
file of its own that pytest collects last, and it needs nothing from the other
tests: it passes alone in a fresh process and after the rest of the suite.
"""
import ctypes

import pytest
import torch

import msa_inputs as mi
from tests import _parity as P

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _noalloc_fn(msa):
    fn = msa.library().msa_sparse_attn_decode_noalloc
    fn.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(msa.msa_dims_t)] + \
        [ctypes.c_void_p] * 4
    fn.restype = ctypes.c_int
    return fn


def test_noalloc_decode_matches_workspace_entry_point_twice():
    import block_sparse_attention_06_gb300 as msa
    fn = _noalloc_fn(msa)
    case = mi.decode_case([3000, 60000, 129, 7000], Hq=64, G=8, D=128, Di=64, topk=16, pool_pages=700,
                          needles_per_group=4, seed=31, device=DEV)
    dims = msa.dims_of(case)
    step = msa.DecodeStep(dims, case.n_rows, case.n_req, case.n_pages, DEV)
    step(case.q, case.q_idx, case.k_cache, case.v_cache, case.kidx_cache, case.block_table, case.seq_lens,
         case.q_pos)
    msa.msa_check(step.err)
    d = dims.c()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    gen = torch.Generator(device=DEV).manual_seed(99)
    for call in range(2):
        q = case.q if call == 0 else torch.randn(case.q.shape, generator=gen, device=DEV).to(torch.bfloat16)
        ref_out, ref_lse = msa.msa_sparse_attn_decode(q, case.k_cache, case.v_cache, step.page_table, step.row_len,
                                                      dims)
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        rc = fn(q.data_ptr(), case.k_cache.data_ptr(), case.v_cache.data_ptr(), step.page_table.data_ptr(),
                step.row_len.data_ptr(), case.n_rows, case.n_pages, ctypes.byref(d), out.data_ptr(), lse.data_ptr(),
                err.data_ptr(), stream)
        assert rc == 0, msa.library().msa_last_error()
        msa.msa_check(err)
        torch.cuda.synchronize()
        P.assert_out(out, ref_out, f"noalloc out (call {call + 1})")
        P.assert_lse(lse, ref_lse, f"noalloc lse (call {call + 1})")


def test_noalloc_largest_batch_matches_workspace_entry_point():
    """B = 31 requests at G = 8, topk = 16, Hq/G = 8, D = 128: the largest batch the
    16 MiB array accepts, so the partials' lse and the per-row merge counters sit at its
    very end.  Short ragged contexts keep the oracle-free comparison quick; two calls in
    a row, the second with new queries."""
    import block_sparse_attention_06_gb300 as msa
    fn = _noalloc_fn(msa)
    lens = [129 + 97 * i for i in range(31)]              # 1 .. 24 pages per request
    case = mi.decode_case(lens, Hq=64, G=8, D=128, Di=64, topk=16, pool_pages=440, needles_per_group=2, seed=37,
                          device=DEV)
    dims = msa.dims_of(case)
    assert msa.msa_workspace_bytes(msa.MSA_OP_DECODE, 31, 0, dims) <= 16 << 20 < \
        msa.msa_workspace_bytes(msa.MSA_OP_DECODE, 32, 0, dims)
    step = msa.DecodeStep(dims, case.n_rows, case.n_req, case.n_pages, DEV)
    step(case.q, case.q_idx, case.k_cache, case.v_cache, case.kidx_cache, case.block_table, case.seq_lens,
         case.q_pos)
    msa.msa_check(step.err)
    d = dims.c()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    gen = torch.Generator(device=DEV).manual_seed(7)
    for call in range(2):
        q = case.q if call == 0 else torch.randn(case.q.shape, generator=gen, device=DEV).to(torch.bfloat16)
        ref_out, ref_lse = msa.msa_sparse_attn_decode(q, case.k_cache, case.v_cache, step.page_table, step.row_len,
                                                      dims)
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        rc = fn(q.data_ptr(), case.k_cache.data_ptr(), case.v_cache.data_ptr(), step.page_table.data_ptr(),
                step.row_len.data_ptr(), case.n_rows, case.n_pages, ctypes.byref(d), out.data_ptr(), lse.data_ptr(),
                err.data_ptr(), stream)
        assert rc == 0, msa.library().msa_last_error()
        msa.msa_check(err)
        torch.cuda.synchronize()
        P.assert_out(out, ref_out, f"noalloc B=31 out (call {call + 1})")
        P.assert_lse(lse, ref_lse, f"noalloc B=31 lse (call {call + 1})")


def test_noalloc_rejects_batches_beyond_the_static_scratch():
    import block_sparse_attention_06_gb300 as msa
    fn = _noalloc_fn(msa)
    dims = msa.Dims(64, 8, 128, 64, 16, 469).c()
    fake = ctypes.c_void_p(0x1000)   # never dereferenced: the size check comes first
    rc = fn(fake, fake, fake, fake, fake, 32, 4096, ctypes.byref(dims), fake, fake, fake, None)
    assert rc == 6   # MSA_ERR_WORKSPACE: 32 * 8 * 16 partials exceed 16 MiB
    assert b"16 MiB" in msa.library().msa_last_error()
