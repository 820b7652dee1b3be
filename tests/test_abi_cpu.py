"""The C ABI without a GPU: the library loads, exports every entry point that
include/msa.h declares, and rejects bad arguments on the host (status codes)
before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "msa.h")


@pytest.fixture(scope="module")
def lib():
    from tests.conftest import build_library
    return ctypes.CDLL(build_library())


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(msa_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_hot_path():
    names = declared_functions()
    for n in ("msa_index_score", "msa_topk_blocks", "msa_build_page_table", "msa_invert_selection",
              "msa_sparse_attn_prefill", "msa_lse_merge", "msa_sparse_attn_decode", "msa_workspace_bytes",
              "msa_check", "msa_status_str", "msa_last_error", "msa_version"):
        assert n in names, n


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"libmsa.so does not export {n}"


class Dims(ctypes.Structure):
    _fields_ = [("Hq", ctypes.c_int32), ("G", ctypes.c_int32), ("D", ctypes.c_int32), ("Di", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("topk", ctypes.c_int32), ("max_blocks", ctypes.c_int32),
                ("sm_scale", ctypes.c_float)]


def good_dims(**kw):
    d = dict(Hq=64, G=8, D=128, Di=64, page_size=128, topk=16, max_blocks=469, sm_scale=0.088)
    d.update(kw)
    return Dims(**d)


FAKE = ctypes.c_void_p(0x1000)   # never dereferenced: validation fails first


def test_status_strings(lib):
    lib.msa_status_str.restype = ctypes.c_char_p
    assert lib.msa_status_str(0) == b"MSA_OK"
    assert lib.msa_status_str(6) == b"MSA_ERR_WORKSPACE"
    lib.msa_version.restype = ctypes.c_int32
    assert lib.msa_version() >= 100


@pytest.mark.parametrize("kw,status", [
    (dict(page_size=64), 2), (dict(topk=33), 2), (dict(topk=0), 1), (dict(Hq=63), 1),
    (dict(Di=48), 2), (dict(G=3, Hq=24), 2), (dict(max_blocks=0), 1),
])
def test_index_score_rejects_bad_dims(lib, kw, status):
    d = good_dims(**kw)
    rc = lib.msa_index_score(FAKE, FAKE, FAKE, FAKE, FAKE, 8, 8, 100, ctypes.byref(d), 0, FAKE, FAKE, None)
    assert rc == status
    lib.msa_last_error.restype = ctypes.c_char_p
    assert lib.msa_last_error()


def test_null_pointers_and_bad_sizes(lib):
    d = good_dims()
    assert lib.msa_index_score(None, FAKE, FAKE, FAKE, FAKE, 8, 8, 100, ctypes.byref(d), 0, FAKE, FAKE, None) == 1
    assert lib.msa_index_score(FAKE, FAKE, FAKE, FAKE, FAKE, 8, 8, 100, ctypes.byref(d), 7, FAKE, FAKE, None) == 1
    assert lib.msa_topk_blocks(FAKE, None, 4, ctypes.byref(d), FAKE, FAKE, None) == 1
    assert lib.msa_topk_blocks(FAKE, FAKE, -1, ctypes.byref(d), FAKE, FAKE, None) == 1
    assert lib.msa_build_page_table(FAKE, FAKE, FAKE, 2, 0, ctypes.byref(d), FAKE, FAKE, FAKE, None) == 1
    assert lib.msa_lse_merge(FAKE, FAKE, None, FAKE, 4, ctypes.byref(d), FAKE, FAKE, FAKE, None) == 1
    assert lib.msa_lse_merge(FAKE, FAKE, FAKE, None, 4, ctypes.byref(d), FAKE, FAKE, FAKE, None) == 1
    assert lib.msa_check(None, None) == 1
    # empty work is a no-op that never touches the device
    assert lib.msa_topk_blocks(None, None, 0, ctypes.byref(d), None, None, None) == 0
    assert lib.msa_sparse_attn_decode(None, None, None, None, None, 0, 10, ctypes.byref(d), None, None, None, 0,
                                      None, None) == 0


def test_attention_shape_limits(lib):
    for kw in (dict(Hq=16, G=8), dict(D=96), dict(sm_scale=0.0)):
        d = good_dims(**kw)
        rc = lib.msa_sparse_attn_prefill(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, 1, 100,
                                         ctypes.byref(d), FAKE, FAKE, FAKE, ctypes.c_size_t(1 << 30), FAKE, None)
        assert rc in (1, 2), kw


def test_workspace_sizes_and_errors(lib):
    lib.msa_workspace_bytes.restype = ctypes.c_size_t
    d = good_dims(max_blocks=533)
    inv = lib.msa_workspace_bytes(0, 8192, 1, ctypes.byref(d))
    # bitmap over (group, block) keys x ceil(rows/32) words + per-key counts, 256-byte aligned
    # bitmap and per-word prefix counts (one int32 per key and 32 rows each), then one count per key
    assert inv == 2 * (((8 * 533 * 256 * 4 + 255) // 256) * 256) + ((8 * 533 * 4 + 255) // 256) * 256
    dec = lib.msa_workspace_bytes(1, 8, 0, ctypes.byref(good_dims()))
    # fp32 partials + their lse + one merge counter per (request, group) row, 256-byte aligned
    assert dec == (((8 * 8 * 16 * 8 * 128 * 4 + 255) // 256) * 256 + ((8 * 8 * 16 * 8 * 4 + 255) // 256) * 256
                   + ((8 * 8 * 4 + 255) // 256) * 256)
    assert lib.msa_workspace_bytes(9, 8, 1, ctypes.byref(d)) == 0
    # fused selection + inversion: the candidate lists (one list of 15 keys per 128-block chunk),
    # 256-byte rounded, then the inversion's workspace
    sel_inv = lib.msa_workspace_bytes(4, 8192, 1, ctypes.byref(d))
    assert sel_inv == ((8192 * 8 * 5 * 15 * 8 + 255) // 256) * 256 + inv
    # ... refused before any launch when too small, misaligned, or for topk > 16
    sel_args = lambda dims, ws, nbytes: (*([FAKE] * 5), 8192, 1, 4096, ctypes.byref(dims), *([FAKE] * 4), ws,
                                         ctypes.c_size_t(nbytes), FAKE, None)
    assert lib.msa_select_invert_prefill(*sel_args(d, FAKE, sel_inv - 1)) == 6
    assert lib.msa_select_invert_prefill(*sel_args(d, ctypes.c_void_p(0x1008), sel_inv)) == 1
    assert lib.msa_select_invert_prefill(*sel_args(good_dims(max_blocks=533, topk=17), FAKE, 1 << 40)) == 2
    # prefill work list: 16-byte header + one {key, first tile} pair per chunk of <= 8 tiles,
    # at most one partial chunk per key plus the entries split into full chunks of 8 x 16 entries
    pre = lib.msa_workspace_bytes(2, 8192, 1, ctypes.byref(d))
    assert pre == 16 + 8 * (8 * 533 + (8192 * 8 * 16 + 127) // 128)
    rc = lib.msa_sparse_attn_prefill(*([FAKE] * 8), 8192, 1, 4096, ctypes.byref(d), FAKE, FAKE, FAKE,
                                     ctypes.c_size_t(pre - 1), FAKE, None)
    assert rc == 6
    # too small a workspace is refused before any launch
    rc = lib.msa_invert_selection(FAKE, FAKE, 8192, 1, ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, ctypes.c_size_t(inv - 1),
                                  FAKE, None)
    assert rc == 6
    rc = lib.msa_sparse_attn_decode(FAKE, FAKE, FAKE, FAKE, FAKE, 8, 4096, ctypes.byref(good_dims()), FAKE, FAKE,
                                    FAKE, ctypes.c_size_t(dec - 1), FAKE, None)
    assert rc == 6
    rc = lib.msa_decode_step(*([FAKE] * 7), 8, 4096, ctypes.byref(good_dims()), *([FAKE] * 6), FAKE,
                             ctypes.c_size_t(dec - 1), FAKE, None)
    assert rc == 6
    # a scan over more than 16384 blocks is refused by the fused decode step
    rc = lib.msa_decode_step(*([FAKE] * 7), 8, 4096, ctypes.byref(good_dims(max_blocks=16385)), *([FAKE] * 6),
                             FAKE, ctypes.c_size_t(1 << 40), FAKE, None)
    assert rc == 2


def test_package_import_fails_loudly_without_library(tmp_path):
    """The binding has no fallback: with the shared library missing, import raises."""
    import subprocess
    import sys
    import shutil
    pkg = os.path.join(ROOT, "block_sparse_attention_06_gb300")
    dst = tmp_path / "block_sparse_attention_06_gb300"
    shutil.copytree(pkg, dst, ignore=shutil.ignore_patterns("libmsa.so", "_build", "__pycache__"))
    code = "import block_sparse_attention_06_gb300"
    res = subprocess.run([sys.executable, "-c", code], cwd=tmp_path, capture_output=True, text=True)
    assert res.returncode != 0 and "libmsa.so is not built" in res.stderr


def test_packed_buffer_layout():
    """The packed staging buffers of DecodeInputs and DecodeStep: each view starts on
    a 256-byte boundary, views do not overlap, and each has its dtype and shape."""
    import torch
    import block_sparse_attention_06_gb300 as m
    specs = [((8, 64, 128), torch.bfloat16), ((8, 8, 64), torch.bfloat16), ((8,), torch.int32), ((3,), torch.int32),
             ((8, 469), torch.int32)]
    offs, n = m._layout(specs)
    assert offs == [0, 131072, 139264, 139520, 139776] and n == 139776 + 15104
    buf = torch.zeros(n, dtype=torch.uint8)
    views = m._views(buf, specs)
    for (shape, dtype), v, o in zip(specs, views, offs):
        assert v.shape == shape and v.dtype == dtype and v.is_contiguous()
        assert v.data_ptr() - buf.data_ptr() == o and o % 256 == 0
    for i, v in enumerate(views):   # writing one view leaves the others untouched
        v.fill_(i + 1)
    for i, v in enumerate(views):
        assert bool((v == i + 1).all())


@pytest.mark.parametrize("hpg,D,n_ent", [(8, 128, 37), (4, 64, 70), (8, 64, 16)])
def test_prefill_partials_layout(hpg, D, n_ent):
    """The prefill partials buffer and its entry-major view: the value of (entry i, head hh,
    column col) sits at the bf16 element that msa.h's formula gives, written out here on its
    own: i * hpg * D + ((col / 8) * hpg + hh) * 8 + col % 8."""
    import torch
    import block_sparse_attention_06_gb300 as m
    shape = m.partials_shape(n_ent, hpg, D)
    assert shape == (n_ent, D // 8, hpg, 8)
    flat = torch.zeros(shape, dtype=torch.float64).reshape(-1)
    for i in range(n_ent):
        for hh in range(hpg):
            for col in range(D):
                at = i * hpg * D + ((col // 8) * hpg + hh) * 8 + col % 8
                flat[at] = i * 1000 + hh * 100 + col * 0.5
    em = m.partials_entry_major(flat.reshape(shape), n_ent, hpg, D)
    want = (torch.arange(n_ent, dtype=torch.float64)[:, None, None] * 1000
            + torch.arange(hpg, dtype=torch.float64)[None, :, None] * 100
            + torch.arange(D, dtype=torch.float64)[None, None, :] * 0.5)
    assert em.shape == (n_ent, hpg, D) and torch.equal(em, want)
    back = m.partials_from_entry_major(want, hpg, D)   # and the inverse rearrangement
    assert back.shape == shape and torch.equal(back.reshape(-1), flat)
