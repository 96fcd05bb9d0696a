"""The C ABI without a GPU: the library loads, exports every symbol msa.h
declares, the ctypes structs match the C layout, and bad arguments are rejected
on the host with nothing enqueued."""
import ctypes as C
import os
import re
import subprocess

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "msa.h")


@pytest.fixture(scope="module")
def abi():
    from block_sparse_attention_02_gb300 import build as b
    b.build()
    from block_sparse_attention_02_gb300 import _abi
    _abi.load()
    return _abi


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(msa_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(abi):
    names = declared_functions()
    assert len(names) >= 11
    lib = abi.load()
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(abi.SIGNATURES), "ctypes signatures must mirror msa.h"
    out = subprocess.run(["nm", "-D", "--defined-only", abi.LIB_PATH], capture_output=True, text=True).stdout
    for n in names:
        assert re.search(rf"\bT {n}$", out, re.M), n


def test_struct_layout_matches_header(abi, tmp_path):
    structs = {"msa_index_args": abi.IndexArgs, "msa_topk_args": abi.TopkArgs,
               "msa_prefill_args": abi.PrefillArgs, "msa_decode_args": abi.DecodeArgs,
               "msa_append_args": abi.AppendArgs, "msa_dense_decode_args": abi.DenseDecodeArgs,
               "msa_dense_prefill_args": abi.DensePrefillArgs}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "msa.h"', "int main(void) {"]
    for cname, py in structs.items():
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for f, _ in py._fields_:
            lines.append(f'printf("{cname} {f} %zu\\n", offsetof({cname}, {f}));')
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    got = {}
    for line in subprocess.check_output([str(exe)], text=True).splitlines():
        s, f, v = line.split()
        got[(s, f)] = int(v)
    for cname, py in structs.items():
        assert got[(cname, "size")] == C.sizeof(py), cname
        for f, _ in py._fields_:
            assert got[(cname, f)] == getattr(py, f).offset, (cname, f)


def test_version_and_status_strings(abi):
    lib = abi.load()
    assert lib.msa_version() >= 100
    assert lib.msa_status_string(abi.MSA_ERR_WORKSPACE) == b"MSA_ERR_WORKSPACE"


FAKE = 0x10000  # never dereferenced: every call below fails validation first


def _index_args(abi, **kw):
    a = abi.IndexArgs()
    a.mode, a.B, a.S, a.Hkv, a.HI, a.dI, a.Bk = abi.MSA_MODE_DECODE, 2, 0, 8, 4, 64, 128
    a.q_idx = a.w = a.k_idx = a.C = a.seq_pt = a.seq_len = FAKE
    a.q_idx_stride[:] = [2048, 256, 64, 0]
    a.w_stride[:] = [32, 4, 0]
    a.k_idx_stride[:] = [65536, 8192, 64]
    a.C_stride[:] = [800, 100, 0]
    a.num_pages, a.max_pages, a.nb_stride = 10, 5, 100
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("field,value,status", [
    ("q_idx", None, 1), ("Bk", 64, 2), ("dI", 32, 2), ("HI", 5, 2), ("HI", 0, 2),
    ("nb_stride", 0, 1), ("num_pages", 0, 1), ("max_pages", 0, 1), ("mode", 7, 1),
    ("q_idx", FAKE + 2, 1),  # misaligned
])
def test_index_score_rejects(abi, field, value, status):
    lib = abi.load()
    a = _index_args(abi, **{field: value})
    assert lib.msa_index_score(C.byref(a), None) == status
    assert lib.msa_last_error_string()


def test_index_score_rejects_bad_strides(abi):
    lib = abi.load()
    a = _index_args(abi)
    a.k_idx_stride[2] = 63   # not a multiple of 8 elements
    assert lib.msa_index_score(C.byref(a), None) == abi.MSA_ERR_INVALID_ARG
    a = _index_args(abi)
    a.mode, a.S = abi.MSA_MODE_PREFILL, 1000
    a.nb_stride = 7          # < ceil(1000 / 128)
    assert lib.msa_index_score(C.byref(a), None) == abi.MSA_ERR_INVALID_ARG


def test_topk_rejects(abi):
    lib = abi.load()
    a = abi.TopkArgs()
    a.mode, a.B, a.S, a.Hkv, a.Bk, a.k = abi.MSA_MODE_DECODE, 1, 0, 8, 128, 0
    a.C = a.sel = a.count = a.seq_len = FAKE
    a.C_stride[:] = [8, 1, 0]
    a.nb_stride = 4
    assert lib.msa_topk_blocks(C.byref(a), None) == abi.MSA_ERR_UNSUPPORTED   # k = 0
    a.k = 65
    assert lib.msa_topk_blocks(C.byref(a), None) == abi.MSA_ERR_UNSUPPORTED
    a.k, a.seq_len = 16, None
    assert lib.msa_topk_blocks(C.byref(a), None) == abi.MSA_ERR_INVALID_ARG


def test_page_table_rejects(abi):
    lib = abi.load()
    f = lib.msa_build_page_table
    assert f(FAKE, FAKE, FAKE, 4, FAKE, 1, 8, 0, 128, FAKE, FAKE, FAKE, None, None) == abi.MSA_ERR_UNSUPPORTED
    assert f(FAKE, FAKE, FAKE, 0, FAKE, 1, 8, 16, 128, FAKE, FAKE, FAKE, None, None) == abi.MSA_ERR_INVALID_ARG
    assert f(None, FAKE, FAKE, 4, FAKE, 1, 8, 16, 128, FAKE, FAKE, FAKE, None, None) == abi.MSA_ERR_INVALID_ARG


def _decode_args(abi, **kw):
    a = abi.DecodeArgs()
    a.B, a.Hq, a.Hkv, a.D, a.Bk, a.k = 2, 48, 8, 128, 128, 16
    a.Q = a.K_pool = a.V_pool = a.pt = a.n = a.last_len = a.O = FAKE
    a.Q_stride[:] = [48 * 128, 128]
    a.kv_stride[:] = [8 * 128 * 128, 128 * 128, 128]
    a.num_pages = 10
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("field,value,status", [
    ("Hq", 47, 2), ("Hq", 80, 2), ("D", 64, 2), ("k", 0, 2), ("K_pool", None, 1), ("num_pages", 0, 1),
])
def test_decode_rejects(abi, field, value, status):
    lib = abi.load()
    a = _decode_args(abi, **{field: value})
    ws = abi.load().msa_sparse_attn_decode_workspace_size(C.byref(_decode_args(abi)))
    assert lib.msa_sparse_attn_decode(C.byref(a), FAKE, ws, None) == status


def test_decode_rejects_small_workspace(abi):
    lib = abi.load()
    a = _decode_args(abi)
    ws = lib.msa_sparse_attn_decode_workspace_size(C.byref(a))
    assert ws >= 2 * 48 * 16 * 129 * 4
    assert lib.msa_sparse_attn_decode(C.byref(a), FAKE, ws - 1, None) == abi.MSA_ERR_WORKSPACE
    assert lib.msa_sparse_attn_decode(C.byref(a), None, ws, None) == abi.MSA_ERR_WORKSPACE


def test_merge_rejects(abi):
    lib = abi.load()
    f = lib.msa_lse_merge
    assert f(FAKE, FAKE, 4, 0, 128, FAKE, None, None, None) == abi.MSA_ERR_UNSUPPORTED
    assert f(FAKE, FAKE, 4, 16, 130, FAKE, None, None, None) == abi.MSA_ERR_UNSUPPORTED
    assert f(FAKE, FAKE, -1, 16, 128, FAKE, None, None, None) == abi.MSA_ERR_INVALID_ARG
    assert f(None, FAKE, 4, 16, 128, FAKE, None, None, None) == abi.MSA_ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_call_without_device_reports_cuda_error(abi):
    lib = abi.load()
    a = _index_args(abi)
    assert lib.msa_index_score(C.byref(a), None) == abi.MSA_ERR_CUDA
    assert b"cuda" in lib.msa_last_error_string().lower()


def test_cache_append_rejects(abi):
    a = abi.AppendArgs()
    a.B, a.Hkv, a.D, a.dI, a.Bk = 2, 2, 128, 64, 64          # Bk must be 128
    assert abi.load().msa_cache_append(C.byref(a), None) == 2
    a.Bk = 128
    assert abi.load().msa_cache_append(C.byref(a), None) == 1   # NULL pointers


def _chunk_index_args(abi, **kw):
    a = abi.IndexArgs()
    a.mode, a.B, a.S, a.Hkv, a.HI, a.dI, a.Bk = abi.MSA_MODE_CHUNK, 2, 4, 8, 4, 64, 128
    a.q_idx = a.w = a.k_idx = a.C = a.seq_pt = a.q_pos = FAKE
    a.q_idx_stride[:] = [8192, 2048, 256, 64]
    a.w_stride[:] = [128, 32, 4]
    a.k_idx_stride[:] = [65536, 8192, 64]      # page pool strides (page, g, t)
    a.C_stride[:] = [4 * 8 * 100, 8 * 100, 100]
    a.num_pages, a.max_pages, a.nb_stride = 10, 100, 100
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("field,value,status", [
    ("q_pos", None, 1), ("seq_pt", None, 1), ("num_pages", 0, 1), ("max_pages", 0, 1), ("nb_stride", 0, 1),
])
def test_chunk_index_rejects(abi, field, value, status):
    lib = abi.load()
    a = _chunk_index_args(abi, **{field: value})
    assert lib.msa_index_score(C.byref(a), None) == status
    assert lib.msa_last_error_string()


def test_chunk_index_rejects_rows_wider_than_the_page_table(abi):
    """nb_stride > max_pages would let the index score and the top-k disagree
    on which sequences they reject, so it is refused on the host."""
    lib = abi.load()
    a = _chunk_index_args(abi, max_pages=99)
    assert lib.msa_index_score(C.byref(a), None) == abi.MSA_ERR_INVALID_ARG
    assert b"max_pages" in lib.msa_last_error_string()


def test_chunk_index_group_stride(abi):
    """A chunk's index pool may share one group (stride 0 at the pool's group
    index 1); a zero page or token stride is rejected."""
    lib = abi.load()
    a = _chunk_index_args(abi)
    a.k_idx_stride[1] = 0
    assert lib.msa_index_score(C.byref(a), None) == abi.MSA_ERR_CUDA      # valid: stops at the missing device
    a = _chunk_index_args(abi)
    a.k_idx_stride[2] = 0
    assert lib.msa_index_score(C.byref(a), None) == abi.MSA_ERR_INVALID_ARG


def test_chunk_topk_and_attention_reject(abi):
    lib = abi.load()
    t = abi.TopkArgs()
    t.mode, t.B, t.S, t.Hkv, t.Bk, t.k = abi.MSA_MODE_CHUNK, 1, 4, 8, 128, 16
    t.C = t.sel = t.count = FAKE
    t.C_stride[:] = [3200, 800, 100]
    t.nb_stride = 100
    assert lib.msa_topk_blocks(C.byref(t), None) == abi.MSA_ERR_INVALID_ARG   # q_pos NULL
    a = abi.PrefillArgs()
    a.B, a.S, a.Hq, a.Hkv, a.D, a.Bk, a.k = 1, 4, 48, 8, 128, 128, 16
    a.Q = a.K = a.V = a.sel = a.count = a.O = FAKE
    a.Q_stride[:] = [4 * 48 * 128, 48 * 128, 128]
    a.K_stride[:] = a.V_stride[:] = [8 * 128 * 128, 128 * 128, 128]
    ws = FAKE
    a.mode = abi.MSA_MODE_DECODE
    assert lib.msa_sparse_attn_prefill(C.byref(a), ws, 1 << 30, None) == abi.MSA_ERR_INVALID_ARG
    a.mode = abi.MSA_MODE_CHUNK
    assert lib.msa_sparse_attn_prefill(C.byref(a), ws, 1 << 30, None) == abi.MSA_ERR_INVALID_ARG   # no seq_pt
    a.seq_pt = a.q_pos = FAKE
    a.max_pages, a.num_pages = 5, (1 << 29) + 1            # page ids must fit the tile descriptor
    assert lib.msa_sparse_attn_prefill(C.byref(a), ws, 1 << 30, None) == abi.MSA_ERR_INVALID_ARG
    a.num_pages = 10
    assert lib.msa_sparse_attn_prefill_workspace_size(C.byref(a), 4) > 0
    a.max_pages = 0
    assert lib.msa_sparse_attn_prefill_workspace_size(C.byref(a), 4) == 0


def _dense_decode_args(abi, **kw):
    a = abi.DenseDecodeArgs()
    a.B, a.Hq, a.Hkv, a.D, a.Bk = 2, 48, 8, 128, 128
    a.Q = a.K_pool = a.V_pool = a.seq_pt = a.seq_len = a.O = FAKE
    a.Q_stride[:] = [48 * 128, 128]
    a.kv_stride[:] = [8 * 128 * 128, 128 * 128, 128]
    a.num_pages, a.max_pages = 10, 5
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("field,value,status", [
    ("Hq", 47, 2), ("D", 64, 2), ("Bk", 64, 2), ("B", 1025, 1), ("seq_pt", None, 1), ("max_pages", 0, 1),
    ("max_pages", 1 << 27, 1), ("num_pages", 0, 1), ("Q", FAKE + 4, 1),
])
def test_dense_decode_rejects(abi, field, value, status):
    lib = abi.load()
    ws = lib.msa_dense_attn_decode_workspace_size(C.byref(_dense_decode_args(abi)))
    assert ws >= 2 * 48 * 2 * 129 * 4
    a = _dense_decode_args(abi, **{field: value})
    assert lib.msa_dense_attn_decode(C.byref(a), FAKE, ws, None) == status
    assert lib.msa_last_error_string()


def test_dense_decode_rejects_small_workspace(abi):
    lib = abi.load()
    a = _dense_decode_args(abi)
    ws = lib.msa_dense_attn_decode_workspace_size(C.byref(a))
    assert lib.msa_dense_attn_decode(C.byref(a), FAKE, ws - 1, None) == abi.MSA_ERR_WORKSPACE
    assert lib.msa_dense_attn_decode(C.byref(a), None, ws, None) == abi.MSA_ERR_WORKSPACE


def test_dense_prefill_rejects(abi):
    lib = abi.load()
    a = abi.DensePrefillArgs()
    a.B, a.S, a.Hq, a.Hkv, a.D = 1, 256, 48, 8, 128
    a.Q = a.K = a.V = a.O = FAKE
    a.Q_stride[:] = [256 * 48 * 128, 48 * 128, 128]
    a.K_stride[:] = a.V_stride[:] = [256 * 8 * 128, 8 * 128, 128]
    a.D = 64
    assert lib.msa_dense_attn_prefill(C.byref(a), None) == abi.MSA_ERR_UNSUPPORTED
    a.D, a.Hq = 128, 80                                  # G = 10
    assert lib.msa_dense_attn_prefill(C.byref(a), None) == abi.MSA_ERR_UNSUPPORTED
    a.Hq, a.V = 48, None
    assert lib.msa_dense_attn_prefill(C.byref(a), None) == abi.MSA_ERR_INVALID_ARG
    a.V = FAKE
    a.K_stride[1] = 100                                  # not a multiple of 8 elements
    assert lib.msa_dense_attn_prefill(C.byref(a), None) == abi.MSA_ERR_INVALID_ARG
