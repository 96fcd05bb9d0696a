"""The decode attention entry point that allocates nothing.

Callers that cannot allocate device memory (a serving loop whose allocator is
frozen after start-up, a plug-in whose host framework owns every allocation)
use msa_sparse_attn_decode_noalloc, which keeps its scratch in the library's
own device array.  Its output must match msa_sparse_attn_decode, the entry point
with a caller workspace, within the decode tolerances, on two calls in a row
that share that array.  This file is collected last on purpose.
"""
import pytest
import torch

from msa_check import LSE_MAX_ABS, O_MAX_ABS, O_MEAN_ABS
from workloads import DecodeWorkload, MSAShape, decode_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msa():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from block_sparse_attention_02_gb300 import build as b
    b.build()
    import block_sparse_attention_02_gb300 as m
    return m


def test_noalloc_matches_workspace_entry_point_twice(msa):
    cases = [
        DecodeWorkload("noalloc_a", lengths=(60001,) * 8, shape=MSAShape(), seed=61),
        # the second call has fewer live splits, so stale scratch from the first call would show
        DecodeWorkload("noalloc_b", lengths=(1, 300, 2049, 129), shape=MSAShape(Hq=16, Hkv=2, k=16), seed=62),
    ]
    for wl in cases:
        inp = decode_inputs(wl, device="cuda")
        ref = msa.decode_step(inp, wl.shape.k)       # index, top-k, page table, workspace attention
        O = torch.empty_like(ref["O"])
        L = torch.empty_like(ref["LSE"])
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        msa.msa_sparse_attn_decode_noalloc(inp["Q"], inp["K_pool"], inp["V_pool"], ref["pt"], ref["n"],
                                           ref["last_len"], O, L, dev_err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0 and int(ref["dev_err"].item()) == 0
        d = (O.float() - ref["O"].float()).abs()
        assert d.max().item() <= O_MAX_ABS and d.mean().item() <= O_MEAN_ABS
        assert (L - ref["LSE"]).abs().max().item() <= LSE_MAX_ABS


def test_noalloc_rejects_sizes_beyond_its_array(msa):
    lib = msa.lib()
    from block_sparse_attention_02_gb300 import _abi
    import ctypes as C
    a = _abi.DecodeArgs()
    a.B, a.Hq, a.Hkv, a.D, a.Bk, a.k = 4096, 48, 8, 128, 128, 64     # ~6.5 GB of scratch
    a.Q = a.K_pool = a.V_pool = a.pt = a.n = a.last_len = a.O = 0x10000
    a.Q_stride[:] = [48 * 128, 128]
    a.kv_stride[:] = [8 * 128 * 128, 128 * 128, 128]
    a.num_pages = 10
    assert lib.msa_sparse_attn_decode_noalloc(C.byref(a), None) == _abi.MSA_ERR_WORKSPACE
    assert b"built-in array" in lib.msa_last_error_string()
