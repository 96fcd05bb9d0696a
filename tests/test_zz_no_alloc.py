"""The decode attention entry point that allocates nothing.

Callers that cannot allocate device memory (a serving loop whose allocator is
frozen after start-up, a plug-in whose host framework owns every allocation)
use msa_sparse_attn_decode_noalloc, which keeps its scratch in the library's
own device array of MSA_NOALLOC_SCRATCH_BYTES.  Its output must match the fp64
oracle (on the selection the GPU made) and msa_sparse_attn_decode, the entry
point with a caller workspace, within the decode tolerances, on calls in a row
that share that array: first the largest batch whose scratch fits the array,
then smaller batches with other (batch, group) layouts, so counters or
partials left by an earlier call would show.  One sequence more than the
largest batch is rejected on the host.  This file is collected last on purpose.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from msa_check import LSE_MAX_ABS, O_MAX_ABS, O_MEAN_ABS, check_attention
from workloads import DecodeWorkload, MSAShape, decode_inputs, ragged_lengths

pytestmark = pytest.mark.gpu

LIMIT = 32 << 20                       # MSA_NOALLOC_SCRATCH_BYTES in msa.h


@pytest.fixture(scope="module")
def msa():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from block_sparse_attention_02_gb300 import build as b
    b.build()
    import block_sparse_attention_02_gb300 as m
    return m


def _largest_batch(msa, sh):
    """The largest B whose decode scratch fits the built-in array."""
    per = msa.msa_sparse_attn_decode_workspace_size(1, sh.Hq, sh.Hkv, sh.k) - 256
    B = (LIMIT - 256) // per
    assert msa.msa_sparse_attn_decode_workspace_size(B, sh.Hq, sh.Hkv, sh.k) <= LIMIT
    assert msa.msa_sparse_attn_decode_workspace_size(B + 1, sh.Hq, sh.Hkv, sh.k) > LIMIT
    return B


def _noalloc(msa, inp, ref):
    O = torch.full_like(ref["O"], float("nan"))
    L = torch.full_like(ref["LSE"], float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    msa.msa_sparse_attn_decode_noalloc(inp["Q"], inp["K_pool"], inp["V_pool"], ref["pt"], ref["n"],
                                       ref["last_len"], O, L, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and int(ref["dev_err"].item()) == 0
    return O, L


def test_noalloc_matches_oracle_and_workspace_entry_point(msa):
    sh = MSAShape()
    Bmax = _largest_batch(msa, sh)
    cases = [
        # the largest batch that fits the array (48 q / 8 KV heads, k = 16)
        DecodeWorkload("noalloc_max", lengths=ragged_lengths(Bmax, 1, 4000, seed=60), shape=sh, seed=60),
        DecodeWorkload("noalloc_a", lengths=(60001,) * 8, shape=sh, seed=61),
        # fewer live splits and another (batch, group) layout than the calls before
        DecodeWorkload("noalloc_b", lengths=(1, 300, 2049, 129), shape=MSAShape(Hq=16, Hkv=2, k=16), seed=62),
    ]
    for wl in cases:
        inp = decode_inputs(wl, device="cuda")
        ref = msa.decode_step(inp, wl.shape.k)       # index, top-k, page table, workspace attention
        O, L = _noalloc(msa, inp, ref)
        # against the entry point with a caller workspace
        d = (O.float() - ref["O"].float()).abs()
        assert d.max().item() <= O_MAX_ABS and d.mean().item() <= O_MEAN_ABS, wl.name
        assert (L - ref["LSE"]).abs().max().item() <= LSE_MAX_ABS, wl.name
        # against the oracle on the selection the GPU made
        h = {n: inp[n].cpu() for n in ("Q", "K_pool", "V_pool", "seq_pt", "seq_len")}
        O_o, L_o = oracle.decode_attend(h["Q"], h["K_pool"], h["V_pool"], h["seq_pt"], h["seq_len"],
                                        ref["sel"].cpu().numpy(), ref["count"].cpu().numpy(),
                                        1.0 / math.sqrt(wl.shape.D))
        check_attention(O.float().cpu().numpy(), L.cpu().numpy(), O_o, L_o)


def test_noalloc_rejects_one_sequence_past_its_array(msa):
    from block_sparse_attention_02_gb300 import _abi
    import ctypes as C
    sh = MSAShape()
    Bmax = _largest_batch(msa, sh)
    lib = msa.lib()
    a = _abi.DecodeArgs()
    a.B, a.Hq, a.Hkv, a.D, a.Bk, a.k = Bmax + 1, sh.Hq, sh.Hkv, 128, 128, sh.k
    a.Q = a.K_pool = a.V_pool = a.pt = a.n = a.last_len = a.O = 0x10000     # never dereferenced
    a.Q_stride[:] = [sh.Hq * 128, 128]
    a.kv_stride[:] = [sh.Hkv * 128 * 128, 128 * 128, 128]
    a.num_pages = 10
    assert lib.msa_sparse_attn_decode_noalloc(C.byref(a), None) == _abi.MSA_ERR_WORKSPACE
    assert b"built-in array" in lib.msa_last_error_string()
    a.B = 4096                                                                # far past it
    assert lib.msa_sparse_attn_decode_noalloc(C.byref(a), None) == _abi.MSA_ERR_WORKSPACE
