"""MiniMax Sparse Attention (MSA) hot path on one GB300 -- Python binding.

Thin ctypes marshalling over ``libmsa.so`` (include/msa.h).  Every function
takes torch CUDA tensors, passes their pointers and element strides to the C
entry point of the same name, and raises ``MSAError`` on a non-OK status.  All
computation runs in the library's sm_103a kernels; there is no fallback path.
PyTorch provides device memory and streams only.

The pipelines at the bottom (``decode_step``, ``prefill_layer`` and
``chunk_layer``) call the entry points in hot-path order: index score -> top-k
-> (decode: page table) -> sparse attention (with its log-sum-exp merge).
"""
from __future__ import annotations

import ctypes as C
from typing import Dict, Optional

import torch

from . import _abi
from ._abi import (MSA_DEVERR_BAD_LEN, MSA_DEVERR_BAD_PAGE, MSA_DEVERR_BAD_SEL, MSA_DEVERR_TIMEOUT,
                   MSA_MODE_CHUNK, MSA_MODE_DECODE, MSA_MODE_PREFILL, MSAError)

__all__ = [
    "msa_index_score", "msa_topk_blocks", "msa_build_page_table", "msa_sparse_attn_prefill",
    "msa_sparse_attn_decode", "msa_sparse_attn_decode_noalloc", "msa_lse_merge", "msa_sparse_attn_prefill_workspace_size",
    "msa_sparse_attn_decode_workspace_size", "msa_cache_append", "decode_step", "prefill_layer", "chunk_layer",
    "msa_dense_attn_decode", "msa_dense_attn_decode_workspace_size", "dense_decode_buffers", "dense_decode_step",
    "msa_dense_attn_prefill", "dense_prefill_layer",
    "lib", "MSAError",
    "MSA_MODE_PREFILL", "MSA_MODE_DECODE", "MSA_MODE_CHUNK", "MSA_DEVERR_TIMEOUT", "MSA_DEVERR_BAD_PAGE",
    "MSA_DEVERR_BAD_SEL", "MSA_DEVERR_BAD_LEN", "Bk", "D", "dI",
]

Bk = 128
D = 128
dI = 64


def lib():
    return _abi.load()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return C.c_void_p(stream.cuda_stream)
    return C.c_void_p(int(stream))


def _inner_contig(t: torch.Tensor, name: str):
    if t.stride(-1) != 1:
        raise ValueError(f"{name}: innermost dimension must be contiguous")


def _strides(t: torch.Tensor, n: int):
    s = list(t.stride()[:-1])
    return (s + [0] * n)[:n]


# ---------------------------------------------------------------------------
# a1. index score
# ---------------------------------------------------------------------------

def msa_index_score(mode: int, q_idx: torch.Tensor, w: torch.Tensor, k_idx: torch.Tensor, C_out: torch.Tensor,
                    *, seq_pt: Optional[torch.Tensor] = None, seq_len: Optional[torch.Tensor] = None,
                    dev_err: Optional[torch.Tensor] = None, stream=None, k: int = 0,
                    sel: Optional[torch.Tensor] = None, count: Optional[torch.Tensor] = None,
                    pt: Optional[torch.Tensor] = None, n: Optional[torch.Tensor] = None,
                    last_len: Optional[torch.Tensor] = None, row_scratch: Optional[torch.Tensor] = None,
                    scratch_zeroed: bool = False, q_pos: Optional[torch.Tensor] = None) -> None:
    """Block scores of the Index Branch into ``C_out`` (see msa.h, a1).

    PREFILL: q_idx [B,S,Hkv,HI,dI], w [B,S,Hkv,HI], k_idx [B,S,Hkv,dI], C_out [B,S,Hkv,nb_stride].
    CHUNK:   q_idx, w, C_out as PREFILL; k_idx pool [P,Hkv,Bk,dI], seq_pt [B,max_pages] int32,
             q_pos [B] int32 (position of each sequence's first chunk query).
    DECODE:  q_idx [B,Hkv,HI,dI], w [B,Hkv,HI], k_idx pool [P,Hkv,Bk,dI], C_out [B,Hkv,nb_stride],
             seq_pt [B,max_pages] int32 (contiguous rows), seq_len [B] int32.
    DECODE with ``sel`` given: the same call also selects (a2) into sel/count and,
    with ``pt`` given, builds the page table (a3) into pt/n/last_len; ``row_scratch``
    is B*Hkv int32 of scratch, cleared by the call unless ``scratch_zeroed`` says
    it is already zero (every error-free call leaves it zero).
    """
    for t, nm in ((q_idx, "q_idx"), (w, "w"), (k_idx, "k_idx"), (C_out, "C")):
        _inner_contig(t, nm)
    a = _abi.IndexArgs()
    a.mode = mode
    a.q_idx, a.w, a.k_idx, a.C = _ptr(q_idx), _ptr(w), _ptr(k_idx), _ptr(C_out)
    a.dev_err = _ptr(dev_err)
    a.nb_stride = C_out.shape[-1]
    if mode in (MSA_MODE_PREFILL, MSA_MODE_CHUNK):
        B, S, Hkv, HI, di = q_idx.shape
        a.B, a.S, a.Hkv, a.HI, a.dI, a.Bk = B, S, Hkv, HI, di, Bk
        a.q_idx_stride[:] = _strides(q_idx, 4)
        a.w_stride[:] = _strides(w, 3)
        a.k_idx_stride[:] = _strides(k_idx, 3)
        a.C_stride[:] = _strides(C_out, 3)
        if mode == MSA_MODE_CHUNK:
            if not (seq_pt.is_contiguous() and q_pos.is_contiguous()):
                raise ValueError("seq_pt and q_pos must be contiguous")
            a.num_pages, a.seq_pt, a.max_pages, a.q_pos = k_idx.shape[0], _ptr(seq_pt), seq_pt.shape[1], _ptr(q_pos)
    else:
        B, Hkv, HI, di = q_idx.shape
        a.B, a.S, a.Hkv, a.HI, a.dI, a.Bk = B, 0, Hkv, HI, di, k_idx.shape[2]
        a.q_idx_stride[:] = _strides(q_idx, 3) + [0]
        a.w_stride[:] = _strides(w, 2) + [0]
        a.k_idx_stride[:] = _strides(k_idx, 3)
        a.C_stride[:] = _strides(C_out, 2) + [0]
        if not seq_pt.is_contiguous():
            raise ValueError("seq_pt must be contiguous")
        a.num_pages = k_idx.shape[0]
        a.seq_pt, a.max_pages, a.seq_len = _ptr(seq_pt), seq_pt.shape[1], _ptr(seq_len)
        if sel is not None:
            for t, nm in ((sel, "sel"), (count, "count"), (row_scratch, "row_scratch")):
                if t is None or not t.is_contiguous():
                    raise ValueError(f"fused selection: {nm} must be a contiguous tensor")
            a.k, a.sel, a.count, a.row_scratch = k, _ptr(sel), _ptr(count), _ptr(row_scratch)
            a.scratch_zeroed = int(bool(scratch_zeroed))
            if pt is not None:
                a.pt, a.n, a.last_len = _ptr(pt), _ptr(n), _ptr(last_len)
    _abi.check(lib().msa_index_score(C.byref(a), _stream(stream)), "msa_index_score")


# ---------------------------------------------------------------------------
# a2. top-k
# ---------------------------------------------------------------------------

def msa_topk_blocks(mode: int, C_in: torch.Tensor, k: int, sel: torch.Tensor, count: torch.Tensor, *,
                    seq_len: Optional[torch.Tensor] = None, dev_err: Optional[torch.Tensor] = None,
                    stream=None, q_pos: Optional[torch.Tensor] = None) -> None:
    """Own block + top-(k-1) earlier blocks per row (see msa.h, a2).

    PREFILL: C_in [B,S,Hkv,nb], sel [B,S,Hkv,k], count [B,S,Hkv].
    CHUNK:   as PREFILL, own block (q_pos[b] + s) // Bk.
    DECODE:  C_in [B,Hkv,nb], seq_len [B], sel [B,Hkv,k], count [B,Hkv].
    """
    _inner_contig(C_in, "C")
    if not (sel.is_contiguous() and count.is_contiguous()):
        raise ValueError("sel and count must be contiguous")
    a = _abi.TopkArgs()
    a.mode, a.k, a.Bk = mode, k, Bk
    a.C, a.sel, a.count, a.dev_err = _ptr(C_in), _ptr(sel), _ptr(count), _ptr(dev_err)
    a.nb_stride = C_in.shape[-1]
    if mode in (MSA_MODE_PREFILL, MSA_MODE_CHUNK):
        a.B, a.S, a.Hkv = C_in.shape[0], C_in.shape[1], C_in.shape[2]
        a.C_stride[:] = _strides(C_in, 3)
        if mode == MSA_MODE_CHUNK:
            a.q_pos = _ptr(q_pos)
    else:
        a.B, a.S, a.Hkv = C_in.shape[0], 0, C_in.shape[1]
        a.C_stride[:] = _strides(C_in, 2) + [0]
        a.seq_len = _ptr(seq_len)
    _abi.check(lib().msa_topk_blocks(C.byref(a), _stream(stream)), "msa_topk_blocks")


# ---------------------------------------------------------------------------
# a3. page table
# ---------------------------------------------------------------------------

def msa_build_page_table(sel: torch.Tensor, count: torch.Tensor, seq_pt: torch.Tensor, seq_len: torch.Tensor,
                         pt: torch.Tensor, n: torch.Tensor, last_len: torch.Tensor, *,
                         dev_err: Optional[torch.Tensor] = None, stream=None) -> None:
    """Flattened (B*Hkv) page table from the selected blocks (see msa.h, a3)."""
    B, Hkv, k = sel.shape
    for t, nm in ((sel, "sel"), (count, "count"), (pt, "pt"), (n, "n"), (last_len, "last_len")):
        if not t.is_contiguous():
            raise ValueError(f"{nm} must be contiguous")
    if not seq_pt.is_contiguous():
        raise ValueError("seq_pt must be contiguous")
    _abi.check(lib().msa_build_page_table(_ptr(sel), _ptr(count), _ptr(seq_pt), seq_pt.shape[1], _ptr(seq_len),
                                          B, Hkv, k, Bk, _ptr(pt), _ptr(n), _ptr(last_len), _ptr(dev_err),
                                          _stream(stream)),
               "msa_build_page_table")


# ---------------------------------------------------------------------------
# a4/a5 sparse attention and a6 merge
# ---------------------------------------------------------------------------

def _prefill_args(Q, K, V, sel, count, O, LSE, softmax_scale, dev_err, seq_pt=None, q_pos=None
                  ) -> _abi.PrefillArgs:
    """PREFILL: K, V [B,S,Hkv,D].  CHUNK (seq_pt and q_pos given): K, V page pools [P,Hkv,Bk,D]."""
    for t, nm in ((Q, "Q"), (K, "K"), (V, "V")):
        _inner_contig(t, nm)
    a = _abi.PrefillArgs()
    a.B, a.S, a.Hq, a.D = Q.shape
    a.Hkv = K.shape[2]
    if seq_pt is not None:
        if not (seq_pt.is_contiguous() and q_pos.is_contiguous()):
            raise ValueError("seq_pt and q_pos must be contiguous")
        a.mode = MSA_MODE_CHUNK
        a.Hkv = K.shape[1]
        a.seq_pt, a.max_pages, a.num_pages, a.q_pos = _ptr(seq_pt), seq_pt.shape[1], K.shape[0], _ptr(q_pos)
    a.Bk = Bk
    a.k = sel.shape[-1]
    a.softmax_scale = softmax_scale
    a.Q, a.K, a.V = _ptr(Q), _ptr(K), _ptr(V)
    a.Q_stride[:] = _strides(Q, 3)
    a.K_stride[:] = _strides(K, 3)
    a.V_stride[:] = _strides(V, 3)
    a.sel, a.count = _ptr(sel), _ptr(count)
    a.O, a.LSE, a.dev_err = _ptr(O), _ptr(LSE), _ptr(dev_err)
    return a


def msa_sparse_attn_prefill_workspace_size(Q, K, sel, chunk_queries: int, max_pages: Optional[int] = None) -> int:
    """Workspace bytes for chunks of ``chunk_queries`` queries; ``max_pages`` (the
    page-table width) selects CHUNK mode, where K is a page pool [P,Hkv,Bk,D]."""
    a = _abi.PrefillArgs()
    a.B, a.S, a.Hq, a.D = Q.shape
    a.Hkv, a.Bk, a.k = K.shape[2], Bk, sel.shape[-1]
    a.Q_stride[:] = _strides(Q, 3)
    a.K_stride[:] = _strides(K, 3)
    a.V_stride[:] = _strides(K, 3)      # V is taken to share K's strides
    if max_pages is not None:
        a.mode, a.Hkv, a.max_pages = MSA_MODE_CHUNK, K.shape[1], int(max_pages)
    return int(lib().msa_sparse_attn_prefill_workspace_size(C.byref(a), int(chunk_queries)))


def msa_sparse_attn_prefill(Q, K, V, sel, count, O, LSE, ws: torch.Tensor, *, softmax_scale: float = 0.0,
                            dev_err=None, stream=None, seq_pt: Optional[torch.Tensor] = None,
                            q_pos: Optional[torch.Tensor] = None) -> None:
    """KV-block-major causal sparse attention (see msa.h, a3'-a4-a6).

    With ``seq_pt`` and ``q_pos`` (CHUNK mode) Q is a chunk of queries at
    positions q_pos[b] + s and K, V are page pools [P,Hkv,Bk,D] indexed by seq_pt."""
    if not (sel.is_contiguous() and count.is_contiguous() and O.is_contiguous()):
        raise ValueError("sel, count and O must be contiguous")
    a = _prefill_args(Q, K, V, sel, count, O, LSE, softmax_scale, dev_err, seq_pt, q_pos)
    _abi.check(lib().msa_sparse_attn_prefill(C.byref(a), _ptr(ws), ws.numel() * ws.element_size(),
                                             _stream(stream)), "msa_sparse_attn_prefill")


def _decode_args(Q, K_pool, V_pool, pt, n, last_len, O, LSE, softmax_scale, dev_err) -> _abi.DecodeArgs:
    for t, nm in ((Q, "Q"), (K_pool, "K_pool"), (V_pool, "V_pool")):
        _inner_contig(t, nm)
    if K_pool.stride() != V_pool.stride():
        raise ValueError("K_pool and V_pool must share strides")
    a = _abi.DecodeArgs()
    a.B, a.Hq, a.D = Q.shape
    a.Hkv, a.Bk = K_pool.shape[1], K_pool.shape[2]
    a.k = pt.shape[-1]
    a.softmax_scale = softmax_scale
    a.Q = _ptr(Q)
    a.Q_stride[:] = _strides(Q, 2)
    a.K_pool, a.V_pool = _ptr(K_pool), _ptr(V_pool)
    a.kv_stride[:] = _strides(K_pool, 3)
    a.num_pages = K_pool.shape[0]
    a.pt, a.n, a.last_len = _ptr(pt), _ptr(n), _ptr(last_len)
    a.O, a.LSE, a.dev_err = _ptr(O), _ptr(LSE), _ptr(dev_err)
    return a


def msa_sparse_attn_decode_workspace_size(B: int, Hq: int, Hkv: int, k: int, D_: int = D) -> int:
    a = _abi.DecodeArgs()
    a.B, a.Hq, a.Hkv, a.k, a.D = B, Hq, Hkv, k, D_
    return int(lib().msa_sparse_attn_decode_workspace_size(C.byref(a)))


def msa_sparse_attn_decode(Q, K_pool, V_pool, pt, n, last_len, O, LSE, ws: torch.Tensor, *,
                           softmax_scale: float = 0.0, dev_err=None, stream=None,
                           scratch_zeroed: bool = False) -> None:
    """Paged sparse attention of one decode step over the flattened page table (see msa.h, a5-a6).

    The workspace's row counters are cleared by the call unless ``scratch_zeroed``
    says they are already zero (every error-free call leaves them zero)."""
    if not (pt.is_contiguous() and n.is_contiguous() and last_len.is_contiguous() and O.is_contiguous()):
        raise ValueError("pt, n, last_len and O must be contiguous")
    a = _decode_args(Q, K_pool, V_pool, pt, n, last_len, O, LSE, softmax_scale, dev_err)
    a.scratch_zeroed = int(bool(scratch_zeroed))
    _abi.check(lib().msa_sparse_attn_decode(C.byref(a), _ptr(ws), ws.numel() * ws.element_size(),
                                            _stream(stream)), "msa_sparse_attn_decode")


def msa_sparse_attn_decode_noalloc(Q, K_pool, V_pool, pt, n, last_len, O, LSE, *, softmax_scale: float = 0.0,
                                   dev_err=None, stream=None) -> None:
    """Same as msa_sparse_attn_decode, for callers that cannot allocate: the
    scratch is the library's built-in device array (see msa.h).  Calls that
    overlap on the GPU share that array and must be serialised."""
    if not (pt.is_contiguous() and n.is_contiguous() and last_len.is_contiguous() and O.is_contiguous()):
        raise ValueError("pt, n, last_len and O must be contiguous")
    a = _decode_args(Q, K_pool, V_pool, pt, n, last_len, O, LSE, softmax_scale, dev_err)
    _abi.check(lib().msa_sparse_attn_decode_noalloc(C.byref(a), _stream(stream)), "msa_sparse_attn_decode_noalloc")


def msa_lse_merge(O_part: torch.Tensor, LSE_part: torch.Tensor, O: torch.Tensor, LSE: Optional[torch.Tensor] = None,
                  *, dev_err=None, stream=None) -> None:
    """O [rows, D] bf16, LSE [rows] from O_part [rows, parts, D] fp32, LSE_part [rows, parts] (see msa.h, a6)."""
    rows, parts, d = O_part.shape
    for t, nm in ((O_part, "O_part"), (LSE_part, "LSE_part"), (O, "O")):
        if not t.is_contiguous():
            raise ValueError(f"{nm} must be contiguous")
    _abi.check(lib().msa_lse_merge(_ptr(O_part), _ptr(LSE_part), rows, parts, d, _ptr(O), _ptr(LSE),
                                   _ptr(dev_err), _stream(stream)), "msa_lse_merge")


# ---------------------------------------------------------------------------
# dense comparator (no index branch, no selection)
# ---------------------------------------------------------------------------

def _dense_decode_args(Q, K_pool, V_pool, seq_pt, seq_len, O, LSE, softmax_scale, dev_err) -> _abi.DenseDecodeArgs:
    for t, nm in ((Q, "Q"), (K_pool, "K_pool"), (V_pool, "V_pool")):
        _inner_contig(t, nm)
    if K_pool.stride() != V_pool.stride():
        raise ValueError("K_pool and V_pool must share strides")
    if not seq_pt.is_contiguous():
        raise ValueError("seq_pt must be contiguous")
    a = _abi.DenseDecodeArgs()
    a.B, a.Hq, a.D = Q.shape
    a.Hkv, a.Bk = K_pool.shape[1], K_pool.shape[2]
    a.softmax_scale = softmax_scale
    a.Q = _ptr(Q)
    a.Q_stride[:] = _strides(Q, 2)
    a.K_pool, a.V_pool = _ptr(K_pool), _ptr(V_pool)
    a.kv_stride[:] = _strides(K_pool, 3)
    a.num_pages = K_pool.shape[0]
    a.seq_pt, a.max_pages, a.seq_len = _ptr(seq_pt), seq_pt.shape[1], _ptr(seq_len)
    a.O, a.LSE, a.dev_err = _ptr(O), _ptr(LSE), _ptr(dev_err)
    return a


def msa_dense_attn_decode_workspace_size(B: int, Hq: int, Hkv: int, max_pages: int) -> int:
    a = _abi.DenseDecodeArgs()
    a.B, a.Hq, a.Hkv, a.D, a.Bk, a.max_pages = B, Hq, Hkv, D, Bk, max_pages
    return int(lib().msa_dense_attn_decode_workspace_size(C.byref(a)))


def msa_dense_attn_decode(Q, K_pool, V_pool, seq_pt, seq_len, O, LSE, ws: torch.Tensor, *,
                          softmax_scale: float = 0.0, dev_err=None, stream=None, scratch_zeroed: bool = False) -> None:
    """Dense comparator of a decode step: every cached token of each sequence (see msa.h)."""
    if not O.is_contiguous():
        raise ValueError("O must be contiguous")
    a = _dense_decode_args(Q, K_pool, V_pool, seq_pt, seq_len, O, LSE, softmax_scale, dev_err)
    a.scratch_zeroed = int(bool(scratch_zeroed))
    _abi.check(lib().msa_dense_attn_decode(C.byref(a), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
               "msa_dense_attn_decode")


def dense_decode_buffers(B: int, Hq: int, Hkv: int, max_pages: int, device) -> Dict[str, torch.Tensor]:
    """Outputs and zero-filled scratch of ``dense_decode_step``."""
    dev = torch.device(device)
    return {
        "O": torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev),
        "LSE": torch.empty(B, Hq, dtype=torch.float32, device=dev),
        "ws": torch.zeros(msa_dense_attn_decode_workspace_size(B, Hq, Hkv, max_pages) // 4 + 64, dtype=torch.float32,
                          device=dev),
        "dev_err": torch.zeros(1, dtype=torch.int32, device=dev),
    }


def dense_decode_step(inp: Dict[str, torch.Tensor], bufs: Optional[Dict[str, torch.Tensor]] = None,
                      softmax_scale: float = 0.0, stream=None, scratch_zeroed: bool = False
                      ) -> Dict[str, torch.Tensor]:
    """The dense comparator of ``decode_step``: attention over every cached token (no index branch)."""
    B, Hq, _ = inp["Q"].shape
    Hkv = inp["K_pool"].shape[1]
    if bufs is None:
        bufs = dense_decode_buffers(B, Hq, Hkv, inp["seq_pt"].shape[1], inp["Q"].device)
    msa_dense_attn_decode(inp["Q"], inp["K_pool"], inp["V_pool"], inp["seq_pt"], inp["seq_len"], bufs["O"],
                          bufs["LSE"], bufs["ws"], softmax_scale=softmax_scale, dev_err=bufs["dev_err"],
                          stream=stream, scratch_zeroed=scratch_zeroed)
    return bufs


def msa_dense_attn_prefill(Q, K, V, O, LSE, *, softmax_scale: float = 0.0, dev_err=None, stream=None) -> None:
    """Dense comparator of a prefill layer: causal GQA attention over every earlier token (see msa.h).

    Q [B,S,Hq,D], K, V [B,S,Hkv,D] bf16; O [B,S,Hq,D] bf16 and LSE [B,S,Hq] fp32 (dense)."""
    for t, nm in ((Q, "Q"), (K, "K"), (V, "V")):
        _inner_contig(t, nm)
    if not O.is_contiguous() or (LSE is not None and not LSE.is_contiguous()):
        raise ValueError("O and LSE must be contiguous")
    a = _abi.DensePrefillArgs()
    a.B, a.S, a.Hq, a.D = Q.shape
    a.Hkv = K.shape[2]
    a.softmax_scale = softmax_scale
    a.Q, a.K, a.V = _ptr(Q), _ptr(K), _ptr(V)
    a.Q_stride[:] = _strides(Q, 3)
    a.K_stride[:] = _strides(K, 3)
    a.V_stride[:] = _strides(V, 3)
    a.O, a.LSE, a.dev_err = _ptr(O), _ptr(LSE), _ptr(dev_err)
    _abi.check(lib().msa_dense_attn_prefill(C.byref(a), _stream(stream)), "msa_dense_attn_prefill")


def dense_prefill_layer(inp: Dict[str, torch.Tensor], bufs: Optional[Dict[str, torch.Tensor]] = None,
                        softmax_scale: float = 0.0, stream=None) -> Dict[str, torch.Tensor]:
    """The dense comparator of ``prefill_layer``: causal attention over every earlier token (no index branch)."""
    B, S, Hq, _ = inp["Q"].shape
    if bufs is None:
        dev = inp["Q"].device
        bufs = {"O": torch.empty(B, S, Hq, D, dtype=torch.bfloat16, device=dev),
                "LSE": torch.empty(B, S, Hq, dtype=torch.float32, device=dev),
                "dev_err": torch.zeros(1, dtype=torch.int32, device=dev)}
    msa_dense_attn_prefill(inp["Q"], inp["K"], inp["V"], bufs["O"], bufs["LSE"], softmax_scale=softmax_scale,
                           dev_err=bufs["dev_err"], stream=stream)
    return bufs


# ---------------------------------------------------------------------------
# the step before a decode step: append the current tokens to the paged caches
# ---------------------------------------------------------------------------

def msa_cache_append(K_new: torch.Tensor, V_new: torch.Tensor, kidx_new: torch.Tensor, K_pool: torch.Tensor,
                     V_pool: torch.Tensor, kidx_pool: torch.Tensor, seq_pt: torch.Tensor, seq_len: torch.Tensor,
                     *, dev_err=None, stream=None) -> None:
    """Writes token L_b - 1 of every sequence into its page (see msa.h, cache append).

    K_new, V_new [B,Hkv,D], kidx_new [B,Hkv,dI] bf16; K_pool, V_pool [P,Hkv,Bk,D] and
    kidx_pool [P,Hkv,Bk,dI] bf16; seq_pt [B,max_pages] int32 (contiguous rows), seq_len [B].
    With 4-D K_new, V_new [B,T,Hkv,D] and kidx_new [B,T,Hkv,dI] the T tokens of each
    sequence go to positions L_b - T .. L_b - 1.
    """
    for t, nm in ((K_new, "K_new"), (V_new, "V_new"), (kidx_new, "kidx_new"), (K_pool, "K_pool"),
                  (V_pool, "V_pool"), (kidx_pool, "kidx_pool")):
        _inner_contig(t, nm)
    if K_pool.stride() != V_pool.stride():
        raise ValueError("K_pool and V_pool must share strides")
    if not seq_pt.is_contiguous():
        raise ValueError("seq_pt must be contiguous")
    a = _abi.AppendArgs()
    if K_new.dim() == 4:   # several tokens per sequence: strides (b, u, g)
        a.B, a.T, a.Hkv, a.D = K_new.shape
        a.new_t_stride[:] = [K_new.stride(1), V_new.stride(1), kidx_new.stride(1)]
        K_new_bg = [K_new.stride(0), K_new.stride(2)]
        V_new_bg = [V_new.stride(0), V_new.stride(2)]
        X_new_bg = [kidx_new.stride(0), kidx_new.stride(2)]
    else:
        a.B, a.Hkv, a.D = K_new.shape
        a.T = 1
        K_new_bg, V_new_bg, X_new_bg = _strides(K_new, 2), _strides(V_new, 2), _strides(kidx_new, 2)
    a.dI, a.Bk = kidx_new.shape[-1], K_pool.shape[2]
    a.K_new, a.V_new, a.kidx_new = _ptr(K_new), _ptr(V_new), _ptr(kidx_new)
    a.K_new_stride[:] = K_new_bg
    a.V_new_stride[:] = V_new_bg
    a.kidx_new_stride[:] = X_new_bg
    a.K_pool, a.V_pool, a.kidx_pool = _ptr(K_pool), _ptr(V_pool), _ptr(kidx_pool)
    a.kv_stride[:] = _strides(K_pool, 3)
    a.kidx_stride[:] = _strides(kidx_pool, 3)
    a.num_pages = K_pool.shape[0]
    a.seq_pt, a.max_pages, a.seq_len = _ptr(seq_pt), seq_pt.shape[1], _ptr(seq_len)
    a.dev_err = _ptr(dev_err)
    _abi.check(lib().msa_cache_append(C.byref(a), _stream(stream)), "msa_cache_append")


# ---------------------------------------------------------------------------
# pipelines (hot-path order; marshalling and buffer allocation only)
# ---------------------------------------------------------------------------

def decode_buffers(B: int, Hq: int, Hkv: int, k: int, nb_stride: int, device) -> Dict[str, torch.Tensor]:
    """Output and scratch buffers of one decode step (allocated by torch, owned by the caller).

    The scratch (``ws``, ``row_scratch``) is zero-filled, so calls may pass
    ``scratch_zeroed=True`` from the first one on."""
    dev = torch.device(device)
    return {
        "C": torch.empty(B, Hkv, nb_stride, dtype=torch.float32, device=dev),
        "sel": torch.empty(B, Hkv, k, dtype=torch.int32, device=dev),
        "count": torch.empty(B, Hkv, dtype=torch.int32, device=dev),
        "pt": torch.empty(B * Hkv, k, dtype=torch.int32, device=dev),
        "n": torch.empty(B * Hkv, dtype=torch.int32, device=dev),
        "last_len": torch.empty(B * Hkv, dtype=torch.int32, device=dev),
        "O": torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev),
        "LSE": torch.empty(B, Hq, dtype=torch.float32, device=dev),
        "ws": torch.zeros(msa_sparse_attn_decode_workspace_size(B, Hq, Hkv, k) // 4 + 64, dtype=torch.float32,
                          device=dev),
        "row_scratch": torch.zeros(B * Hkv, dtype=torch.int32, device=dev),
        "dev_err": torch.zeros(1, dtype=torch.int32, device=dev),
    }


def decode_step(inp: Dict[str, torch.Tensor], k: int, bufs: Optional[Dict[str, torch.Tensor]] = None,
                softmax_scale: float = 0.0, stream=None, fused: bool = True,
                scratch_zeroed: bool = False) -> Dict[str, torch.Tensor]:
    """One MSA decode step: a1 index score -> a2 top-k -> a3 page table -> a5/a6 attention.

    ``inp`` holds Q, q_idx, w, kidx_pool, K_pool, V_pool, seq_pt, seq_len (device tensors).
    With ``fused`` (default) a1-a3 run in one index-score call; otherwise the
    four entry points are called one by one.  ``scratch_zeroed`` skips the
    counter clears (valid with ``decode_buffers`` scratch that every previous
    call left zero, i.e. no device error was raised).
    """
    B, Hq, _ = inp["Q"].shape
    Hkv = inp["K_pool"].shape[1]
    if bufs is None:
        bufs = decode_buffers(B, Hq, Hkv, k, inp["seq_pt"].shape[1], inp["Q"].device)
    e = bufs["dev_err"]
    if fused:
        msa_index_score(MSA_MODE_DECODE, inp["q_idx"], inp["w"], inp["kidx_pool"], bufs["C"], seq_pt=inp["seq_pt"],
                        seq_len=inp["seq_len"], dev_err=e, stream=stream, k=k, sel=bufs["sel"],
                        count=bufs["count"], pt=bufs["pt"], n=bufs["n"], last_len=bufs["last_len"],
                        row_scratch=bufs["row_scratch"], scratch_zeroed=scratch_zeroed)
    else:
        msa_index_score(MSA_MODE_DECODE, inp["q_idx"], inp["w"], inp["kidx_pool"], bufs["C"], seq_pt=inp["seq_pt"],
                        seq_len=inp["seq_len"], dev_err=e, stream=stream)
        msa_topk_blocks(MSA_MODE_DECODE, bufs["C"], k, bufs["sel"], bufs["count"], seq_len=inp["seq_len"],
                        dev_err=e, stream=stream)
        msa_build_page_table(bufs["sel"], bufs["count"], inp["seq_pt"], inp["seq_len"], bufs["pt"], bufs["n"],
                             bufs["last_len"], dev_err=e, stream=stream)
    msa_sparse_attn_decode(inp["Q"], inp["K_pool"], inp["V_pool"], bufs["pt"], bufs["n"], bufs["last_len"],
                           bufs["O"], bufs["LSE"], bufs["ws"], softmax_scale=softmax_scale, dev_err=e,
                           stream=stream, scratch_zeroed=scratch_zeroed)
    return bufs


def prefill_buffers(B: int, S: int, Hq: int, Hkv: int, k: int, device, ws_bytes: int) -> Dict[str, torch.Tensor]:
    dev = torch.device(device)
    nb = (S + Bk - 1) // Bk
    return {
        "C": torch.empty(B, S, Hkv, nb, dtype=torch.float32, device=dev),
        "sel": torch.empty(B, S, Hkv, k, dtype=torch.int32, device=dev),
        "count": torch.empty(B, S, Hkv, dtype=torch.int32, device=dev),
        "O": torch.empty(B, S, Hq, D, dtype=torch.bfloat16, device=dev),
        "LSE": torch.empty(B, S, Hq, dtype=torch.float32, device=dev),
        "ws": torch.empty((ws_bytes + 15) // 16 * 4, dtype=torch.float32, device=dev),
        "dev_err": torch.zeros(1, dtype=torch.int32, device=dev),
    }


def prefill_layer(inp: Dict[str, torch.Tensor], k: int, bufs: Optional[Dict[str, torch.Tensor]] = None,
                  ws_bytes: Optional[int] = None, softmax_scale: float = 0.0, stream=None
                  ) -> Dict[str, torch.Tensor]:
    """One MSA prefill layer: a1 index score -> a2 top-k -> a3'/a4/a6 KV-block-major attention.

    ``inp`` holds Q, K, V, q_idx, k_idx, w (device tensors).
    """
    B, S, Hq, _ = inp["Q"].shape
    Hkv = inp["K"].shape[2]
    if bufs is None:
        if ws_bytes is None:
            sel_probe = torch.empty(1, 1, 1, k, dtype=torch.int32)
            ws_bytes = msa_sparse_attn_prefill_workspace_size(inp["Q"], inp["K"], sel_probe, min(S, 8192) * B)
        bufs = prefill_buffers(B, S, Hq, Hkv, k, inp["Q"].device, ws_bytes)
    e = bufs["dev_err"]
    msa_index_score(MSA_MODE_PREFILL, inp["q_idx"], inp["w"], inp["k_idx"], bufs["C"], dev_err=e, stream=stream)
    msa_topk_blocks(MSA_MODE_PREFILL, bufs["C"], k, bufs["sel"], bufs["count"], dev_err=e, stream=stream)
    msa_sparse_attn_prefill(inp["Q"], inp["K"], inp["V"], bufs["sel"], bufs["count"], bufs["O"], bufs["LSE"],
                            bufs["ws"], softmax_scale=softmax_scale, dev_err=e, stream=stream)
    return bufs


def chunk_buffers(B: int, S: int, Hq: int, Hkv: int, k: int, nb: int, device, ws_bytes: int
                  ) -> Dict[str, torch.Tensor]:
    """Outputs and scratch of ``chunk_layer`` (score rows of ``nb`` blocks)."""
    bufs = prefill_buffers(B, S, Hq, Hkv, k, device, ws_bytes)
    bufs["C"] = torch.empty(B, S, Hkv, nb, dtype=torch.float32, device=torch.device(device))
    return bufs


def chunk_layer(inp: Dict[str, torch.Tensor], k: int, bufs: Optional[Dict[str, torch.Tensor]] = None,
                ws_bytes: Optional[int] = None, softmax_scale: float = 0.0, stream=None
                ) -> Dict[str, torch.Tensor]:
    """One MSA layer over a chunk of S queries per sequence on a paged cache
    (chunked prefill over a cached prefix, or several decode tokens per
    sequence): a1 index score -> a2 top-k -> a3'/a4/a6 KV-block-major attention.

    ``inp`` holds Q [B,S,Hq,D], q_idx [B,S,Hkv,HI,dI], w [B,S,Hkv,HI], the page
    pools K_pool, V_pool [P,Hkv,Bk,D] and kidx_pool [P,Hkv,Bk,dI], seq_pt
    [B,max_pages] and q_pos [B] int32 (the chunk's own tokens already in the
    pages).  Score rows span max_pages blocks unless ``bufs`` says otherwise.
    """
    B, S, Hq, _ = inp["Q"].shape
    Hkv = inp["K_pool"].shape[1]
    max_pages = inp["seq_pt"].shape[1]
    if bufs is None:
        if ws_bytes is None:
            sel_probe = torch.empty(1, 1, 1, k, dtype=torch.int32)
            ws_bytes = msa_sparse_attn_prefill_workspace_size(inp["Q"], inp["K_pool"], sel_probe,
                                                              min(S, 8192) * B, max_pages=max_pages)
        bufs = chunk_buffers(B, S, Hq, Hkv, k, max_pages, inp["Q"].device, ws_bytes)
    e = bufs["dev_err"]
    msa_index_score(MSA_MODE_CHUNK, inp["q_idx"], inp["w"], inp["kidx_pool"], bufs["C"], seq_pt=inp["seq_pt"],
                    q_pos=inp["q_pos"], dev_err=e, stream=stream)
    msa_topk_blocks(MSA_MODE_CHUNK, bufs["C"], k, bufs["sel"], bufs["count"], q_pos=inp["q_pos"], dev_err=e,
                    stream=stream)
    msa_sparse_attn_prefill(inp["Q"], inp["K_pool"], inp["V_pool"], bufs["sel"], bufs["count"], bufs["O"],
                            bufs["LSE"], bufs["ws"], softmax_scale=softmax_scale, dev_err=e, stream=stream,
                            seq_pt=inp["seq_pt"], q_pos=inp["q_pos"])
    return bufs
