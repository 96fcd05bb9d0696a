"""fp64 CPU oracle of the MSA hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference arms may import this package.  The product path (the CUDA library
and its Python binding) never imports, links or calls anything here, and this
package never touches the CUDA path.

The arithmetic lives in ``msa_oracle.c`` (plain C, fp64, OpenMP over rows);
this module builds it with gcc and marshals numpy arrays in and out.  bf16
inputs are passed as their raw 16-bit patterns and widened exactly in C.

Functions and the passages they follow (page title and passage):

* ``prefill_scores`` / ``decode_scores`` -- block scores of the Index Branch
  ("MiniMax M3: Como la atencion dispersa hace practicos a los agentes de largo
  alcance", MSA paragraph and figure caption); the pages print no formula, the
  library and this oracle both take:
  s_t = sum_h w_h ReLU(q_idx_h . k_idx_t), c_j = max over block j.
* ``select`` -- own block + top-(k-1) earlier blocks by (score desc, index asc)
  (same page, bullet "Costo predecible": Bk = 128, k = 16).
* ``prefill_attend`` / ``decode_attend`` -- exact softmax attention over the
  selected blocks' uncompressed K/V (M2-report article, section "MiniMax Sparse
  Attention (MSA) y escalado subcuadratico entrante").
* ``lse_merge`` -- log-sum-exp recombination of per-block partials (M3 serving
  report post, paragraph "KV-Block-Major").
* ``page_table`` -- decode page table from the selected blocks with the KV
  group flattened into the batch (same post, paragraph "MSA con paged
  attention").
* ``cache_append`` -- the step before a decode step: the current token's K, V
  and index key written into the fixed-size pages (same paragraph; the token
  is in the cache before the step).  Plain numpy copies.
* ``chunk_layer`` -- a chunk of S queries per sequence over a paged cache:
  chunked prefill after a cached prefix ("MiniMax M3: MoE de 428B con 1M de
  contexto en Blackwell", section "Como se sirve en inferencia open source?",
  the serving command's 8,192-token prefill chunks; the serving post's
  measurement paragraph, a 60,000-token cached prefix), and with a small S the
  decode of several tokens per sequence (the M2-report article names
  multi-token prediction for speculative decoding).  No new arithmetic: a
  chunk query at position p sees exactly what a decode query of a sequence of
  length p + 1 sees over the same pages, so query offset s of every sequence
  is one call of the decode step functions above with lengths q_pos[b] + s + 1.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "msa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile msa_oracle.c into liboracle.so with gcc (-O2, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_i, _l, _d = C.c_int, C.c_int64, C.c_double


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = C.CDLL(_LIB)
            L.orc_num_threads.restype = _i
            L.orc_set_num_threads.argtypes = [_i]
            L.orc_prefill_scores.argtypes = [_i, _i, _i, _i, _i, _i, _u16p, _u16p, _f32p,
                                             _l, _i64p, _i, _f64p]
            L.orc_decode_scores.argtypes = [_i, _i, _i, _i, _i, _u16p, _f32p, _u16p,
                                            _i32p, _i, _i32p, _i, _f64p]
            L.orc_select.argtypes = [_l, _i, _f64p, _i32p, _i, _i32p, _i32p, _f64p, _f64p]
            L.orc_prefill_attend.argtypes = [_i, _i, _i, _i, _i, _i, _d, _u16p, _u16p, _u16p,
                                             _l, _i64p, _i, _i32p, _i32p, _f64p, _f64p]
            L.orc_decode_attend.argtypes = [_i, _i, _i, _i, _i, _d, _u16p, _u16p, _u16p,
                                            _i32p, _i, _i32p, _i, _i32p, _i32p, _f64p, _f64p]
            L.orc_lse_merge.argtypes = [_l, _i, _i, _f64p, _f64p, _f64p, _f64p]
            L.orc_page_table.argtypes = [_i, _i, _i, _i, _i32p, _i32p, _i32p, _i, _i32p,
                                         _i32p, _i32p, _i32p]
            _lib = L
    return _lib


def num_threads() -> int:
    return lib().orc_num_threads()


def set_num_threads(n: int) -> None:
    lib().orc_set_num_threads(int(n))


# ---------------------------------------------------------------------------
# marshalling helpers (no arithmetic of the method)
# ---------------------------------------------------------------------------

def _np(t):
    """torch tensor or array -> contiguous numpy array on the host."""
    if hasattr(t, "detach"):
        import torch
        t = t.detach()
        if t.dtype == torch.bfloat16:
            return np.ascontiguousarray(t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16))
        return np.ascontiguousarray(t.cpu().contiguous().numpy())
    return np.ascontiguousarray(t)


def _u16(t):
    a = _np(t)
    assert a.dtype == np.uint16, a.dtype
    return a


def _f32(t):
    return np.ascontiguousarray(_np(t), dtype=np.float32)


def _i32(t):
    return np.ascontiguousarray(_np(t), dtype=np.int32)


def _i64(t):
    return np.ascontiguousarray(_np(t), dtype=np.int64)


# ---------------------------------------------------------------------------
# step functions
# ---------------------------------------------------------------------------

def prefill_scores(q_idx, k_idx, w, Bk: int, rows=None):
    """Block scores C [nrows, Hkv, nb] (fp64) for prefill query rows b*S + i."""
    qi, ki, ww = _u16(q_idx), _u16(k_idx), _f32(w)
    B, S, Hkv, HI, dI = qi.shape
    nb = (S + Bk - 1) // Bk
    rows = np.arange(B * S, dtype=np.int64) if rows is None else _i64(rows)
    out = np.empty((len(rows), Hkv, nb), dtype=np.float64)
    lib().orc_prefill_scores(B, S, Hkv, HI, dI, Bk, qi, ki, ww, len(rows), rows, nb, out)
    return out


def decode_scores(q_idx, w, kidx_pool, seq_pt, seq_len, nb_stride: int = None):
    """Block scores C [B, Hkv, nb_stride] (fp64) of one decode step over paged k_idx."""
    qi, ww, kp = _u16(q_idx), _f32(w), _u16(kidx_pool)
    pt, sl = _i32(seq_pt), _i32(seq_len)
    B, Hkv, HI, dI = qi.shape
    Bk = kp.shape[2]
    nb_stride = pt.shape[1] if nb_stride is None else nb_stride
    out = np.empty((B, Hkv, nb_stride), dtype=np.float64)
    lib().orc_decode_scores(B, Hkv, HI, dI, Bk, qi, ww, kp, pt, pt.shape[1], sl, nb_stride, out)
    return out


def select(Cs, own, k: int):
    """Selection per row of scores.  Cs [..., nb] fp64, own [...] int.

    Returns (sel [..., k] int32 ascending, -1 padded; count [...] int32;
    c_last [...]; c_next [...]) where c_last / c_next are the scores of the last
    kept and first dropped earlier block (NaN when nothing is dropped).
    """
    Cs = np.ascontiguousarray(Cs, dtype=np.float64)
    lead = Cs.shape[:-1]
    nb = Cs.shape[-1]
    flat = Cs.reshape(-1, nb)
    o = np.ascontiguousarray(np.broadcast_to(np.asarray(own, dtype=np.int32), lead).reshape(-1))
    n = flat.shape[0]
    sel = np.empty((n, k), dtype=np.int32)
    cnt = np.empty(n, dtype=np.int32)
    cl = np.empty(n, dtype=np.float64)
    cn = np.empty(n, dtype=np.float64)
    lib().orc_select(n, nb, flat, o, k, sel, cnt, cl, cn)
    return sel.reshape(*lead, k), cnt.reshape(lead), cl.reshape(lead), cn.reshape(lead)


def prefill_attend(Q, K, V, sel, count, Bk: int, scale: float, rows=None):
    """Sparse attention for prefill rows with a given selection.

    sel [nrows, Hkv, k], count [nrows, Hkv].  Returns O [nrows, Hq, D], LSE [nrows, Hq].
    """
    q, kk, vv = _u16(Q), _u16(K), _u16(V)
    B, S, Hq, D = q.shape
    Hkv = kk.shape[2]
    rows = np.arange(B * S, dtype=np.int64) if rows is None else _i64(rows)
    s, c = _i32(sel), _i32(count)
    k = s.shape[-1]
    assert s.shape == (len(rows), Hkv, k) and c.shape == (len(rows), Hkv)
    O = np.empty((len(rows), Hq, D), dtype=np.float64)
    LSE = np.empty((len(rows), Hq), dtype=np.float64)
    lib().orc_prefill_attend(B, S, Hq, Hkv, D, Bk, float(scale), q, kk, vv, len(rows), rows, k,
                             s, c, O, LSE)
    return O, LSE


def decode_attend(Q, K_pool, V_pool, seq_pt, seq_len, sel, count, scale: float):
    """Sparse attention of one decode step.  Returns O [B, Hq, D], LSE [B, Hq]."""
    q, kp, vp = _u16(Q), _u16(K_pool), _u16(V_pool)
    pt, sl, s, c = _i32(seq_pt), _i32(seq_len), _i32(sel), _i32(count)
    B, Hq, D = q.shape
    Hkv, Bk = kp.shape[1], kp.shape[2]
    k = s.shape[-1]
    O = np.empty((B, Hq, D), dtype=np.float64)
    LSE = np.empty((B, Hq), dtype=np.float64)
    lib().orc_decode_attend(B, Hq, Hkv, D, Bk, float(scale), q, kp, vp, pt, pt.shape[1], sl, k,
                            s, c, O, LSE)
    return O, LSE


def lse_merge(Op, LSEp):
    """Merge partials Op [rows, parts, D], LSEp [rows, parts] -> O [rows, D], LSE [rows]."""
    op = np.ascontiguousarray(Op, dtype=np.float64)
    lp = np.ascontiguousarray(LSEp, dtype=np.float64)
    rows, parts, D = op.shape
    O = np.empty((rows, D), dtype=np.float64)
    LSE = np.empty(rows, dtype=np.float64)
    lib().orc_lse_merge(rows, parts, D, op, lp, O, LSE)
    return O, LSE


def page_table(sel, count, seq_pt, seq_len, Bk: int):
    """Decode page table rows r = b*Hkv + g: (pt [B*Hkv, k], n [B*Hkv], last_len [B*Hkv])."""
    s, c, pt, sl = _i32(sel), _i32(count), _i32(seq_pt), _i32(seq_len)
    B, Hkv, k = s.shape
    out_pt = np.empty((B * Hkv, k), dtype=np.int32)
    n = np.empty(B * Hkv, dtype=np.int32)
    ll = np.empty(B * Hkv, dtype=np.int32)
    lib().orc_page_table(B, Hkv, k, Bk, s, c, pt, pt.shape[1], sl, out_pt, n, ll)
    return out_pt, n, ll


def own_blocks_prefill(S: int, Bk: int, rows):
    """Own block b_i = floor(i / Bk) of prefill rows b*S + i (index bookkeeping)."""
    r = _i64(rows)
    return ((r % S) // Bk).astype(np.int32)


def own_blocks_decode(seq_len, Bk: int):
    """Own block (L_b - 1) // Bk of each decode sequence (index bookkeeping)."""
    return ((_i64(seq_len) - 1) // Bk).astype(np.int32)


def cache_append(K_new, V_new, kidx_new, K_pool, V_pool, kidx_pool, seq_pt, seq_len, Bk: int,
                 shared_index: bool = False):
    """The three pools after the new tokens of every sequence b are written into
    their page slots (raw 16-bit patterns, copies; the inputs are not
    modified).  K_new [B, Hkv, D] is one token per sequence, at position
    L_b - 1; K_new [B, T, Hkv, D] is T tokens, token u at position L_b - T + u.
    Position p is slot p % Bk of page seq_pt[b][p // Bk].  A sequence whose
    length is below T or outside [1, max_pages * Bk] is left out, and so is a
    token whose page id is outside the pool; ``skipped`` lists the sequences
    (one token) or the (b, u) tokens (several) left out.  With
    ``shared_index`` the index-key pool is one pool for all groups and takes
    group 0's key."""
    K, V, X = _u16(K_pool).copy(), _u16(V_pool).copy(), _u16(kidx_pool).copy()
    kn, vn, xn = _u16(K_new), _u16(V_new), _u16(kidx_new)
    one = kn.ndim == 3
    if one:
        kn, vn, xn = kn[:, None], vn[:, None], xn[:, None]
    pt, sl = _i32(seq_pt), _i32(seq_len)
    P, max_pages = K.shape[0], pt.shape[1]
    T = kn.shape[1]
    skipped = []
    for b in range(sl.shape[0]):
        L = int(sl[b])
        if L < T or L < 1 or L > max_pages * Bk:
            skipped += [b] if one else [(b, u) for u in range(T)]
            continue
        for u in range(T):
            pos = L - T + u
            page = int(pt[b, pos // Bk])
            if page < 0 or page >= P:
                skipped.append(b if one else (b, u))
                continue
            t = pos % Bk
            K[page, :, t, :] = kn[b, u]
            V[page, :, t, :] = vn[b, u]
            X[page, :, t, :] = xn[b, u] if not shared_index else xn[b, u, 0]
    return K, V, X, skipped


def chunk_scores(q_idx, w, kidx_pool, seq_pt, q_pos, Bk: int = 128):
    """Block scores C [B, S, Hkv, nbT] (fp64) of a chunk's queries at positions
    q_pos[b] + s over the paged index keys (nbT = blocks of the longest
    context): offset s is the decode score of a sequence of length q_pos[b] + s + 1."""
    qi, ww, qp = _u16(q_idx), _f32(w), _i64(q_pos)
    B, S = qi.shape[:2]
    nbT = int(((qp + S - 1) // Bk).max()) + 1
    return np.stack([decode_scores(qi[:, s], ww[:, s], kidx_pool, seq_pt, (qp + s + 1).astype(np.int32), nbT)
                     for s in range(S)], axis=1)


def chunk_own_blocks(q_pos, S: int, Bk: int = 128):
    """Own block (q_pos[b] + s) // Bk of each chunk query, [B, S] (index bookkeeping)."""
    qp = _i64(q_pos)
    return ((qp[:, None] + np.arange(S)[None, :]) // Bk).astype(np.int32)


def chunk_attend(Q, K_pool, V_pool, seq_pt, q_pos, sel, count, scale: float, Bk: int = 128):
    """Attention of a chunk's queries over the given selection (sel [B,S,Hkv,k],
    count [B,S,Hkv]): offset s is the decode attention of a sequence of length
    q_pos[b] + s + 1.  Returns O [B,S,Hq,D], LSE [B,S,Hq] (fp64)."""
    q, qp, sl, c = _u16(Q), _i64(q_pos), _i32(sel), _i32(count)
    S = q.shape[1]
    outs = [decode_attend(q[:, s], K_pool, V_pool, seq_pt, (qp + s + 1).astype(np.int32), sl[:, s], c[:, s], scale)
            for s in range(S)]
    return np.stack([o for o, _ in outs], axis=1), np.stack([l for _, l in outs], axis=1)


def chunk_layer(Q, q_idx, w, K_pool, V_pool, kidx_pool, seq_pt, q_pos, k: int, scale: float, Bk: int = 128):
    """Index scores, selection and attention of a chunk of S queries per
    sequence at positions q_pos[b] + s over a paged cache holding each
    sequence's q_pos[b] + S tokens.

    Q [B,S,Hq,D], q_idx [B,S,Hkv,HI,dI] (bf16), w [B,S,Hkv,HI] fp32, pools
    [P,Hkv,Bk,*], seq_pt [B,max_pages], q_pos [B].  Returns a dict with C
    [B,S,Hkv,nbT] (nbT = blocks of the longest context), sel [B,S,Hkv,k],
    count [B,S,Hkv], c_last / c_next (as ``select``), O [B,S,Hq,D] and LSE
    [B,S,Hq] (fp64).
    """
    Cs = chunk_scores(q_idx, w, kidx_pool, seq_pt, q_pos, Bk)
    B, S, Hkv = Cs.shape[:3]
    own = np.repeat(chunk_own_blocks(q_pos, S, Bk)[..., None], Hkv, axis=2)
    sel, cnt, cl, cn = select(Cs, own, k)
    O, LSE = chunk_attend(Q, K_pool, V_pool, seq_pt, q_pos, sel, cnt, scale, Bk)
    return {"C": Cs, "sel": sel, "count": cnt, "c_last": cl, "c_next": cn, "O": O, "LSE": LSE}
