"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each pin is chosen so that a plausible mistake in the oracle (a dropped term, a
wrong sign or index, a transposed operand, a wrong head-to-group map, an
off-by-one in causality or in the selection order) fails at least one test:

* dense limit   -- with k >= number of blocks MSA is dense causal GQA attention;
                   checked against a numpy matrix-form softmax and against
                   torch's fp64 scaled-dot-product attention.
* merge         -- LSE merge of a split softmax equals one softmax.
* top-k         -- selection equals an exhaustive sort by (-score, index).
* closed forms  -- one-hot index vectors give hand-derivable block scores;
                   one key gives O = V, LSE = z; equal keys give the mean of V.
* cross-path    -- decode at length L equals prefill row L-1; page order and
                   the flattened (B*Hkv) page table do not change the result;
                   a chunk over paged caches equals the same rows of a prefill
                   of the whole context, and a one-token chunk equals decode
                   (whose C code reads the pages itself).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from workloads import (ChunkWorkload, DecodeWorkload, MSAShape, PrefillWorkload, chunk_inputs, decode_inputs,
                       prefill_inputs, workload)


def f64(t):
    return t.detach().cpu().double().numpy()


def dense_causal_gqa_numpy(Q, K, V, scale):
    """Dense causal GQA attention in matrix form: softmax(scale Q K^T + mask) V."""
    q, k, v = f64(Q), f64(K), f64(V)
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    O = np.zeros((B, S, Hq, D))
    LSE = np.zeros((B, S, Hq))
    mask = np.triu(np.ones((S, S), dtype=bool), 1)
    for b in range(B):
        for hq in range(Hq):
            g = hq // G
            z = scale * q[b, :, hq, :] @ k[b, :, g, :].T
            z[mask] = -np.inf
            m = z.max(axis=1, keepdims=True)
            e = np.exp(z - m)
            l = e.sum(axis=1, keepdims=True)
            O[b, :, hq, :] = (e / l) @ v[b, :, g, :]
            LSE[b, :, hq] = (m + np.log(l))[:, 0]
    return O, LSE


def run_prefill_oracle(inp, sh, rows=None):
    B, S = inp["Q"].shape[:2]
    rows = np.arange(B * S, dtype=np.int64) if rows is None else rows
    C = oracle.prefill_scores(inp["q_idx"], inp["k_idx"], inp["w"], sh.Bk, rows)
    own = oracle.own_blocks_prefill(S, sh.Bk, rows)
    sel, cnt, _, _ = oracle.select(C, own[:, None], sh.k)
    O, LSE = oracle.prefill_attend(inp["Q"], inp["K"], inp["V"], sel, cnt, sh.Bk,
                                   1.0 / math.sqrt(sh.D), rows)
    return C, sel, cnt, O, LSE


# ---------------------------------------------------------------------------
# P1: dense limit
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("wl", [
    workload("prefill_tiny_s2048_k16"),
    # GQA with ragged tail: G = 3, two KV groups, S not a multiple of Bk
    PrefillWorkload("gqa_ragged", B=2, S=300, shape=MSAShape(Hq=6, Hkv=2, HI=2, k=3), seed=11),
])
def test_dense_limit_equals_causal_gqa(wl):
    sh = wl.shape
    assert sh.k >= wl.nb
    inp = prefill_inputs(wl)
    C, sel, cnt, O, LSE = run_prefill_oracle(inp, sh)
    B, S = wl.B, wl.S
    own = (np.arange(S) // sh.Bk)
    # every row keeps all blocks 0..b_i
    cnt = cnt.reshape(B, S, sh.Hkv)
    assert np.array_equal(cnt, np.broadcast_to((own + 1)[None, :, None], cnt.shape))
    Od, LSEd = dense_causal_gqa_numpy(inp["Q"], inp["K"], inp["V"], 1.0 / math.sqrt(sh.D))
    np.testing.assert_allclose(O.reshape(Od.shape), Od, rtol=0, atol=1e-12)
    np.testing.assert_allclose(LSE.reshape(LSEd.shape), LSEd, rtol=0, atol=1e-12)
    # second, independent check: torch fp64 SDPA with repeated KV heads
    G = sh.G
    q = inp["Q"].double().permute(0, 2, 1, 3)
    k = inp["K"].double().repeat_interleave(G, dim=2).permute(0, 2, 1, 3)
    v = inp["V"].double().repeat_interleave(G, dim=2).permute(0, 2, 1, 3)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True,
                                                           scale=1.0 / math.sqrt(sh.D))
    np.testing.assert_allclose(O.reshape(Od.shape), ref.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# P2: merge of a split softmax equals one softmax
# ---------------------------------------------------------------------------

def test_merge_equals_single_softmax():
    rng = np.random.default_rng(5)
    rows, n, D = 64, 300, 16
    z = rng.normal(size=(rows, n)) * 3.0
    Vv = rng.normal(size=(n, D))
    parts = 7
    Op = np.full((rows, parts, D), np.nan)     # empty parts hold garbage on purpose
    LSEp = np.full((rows, parts), -np.inf)
    for r in range(rows):
        # random cut points; some parts end up empty
        cuts = np.sort(rng.integers(0, n + 1, size=parts - 1))
        bounds = np.concatenate([[0], cuts, [n]])
        for p in range(parts):
            a, b = bounds[p], bounds[p + 1]
            if a == b:
                continue
            zz = z[r, a:b]
            m = zz.max()
            e = np.exp(zz - m)
            Op[r, p] = (e / e.sum()) @ Vv[a:b]
            LSEp[r, p] = m + np.log(e.sum())
    O, LSE = oracle.lse_merge(Op, LSEp)
    m = z.max(axis=1, keepdims=True)
    e = np.exp(z - m)
    np.testing.assert_allclose(O, (e / e.sum(axis=1, keepdims=True)) @ Vv, rtol=0, atol=1e-12)
    np.testing.assert_allclose(LSE, (m + np.log(e.sum(axis=1, keepdims=True)))[:, 0], rtol=0, atol=1e-12)


def test_merge_all_empty_row():
    O, LSE = oracle.lse_merge(np.full((1, 3, 4), np.nan), np.full((1, 3), -np.inf))
    assert np.all(O == 0) and LSE[0] == -np.inf


def test_attend_per_block_then_merge_equals_attend_all():
    """Attention restricted to each selected block, LSE-merged, equals attention over all of them."""
    wl = PrefillWorkload("split", B=1, S=700, shape=MSAShape(Hq=4, Hkv=2, HI=2, k=6), seed=21)
    sh = wl.shape
    inp = prefill_inputs(wl)
    rows = np.array([0, 127, 128, 350, 699], dtype=np.int64)
    C, sel, cnt, O, LSE = run_prefill_oracle(inp, sh, rows)
    k = sh.k
    Op = np.zeros((len(rows), sh.Hq, k, sh.D))
    LSEp = np.full((len(rows), sh.Hq, k), -np.inf)
    for s in range(k):
        sel1 = np.full_like(sel, -1)
        sel1[..., 0] = sel[..., s]
        cnt1 = (cnt > s).astype(np.int32)
        o1, l1 = oracle.prefill_attend(inp["Q"], inp["K"], inp["V"], sel1, cnt1, sh.Bk,
                                       1.0 / math.sqrt(sh.D), rows)
        Op[:, :, s] = o1
        LSEp[:, :, s] = l1
    Om, LSEm = oracle.lse_merge(Op.reshape(-1, k, sh.D), LSEp.reshape(-1, k))
    np.testing.assert_allclose(Om.reshape(O.shape), O, rtol=0, atol=1e-12)
    np.testing.assert_allclose(LSEm.reshape(LSE.shape), LSE, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# P3: selection equals an exhaustive sort
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("k", [1, 2, 4, 16])
def test_select_equals_exhaustive_sort(k):
    rng = np.random.default_rng(100 + k)
    rows, nb = 400, 40
    C = rng.integers(0, 8, size=(rows, nb)).astype(np.float64) / 8.0  # heavy ties
    own = rng.integers(0, nb, size=rows).astype(np.int32)
    sel, cnt, cl, cn = oracle.select(C, own, k)
    for r in range(rows):
        n = own[r]
        order = sorted(range(n), key=lambda j: (-C[r, j], j))
        keep = sorted(order[:k - 1]) + [n]
        assert cnt[r] == len(keep)
        assert list(sel[r, :cnt[r]]) == keep
        assert np.all(sel[r, cnt[r]:] == -1)
        if n > k - 1:
            if k >= 2:
                assert cl[r] == C[r, order[k - 2]]
            else:
                assert np.isnan(cl[r])
            assert cn[r] == C[r, order[k - 1]]
        else:
            assert np.isnan(cl[r]) and np.isnan(cn[r])


def test_select_ignores_future_and_own_scores():
    C = np.array([[0.1, 0.9, 0.5, 100.0, 200.0]])
    sel, cnt, _, _ = oracle.select(C, np.array([3], dtype=np.int32), 3)
    # candidates are blocks 0..2 only: top-2 = {1, 2}, plus own block 3
    assert list(sel[0]) == [1, 2, 3] and cnt[0] == 3


# ---------------------------------------------------------------------------
# P4: closed forms
# ---------------------------------------------------------------------------

def test_index_score_onehot_closed_form():
    """One-hot index vectors: q_idx_h = a_h e_{d_h}, k_idx_t = x_t e_{e_t}.

    Then q_idx_h . k_idx_t = a_h x_t [d_h == e_t] and
    s_t = sum_h w_h max(0, a_h x_t [d_h == e_t]).  Values are exact in bf16.
    """
    Bk, HI, dI = 4, 2, 64
    S = 3 * Bk
    q_idx = torch.zeros(1, S, 1, HI, dI, dtype=torch.bfloat16)
    k_idx = torch.zeros(1, S, 1, dI, dtype=torch.bfloat16)
    w = torch.zeros(1, S, 1, HI)
    i = S - 1                      # query in block 2: blocks 0 and 1 are scored
    q_idx[0, i, 0, 0, 3] = 1.0     # head 0 looks at dim 3 with a = 1
    q_idx[0, i, 0, 1, 5] = -2.0    # head 1 looks at dim 5 with a = -2
    w[0, i, 0] = torch.tensor([0.75, 0.5])
    tokens = {  # t: (dim, x)
        0: (3, 0.5), 1: (5, -1.0), 2: (3, -4.0), 3: (7, 8.0),      # block 0
        4: (5, 0.25), 5: (3, 0.125), 6: (5, -0.5), 7: (3, 0.25),   # block 1
        8: (3, 64.0), 9: (5, -64.0), 10: (3, 1.0), 11: (3, 1.0),   # own block (not scored)
    }
    for t, (d, x) in tokens.items():
        k_idx[0, t, 0, d] = x
    # hand derivation
    # block 0: t0: 0.75*max(0, 0.5) = 0.375; t1: 0.5*max(0, -2*-1) = 1.0;
    #          t2: 0.75*max(0, -4) = 0;       t3: dim 7 matches no head -> 0.   max = 1.0
    # block 1: t4: 0.5*max(0, -2*0.25) = 0;  t5: 0.75*0.125 = 0.09375;
    #          t6: 0.5*max(0, -2*-0.5) = 0.5; t7: 0.75*0.25 = 0.1875.           max = 0.5
    C = oracle.prefill_scores(q_idx, k_idx, w, Bk, rows=np.array([i]))
    assert C.shape == (1, 1, 3)
    assert C[0, 0, 0] == 1.0 and C[0, 0, 1] == 0.5 and C[0, 0, 2] == -np.inf


def test_index_score_negative_dots_contribute_zero():
    Bk, HI, dI = 2, 3, 64
    q_idx = torch.zeros(1, 4, 1, HI, dI, dtype=torch.bfloat16)
    k_idx = torch.zeros(1, 4, 1, dI, dtype=torch.bfloat16)
    w = torch.ones(1, 4, 1, HI)
    q_idx[0, 3, 0, :, 0] = torch.tensor([1.0, -1.0, 2.0])
    k_idx[0, 0, 0, 0] = 1.0    # dots (1, -1, 2): ReLU keeps 1 + 2 = 3
    k_idx[0, 1, 0, 0] = -1.0   # dots (-1, 1, -2): ReLU keeps 1
    C = oracle.prefill_scores(q_idx, k_idx, w, Bk, rows=np.array([3]))
    assert C[0, 0, 0] == 3.0


def test_attention_single_key_closed_form():
    """Query 0 sees only token 0: O = V_0, LSE = scale * Q_0 . K_0."""
    wl = PrefillWorkload("one", B=1, S=5, shape=MSAShape(Hq=4, Hkv=2, HI=2, k=2), seed=3)
    sh = wl.shape
    inp = prefill_inputs(wl)
    _, _, _, O, LSE = run_prefill_oracle(inp, sh, rows=np.array([0]))
    q, k, v = f64(inp["Q"]), f64(inp["K"]), f64(inp["V"])
    for hq in range(sh.Hq):
        g = hq // sh.G
        np.testing.assert_array_equal(O[0, hq], v[0, 0, g])
        z = sum(q[0, 0, hq, d] * k[0, 0, g, d] for d in range(sh.D)) / math.sqrt(sh.D)
        assert abs(LSE[0, hq] - z) < 1e-14


def test_attention_equal_keys_closed_form():
    """All keys equal: uniform weights, O = mean of V over t <= i, LSE = z + ln(i + 1)."""
    wl = PrefillWorkload("eq", B=1, S=300, shape=MSAShape(Hq=2, Hkv=1, HI=2, k=3), seed=4)
    sh = wl.shape
    inp = prefill_inputs(wl)
    inp["K"][:] = inp["K"][0, 0]
    rows = np.array([0, 1, 127, 128, 299], dtype=np.int64)
    _, _, _, O, LSE = run_prefill_oracle(inp, sh, rows)
    q, k, v = f64(inp["Q"]), f64(inp["K"]), f64(inp["V"])
    for r, i in enumerate(rows):
        for hq in range(sh.Hq):
            mean = v[0, :i + 1, 0].sum(axis=0) / (i + 1)
            np.testing.assert_allclose(O[r, hq], mean, rtol=0, atol=1e-13)
            z = float(np.dot(q[0, i, hq], k[0, 0, 0])) / math.sqrt(sh.D)
            assert abs(LSE[r, hq] - (z + math.log(i + 1))) < 1e-12


# ---------------------------------------------------------------------------
# P5: cross-path invariants
# ---------------------------------------------------------------------------

def _decode_from_prefill(inp, sh, b, L, perm_seed):
    """Page tokens 0..L-1 of prefill sequence b into a shuffled pool (tensor plumbing only)."""
    npg = (L + sh.Bk - 1) // sh.Bk
    perm = torch.randperm(npg, generator=torch.Generator().manual_seed(perm_seed))
    P = npg
    Kp = torch.zeros(P, sh.Hkv, sh.Bk, sh.D, dtype=torch.bfloat16)
    Vp = torch.zeros_like(Kp)
    KIp = torch.zeros(P, sh.Hkv, sh.Bk, sh.dI, dtype=torch.bfloat16)
    for j in range(npg):
        t0, t1 = j * sh.Bk, min(L, (j + 1) * sh.Bk)
        p = int(perm[j])
        Kp[p, :, :t1 - t0] = inp["K"][b, t0:t1].transpose(0, 1)
        Vp[p, :, :t1 - t0] = inp["V"][b, t0:t1].transpose(0, 1)
        KIp[p, :, :t1 - t0] = inp["k_idx"][b, t0:t1].transpose(0, 1)
    return {
        "Q": inp["Q"][b, L - 1][None].contiguous(),
        "q_idx": inp["q_idx"][b, L - 1][None].contiguous(),
        "w": inp["w"][b, L - 1][None].contiguous(),
        "K_pool": Kp, "V_pool": Vp, "kidx_pool": KIp,
        "seq_pt": perm.to(torch.int32)[None].contiguous(),
        "seq_len": torch.tensor([L], dtype=torch.int32),
    }


def run_decode_oracle(d, sh, nb_stride=None):
    C = oracle.decode_scores(d["q_idx"], d["w"], d["kidx_pool"], d["seq_pt"], d["seq_len"], nb_stride)
    own = oracle.own_blocks_decode(d["seq_len"], sh.Bk)
    sel, cnt, _, _ = oracle.select(C, own[:, None], sh.k)
    O, LSE = oracle.decode_attend(d["Q"], d["K_pool"], d["V_pool"], d["seq_pt"], d["seq_len"],
                                  sel, cnt, 1.0 / math.sqrt(sh.D))
    return C, sel, cnt, O, LSE


@pytest.mark.parametrize("L", [1, 128, 129, 500, 700])
def test_decode_equals_last_prefill_row(L):
    wl = PrefillWorkload("xpath", B=2, S=700, shape=MSAShape(k=3), seed=7)
    sh = wl.shape
    inp = prefill_inputs(wl)
    b = 1
    row = np.array([b * wl.S + L - 1], dtype=np.int64)
    Cp, selp, cntp, Op, LSEp = run_prefill_oracle(inp, sh, row)
    d = _decode_from_prefill(inp, sh, b, L, perm_seed=L)
    nb = (L + sh.Bk - 1) // sh.Bk
    Cd, seld, cntd, Od, LSEd = run_decode_oracle(d, sh)
    np.testing.assert_array_equal(Cd[0, :, :nb], Cp[0, :, :nb])
    np.testing.assert_array_equal(seld[0], selp[0])
    np.testing.assert_array_equal(cntd[0], cntp[0])
    np.testing.assert_allclose(Od[0], Op[0], rtol=0, atol=1e-13)
    np.testing.assert_allclose(LSEd[0], LSEp[0], rtol=0, atol=1e-12)


def test_decode_page_permutation_invariance():
    wl = PrefillWorkload("perm", B=1, S=1000, shape=MSAShape(k=4), seed=8)
    sh = wl.shape
    inp = prefill_inputs(wl)
    res = [run_decode_oracle(_decode_from_prefill(inp, sh, 0, 1000, perm_seed=s), sh) for s in (1, 2)]
    for a, b in zip(res[0], res[1]):
        np.testing.assert_array_equal(a, b)


def test_page_table_flattened_rows_equal_per_group():
    """Attention through the flattened (B*Hkv) page table equals per-(b, g) attention.

    Every row r = b*Hkv + g is treated as a sequence of its own with one KV head:
    pages pt[r][0..n), length (n-1)*Bk + last_len, and its G query heads.
    """
    wl = DecodeWorkload("pt", lengths=(1, 200, 1000, 1300), shape=MSAShape(k=4), seed=9)
    sh = wl.shape
    d = decode_inputs(wl)
    C, sel, cnt, O, LSE = run_decode_oracle(d, sh)
    pt, n, last = oracle.page_table(sel, cnt, d["seq_pt"], d["seq_len"], sh.Bk)
    assert np.array_equal(n, cnt.reshape(-1))
    G = sh.G
    for r in range(wl.B * sh.Hkv):
        b, g = divmod(r, sh.Hkv)
        assert np.all(pt[r, n[r]:] == -1)
        dd = {
            "Q": d["Q"][b, g * G:(g + 1) * G][None].contiguous(),
            "K_pool": d["K_pool"][:, g:g + 1].contiguous(),
            "V_pool": d["V_pool"][:, g:g + 1].contiguous(),
        }
        L_r = (int(n[r]) - 1) * sh.Bk + int(last[r])
        sel_r = np.arange(sh.k, dtype=np.int32)[None, None]
        sel_r = np.where(sel_r < n[r], sel_r, -1).astype(np.int32)
        o, l = oracle.decode_attend(dd["Q"], dd["K_pool"], dd["V_pool"],
                                    pt[r][None].copy(), np.array([L_r], dtype=np.int32),
                                    sel_r, np.array([[n[r]]], dtype=np.int32), 1.0 / math.sqrt(sh.D))
        np.testing.assert_allclose(o[0], O[b, g * G:(g + 1) * G], rtol=0, atol=1e-13)
        np.testing.assert_allclose(l[0], LSE[b, g * G:(g + 1) * G], rtol=0, atol=1e-12)


def test_decode_own_block_and_last_len():
    wl = DecodeWorkload("own", lengths=(1, 128, 129, 60001), shape=MSAShape(k=16), seed=10)
    sh = wl.shape
    d = decode_inputs(wl)
    C, sel, cnt, O, LSE = run_decode_oracle(d, sh)
    _, n, last = oracle.page_table(sel, cnt, d["seq_pt"], d["seq_len"], sh.Bk)
    # L = 1: own block 0, nothing scored; L = 128: own block 0 full; L = 129: own block 1 holds 1 token;
    # L = 60001: own block 468 holds 97 tokens (60001 - 468*128)
    assert list(last.reshape(4, sh.Hkv)[:, 0]) == [1, 128, 1, 97]
    assert list(cnt[:, 0]) == [1, 1, 2, 16]
    assert np.all(C[0] == -np.inf) and np.all(C[3, :, 468:] == -np.inf) and np.all(np.isfinite(C[3, :, :468]))


def test_cache_append_slots_by_hand():
    """Token L-1 lands in slot (L-1) % 128 of page seq_pt[b][(L-1) // 128], in
    every group, and nothing else changes: lengths 1, 128, 129 and 300 give
    (block 0, slot 0), (0, 127), (1, 0) and (2, 43) by hand; a length of 0 and a
    page id outside the pool are skipped."""
    P, Hkv, Bk, D, dI = 8, 2, 128, 16, 8
    K = np.zeros((P, Hkv, Bk, D), dtype=np.uint16)
    V = np.zeros((P, Hkv, Bk, D), dtype=np.uint16)
    X = np.zeros((P, Hkv, Bk, dI), dtype=np.uint16)
    seq_pt = np.array([[5, 1, 2], [3, 0, 4], [6, 7, 2], [2, 4, 1], [0, 1, 3], [4, 99, 5]], dtype=np.int32)
    seq_len = np.array([1, 128, 129, 300, 0, 200], dtype=np.int32)
    B = seq_len.shape[0]
    kn = (np.arange(B * Hkv * D, dtype=np.uint16) + 1).reshape(B, Hkv, D)
    vn = (np.arange(B * Hkv * D, dtype=np.uint16) + 1000).reshape(B, Hkv, D)
    xn = (np.arange(B * Hkv * dI, dtype=np.uint16) + 2000).reshape(B, Hkv, dI)
    K2, V2, X2, skipped = oracle.cache_append(kn, vn, xn, K, V, X, seq_pt, seq_len, Bk)
    assert skipped == [4, 5]   # length 0; page 99 is outside the pool of 8
    expect = {0: (5, 0), 1: (3, 127), 2: (7, 0), 3: (1, 43)}   # b -> (page, slot)
    for b, (page, t) in expect.items():
        for g in range(Hkv):
            assert np.array_equal(K2[page, g, t], kn[b, g])
            assert np.array_equal(V2[page, g, t], vn[b, g])
            assert np.array_equal(X2[page, g, t], xn[b, g])
    written = np.zeros((P, Hkv, Bk), dtype=bool)
    for page, t in expect.values():
        written[page, :, t] = True
    assert not K2[~written].any() and not V2[~written].any() and not X2[~written].any()


def test_cache_append_tokens_by_hand():
    """T = 3 tokens per sequence land at positions L-3, L-2, L-1: lengths 5, 130
    and 256 give (page, slot) pairs worked out by hand across page boundaries;
    a length below T skips the sequence, and a token whose page id is outside
    the pool is skipped alone."""
    P, Hkv, Bk, D, dI, T = 8, 2, 128, 16, 8, 3
    K = np.zeros((P, Hkv, Bk, D), dtype=np.uint16)
    V = np.zeros((P, Hkv, Bk, D), dtype=np.uint16)
    X = np.zeros((P, Hkv, Bk, dI), dtype=np.uint16)
    seq_pt = np.array([[5, 1, 2], [3, 0, 4], [6, 7, 2], [2, 4, 1], [0, 99, 3]], dtype=np.int32)
    seq_len = np.array([5, 130, 256, 2, 129], dtype=np.int32)
    B = seq_len.shape[0]
    kn = (np.arange(B * T * Hkv * D, dtype=np.uint16) + 1).reshape(B, T, Hkv, D)
    vn = (np.arange(B * T * Hkv * D, dtype=np.uint16) + 3000).reshape(B, T, Hkv, D)
    xn = (np.arange(B * T * Hkv * dI, dtype=np.uint16) + 7000).reshape(B, T, Hkv, dI)
    K2, V2, X2, skipped = oracle.cache_append(kn, vn, xn, K, V, X, seq_pt, seq_len, Bk)
    # b = 3: length 2 < T; b = 4: positions 126, 127 on page 0, position 128 on page 99 (outside)
    assert skipped == [(3, 0), (3, 1), (3, 2), (4, 2)]
    expect = {(0, 0): (5, 2), (0, 1): (5, 3), (0, 2): (5, 4),          # positions 2, 3, 4
              (1, 0): (3, 127), (1, 1): (0, 0), (1, 2): (0, 1),        # positions 127, 128, 129
              (2, 0): (7, 125), (2, 1): (7, 126), (2, 2): (7, 127),    # positions 253, 254, 255
              (4, 0): (0, 126), (4, 1): (0, 127)}                      # positions 126, 127
    for (b, u), (page, t) in expect.items():
        for g in range(Hkv):
            assert np.array_equal(K2[page, g, t], kn[b, u, g])
            assert np.array_equal(V2[page, g, t], vn[b, u, g])
            assert np.array_equal(X2[page, g, t], xn[b, u, g])
    written = np.zeros((P, Hkv, Bk), dtype=bool)
    for page, t in expect.values():
        written[page, :, t] = True
    assert not K2[~written].any() and not V2[~written].any() and not X2[~written].any()


def _paged(x, perm, Bk):
    """[B, T, Hkv, X] -> page pool [B * ceil(T/Bk), Hkv, Bk, X] (zero tail) and
    seq_pt [B, ceil(T/Bk)]: block j of sequence b goes to page perm[b*n + j]."""
    B, T, Hkv, X = x.shape
    n = (T + Bk - 1) // Bk
    pad = torch.zeros(B, n * Bk, Hkv, X, dtype=x.dtype)
    pad[:, :T] = x
    blocks = pad.view(B, n, Bk, Hkv, X).permute(0, 1, 3, 2, 4).reshape(B * n, Hkv, Bk, X)
    pool = torch.empty_like(blocks)
    pool[perm] = blocks
    return pool, perm.view(B, n).to(torch.int32)


@pytest.mark.parametrize("q_pos,S", [((0, 0), 700), ((300, 451), 249), ((128, 64), 64), ((699, 500), 1)])
def test_chunk_layer_equals_prefill_rows(q_pos, S):
    """A chunk at positions q_pos[b] + s over shuffled pages gives, bit for bit,
    the scores, selection and attention of those rows of a prefill of the
    whole context (contiguous tensors, no pages)."""
    sh = MSAShape(Hq=12, Hkv=2, HI=3, k=3)
    wl = PrefillWorkload("pin_chunk", B=2, S=700, shape=sh, seed=91)
    inp = prefill_inputs(wl)
    T, Bk = wl.S, sh.Bk
    perm = torch.randperm(2 * ((T + Bk - 1) // Bk), generator=torch.Generator().manual_seed(5))
    K_pool, seq_pt = _paged(inp["K"], perm, Bk)
    V_pool, _ = _paged(inp["V"], perm, Bk)
    X_pool, _ = _paged(inp["k_idx"], perm, Bk)
    qp = np.array(q_pos, dtype=np.int64)
    idx = torch.as_tensor(qp[:, None] + np.arange(S)[None, :])
    take = lambda t: torch.stack([t[b, idx[b]] for b in range(2)])
    scale = 1 / math.sqrt(sh.D)
    r = oracle.chunk_layer(take(inp["Q"]), take(inp["q_idx"]), take(inp["w"]), K_pool, V_pool, X_pool, seq_pt,
                           torch.as_tensor(qp, dtype=torch.int32), sh.k, scale, Bk)
    rows = (np.arange(2)[:, None] * T + idx.numpy()).reshape(-1)
    Cp = oracle.prefill_scores(inp["q_idx"], inp["k_idx"], inp["w"], Bk, rows)
    nbc = r["C"].shape[-1]
    assert np.array_equal(r["C"].reshape(-1, sh.Hkv, nbc), Cp[:, :, :nbc])
    assert np.all(Cp[:, :, nbc:] == -np.inf)
    own = np.repeat(oracle.own_blocks_prefill(T, Bk, rows), sh.Hkv).reshape(-1, sh.Hkv)
    sel, cnt, _, _ = oracle.select(Cp, own, sh.k)
    assert np.array_equal(r["sel"].reshape(sel.shape), sel) and np.array_equal(r["count"].reshape(cnt.shape), cnt)
    O, LSE = oracle.prefill_attend(inp["Q"], inp["K"], inp["V"], sel, cnt, Bk, scale, rows)
    assert np.array_equal(r["O"].reshape(O.shape), O) and np.array_equal(r["LSE"].reshape(LSE.shape), LSE)


def test_chunk_layer_brute_force_numpy():
    """Every block score and the attention of a few chunk queries, written out
    in numpy from the definitions with explicit page reads (token t of sequence
    b is slot t % Bk of page seq_pt[b][t // Bk]), against the chunk oracle."""
    sh = MSAShape(Hq=6, Hkv=2, HI=2, k=3)
    wl = ChunkWorkload("pin_chunk_numpy", prefix=(130, 5, 383), S=3, shape=sh, seed=93)
    inp = chunk_inputs(wl)
    scale = 1 / math.sqrt(sh.D)
    r = oracle.chunk_layer(inp["Q"], inp["q_idx"], inp["w"], inp["K_pool"], inp["V_pool"], inp["kidx_pool"],
                           inp["seq_pt"], inp["q_pos"], sh.k, scale, sh.Bk)
    qi, w, Q = f64(inp["q_idx"]), f64(inp["w"]), f64(inp["Q"])
    Kp, Vp, Xp = f64(inp["K_pool"]), f64(inp["V_pool"]), f64(inp["kidx_pool"])
    pt = inp["seq_pt"].numpy()
    for b in range(wl.B):
        for s in range(wl.S):
            p = wl.prefix[b] + s
            own = p // sh.Bk
            for g in range(sh.Hkv):
                c = np.full(r["C"].shape[-1], -np.inf)
                for j in range(own):
                    keys = Xp[pt[b, j], g]                               # [Bk, dI]
                    st = sum(w[b, s, g, h] * np.maximum(keys @ qi[b, s, g, h], 0.0) for h in range(sh.HI))
                    c[j] = st.max()
                assert np.allclose(r["C"][b, s, g], c, rtol=1e-12, atol=0) and \
                    np.array_equal(np.isneginf(r["C"][b, s, g]), np.isneginf(c))
                ts = [t for j in r["sel"][b, s, g] if j >= 0 for t in range(j * sh.Bk, (j + 1) * sh.Bk) if t <= p]
                Kt = np.stack([Kp[pt[b, t // sh.Bk], g, t % sh.Bk] for t in ts])
                Vt = np.stack([Vp[pt[b, t // sh.Bk], g, t % sh.Bk] for t in ts])
                for hh in range(sh.G):
                    hq = g * sh.G + hh
                    z = scale * (Kt @ Q[b, s, hq])
                    m = z.max()
                    e = np.exp(z - m)
                    assert np.allclose(r["O"][b, s, hq], e @ Vt / e.sum(), rtol=1e-10, atol=1e-13)
                    assert abs(r["LSE"][b, s, hq] - (m + math.log(e.sum()))) < 1e-10
