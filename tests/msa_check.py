"""Comparison rules between the CUDA path and the fp64 oracle.

Tolerances (each with the arithmetic it follows from):

* block scores: fp32 accumulation of HI * dI = 256 bf16 products per token
  errs by at most ~256 * 2^-24 (1.5e-5) relative to the sum of the terms'
  magnitudes; |C_gpu - C_oracle| <= SCORE_ATOL + SCORE_RTOL * |C_oracle| leaves
  margin, and the -inf entries (own block, future blocks, padding) must
  coincide exactly.
* selection: bit-exact wherever the oracle's gap between the last kept and the
  first dropped earlier block exceeds SEL_REL relative; at a near-tie any set
  containing every block clearly above the cut and only blocks clearly not
  below it is accepted (same size, ascending, own block last).
* attention output (bf16, fp32 accumulation): max-abs <= 1e-2 and mean-abs
  <= 1e-3 against the oracle run on the GPU's own selection (the bf16 output
  alone rounds by up to 2^-9 relative); LSE max-abs <= 1e-3 (an fp32
  log-sum-exp of <= 2048 terms with |z| of order 10 errs by ~1e-5).
* integer / index work (page table, counts): bit-exact.
"""
from __future__ import annotations

import math

import numpy as np

import oracle

SCORE_ATOL = 1e-4
SCORE_RTOL = 1e-4
SEL_REL = 1e-3
O_MAX_ABS = 1e-2
O_MEAN_ABS = 1e-3
LSE_MAX_ABS = 1e-3


def check_scores(C_gpu, C_orc, ncheck=None):
    """C_gpu (fp32) and C_orc (fp64) of the same shape; compare the first ncheck entries of each row."""
    g = np.asarray(C_gpu, dtype=np.float64)
    o = np.asarray(C_orc, dtype=np.float64)
    if ncheck is not None:
        g, o = g[..., :ncheck], o[..., :ncheck]
    assert g.shape == o.shape, (g.shape, o.shape)
    inf_g, inf_o = np.isneginf(g), np.isneginf(o)
    assert np.array_equal(inf_g, inf_o), f"-inf pattern differs at {np.argwhere(inf_g != inf_o)[:5]}"
    fin = ~inf_o
    err = np.abs(g[fin] - o[fin])
    lim = SCORE_ATOL + SCORE_RTOL * np.abs(o[fin])
    bad = err > lim
    assert not bad.any(), f"{bad.sum()} scores out of tolerance, worst {err.max():.3e}"
    return float(err.max()) if err.size else 0.0


def check_selection(sel_gpu, cnt_gpu, C_orc, own, k, rel=SEL_REL):
    """Selection of the CUDA path against the oracle's, with the near-tie rule.

    sel_gpu [R, k], cnt_gpu [R], C_orc [R, nb] (fp64 oracle scores), own [R].
    Returns (rows compared exactly, rows at a near-tie).
    """
    sel_gpu = np.asarray(sel_gpu).reshape(-1, k)
    cnt_gpu = np.asarray(cnt_gpu).reshape(-1)
    C_orc = np.asarray(C_orc, dtype=np.float64).reshape(len(cnt_gpu), -1)
    own = np.asarray(own).reshape(-1)
    sel_o, cnt_o, c_last, c_next = oracle.select(C_orc, own.astype(np.int32), k)
    assert np.array_equal(cnt_gpu, cnt_o), "selected counts differ"
    exact = tie = 0
    for r in range(len(cnt_o)):
        c = int(cnt_o[r])
        s = sel_gpu[r, :c]
        assert np.all(sel_gpu[r, c:] == -1), f"row {r}: padding is not -1"
        if math.isnan(c_last[r]) or (c_last[r] - c_next[r]) > rel * max(abs(c_last[r]), 1e-30):
            if not np.array_equal(s, sel_o[r, :c]):
                raise AssertionError(f"row {r}: selection {s.tolist()} != oracle {sel_o[r, :c].tolist()}")
            exact += 1
            continue
        tie += 1
        assert np.all(np.diff(s) > 0), f"row {r}: not ascending"
        assert s[-1] == own[r], f"row {r}: own block not last"
        picked = set(s[:-1].tolist())
        cand = C_orc[r, :own[r]]
        hi = c_last[r] + rel * max(abs(c_last[r]), 1e-30)
        lo = c_next[r] - rel * max(abs(c_next[r]), 1e-30)
        must = set(np.nonzero(cand > hi)[0].tolist())
        may = set(np.nonzero(cand >= lo)[0].tolist())
        assert must <= picked <= may, f"row {r}: near-tie selection outside the accepted band"
    return exact, tie


def check_attention(O_gpu, LSE_gpu, O_orc, LSE_orc):
    og = np.asarray(O_gpu, dtype=np.float64)
    oo = np.asarray(O_orc, dtype=np.float64)
    assert og.shape == oo.shape, (og.shape, oo.shape)
    err = np.abs(og - oo)
    assert np.isfinite(og).all(), "non-finite attention output"
    assert err.max() <= O_MAX_ABS, f"max-abs {err.max():.3e} > {O_MAX_ABS}"
    assert err.mean() <= O_MEAN_ABS, f"mean-abs {err.mean():.3e} > {O_MEAN_ABS}"
    lg = np.asarray(LSE_gpu, dtype=np.float64)
    lo = np.asarray(LSE_orc, dtype=np.float64)
    lerr = np.abs(lg - lo)
    assert lerr.max() <= LSE_MAX_ABS, f"LSE max-abs {lerr.max():.3e} > {LSE_MAX_ABS}"
    return float(err.max()), float(err.mean()), float(lerr.max())
