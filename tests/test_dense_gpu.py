"""The dense comparator (attention over every token, no index branch) against
the fp64 oracle, through the C ABI, on a GB300.

The oracle's attention with every block of a row selected is pinned to a
brute-force dense causal GQA attention (the dense-limit pin), so the dense
calls are compared with oracle.decode_attend / oracle.prefill_attend given the
full selection.  Decode cases: ragged lengths (1 token, partial and full last
pages), GQA ratios 1, 6 and 8, the concurrency-8 step over 60,001 tokens, the
1M-token step, a sample of the ragged batch of 64, a page id outside the
pool, a sequence whose length is outside the pages, and repeated calls on the
same scratch.  Prefill cases: the tiny 2,048-token layer, ragged lengths
(1, 300, 513, 700, 1000 tokens), GQA ratios 1, 3, 4, 6 and 8 (odd ratios leave
a head without a partner), sampled rows of the MSA head shape at 4,096 and
131,072 tokens, and agreement with MSA's own prefill layer when k covers
every block.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from msa_check import check_attention
from workloads import DecodeWorkload, MSAShape, decode_inputs, workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msa():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from block_sparse_attention_02_gb300 import build as b
    b.build()
    import block_sparse_attention_02_gb300 as m
    return m


def full_selection(seq_len, Hkv, Bk=128, skip=()):
    """Every block of every (b, g) row, ascending (index bookkeeping); (b, j)
    pairs in ``skip`` are left out."""
    L = np.asarray(seq_len, dtype=np.int64)
    nb = (L + Bk - 1) // Bk
    k = int(max(nb.max(), 1))
    sel = np.full((len(L), Hkv, k), -1, dtype=np.int32)
    cnt = np.zeros((len(L), Hkv), dtype=np.int32)
    for b, n in enumerate(nb):
        js = [j for j in range(int(n)) if (b, j) not in skip]
        sel[b, :, :len(js)] = js
        cnt[b, :] = len(js)
    return sel, cnt


def run_dense(msa, inp, expect_err=0):
    bufs = msa.dense_decode_step(inp)
    torch.cuda.synchronize()
    err = int(bufs["dev_err"].item())
    assert err == expect_err, f"device error word {err:#x}, expected {expect_err:#x}"
    return bufs


def host_subset(inp_dev, bs):
    """Host copy of sequences ``bs`` with their pages compacted (tensor plumbing, no arithmetic)."""
    pages = sorted({int(p) for b in bs for p in inp_dev["seq_pt"][b].tolist() if p >= 0})
    remap = torch.full((inp_dev["K_pool"].shape[0],), -1, dtype=torch.int32)
    remap[torch.tensor(pages)] = torch.arange(len(pages), dtype=torch.int32)
    idx = torch.tensor(pages, device=inp_dev["K_pool"].device)
    spt = inp_dev["seq_pt"][bs].cpu().clone()
    spt[spt >= 0] = remap[spt[spt >= 0].long()]
    return {"Q": inp_dev["Q"][bs].cpu(), "K_pool": inp_dev["K_pool"].index_select(0, idx).cpu(),
            "V_pool": inp_dev["V_pool"].index_select(0, idx).cpu(), "seq_pt": spt,
            "seq_len": inp_dev["seq_len"][bs].cpu()}


def check_dense_decode(msa, wl, inp, bufs, bs=None):
    sh = wl.shape
    bs = list(range(wl.B)) if bs is None else list(bs)
    h = host_subset(inp, bs)
    sel, cnt = full_selection(h["seq_len"].numpy(), sh.Hkv, sh.Bk)
    O_o, L_o = oracle.decode_attend(h["Q"], h["K_pool"], h["V_pool"], h["seq_pt"], h["seq_len"], sel, cnt,
                                    1.0 / math.sqrt(sh.D))
    return check_attention(bufs["O"].float().cpu().numpy()[bs], bufs["LSE"].cpu().numpy()[bs], O_o, L_o)


SMALL = [
    DecodeWorkload("dense_edges", lengths=(1, 2, 127, 128, 129, 255, 256, 257, 1000, 2049, 5000),
                   shape=MSAShape(), seed=81),
    DecodeWorkload("dense_gqa1", lengths=(300, 4100, 777), shape=MSAShape(Hq=8, Hkv=8), seed=82),
    DecodeWorkload("dense_gqa8", lengths=(9000, 1, 640), shape=MSAShape(Hq=16, Hkv=2), seed=83),
    DecodeWorkload("dense_one_row", lengths=(70000,), shape=MSAShape(Hq=6, Hkv=1), seed=84),
]


@pytest.mark.parametrize("wl", SMALL, ids=[w.name for w in SMALL])
def test_dense_decode_small(msa, wl):
    inp = decode_inputs(wl, device="cuda")
    bufs = run_dense(msa, inp)
    errs = check_dense_decode(msa, wl, inp, bufs)
    print(f"{wl.name}: O max/mean {errs[0]:.2e}/{errs[1]:.2e}, LSE {errs[2]:.2e}")


@pytest.mark.parametrize("name", ["decode_b8_l60001", "decode_b1_l1048576"])
def test_dense_decode_full_size(msa, name):
    wl = workload(name)
    inp = decode_inputs(wl, device="cuda")
    bufs = run_dense(msa, inp)
    errs = check_dense_decode(msa, wl, inp, bufs)
    print(f"{name} dense: O max/mean {errs[0]:.2e}/{errs[1]:.2e}, LSE {errs[2]:.2e}")


def test_dense_decode_ragged_b64_sampled(msa):
    wl = workload("decode_ragged_b64")
    inp = decode_inputs(wl, device="cuda")
    bufs = run_dense(msa, inp)
    L = np.array(wl.lengths)
    rng = np.random.default_rng(1)
    sample = sorted({int(L.argmin()), int(L.argmax())} | set(rng.choice(wl.B, 4, replace=False).tolist()))
    check_dense_decode(msa, wl, inp, bufs, sample)


def test_dense_decode_bad_page_and_length(msa):
    """A page id outside the pool is left out (the oracle over the remaining
    blocks); a sequence of length 0 gets O = 0 and LSE = -inf; both flagged."""
    wl = DecodeWorkload("dense_bad", lengths=(1000, 1000, 700), shape=MSAShape(Hq=12, Hkv=2), seed=85)
    inp = decode_inputs(wl, device="cuda")
    inp["seq_pt"][1, 2] = inp["K_pool"].shape[0] + 5
    inp["seq_len"][2] = 0
    bufs = run_dense(msa, inp, expect_err=msa.MSA_DEVERR_BAD_PAGE | msa.MSA_DEVERR_BAD_LEN)
    assert torch.all(bufs["O"][2] == 0) and torch.all(bufs["LSE"][2] == -math.inf)
    h = {n: inp[n].cpu() for n in ("Q", "K_pool", "V_pool", "seq_pt", "seq_len")}
    h["seq_pt"][1, 2] = 0                                  # never read: block 2 of sequence 1 is left out
    sel, cnt = full_selection(h["seq_len"].numpy()[:2], wl.shape.Hkv, skip={(1, 2)})
    O_o, L_o = oracle.decode_attend(h["Q"][:2], h["K_pool"], h["V_pool"], h["seq_pt"][:2], h["seq_len"][:2], sel,
                                    cnt, 1.0 / math.sqrt(wl.shape.D))
    check_attention(bufs["O"][:2].float().cpu().numpy(), bufs["LSE"][:2].cpu().numpy(), O_o, L_o)


def test_dense_decode_repeated_calls_on_zeroed_scratch(msa):
    """scratch_zeroed: the row counters left zero by each call serve the next
    call, whose outputs are bit-identical."""
    wl = SMALL[0]
    inp = decode_inputs(wl, device="cuda")
    ref = run_dense(msa, inp)
    bufs = msa.dense_decode_buffers(wl.B, wl.shape.Hq, wl.shape.Hkv, inp["seq_pt"].shape[1], "cuda")
    for _ in range(3):
        msa.dense_decode_step(inp, bufs, scratch_zeroed=True)
        torch.cuda.synchronize()
        assert int(bufs["dev_err"].item()) == 0
        assert torch.equal(bufs["O"], ref["O"]) and torch.equal(bufs["LSE"], ref["LSE"])


# ---------------------------------------------------------------------------
# dense prefill
# ---------------------------------------------------------------------------

def prefill_full_selection(rows, S, Hkv, Bk=128):
    """Every block up to the own one, for prefill rows b*S + i (index bookkeeping)."""
    rows = np.asarray(rows, dtype=np.int64)
    own = (rows % S) // Bk
    k = int(max((S - 1) // Bk + 1, 1))
    sel = np.full((len(rows), Hkv, k), -1, dtype=np.int32)
    cnt = np.zeros((len(rows), Hkv), dtype=np.int32)
    for x, o in enumerate(own):
        sel[x, :, :o + 1] = np.arange(o + 1)
        cnt[x, :] = o + 1
    return sel, cnt


def check_dense_prefill(msa, wl, inp, rows=None):
    sh = wl.shape
    bufs = msa.dense_prefill_layer(inp)
    torch.cuda.synchronize()
    assert int(bufs["dev_err"].item()) == 0
    rows = np.arange(wl.B * wl.S) if rows is None else np.asarray(rows, dtype=np.int64)
    sel, cnt = prefill_full_selection(rows, wl.S, sh.Hkv, sh.Bk)
    h = {n: inp[n].cpu() for n in ("Q", "K", "V")}
    O_o, L_o = oracle.prefill_attend(h["Q"], h["K"], h["V"], sel, cnt, sh.Bk, 1.0 / math.sqrt(sh.D), rows)
    Og = bufs["O"].view(wl.B * wl.S, sh.Hq, sh.D)[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    Lg = bufs["LSE"].view(wl.B * wl.S, sh.Hq)[torch.from_numpy(rows).cuda()].cpu().numpy()
    return check_attention(Og, Lg, O_o, L_o)


def _prefill_cases():
    from workloads import PrefillWorkload
    return [
        PrefillWorkload("dense_tiny_s2048", B=1, S=2048, shape=MSAShape(Hq=4, Hkv=1, HI=2, k=16), seed=0),
        PrefillWorkload("dense_ragged_s300_g6", B=2, S=300, shape=MSAShape(Hq=12, Hkv=2), seed=86),
        PrefillWorkload("dense_g1", B=1, S=700, shape=MSAShape(Hq=4, Hkv=4), seed=87),
        PrefillWorkload("dense_g3", B=1, S=513, shape=MSAShape(Hq=6, Hkv=2), seed=88),
        PrefillWorkload("dense_g8", B=2, S=1000, shape=MSAShape(Hq=16, Hkv=2), seed=89),
        PrefillWorkload("dense_short", B=3, S=1, shape=MSAShape(Hq=12, Hkv=2), seed=90),
    ]


@pytest.mark.parametrize("wl", _prefill_cases(), ids=lambda w: w.name)
def test_dense_prefill_small(msa, wl):
    from workloads import prefill_inputs
    inp = prefill_inputs(wl, device="cuda")
    errs = check_dense_prefill(msa, wl, inp)
    print(f"{wl.name}: O max/mean {errs[0]:.2e}/{errs[1]:.2e}, LSE {errs[2]:.2e}")


def test_dense_prefill_equals_msa_with_every_block(msa):
    """With k covering every block, MSA's prefill layer is dense attention:
    the dense comparator agrees with it within the output tolerances."""
    from workloads import PrefillWorkload, prefill_inputs
    wl = PrefillWorkload("dense_vs_msa", B=1, S=2048, shape=MSAShape(Hq=12, Hkv=2, k=16), seed=91)
    inp = prefill_inputs(wl, device="cuda")
    d = msa.dense_prefill_layer(inp)
    s = msa.prefill_layer(inp, 16)
    torch.cuda.synchronize()
    assert int(s["dev_err"].item()) == 0 and int(d["dev_err"].item()) == 0
    assert torch.all(s["count"] == (torch.arange(wl.S, device="cuda") // 128 + 1).view(1, -1, 1))
    diff = (d["O"].float() - s["O"].float()).abs()
    assert diff.max().item() <= 1e-2 and diff.mean().item() <= 1e-3
    assert (d["LSE"] - s["LSE"]).abs().max().item() <= 1e-3


@pytest.mark.parametrize("S,nrows", [(4096, 64), (131072, 8)], ids=["s4096", "s131072"])
def test_dense_prefill_msa_shape_sampled_rows(msa, S, nrows):
    """The MSA head shape (48 q / 8 KV heads) on sampled rows: the first and
    last query, block boundaries and random rows."""
    from dataclasses import replace
    from workloads import prefill_inputs
    wl = replace(workload("prefill_s131072"), name=f"dense_s{S}", S=S)
    inp = prefill_inputs(wl, device="cuda")
    rng = np.random.default_rng(S)
    rows = sorted({0, 127, 128, S - 1, S // 2} | set(rng.integers(0, S, nrows - 5).tolist()))
    errs = check_dense_prefill(msa, wl, inp, rows)
    print(f"dense prefill S={S} rows {len(rows)}: O max/mean {errs[0]:.2e}/{errs[1]:.2e}, LSE {errs[2]:.2e}")
