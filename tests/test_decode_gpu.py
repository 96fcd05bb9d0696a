"""Decode path (a1 index score -> a2 top-k -> a3 page table -> a5/a6 attention)
against the fp64 oracle, through the C ABI, on a GB300.

Small cases cover ragged lengths (1 token, partial and full own blocks, fewer
than k earlier blocks), GQA ratios 1/6/8, HI = 1..4 and k = 1/4/16/64.  The
full-size cases run the decode step at concurrency 8 over a 60,000-token cached
prefix, the 1M-token batch-1 step, and the ragged batch of 64 (checked on a
sample of its sequences, which the oracle computes one by one).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from msa_check import O_MAX_ABS, O_MEAN_ABS, check_attention, check_scores, check_selection
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


def run_gpu(msa, inp, k, fused=True):
    bufs = msa.decode_step(inp, k, fused=fused)
    torch.cuda.synchronize()
    assert int(bufs["dev_err"].item()) == 0, f"device error word {int(bufs['dev_err'].item()):#x}"
    return {n: t.cpu() for n, t in bufs.items() if n != "ws"}


def check_decode(msa, wl, inp_dev, k, seq_subset=None):
    """Full GPU step, then oracle checks on all (or a subset of) sequences."""
    sh = wl.shape
    out = run_gpu(msa, inp_dev, k)
    small = ("Q", "q_idx", "w", "seq_pt", "seq_len")
    inp = {n: inp_dev[n].cpu() for n in small}
    bs = list(range(wl.B)) if seq_subset is None else list(seq_subset)
    if seq_subset is not None:
        # compact host copy of the sampled sequences (tensor plumbing, no arithmetic)
        pages = sorted({int(p) for b in bs for p in inp["seq_pt"][b].tolist() if p >= 0})
        remap = torch.full((inp_dev["K_pool"].shape[0],), -1, dtype=torch.int32)
        remap[torch.tensor(pages)] = torch.arange(len(pages), dtype=torch.int32)
        idx = torch.tensor(pages, device=inp_dev["K_pool"].device)
        sub = {
            "Q": inp["Q"][bs], "q_idx": inp["q_idx"][bs], "w": inp["w"][bs],
            "kidx_pool": inp_dev["kidx_pool"].index_select(0, idx).cpu(),
            "K_pool": inp_dev["K_pool"].index_select(0, idx).cpu(),
            "V_pool": inp_dev["V_pool"].index_select(0, idx).cpu(),
            "seq_len": inp["seq_len"][bs],
        }
        spt = inp["seq_pt"][bs].clone()
        spt[spt >= 0] = remap[spt[spt >= 0].long()]
        sub["seq_pt"] = spt
        inp = sub
    else:
        for n in ("kidx_pool", "K_pool", "V_pool"):
            inp[n] = inp_dev[n].cpu()
    nb_stride = out["C"].shape[-1]
    C_orc = oracle.decode_scores(inp["q_idx"], inp["w"], inp["kidx_pool"], inp["seq_pt"], inp["seq_len"], nb_stride)
    C_gpu = out["C"].numpy()[bs]
    check_scores(C_gpu, C_orc)
    own = oracle.own_blocks_decode(inp["seq_len"], sh.Bk)
    own_rows = np.repeat(own, sh.Hkv)
    sel_gpu = out["sel"].numpy()[bs]
    cnt_gpu = out["count"].numpy()[bs]
    exact, tie = check_selection(sel_gpu.reshape(-1, k), cnt_gpu.reshape(-1), C_orc.reshape(-1, nb_stride),
                                 own_rows, k)
    # page table: bit-exact against the oracle's construction from the GPU selection
    pt_o, n_o, ll_o = oracle.page_table(out["sel"].numpy(), out["count"].numpy(), inp_dev["seq_pt"].cpu(),
                                        inp_dev["seq_len"].cpu(), sh.Bk)
    assert np.array_equal(out["pt"].numpy(), pt_o)
    assert np.array_equal(out["n"].numpy(), n_o)
    assert np.array_equal(out["last_len"].numpy(), ll_o)
    # attention on the GPU's own selection
    O_o, LSE_o = oracle.decode_attend(inp["Q"], inp["K_pool"], inp["V_pool"], inp["seq_pt"], inp["seq_len"],
                                      sel_gpu, cnt_gpu, 1.0 / math.sqrt(sh.D))
    O_g = out["O"].float().numpy()[bs]
    L_g = out["LSE"].numpy()[bs]
    errs = check_attention(O_g, L_g, O_o, LSE_o)
    return exact, tie, errs


SMALL = [
    DecodeWorkload("edge_lengths", lengths=(1, 2, 127, 128, 129, 255, 256, 257, 1000, 2049, 5000),
                   shape=MSAShape(), seed=31),
    DecodeWorkload("gqa1_hi1", lengths=(300, 4100, 777), shape=MSAShape(Hq=8, Hkv=8, HI=1, k=4), seed=32),
    DecodeWorkload("gqa8_hi3", lengths=(9000, 1, 640), shape=MSAShape(Hq=16, Hkv=2, HI=3, k=16), seed=33),
    DecodeWorkload("k1", lengths=(3000, 129), shape=MSAShape(Hq=12, Hkv=2, HI=2, k=1), seed=34),
    DecodeWorkload("k64", lengths=(20000, 8000, 64 * 128 + 5), shape=MSAShape(Hq=24, Hkv=4, k=64), seed=35),
    DecodeWorkload("unshuffled", lengths=(2500,) * 3, shape=MSAShape(), seed=36, shuffle_pages=False),
    DecodeWorkload("gqa3", lengths=(5000, 130, 1500), shape=MSAShape(Hq=9, Hkv=3, k=8), seed=37),
]


@pytest.mark.parametrize("wl", SMALL, ids=[w.name for w in SMALL])
def test_decode_small(msa, wl):
    inp = decode_inputs(wl, device="cuda")
    exact, tie, errs = check_decode(msa, wl, inp, wl.shape.k)
    print(f"{wl.name}: exact rows {exact}, near-tie rows {tie}, O max/mean {errs[0]:.2e}/{errs[1]:.2e}")


def test_decode_b8_l60001(msa):
    wl = workload("decode_b8_l60001")
    inp = decode_inputs(wl, device="cuda")
    exact, tie, errs = check_decode(msa, wl, inp, wl.shape.k)
    assert exact + tie == 64
    print(f"decode_b8_l60001: exact rows {exact}, near-tie rows {tie}, errs {errs}")


def test_decode_b1_l1048576(msa):
    wl = workload("decode_b1_l1048576")
    inp = decode_inputs(wl, device="cuda")
    exact, tie, errs = check_decode(msa, wl, inp, wl.shape.k)
    print(f"decode_b1_l1048576: exact rows {exact}, near-tie rows {tie}, errs {errs}")


def test_decode_ragged_b64_sampled(msa):
    wl = workload("decode_ragged_b64")
    inp = decode_inputs(wl, device="cuda")
    L = np.array(wl.lengths)
    rng = np.random.default_rng(0)
    sample = sorted({int(L.argmin()), int(L.argmax())} | set(rng.choice(wl.B, 4, replace=False).tolist()))
    exact, tie, errs = check_decode(msa, wl, inp, wl.shape.k, seq_subset=sample)
    print(f"decode_ragged_b64 sample {sample}: exact rows {exact}, near-tie rows {tie}, errs {errs}")


def test_decode_is_deterministic(msa):
    wl = workload("decode_b8_l60001")
    inp = decode_inputs(wl, device="cuda")
    a = run_gpu(msa, inp, 16)
    b = run_gpu(msa, inp, 16)
    for n in ("C", "sel", "count", "pt", "O", "LSE"):
        assert torch.equal(a[n], b[n]), n


@pytest.mark.parametrize("wl", SMALL[:2] + [workload("decode_b8_l60001")], ids=lambda w: w.name)
def test_scratch_zeroed_calls_leave_counters_zero(msa, wl):
    """With scratch_zeroed the counter clears are skipped: repeated calls on the
    same zero-filled scratch give the bits of the default calls and leave every
    row counter (row_scratch and the workspace's counter words) zero."""
    sh = wl.shape
    inp = decode_inputs(wl, device="cuda")
    ref = run_gpu(msa, inp, sh.k)
    bufs = msa.decode_buffers(wl.B, sh.Hq, sh.Hkv, sh.k, inp["seq_pt"].shape[1], "cuda")
    off = wl.B * sh.Hq * sh.k * (sh.D + 1)          # counter words follow the partials and LSEs (4-byte units)
    for _ in range(3):
        msa.decode_step(inp, sh.k, bufs, scratch_zeroed=True)
        torch.cuda.synchronize()
        assert int(bufs["dev_err"].item()) == 0
        for n in ("C", "sel", "count", "pt", "n", "last_len", "O", "LSE"):
            assert torch.equal(bufs[n].cpu(), ref[n]), n
        assert int(bufs["row_scratch"].abs().sum().item()) == 0
        assert int(bufs["ws"].view(torch.int32)[off: off + wl.B * sh.Hkv].abs().sum().item()) == 0


def test_decode_bad_page_is_reported_not_read(msa):
    """A page id outside the pool is skipped and flagged; nothing faults."""
    wl = DecodeWorkload("badpage", lengths=(1000, 1000), shape=MSAShape(), seed=37)
    inp = decode_inputs(wl, device="cuda")
    inp["seq_pt"][1, 2] = inp["K_pool"].shape[0] + 5
    bufs = msa.decode_step(inp, 16)
    torch.cuda.synchronize()
    assert int(bufs["dev_err"].item()) & msa.MSA_DEVERR_BAD_PAGE
    C = bufs["C"].cpu()
    assert torch.isneginf(C[1, :, 2]).all()
    assert torch.isfinite(bufs["O"].float()).all()


def test_standalone_lse_merge(msa):
    """msa_lse_merge on random partials with empty parts against the oracle merge."""
    g = torch.Generator(device="cuda").manual_seed(5)
    rows, parts, D = 1000, 16, 128
    # partials at the scale of attention outputs over V ~ N(0, 1)/sqrt(D), the
    # scale the stated max-abs / mean-abs output bounds are for
    Op = torch.randn(rows, parts, D, device="cuda", generator=g) / math.sqrt(D)
    Lp = torch.randn(rows, parts, device="cuda", generator=g) * 4
    Lp[torch.rand(rows, parts, device="cuda", generator=g) < 0.2] = -float("inf")
    Lp[7] = -float("inf")                       # a row with nothing in it
    O = torch.empty(rows, D, dtype=torch.bfloat16, device="cuda")
    L = torch.empty(rows, device="cuda")
    msa.msa_lse_merge(Op, Lp, O, L)
    torch.cuda.synchronize()
    Oo, Lo = oracle.lse_merge(Op.cpu().double().numpy(), Lp.cpu().double().numpy())
    fin = np.isfinite(Lo)
    assert np.array_equal(np.isneginf(L.cpu().numpy()), ~fin)
    og = O.float().cpu().numpy().astype(np.float64)
    err = np.abs(og - Oo)
    # the stated output bounds, and per element the bf16 rounding of the
    # output (at most 2^-9 relative) plus fp32 arithmetic over 16 parts
    assert err.max() <= O_MAX_ABS and err.mean() <= O_MEAN_ABS, (err.max(), err.mean())
    assert np.all(err <= 2.0 ** -8 * np.abs(Oo) + 1e-5), err.max()
    np.testing.assert_allclose(L.cpu().numpy()[fin], Lo[fin], rtol=0, atol=1e-4)
    assert torch.all(O[7] == 0)


@pytest.mark.parametrize("wl", SMALL[:3] + [workload("decode_b8_l60001")], ids=lambda w: w.name)
def test_fused_selection_equals_standalone_entry_points(msa, wl):
    """a2/a3 fused into the index-score call give the same bits as msa_topk_blocks + msa_build_page_table."""
    inp = decode_inputs(wl, device="cuda")
    f = run_gpu(msa, inp, wl.shape.k, fused=True)
    u = run_gpu(msa, inp, wl.shape.k, fused=False)
    for n in ("C", "sel", "count", "pt", "n", "last_len", "O", "LSE"):
        assert torch.equal(f[n], u[n]), n


def test_decode_b1_l1048576_unfused(msa):
    """The standalone top-k (CTA per long row) and page table at 1M tokens."""
    wl = workload("decode_b1_l1048576")
    inp = decode_inputs(wl, device="cuda")
    f = run_gpu(msa, inp, wl.shape.k, fused=True)
    u = run_gpu(msa, inp, wl.shape.k, fused=False)
    for n in ("sel", "count", "pt", "n", "last_len"):
        assert torch.equal(f[n], u[n]), n


@pytest.mark.parametrize("wl", SMALL[:4] + [workload("decode_b1_l1048576"), workload("decode_ragged_b64")],
                         ids=lambda w: w.name)
def test_standalone_topk_and_page_table_match_oracle(msa, wl):
    """msa_topk_blocks and msa_build_page_table called on their own, against
    oracle.select and oracle.page_table run on the same fp32 scores: the
    selection is then unique, so both must agree bit for bit (warp-per-row
    rows, and CTA-per-row rows of more than 2048 blocks at 1M tokens and in
    the ragged batch)."""
    sh = wl.shape
    inp = decode_inputs(wl, device="cuda")
    u = run_gpu(msa, inp, sh.k, fused=False)
    seq_len = inp["seq_len"].cpu()
    own = np.repeat(oracle.own_blocks_decode(seq_len, sh.Bk), sh.Hkv)
    C = u["C"].numpy().astype(np.float64).reshape(wl.B * sh.Hkv, -1)
    sel_o, cnt_o, _, _ = oracle.select(C, own.astype(np.int32), sh.k)
    assert np.array_equal(u["count"].numpy().reshape(-1), cnt_o)
    assert np.array_equal(u["sel"].numpy().reshape(-1, sh.k), sel_o)
    pt_o, n_o, ll_o = oracle.page_table(sel_o.reshape(wl.B, sh.Hkv, sh.k), cnt_o.reshape(wl.B, sh.Hkv),
                                        inp["seq_pt"].cpu(), seq_len, sh.Bk)
    assert np.array_equal(u["pt"].numpy(), pt_o)
    assert np.array_equal(u["n"].numpy(), n_o)
    assert np.array_equal(u["last_len"].numpy(), ll_o)


LONG_ROWS = (2049, 5000, 8191, 8192, 8193, 20000, 65536, 70000)


@pytest.mark.parametrize("k", [16, 64])
@pytest.mark.parametrize("ties", [False, True], ids=["distinct", "few_values"])
def test_topk_long_rows_match_oracle(msa, k, ties):
    """msa_topk_blocks on decode rows of more than 2048 blocks (one CTA per
    row: its warps select the best of slices of 1024 or 2048 blocks, the
    slices' picks are ranked together; past 65,536 blocks successive
    arg-max), against oracle.select on the same fp32 scores.  Own-block
    counts sit on both sides of each switch; k = 64 makes the warp select keep
    every candidate of a slice; rows of a few distinct values put thousands
    of ties at the threshold (broken by block index)."""
    g = torch.Generator().manual_seed(71 + k + int(ties))
    own = torch.tensor(LONG_ROWS, dtype=torch.int64)
    B, Hkv = len(LONG_ROWS), 2
    nb = int(own.max()) + 1
    C = torch.randn(B, Hkv, nb, generator=g)
    if ties:
        C = torch.round(C * 2) / 2
    seq_len = (own * 128 + 1 + torch.arange(B) * 13 % 128).to(torch.int32)   # own block (L - 1) // 128
    assert torch.equal((seq_len.long() - 1) // 128, own)
    sel = torch.empty(B, Hkv, k, dtype=torch.int32, device="cuda")
    count = torch.empty(B, Hkv, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    msa.msa_topk_blocks(msa.MSA_MODE_DECODE, C.cuda(), k, sel, count, seq_len=seq_len.cuda(), dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    sel_o, cnt_o, _, _ = oracle.select(C.double().numpy(), np.repeat(own.numpy(), Hkv).reshape(B, Hkv), k)
    assert np.array_equal(count.cpu().numpy(), cnt_o)
    assert np.array_equal(sel.cpu().numpy(), sel_o)


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("bad,shared", [(False, False), (True, False), (False, True)],
                         ids=["valid", "bad_len_and_page", "shared_index_pool"])
def test_cache_append_matches_oracle(msa, bad, shared):
    """msa_cache_append writes token L-1 of every sequence into its page slot,
    bit for bit as the oracle's copies; a bad length or page id is flagged and
    that sequence writes nothing; a shared index-key pool (group stride 0)
    takes group 0's key."""
    g = torch.Generator(device="cuda").manual_seed(61)
    P, Hkv, Bk_, D_, dI_, mp = 64, 8, 128, 128, 64, 8
    seq_len = torch.tensor([1, 127, 128, 129, 700, 1024], dtype=torch.int32, device="cuda")
    B = seq_len.shape[0]
    pools = [torch.randn(P, Hkv, Bk_, d, generator=g, device="cuda").to(torch.bfloat16) for d in (D_, D_, dI_)]
    new = [torch.randn(B, Hkv, d, generator=g, device="cuda").to(torch.bfloat16) for d in (D_, D_, dI_)]
    seq_pt = torch.randperm(P, generator=g, device="cuda")[: B * mp].view(B, mp).to(torch.int32).contiguous()
    if bad:
        seq_len[0] = 0                                   # not a valid length
        seq_pt[3, (129 - 1) // 128] = P + 3              # page id outside the pool
    if shared:   # one index pool for all groups, seen through a broadcast view
        pools[2] = pools[2][:, :1].expand(-1, Hkv, -1, -1)
    K2, V2, X2, skipped = oracle.cache_append(*new, *pools, seq_pt, seq_len, 128, shared_index=shared)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    msa.msa_cache_append(*new, *pools, seq_pt, seq_len, dev_err=err)
    torch.cuda.synchronize()
    for got, want in zip(pools, (K2, V2, X2)):
        assert np.array_equal(_bits(got), want)
    e = int(err.item())
    if bad:
        assert skipped == [0, 3]
        assert e & msa.MSA_DEVERR_BAD_LEN and e & msa.MSA_DEVERR_BAD_PAGE
    else:
        assert skipped == [] and e == 0


SHARED_INDEX = [
    DecodeWorkload("shared_edges", lengths=(1, 2, 127, 128, 129, 257, 1000, 2049, 5000), shape=MSAShape(), seed=62),
    DecodeWorkload("shared_hkv4", lengths=(3000, 20000, 640), shape=MSAShape(Hq=24, Hkv=4, k=16), seed=63),
    # rows of more than 2048 blocks: a sequence's 8 group rows complete together and are selected by the
    # top-k kernel after the scores (one CTA per row)
    DecodeWorkload("shared_long", lengths=(300000, 270000, 1000), shape=MSAShape(), seed=64),
]


@pytest.mark.parametrize("wl", SHARED_INDEX, ids=[w.name for w in SHARED_INDEX])
def test_decode_shared_index_keys(msa, wl):
    """One index-key pool for all KV groups (k_idx group stride 0, the lighter
    index): each (page) block is scored for every group in one pass; scores,
    selection, page table and attention match the oracle on the broadcast pool."""
    inp = decode_inputs(wl, device="cuda")
    base = inp["kidx_pool"][:, :1]
    inp["kidx_pool"] = base.expand(-1, wl.shape.Hkv, -1, -1)
    assert inp["kidx_pool"].stride(1) == 0
    exact, tie, errs = check_decode(msa, wl, inp, wl.shape.k)
    print(f"{wl.name}: exact rows {exact}, near-tie rows {tie}, O max/mean {errs[0]:.2e}/{errs[1]:.2e}")
