"""A chunk of queries over a paged cache (MSA_MODE_CHUNK: chunked prefill
after a cached prefix, and decode of several tokens per sequence) against the
fp64 oracle, through the C ABI, on a GB300.

Cases cover ragged prefixes that are not multiples of 64 or 128 (query items
that straddle a block boundary), prefixes shorter than one block, chunks with
ragged tails, the MSA head shape, HI = 3 with k = 64, one index-key pool
shared by all KV groups, and rejected sequences and pages.  A chunk that starts
at position 0 over pages must reproduce the contiguous prefill bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from msa_check import check_attention, check_scores, check_selection
from workloads import ChunkWorkload, MSAShape, PrefillWorkload, chunk_inputs, prefill_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msa():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from block_sparse_attention_02_gb300 import build as b
    b.build()
    import block_sparse_attention_02_gb300 as m
    return m


def run_chunk(msa, inp, k, ws_bytes=None, expect_err=0):
    bufs = msa.chunk_layer(inp, k, ws_bytes=ws_bytes)
    torch.cuda.synchronize()
    err = int(bufs["dev_err"].item())
    assert err == expect_err, f"device error word {err:#x}, expected {expect_err:#x}"
    return bufs


def check_chunk(msa, wl, inp_dev, bufs=None):
    sh = wl.shape
    if bufs is None:
        bufs = run_chunk(msa, inp_dev, sh.k)
    inp = {n: t.cpu() for n, t in inp_dev.items()}
    B, S = wl.B, wl.S
    Co = oracle.chunk_scores(inp["q_idx"], inp["w"], inp["kidx_pool"], inp["seq_pt"], inp["q_pos"], sh.Bk)
    nbo = Co.shape[-1]
    Cg = bufs["C"].cpu().numpy()
    check_scores(Cg[..., :nbo], Co)
    assert np.all(Cg[..., nbo:] == -np.inf), "entries past the longest context must be -inf"
    own = np.repeat(oracle.chunk_own_blocks(inp["q_pos"], S, sh.Bk)[..., None], sh.Hkv, axis=2)
    sel = bufs["sel"].cpu().numpy()
    cnt = bufs["count"].cpu().numpy()
    exact, tie = check_selection(sel.reshape(-1, sh.k), cnt.reshape(-1), Co.reshape(-1, nbo), own.reshape(-1),
                                 sh.k)
    Oo, Lo = oracle.chunk_attend(inp["Q"], inp["K_pool"], inp["V_pool"], inp["seq_pt"], inp["q_pos"], sel, cnt,
                                 1.0 / math.sqrt(sh.D), sh.Bk)
    errs = check_attention(bufs["O"].float().cpu().numpy(), bufs["LSE"].cpu().numpy(), Oo, Lo)
    return exact, tie, errs, bufs


CASES = [
    # ragged prefixes 300 / 1000 (not multiples of 64): items straddle blocks
    ChunkWorkload("ragged_b2", prefix=(300, 1000), S=200, shape=MSAShape(Hq=12, Hkv=2, k=4), seed=61),
    # MSA head shape, a 1,000-query chunk after 3,000 cached tokens
    ChunkWorkload("msa_shape", prefix=(3000,), S=1000, shape=MSAShape(), seed=62),
    # several decode tokens per sequence; a prefix shorter than one block
    ChunkWorkload("verify_s4", prefix=(1000, 129, 4000, 60), S=4, shape=MSAShape(Hq=12, Hkv=2, k=4), seed=63),
    ChunkWorkload("verify_msa_s2", prefix=(60000, 20000), S=2, shape=MSAShape(), seed=64),
    # k = 64 over ~80 blocks, HI = 3
    ChunkWorkload("hi3_k64", prefix=(9000,), S=1300, shape=MSAShape(Hq=16, Hkv=2, HI=3, k=64), seed=65),
    # one query: a decode step through the chunk path
    ChunkWorkload("single_token", prefix=(777, 5), S=1, shape=MSAShape(Hq=12, Hkv=2, k=4), seed=66),
    # 8 tokens per sequence straddling block boundaries (tokens of one sequence
    # with different own blocks), HI = 3, a prefix inside block 0
    ChunkWorkload("straddle_s8_hi3", prefix=(125, 1020, 250, 3), S=8, shape=MSAShape(Hq=12, Hkv=2, HI=3, k=4),
                  seed=75),
    # 5 tokens, MSA head shape, prefixes whose tokens cross a block boundary (60,030 + 2 = 60,032 = 469 * 128)
    ChunkWorkload("verify_msa_s5", prefix=(60030, 383), S=5, shape=MSAShape(), seed=76),
]


@pytest.mark.parametrize("wl", CASES, ids=[w.name for w in CASES])
def test_chunk_matches_oracle(msa, wl):
    inp = chunk_inputs(wl, device="cuda")
    exact, tie, errs, _ = check_chunk(msa, wl, inp)
    print(f"{wl.name}: exact rows {exact}, near-tie rows {tie}, O max/mean {errs[0]:.2e}/{errs[1]:.2e}")


def test_chunk_shared_index_pool(msa):
    """One index-key pool for all KV groups (group stride 0)."""
    wl = ChunkWorkload("shared", prefix=(2000, 700), S=300, shape=MSAShape(Hq=48, Hkv=8, k=8), seed=67)
    inp = chunk_inputs(wl, device="cuda")
    inp["kidx_pool"] = inp["kidx_pool"][:, :1].expand(-1, wl.shape.Hkv, -1, -1)
    assert inp["kidx_pool"].stride(1) == 0
    check_chunk(msa, wl, inp)


def test_chunk_few_tokens_shared_index_pool(msa):
    """A few tokens per sequence with one index-key pool for all KV groups
    (scored by the prefill kernel's few-query variant)."""
    wl = ChunkWorkload("shared_s4", prefix=(2000, 700), S=4, shape=MSAShape(Hq=48, Hkv=8, k=8), seed=77)
    inp = chunk_inputs(wl, device="cuda")
    inp["kidx_pool"] = inp["kidx_pool"][:, :1].expand(-1, wl.shape.Hkv, -1, -1)
    assert inp["kidx_pool"].stride(1) == 0
    check_chunk(msa, wl, inp)


def test_chunk_from_position_zero_equals_prefill(msa):
    """q_pos = 0 over shuffled pages: the same bits as the contiguous prefill."""
    sh = MSAShape(Hq=12, Hkv=2, k=6)
    wl = PrefillWorkload("pos0", B=2, S=1500, shape=sh, seed=68)
    inp = prefill_inputs(wl, device="cuda")
    ref = msa.prefill_layer(inp, sh.k)
    Bk, n = sh.Bk, (wl.S + sh.Bk - 1) // sh.Bk
    perm = torch.randperm(wl.B * n, generator=torch.Generator().manual_seed(3)).cuda()

    def paged(x):
        pad = torch.zeros(wl.B, n * Bk, *x.shape[2:], dtype=x.dtype, device=x.device)
        pad[:, :wl.S] = x
        blocks = pad.view(wl.B, n, Bk, *x.shape[2:]).transpose(2, 3).reshape(wl.B * n, x.shape[2], Bk, -1)
        pool = torch.empty_like(blocks)
        pool[perm] = blocks
        return pool

    cin = {"Q": inp["Q"], "q_idx": inp["q_idx"], "w": inp["w"], "K_pool": paged(inp["K"]),
           "V_pool": paged(inp["V"]), "kidx_pool": paged(inp["k_idx"]),
           "seq_pt": perm.view(wl.B, n).to(torch.int32).contiguous(),
           "q_pos": torch.zeros(wl.B, dtype=torch.int32, device="cuda")}
    got = run_chunk(msa, cin, sh.k)
    torch.cuda.synchronize()
    assert int(ref["dev_err"].item()) == 0
    assert torch.equal(got["C"], ref["C"])
    for name in ("sel", "count", "O", "LSE"):
        assert torch.equal(got[name], ref[name]), name


def test_chunk_small_workspace_is_bit_identical(msa):
    wl = ChunkWorkload("ws", prefix=(5000, 2500), S=900, shape=MSAShape(Hq=12, Hkv=2, k=8), seed=69)
    inp = chunk_inputs(wl, device="cuda")
    sel_probe = torch.empty(1, 1, 1, wl.shape.k, dtype=torch.int32)
    small = msa.msa_sparse_attn_prefill_workspace_size(inp["Q"], inp["K_pool"], sel_probe, 257,
                                                       max_pages=wl.max_pages)
    a = run_chunk(msa, inp, wl.shape.k)
    b = run_chunk(msa, inp, wl.shape.k, ws_bytes=small)
    for name in ("sel", "count", "O", "LSE"):
        assert torch.equal(a[name], b[name]), name


@pytest.mark.parametrize("S", [100, 4], ids=["kv_block_major", "decode_path"])
def test_chunk_rejected_sequence_and_page(msa, S):
    """A sequence whose chunk leaves the pages gets count 0, zero output and
    LSE -inf (MSA_DEVERR_BAD_LEN); a page id outside the pool is reported
    (MSA_DEVERR_BAD_PAGE) and the other sequences are unaffected.  S = 4 runs
    the attention through the decode kernel."""
    wl = ChunkWorkload("bad", prefix=(1000, 600, 300), S=S, shape=MSAShape(Hq=12, Hkv=2, k=4), seed=70)
    inp = chunk_inputs(wl, device="cuda")
    good = run_chunk(msa, inp, wl.shape.k)
    bad = dict(inp)
    bad["q_pos"] = inp["q_pos"].clone()
    bad["q_pos"][1] = wl.max_pages * wl.shape.Bk          # the chunk would end past the page table
    bufs = run_chunk(msa, bad, wl.shape.k, expect_err=msa.MSA_DEVERR_BAD_LEN)
    assert int(bufs["count"][1].abs().sum().item()) == 0
    assert torch.all(bufs["O"][1] == 0) and torch.all(bufs["LSE"][1] == -math.inf)
    for name in ("count", "sel", "O", "LSE"):
        assert torch.equal(bufs[name][0], good[name][0]) and torch.equal(bufs[name][2], good[name][2]), name
    bad = dict(inp)
    bad["seq_pt"] = inp["seq_pt"].clone()
    bad["seq_pt"][2, 0] = inp["K_pool"].shape[0] + 7        # block 0 of sequence 2: no such page
    bufs = run_chunk(msa, bad, wl.shape.k, expect_err=msa.MSA_DEVERR_BAD_PAGE)
    for name in ("count", "sel", "O", "LSE"):
        assert torch.equal(bufs[name][0], good[name][0]) and torch.equal(bufs[name][1], good[name][1]), name
    # the block on the missing page is not loaded: -inf in every row of that sequence
    assert torch.isneginf(bufs["C"][2, :, :, 0]).all()
    assert torch.equal(bufs["C"][2, :, :, 1:], good["C"][2, :, :, 1:])


def test_chunk_few_queries_run_through_the_decode_kernel(msa):
    """S <= 8 with a dense Q: the workspace is that of the decode path (page
    table and fp32 partials of B*S*Hq*k parts) whatever the query chunk, and
    the outputs match the oracle (checked in the verify cases above); here a
    4-token verification at the MSA shape also agrees with four one-token
    chunk calls at consecutive positions, which take the same path."""
    wl = ChunkWorkload("few", prefix=(5000, 777), S=4, shape=MSAShape(), seed=74)
    inp = chunk_inputs(wl, device="cuda")
    sel_probe = torch.empty(1, 1, 1, wl.shape.k, dtype=torch.int32)
    a = msa.msa_sparse_attn_prefill_workspace_size(inp["Q"], inp["K_pool"], sel_probe, 1, max_pages=wl.max_pages)
    b = msa.msa_sparse_attn_prefill_workspace_size(inp["Q"], inp["K_pool"], sel_probe, 8, max_pages=wl.max_pages)
    assert a == b >= wl.B * wl.S * wl.shape.Hq * wl.shape.k * (wl.shape.D + 1) * 4
    whole = run_chunk(msa, inp, wl.shape.k)
    for s in range(wl.S):
        one = dict(inp, Q=inp["Q"][:, s:s + 1].contiguous(), q_idx=inp["q_idx"][:, s:s + 1].contiguous(),
                   w=inp["w"][:, s:s + 1].contiguous(), q_pos=inp["q_pos"] + s)
        got = run_chunk(msa, one, wl.shape.k)
        for name in ("sel", "count", "O", "LSE"):
            assert torch.equal(got[name][:, 0], whole[name][:, s]), (name, s)


def test_chunk_rejects_a_sequence_whose_last_query_leaves_the_pages(msa):
    """The first query of sequence 1 is inside the page table and the last is
    not: index score and top-k reject the sequence as a whole (count 0, zero
    output, LSE -inf, MSA_DEVERR_BAD_LEN); the other sequences are unchanged."""
    wl = ChunkWorkload("bad_tail", prefix=(1000, 600, 300), S=100, shape=MSAShape(Hq=12, Hkv=2, k=4), seed=73)
    inp = chunk_inputs(wl, device="cuda")
    good = run_chunk(msa, inp, wl.shape.k)
    bad = dict(inp)
    bad["q_pos"] = inp["q_pos"].clone()
    bad["q_pos"][1] = wl.max_pages * wl.shape.Bk - wl.S // 2
    bufs = run_chunk(msa, bad, wl.shape.k, expect_err=msa.MSA_DEVERR_BAD_LEN)
    assert torch.isneginf(bufs["C"][1]).all()
    assert int(bufs["count"][1].abs().sum().item()) == 0 and torch.all(bufs["sel"][1] == -1)
    assert torch.all(bufs["O"][1] == 0) and torch.all(bufs["LSE"][1] == -math.inf)
    for name in ("C", "count", "sel", "O", "LSE"):
        assert torch.equal(bufs[name][0], good[name][0]) and torch.equal(bufs[name][2], good[name][2]), name


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("shared", [False, True], ids=["per_group", "shared_index_pool"])
def test_chunk_append_then_layer(msa, shared):
    """The chunk's own tokens, cleared from the pages and appended back with one
    msa_cache_append call (T = S tokens per sequence, crossing page
    boundaries), restore the pools bit for bit (the oracle's copies agree), and
    the layer over them gives the same bits as before."""
    wl = ChunkWorkload("append", prefix=(300, 1000, 127), S=200, shape=MSAShape(Hq=12, Hkv=2, k=4), seed=71)
    inp = chunk_inputs(wl, device="cuda")
    if shared:
        inp["kidx_pool"] = inp["kidx_pool"][:, :1].expand(-1, wl.shape.Hkv, -1, -1)
    ref = run_chunk(msa, inp, wl.shape.k)
    pos = inp["q_pos"].long()[:, None] + torch.arange(wl.S, device="cuda")[None, :]
    pages = torch.gather(inp["seq_pt"].long(), 1, pos // wl.shape.Bk)
    slots = pos % wl.shape.Bk
    names = ("K_pool", "V_pool", "kidx_pool")
    new = [inp[n][pages, :, slots].contiguous() for n in names]       # [B, S, Hkv, d]
    cleared = {n: inp[n].clone() if not (shared and n == "kidx_pool") else inp[n][:, :1].clone() for n in names}
    for n in names:
        cleared[n][pages, :, slots] = 0
    if shared:
        cleared["kidx_pool"] = cleared["kidx_pool"].expand(-1, wl.shape.Hkv, -1, -1)
    want = oracle.cache_append(*[t.cpu() for t in new], *[cleared[n].cpu() for n in names], inp["seq_pt"].cpu(),
                               inp["seq_len"].cpu(), wl.shape.Bk, shared_index=shared)
    assert want[3] == []
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    msa.msa_cache_append(*new, *[cleared[n] for n in names], inp["seq_pt"], inp["seq_len"], dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for n, w in zip(names, want[:3]):
        assert np.array_equal(_bits(cleared[n]), w), n
        assert torch.equal(cleared[n], inp[n]), n
    got = run_chunk(msa, dict(inp, **cleared), wl.shape.k)
    for name in ("C", "sel", "count", "O", "LSE"):
        assert torch.equal(got[name], ref[name]), name


def test_chunk_append_rejects_short_sequence_and_bad_page(msa):
    """A sequence shorter than T writes nothing (MSA_DEVERR_BAD_LEN); a token
    whose page id is outside the pool is skipped alone (MSA_DEVERR_BAD_PAGE);
    the pools match the oracle's copies bit for bit."""
    g = torch.Generator(device="cuda").manual_seed(72)
    P, Hkv, D_, dI_, mp, T = 32, 2, 128, 64, 4, 5
    seq_len = torch.tensor([3, 130, 300, 129], dtype=torch.int32, device="cuda")
    B = seq_len.shape[0]
    pools = [torch.randn(P, Hkv, 128, d, generator=g, device="cuda").to(torch.bfloat16) for d in (D_, D_, dI_)]
    new = [torch.randn(B, T, Hkv, d, generator=g, device="cuda").to(torch.bfloat16) for d in (D_, D_, dI_)]
    seq_pt = torch.randperm(P, generator=g, device="cuda")[: B * mp].view(B, mp).to(torch.int32).contiguous()
    seq_pt[3, 1] = P + 9                                  # position 128 of sequence 3: no such page
    K2, V2, X2, skipped = oracle.cache_append(*[t.cpu() for t in new], *[t.cpu() for t in pools], seq_pt.cpu(),
                                              seq_len.cpu(), 128)
    assert skipped == [(0, u) for u in range(T)] + [(3, 4)]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    msa.msa_cache_append(*new, *pools, seq_pt, seq_len, dev_err=err)
    torch.cuda.synchronize()
    for got, want in zip(pools, (K2, V2, X2)):
        assert np.array_equal(_bits(got), want)
    assert int(err.item()) == msa.MSA_DEVERR_BAD_LEN | msa.MSA_DEVERR_BAD_PAGE
