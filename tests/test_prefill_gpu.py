"""Prefill path (a1 index score -> a2 top-k -> a3'/a4/a6 KV-block-major sparse
attention) against the fp64 oracle, through the C ABI, on a GB300.

Small cases cover ragged sequence lengths (tails that are not a multiple of
Bk), batch > 1, GQA ratios 1/6/8, HI = 1..4 and k = 1/4/16/64, the tiny
workload at k = 4 and at k = 16 (which covers every block, i.e. dense causal
GQA), and chunked processing with a small workspace.  The long prefill
(S = 131,072) runs in full on the GPU and is checked on sampled query rows,
which the oracle computes one by one.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from msa_check import check_attention, check_scores, check_selection
from workloads import MSAShape, PrefillWorkload, prefill_inputs, workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msa():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from block_sparse_attention_02_gb300 import build as b
    b.build()
    import block_sparse_attention_02_gb300 as m
    return m


def run_gpu(msa, inp, k, ws_bytes=None):
    bufs = msa.prefill_layer(inp, k, ws_bytes=ws_bytes)
    torch.cuda.synchronize()
    assert int(bufs["dev_err"].item()) == 0, f"device error word {int(bufs['dev_err'].item()):#x}"
    return bufs


def check_prefill(msa, wl, inp_dev, rows=None, ws_bytes=None, bufs=None):
    sh = wl.shape
    if bufs is None:
        bufs = run_gpu(msa, inp_dev, sh.k, ws_bytes)
    B, S = wl.B, wl.S
    rows = np.arange(B * S, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    inp = {n: t.cpu() for n, t in inp_dev.items() if n in ("Q", "K", "V", "q_idx", "k_idx", "w")}
    nb = wl.nb
    Cg = bufs["C"].reshape(B * S, sh.Hkv, nb)[torch.as_tensor(rows, device=bufs["C"].device)].cpu().numpy()
    Co = oracle.prefill_scores(inp["q_idx"], inp["k_idx"], inp["w"], sh.Bk, rows)
    check_scores(Cg, Co)
    own = np.repeat(oracle.own_blocks_prefill(S, sh.Bk, rows), sh.Hkv)
    ridx = torch.as_tensor(rows, device=bufs["sel"].device)
    sel = bufs["sel"].reshape(B * S, sh.Hkv, sh.k)[ridx].cpu().numpy()
    cnt = bufs["count"].reshape(B * S, sh.Hkv)[ridx].cpu().numpy()
    exact, tie = check_selection(sel.reshape(-1, sh.k), cnt.reshape(-1), Co.reshape(len(own), -1), own, sh.k)
    Oo, Lo = oracle.prefill_attend(inp["Q"], inp["K"], inp["V"], sel, cnt, sh.Bk, 1.0 / math.sqrt(sh.D), rows)
    Og = bufs["O"].reshape(B * S, sh.Hq, sh.D)[ridx].float().cpu().numpy()
    Lg = bufs["LSE"].reshape(B * S, sh.Hq)[ridx].cpu().numpy()
    errs = check_attention(Og, Lg, Oo, Lo)
    return exact, tie, errs, bufs


SMALL = [
    workload("prefill_tiny_s2048"),
    workload("prefill_tiny_s2048_k16"),
    PrefillWorkload("ragged_b2", B=2, S=1000, shape=MSAShape(Hq=12, Hkv=2, k=4), seed=41),
    PrefillWorkload("gqa8_hi3", B=1, S=1500, shape=MSAShape(Hq=16, Hkv=2, HI=3, k=6), seed=42),
    PrefillWorkload("gqa1_hi1", B=1, S=700, shape=MSAShape(Hq=4, Hkv=4, HI=1, k=2), seed=43),
    PrefillWorkload("k1", B=1, S=640, shape=MSAShape(Hq=6, Hkv=1, HI=2, k=1), seed=44),
    PrefillWorkload("k64_long", B=1, S=9000, shape=MSAShape(Hq=12, Hkv=2, k=64), seed=45),
    PrefillWorkload("msa_shape_s4096", B=1, S=4096, shape=MSAShape(), seed=46),
    PrefillWorkload("tail_1", B=3, S=129, shape=MSAShape(Hq=12, Hkv=2, k=16), seed=47),
    # shorter than one key block: no index pass runs, every score row is -inf
    PrefillWorkload("edge_s1", B=2, S=1, shape=MSAShape(Hq=12, Hkv=2, k=4), seed=48),
    PrefillWorkload("edge_s64", B=1, S=64, shape=MSAShape(), seed=49),
    # one query block pair with a partial second 64-query block
    PrefillWorkload("edge_s200_hi2", B=2, S=200, shape=MSAShape(Hq=12, Hkv=2, HI=2, k=2), seed=50),
    # GQA ratios 5 and 3: an entry's packed partial rows are G * 16 bytes per column chunk
    PrefillWorkload("gqa5", B=1, S=900, shape=MSAShape(Hq=10, Hkv=2, k=5), seed=51),
    PrefillWorkload("gqa3_b2", B=2, S=700, shape=MSAShape(Hq=9, Hkv=3, k=3), seed=52),
]


@pytest.mark.parametrize("wl", SMALL, ids=[w.name for w in SMALL])
def test_prefill_small(msa, wl):
    inp = prefill_inputs(wl, device="cuda")
    exact, tie, errs, _ = check_prefill(msa, wl, inp)
    print(f"{wl.name}: exact rows {exact}, near-tie rows {tie}, O max/mean {errs[0]:.2e}/{errs[1]:.2e}")


def test_dense_limit_matches_dense_gqa(msa):
    """k >= number of blocks: the sparse path is dense causal GQA attention."""
    wl = workload("prefill_tiny_s2048_k16")
    sh = wl.shape
    inp = prefill_inputs(wl, device="cuda")
    bufs = run_gpu(msa, inp, sh.k)
    q = inp["Q"].double().permute(0, 2, 1, 3)
    kk = inp["K"].double().repeat_interleave(sh.G, dim=2).permute(0, 2, 1, 3)
    vv = inp["V"].double().repeat_interleave(sh.G, dim=2).permute(0, 2, 1, 3)
    ref = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, is_causal=True, scale=1 / math.sqrt(sh.D))
    err = (bufs["O"].double() - ref.permute(0, 2, 1, 3)).abs()
    assert err.max().item() <= 1e-2 and err.mean().item() <= 1e-3


def test_chunked_workspace_is_bit_identical(msa):
    """A workspace that forces many query chunks gives the same bits as one chunk."""
    wl = PrefillWorkload("chunks", B=2, S=3000, shape=MSAShape(Hq=12, Hkv=2, k=8), seed=48)
    sh = wl.shape
    inp = prefill_inputs(wl, device="cuda")
    sel_probe = torch.empty(1, 1, 1, sh.k, dtype=torch.int32)
    big = msa.msa_sparse_attn_prefill_workspace_size(inp["Q"], inp["K"], sel_probe, wl.B * wl.S)
    small = msa.msa_sparse_attn_prefill_workspace_size(inp["Q"], inp["K"], sel_probe, 333)
    a = run_gpu(msa, inp, sh.k, big)
    b = run_gpu(msa, inp, sh.k, small)
    assert torch.equal(a["O"], b["O"]) and torch.equal(a["LSE"], b["LSE"])
    check_prefill(msa, wl, inp, bufs=b)


def test_prefill_is_deterministic(msa):
    wl = PrefillWorkload("det", B=1, S=5000, shape=MSAShape(), seed=49)
    inp = prefill_inputs(wl, device="cuda")
    a = run_gpu(msa, inp, 16)
    b = run_gpu(msa, inp, 16)
    for n in ("C", "sel", "count", "O", "LSE"):
        assert torch.equal(a[n], b[n]), n


def sampled_rows(S, Bk, n_random, seed):
    """Blocks 0-1, every 128th block boundary, the last block, and random rows."""
    rng = np.random.default_rng(seed)
    r = set(range(0, 2 * Bk, 37)) | {S - 1, S - 2, S - Bk}
    r |= {x for x in range(0, S, 128 * Bk)} | {x + Bk - 1 for x in range(0, S, 128 * Bk) if x + Bk - 1 < S}
    r |= set(rng.integers(0, S, n_random).tolist())
    return np.array(sorted(r), dtype=np.int64)


def test_prefill_s131072_sampled(msa):
    wl = workload("prefill_s131072")
    inp = prefill_inputs(wl, device="cuda")
    rows = sampled_rows(wl.S, wl.shape.Bk, 24, seed=1)
    exact, tie, errs, _ = check_prefill(msa, wl, inp, rows=rows)
    print(f"prefill_s131072: {len(rows)} sampled rows, exact {exact}, near-tie {tie}, errs {errs}")


def test_prefill_shared_index_keys(msa):
    """One k_idx for all KV groups (group stride 0): scores, selection and
    attention match the oracle on the broadcast tensor."""
    wl = PrefillWorkload("shared_k_idx", B=2, S=1000, shape=MSAShape(Hq=12, Hkv=2, k=4), seed=64)
    inp = prefill_inputs(wl, device="cuda")
    inp["k_idx"] = inp["k_idx"][:, :, :1].expand(-1, -1, wl.shape.Hkv, -1)
    assert inp["k_idx"].stride(2) == 0
    exact, tie, errs, _ = check_prefill(msa, wl, inp)
    print(f"shared k_idx: exact rows {exact}, near-tie rows {tie}, O max/mean {errs[0]:.2e}/{errs[1]:.2e}")
