"""The bench's host-side accounting, on CPU: the algorithmic work the roofline
numbers divide by, worked out by hand on tiny cases, and the oracle baselines
on small workloads."""
import math

import torch

import bench
from workloads import ChunkWorkload, DecodeWorkload, MSAShape, PrefillWorkload, chunk_inputs, prefill_inputs


def test_attention_flops_count_visible_keys():
    """4*D*G per visible (query, group, key): one sequence at position 130 with
    blocks {0, 1} sees 128 + 3 keys; one at 300 with {0, 2, 3} sees 128 + 45 + 0;
    -1 slots count nothing."""
    sel = torch.tensor([[[[0, 1, -1]]], [[[0, 2, 3]]]], dtype=torch.int32)   # [B=2, S=1, Hkv=1, k=3]
    cnt = torch.tensor([[[2]], [[3]]], dtype=torch.int32)
    q_pos = torch.tensor([130, 300], dtype=torch.int32)
    D, G = 128, 6
    assert bench.prefill_attention_flops(sel, cnt, 1, 128, G, D, q_pos) == (131 + 173) * 4 * D * G
    # a prefill (positions 0..S-1): query 200 with blocks {0, 1} sees 128 + 73 keys
    sel2 = torch.full((1, 201, 1, 2), -1, dtype=torch.int32)
    sel2[0, 200, 0] = torch.tensor([0, 1])
    assert bench.prefill_attention_flops(sel2, None, 201, 128, 1, 1) == (128 + 73) * 4


def test_decode_bytes_by_hand():
    """lengths 129 and 300, Hkv = 2, k = 2, dI = 64, D = 128: index keys of
    blocks before the own one (1 and 2 blocks per group), the selected K/V
    tokens (one earlier block + the own block's valid tokens), q_idx/w/C and
    Q/O."""
    sh = MSAShape(Hq=4, Hkv=2, HI=4, k=2)
    wl = DecodeWorkload("t", lengths=(129, 300), shape=sh, seed=0)
    got = bench.decode_algorithmic_bytes(wl)
    idx = 2 * (1 + 2) * 128 * 64 * 2
    small = 2 * 2 * (4 * 64 * 2 + 4 * 4) + 2 * 2 * 3 * 4
    kv = 2 * ((128 + 1) + (128 + 44)) * 128 * 2 * 2
    qo = 2 * 4 * 128 * 2 * 2
    assert got == {"index_kernel": idx + small, "step": idx + small + kv + qo}
    shared = bench.decode_algorithmic_bytes(wl, shared_index=True)
    assert shared["index_kernel"] == (1 + 2) * 128 * 64 * 2 + small


def test_oracle_baselines_on_small_workloads():
    """The sampled oracle rates run on CPU and describe their sample."""
    sh = MSAShape(Hq=4, Hkv=1, HI=2, k=4)
    pw = PrefillWorkload("p", B=1, S=512, shape=sh, seed=1)
    r = bench.cpu_prefill_baseline(pw, prefill_inputs(pw), budget_s=0.05)
    assert r["value"] > 0 and r["kind"] == "oracle" and "query rows" in r["sample"]
    cw = ChunkWorkload("c", prefix=(300, 40), S=3, shape=sh, seed=2)
    r = bench.cpu_chunk_baseline(cw, chunk_inputs(cw), budget_s=0.05)
    assert r["value"] > 0 and "query offsets" in r["sample"]
    assert math.isfinite(r["value"])


def test_dense_comparator_work_by_hand():
    """Dense decode reads every cached K and V token once (plus Q, O); a dense
    causal prefill does 4*D FLOPs per (query head, visible key), S(S+1)/2 keys
    per head."""
    sh = MSAShape(Hq=4, Hkv=2, HI=4, k=2)
    wl = DecodeWorkload("t", lengths=(129, 300), shape=sh, seed=0)
    assert bench.dense_decode_bytes(wl) == (129 + 300) * 2 * 128 * 2 * 2 + 2 * 4 * 128 * 2 * 2
    pw = PrefillWorkload("p", B=2, S=3, shape=sh, seed=0)
    assert bench.dense_prefill_flops(pw) == 4 * 128 * 4 * 2 * (1 + 2 + 3)


def test_decode_baseline_reports_one_thread_rate():
    sh = MSAShape(Hq=4, Hkv=1, HI=2, k=4)
    wl = DecodeWorkload("d", lengths=(300, 129), shape=sh, seed=3)
    from workloads import decode_inputs
    r = bench.cpu_decode_baseline(wl, decode_inputs(wl), budget_s=0.05)
    assert r["value"] > 0 and r["value_1_thread"] > 0 and "single" not in r["sample"]
