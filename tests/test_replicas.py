"""The N > 1 host logic on CPU with two gloo ranks.

The MSA hot path shards by sequence (decode) or by KV group with no collective
in the data path; bench.py runs one replica per GPU and only aggregates timings
(barrier + max over ranks).  Here two gloo processes check bench.py's
aggregation (max over ranks) and that the computation is separable the way the
replicas split it: a decode batch and a chunk batch (several queries per
sequence over the paged cache) split by sequence across ranks give exactly the
results of the unsplit batches.  The per-rank results come from the oracle
(all-gathered only for the check), so this covers the sharding and the bench's
aggregation, not the CUDA library; the library's per-sequence independence is
covered by the GPU tests (a sequence's outputs do not change when other
sequences of the batch are rejected or change).
"""
import math
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import oracle
    from workloads import ChunkWorkload, DecodeWorkload, MSAShape, chunk_inputs, decode_inputs

    # timing aggregation: every rank sees the max
    mx = bench.max_over_ranks(float(10 + rank), world)
    # decode batch sharded by sequence: rank r owns sequences r, r + world, ...
    wl = DecodeWorkload("replica", lengths=(300, 1000, 2049, 129), shape=MSAShape(Hq=12, Hkv=2, k=4), seed=71)
    inp = decode_inputs(wl)
    mine = list(range(rank, wl.B, world))
    sub = {n: inp[n][mine] for n in ("Q", "q_idx", "w", "seq_pt", "seq_len")}
    sub.update({n: inp[n] for n in ("kidx_pool", "K_pool", "V_pool")})
    C = oracle.decode_scores(sub["q_idx"], sub["w"], sub["kidx_pool"], sub["seq_pt"], sub["seq_len"])
    own = oracle.own_blocks_decode(sub["seq_len"], wl.shape.Bk)
    sel, cnt, _, _ = oracle.select(C, own[:, None], wl.shape.k)
    O, _ = oracle.decode_attend(sub["Q"], sub["K_pool"], sub["V_pool"], sub["seq_pt"], sub["seq_len"], sel, cnt,
                                1.0 / math.sqrt(wl.shape.D))
    gathered = [None] * world
    dist.all_gather_object(gathered, (mine, O))
    # chunk batch sharded the same way
    cw = ChunkWorkload("replica_chunk", prefix=(300, 1000, 129, 40), S=3, shape=MSAShape(Hq=12, Hkv=2, k=4), seed=72)
    cin = chunk_inputs(cw)
    cmine = list(range(rank, cw.B, world))
    r = oracle.chunk_layer(cin["Q"][cmine], cin["q_idx"][cmine], cin["w"][cmine], cin["K_pool"], cin["V_pool"],
                           cin["kidx_pool"], cin["seq_pt"][cmine], cin["q_pos"][cmine], cw.shape.k,
                           1.0 / math.sqrt(cw.shape.D), cw.shape.Bk)
    cgathered = [None] * world
    dist.all_gather_object(cgathered, (cmine, r["O"]))
    if rank == 0:
        np.save(os.path.join(out_dir, "max.npy"), np.array([mx]))
        full = np.zeros((wl.B,) + O.shape[1:])
        for idx, o in gathered:
            full[idx] = o
        np.save(os.path.join(out_dir, "sharded.npy"), full)
        cfull = np.zeros((cw.B,) + r["O"].shape[1:])
        for idx, o in cgathered:
            cfull[idx] = o
        np.save(os.path.join(out_dir, "sharded_chunk.npy"), cfull)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    assert float(np.load(tmp_path / "max.npy")[0]) == 11.0
    sys.path.insert(0, ROOT)
    import oracle
    from workloads import ChunkWorkload, DecodeWorkload, MSAShape, chunk_inputs, decode_inputs
    wl = DecodeWorkload("replica", lengths=(300, 1000, 2049, 129), shape=MSAShape(Hq=12, Hkv=2, k=4), seed=71)
    inp = decode_inputs(wl)
    C = oracle.decode_scores(inp["q_idx"], inp["w"], inp["kidx_pool"], inp["seq_pt"], inp["seq_len"])
    own = oracle.own_blocks_decode(inp["seq_len"], wl.shape.Bk)
    sel, cnt, _, _ = oracle.select(C, own[:, None], wl.shape.k)
    O, _ = oracle.decode_attend(inp["Q"], inp["K_pool"], inp["V_pool"], inp["seq_pt"], inp["seq_len"], sel, cnt,
                                1.0 / math.sqrt(wl.shape.D))
    np.testing.assert_array_equal(np.load(tmp_path / "sharded.npy"), O)
    cw = ChunkWorkload("replica_chunk", prefix=(300, 1000, 129, 40), S=3, shape=MSAShape(Hq=12, Hkv=2, k=4), seed=72)
    cin = chunk_inputs(cw)
    r = oracle.chunk_layer(cin["Q"], cin["q_idx"], cin["w"], cin["K_pool"], cin["V_pool"], cin["kidx_pool"],
                           cin["seq_pt"], cin["q_pos"], cw.shape.k, 1.0 / math.sqrt(cw.shape.D), cw.shape.Bk)
    np.testing.assert_array_equal(np.load(tmp_path / "sharded_chunk.npy"), r["O"])
