"""The replicas' data split through the CUDA library: two processes (gloo
ranks) each run the library's decode step and chunk layer on their share of
the sequences, and the gathered outputs equal the library's unsplit run bit
for bit and the oracle within the stated tolerances.

On a box with one GPU both ranks use device 0: their kernels are independent
(no rank waits on another's kernels; the only exchange is gloo on CPU tensors
after the GPU work), so this is the same data path bench.py runs with one
replica per GPU.
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

pytestmark = pytest.mark.gpu

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
    torch.cuda.set_device(0)
    import block_sparse_attention_02_gb300 as msa
    from workloads import ChunkWorkload, DecodeWorkload, MSAShape, chunk_inputs, decode_inputs

    wl = DecodeWorkload("replica_gpu", lengths=(3000, 777, 60001, 129, 20000), shape=MSAShape(), seed=91)
    inp = decode_inputs(wl, device="cuda")
    mine = list(range(rank, wl.B, world))
    sub = {n: (inp[n][mine].contiguous() if n in ("Q", "q_idx", "w", "seq_pt", "seq_len") else inp[n]) for n in inp}
    out = msa.decode_step(sub, wl.shape.k)
    torch.cuda.synchronize()
    assert int(out["dev_err"].item()) == 0
    got = [None] * world
    dist.all_gather_object(got, (mine, out["O"].cpu(), out["LSE"].cpu(), out["sel"].cpu()))

    cw = ChunkWorkload("replica_gpu_chunk", prefix=(300, 1000, 129, 5000), S=4, shape=MSAShape(), seed=92)
    cin = chunk_inputs(cw, device="cuda")
    cmine = list(range(rank, cw.B, world))
    csub = {n: (cin[n][cmine].contiguous() if n in ("Q", "q_idx", "w", "seq_pt", "q_pos", "seq_len") else cin[n])
            for n in cin}
    cout = msa.chunk_layer(csub, cw.shape.k)
    torch.cuda.synchronize()
    assert int(cout["dev_err"].item()) == 0
    cgot = [None] * world
    dist.all_gather_object(cgot, (cmine, cout["O"].cpu(), cout["LSE"].cpu()))
    if rank == 0:
        torch.save({"decode": got, "chunk": cgot}, os.path.join(out_dir, "shards.pt"))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_split_by_sequence_match_unsplit_run(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    sys.path.insert(0, ROOT)
    from block_sparse_attention_02_gb300 import build as b
    b.build()
    mp.start_processes(_worker, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    import block_sparse_attention_02_gb300 as msa
    import oracle
    from msa_check import check_attention
    from workloads import ChunkWorkload, DecodeWorkload, MSAShape, chunk_inputs, decode_inputs
    shards = torch.load(tmp_path / "shards.pt")

    wl = DecodeWorkload("replica_gpu", lengths=(3000, 777, 60001, 129, 20000), shape=MSAShape(), seed=91)
    inp = decode_inputs(wl, device="cuda")
    full = msa.decode_step(inp, wl.shape.k)
    torch.cuda.synchronize()
    O = torch.empty_like(full["O"].cpu())
    L = torch.empty_like(full["LSE"].cpu())
    sel = torch.empty_like(full["sel"].cpu())
    for idx, o, lse, s in shards["decode"]:
        O[idx], L[idx], sel[idx] = o, lse, s
    assert torch.equal(O, full["O"].cpu()) and torch.equal(L, full["LSE"].cpu()) and torch.equal(sel, full["sel"].cpu())
    h = {n: inp[n].cpu() for n in ("Q", "K_pool", "V_pool", "seq_pt", "seq_len")}
    O_o, L_o = oracle.decode_attend(h["Q"], h["K_pool"], h["V_pool"], h["seq_pt"], h["seq_len"], sel.numpy(),
                                    full["count"].cpu().numpy(), 1.0 / math.sqrt(wl.shape.D))
    check_attention(O.float().numpy(), L.numpy(), O_o, L_o)

    cw = ChunkWorkload("replica_gpu_chunk", prefix=(300, 1000, 129, 5000), S=4, shape=MSAShape(), seed=92)
    cin = chunk_inputs(cw, device="cuda")
    cfull = msa.chunk_layer(cin, cw.shape.k)
    torch.cuda.synchronize()
    CO = torch.empty_like(cfull["O"].cpu())
    CL = torch.empty_like(cfull["LSE"].cpu())
    for idx, o, lse in shards["chunk"]:
        CO[idx], CL[idx] = o, lse
    assert torch.equal(CO, cfull["O"].cpu()) and torch.equal(CL, cfull["LSE"].cpu())
    assert np.isfinite(CO.float().numpy()).all()
