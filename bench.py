"""Benchmark of the MSA layer hot path on one GB300 (or N replicas).

Default workload: one MSA decode step at concurrency 8 over a 60,000-token
cached prefix (B = 8, L = 60,001, Hq = 48, Hkv = 8, D = 128, index 4 x 64,
Bk = 128, k = 16, shuffled 128-token pages).  A step runs the whole hot path:
index score -> top-k -> page table -> paged sparse attention -> LSE merge.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--also NAMES] [--no-cpu-baseline]

The default run also times the other full-size workloads of the metric, one
after the other, each with its own warm-up, timed steps, roofline, clocks and
oracle baseline: one 131,072-token prefill layer (``prefill_s131072``), the
1M-token decode step (``decode_b1_l1048576``) and the ragged decode batch of
64 sequences (``decode_ragged_b64``).  Then the dense comparator (attention
over every token, no index branch: the baseline the pages quote MSA's
speedups against) on the concurrency-8 and 1M decode inputs and the
131,072-token prefill inputs ("dense:<workload>"), and "msa_vs_dense" holds
the same-box ratios of MSA tokens/s to dense tokens/s.  They appear under
"workloads" in the same JSON line; the top-level ``value`` stays the
concurrency-8 decode step.

Prints one JSON line (rank 0).  ``value`` is decode tokens/s (sequences
advanced by one token per second, all ranks), timed with CUDA events on the
launching stream over exactly K steps bracketed by barrier + synchronize.  The
default step reads 557 MB (the 491 MB of index keys alone exceed the 129 MB
L2), so nothing is flushed; a step that reads less than twice the L2 (one
index-key pool shared by the KV groups at this size) has a 258 MB buffer
read before each step, outside the timed region, and its per-step event
times are summed.  ``roofline`` reports the dominant kernel (decode index
scoring): algorithmic bytes per launch / its mean event-timed duration against
the measured HBM copy bandwidth.  ``e2e`` repeats the step through the same C
ABI with the step's inputs copied from pinned host memory and its outputs read
back inside the timed region (inputs and outputs each packed in one buffer:
one copy each way per step).  ``cpu_baseline`` times the fp64 oracle on a
bounded sample of the same workload on the host cores.

``--impl reference`` times the oracle itself (the only reference this method
has: the pages ship no code) on the same workload and prints the same line
with "impl": "reference": whole decode steps, or, for the prefill and chunk
layers, bounded samples of each layer (uniformly drawn query rows; the first
query offsets of a chunk).  Under torchrun only rank 0 runs it.

``--workload prefill_s131072`` times one prefill layer instead (tokens/s =
B*S per layer), with the tensor-core roofline of the sparse attention.
``--workload chunk_b1_p60000_s8192`` (an 8,192-token prefill chunk after a
60,000-token cached prefix) and ``--workload verify_b8_p60000_s4`` (4 decode
tokens per sequence at concurrency 8) time one layer over a paged cache.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MSA layer prefill & decode tokens/s on 1 GB300; % of HBM / bf16 TC roofline"
UNIT = "tokens/s"
L2_BYTES = 129 * 1024 * 1024


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "src": "fallback"}


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def source_hash(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def read_profile_traffic(name: str, kernel_files):
    """dram bytes per launch from a committed ncu summary, if it matches the current kernel source."""
    p = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(p):
        return None, "no profile"
    kv = {}
    for line in open(p):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("source_sha256_16") != source_hash(kernel_files):
        return None, "kernel changed since the capture"
    try:
        return float(kv["dram_bytes_per_launch"]), os.path.relpath(p, ROOT)
    except (KeyError, ValueError):
        return None, "no dram bytes in profile"


# ---------------------------------------------------------------------------
# decode workload
# ---------------------------------------------------------------------------

PREFILL_ATTN_FILES = ["block_sparse_attention_02_gb300/csrc/attn_prefill.cu",
                      "block_sparse_attention_02_gb300/csrc/msa_ptx.cuh"]
DENSE_FILES = {k: [f"block_sparse_attention_02_gb300/csrc/dense_{k}.cu", "block_sparse_attention_02_gb300/csrc/msa_ptx.cuh"]
               for k in ("decode", "prefill")}
DECODE_INDEX_FILES = ["block_sparse_attention_02_gb300/csrc/index_decode.cu",
                      "block_sparse_attention_02_gb300/csrc/msa_ptx.cuh",
                      "block_sparse_attention_02_gb300/csrc/select_warp.cuh"]


def decode_algorithmic_bytes(wl, shared_index=False):
    """Algorithmic HBM bytes of one decode step (unmasked, selected work only).
    With ``shared_index`` one index-key pool serves every KV group."""
    sh = wl.shape
    idx = 0
    kv = 0
    for L in wl.lengths:
        own = (L - 1) // sh.Bk
        idx += (1 if shared_index else sh.Hkv) * own * sh.Bk * sh.dI * 2   # k_idx of every scored block
        nsel = min(own, sh.k - 1)
        kv += sh.Hkv * (nsel * sh.Bk + (L - own * sh.Bk)) * sh.D * 2 * 2   # selected K and V tokens
    small_idx = wl.B * sh.Hkv * (sh.HI * sh.dI * 2 + sh.HI * 4) + wl.B * sh.Hkv * max(
        (L + sh.Bk - 1) // sh.Bk for L in wl.lengths) * 4          # q_idx, w, C
    q_o = wl.B * sh.Hq * sh.D * 2 * 2                              # Q read, O written
    return {"index_kernel": idx + small_idx, "step": idx + small_idx + kv + q_o}


class L2Flush:
    """Times steps on one stream.  Without a flush, one event pair brackets all
    K steps.  With a flush (a step whose bytes do not clearly exceed the L2),
    a buffer of twice the L2 is read before every step, outside the timed
    region, and the per-step event times are summed.  A read, not a write: a
    rewritten buffer would leave the L2 full of dirty lines whose write-back
    (up to the L2's 129 MB) would then be charged to the timed step."""

    def __init__(self, enabled, device="cuda"):
        import torch
        self.enabled = enabled
        self.buf = torch.zeros(2 * L2_BYTES // 4, dtype=torch.int32, device=device) if enabled else None

    def flush(self):
        if self.enabled:
            self.buf.sum()

    def time(self, fn, K, stream):
        """Total device milliseconds of K calls of ``fn`` on ``stream``."""
        import torch
        if not self.enabled:
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            for _ in range(K):
                fn()
            e.record(stream)
            torch.cuda.synchronize()
            return s.elapsed_time(e)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for s, e in evs:
            self.flush()
            s.record(stream)
            fn()
            e.record(stream)
        torch.cuda.synchronize()
        return sum(s.elapsed_time(e) for s, e in evs)


def pack_tensors(ts, device):
    """Copies the tensors into one contiguous byte buffer (256-byte aligned
    offsets) and returns it with views of the same shapes and dtypes into it."""
    import torch
    offs, total = {}, 0
    for n, t in ts.items():
        offs[n] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    pack = torch.zeros(total, dtype=torch.uint8, device=device)   # alignment padding stays zero
    views = {}
    for n, t in ts.items():
        nbytes = t.numel() * t.element_size()
        v = pack[offs[n]: offs[n] + nbytes].view(t.dtype).view(t.shape)
        v.copy_(t)
        views[n] = v
    return pack, views


def run_decode_ours(args, wl, world, rank):
    import torch
    import block_sparse_attention_02_gb300 as msa
    from workloads import decode_inputs
    sh = wl.shape
    inp = decode_inputs(wl, device="cuda")
    if args.shared_index:   # one index-key pool for all KV groups: group stride 0
        inp["kidx_pool"] = inp["kidx_pool"][:, :1].expand(-1, sh.Hkv, -1, -1)
    bufs = msa.decode_buffers(wl.B, sh.Hq, sh.Hkv, sh.k, inp["seq_pt"].shape[1], "cuda")
    stream = torch.cuda.current_stream()
    # The per-step inputs (Q, q_idx, w, seq_pt, seq_len) and outputs (O, LSE)
    # each live in one contiguous device buffer, so that a step's host
    # round trip is one copy in and one copy out (the page pools stay resident).
    step_in = ("Q", "q_idx", "w", "seq_pt", "seq_len")
    in_pack, in_views = pack_tensors({n: inp[n] for n in step_in}, "cuda")
    inp.update(in_views)
    out_pack, out_views = pack_tensors({n: bufs[n] for n in ("O", "LSE")}, "cuda")
    bufs.update(out_views)

    def make_parts(inp, bufs):
        def index_part():
            # a1 index score with a2 selection and a3 page table fused into the same kernel
            msa.msa_index_score(msa.MSA_MODE_DECODE, inp["q_idx"], inp["w"], inp["kidx_pool"], bufs["C"],
                                seq_pt=inp["seq_pt"], seq_len=inp["seq_len"], dev_err=bufs["dev_err"], k=sh.k,
                                sel=bufs["sel"], count=bufs["count"], pt=bufs["pt"], n=bufs["n"],
                                last_len=bufs["last_len"], row_scratch=bufs["row_scratch"], scratch_zeroed=True)

        def rest_part():
            e = bufs["dev_err"]
            msa.msa_sparse_attn_decode(inp["Q"], inp["K_pool"], inp["V_pool"], bufs["pt"], bufs["n"],
                                       bufs["last_len"], bufs["O"], bufs["LSE"], bufs["ws"], dev_err=e,
                                       scratch_zeroed=True)

        def step():
            index_part()
            rest_part()
        return index_part, rest_part, step

    index_part, rest_part, step = make_parts(inp, bufs)

    # warm up eagerly (sets kernel attributes), then capture the whole step in one CUDA graph
    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize()
    graphs = True
    try:
        g_step = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_step):
            step()
        run_step = g_step.replay
    except Exception:  # capture unavailable: launch directly
        graphs = False
        run_step = step
    for _ in range(args.warmup):
        run_step()
    torch.cuda.synchronize()
    assert int(bufs["dev_err"].item()) == 0, "device error during warm-up"

    K = args.steps
    alg = decode_algorithmic_bytes(wl, args.shared_index)
    # a step that reads less than twice the L2 could be served from it on the next step
    l2 = L2Flush(alg["step"] < 2 * L2_BYTES)
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    step_total = l2.time(run_step, K, stream)
    barrier(world)
    clocks = sampler.stop()
    total_ms = max_over_ranks(step_total, world)
    assert int(bufs["dev_err"].item()) == 0, "device error during the timed steps"

    # ---- per-call breakdown (separate pass, one graph per C-ABI call; not part of `value`) ----
    # The cache append (the step before a decode step) rewrites each sequence's
    # current token with the values it already holds, so the cache is unchanged.
    L = inp["seq_len"].long()
    pages = inp["seq_pt"].long().gather(1, ((L - 1) // sh.Bk).view(-1, 1)).view(-1)
    slot = (L - 1) % sh.Bk
    new_tok = [pool[pages, :, slot, :].contiguous() for pool in (inp["K_pool"], inp["V_pool"], inp["kidx_pool"])]
    calls = {
        "cache_append (the step before)": lambda: msa.msa_cache_append(*new_tok, inp["K_pool"], inp["V_pool"],
                                                                        inp["kidx_pool"], inp["seq_pt"],
                                                                        inp["seq_len"], dev_err=bufs["dev_err"]),
        "index_score+topk+page_table": index_part,
        "topk (standalone)": lambda: msa.msa_topk_blocks(msa.MSA_MODE_DECODE, bufs["C"], sh.k, bufs["sel"],
                                                         bufs["count"], seq_len=inp["seq_len"],
                                                         dev_err=bufs["dev_err"]),
        "page_table (standalone)": lambda: msa.msa_build_page_table(bufs["sel"], bufs["count"], inp["seq_pt"],
                                                                    inp["seq_len"], bufs["pt"], bufs["n"],
                                                                    bufs["last_len"], dev_err=bufs["dev_err"]),
        "attention+merge": lambda: msa.msa_sparse_attn_decode(inp["Q"], inp["K_pool"], inp["V_pool"], bufs["pt"],
                                                              bufs["n"], bufs["last_len"], bufs["O"], bufs["LSE"],
                                                              bufs["ws"], dev_err=bufs["dev_err"],
                                                              scratch_zeroed=True),
    }
    per_call = {}
    try:
        gs = {}
        for name, f in calls.items():
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                f()
            gs[name] = g
        runs = [gs[n].replay for n in calls]
    except Exception:
        runs = list(calls.values())
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in runs]
           for _ in range(K)]
    torch.cuda.synchronize()
    for i in range(K):
        for j, f in enumerate(runs):
            l2.flush()
            evs[i][j][0].record(stream)
            f()
            evs[i][j][1].record(stream)
    torch.cuda.synchronize()
    for j, name in enumerate(calls):
        per_call[name] = statistics.mean(evs[i][j][0].elapsed_time(evs[i][j][1]) for i in range(K))
    # the dominant kernel's time: its own graph (one launch of the fused index kernel)
    idx_ms = per_call["index_score+topk+page_table"]
    rest_ms = per_call["attention+merge"]

    # ---- end to end through the C ABI with host buffers ----
    # Every step copies its inputs in from pinned host memory and its O and
    # LSE out.  Without an L2 flush the copies are pipelined: two sets of
    # device packs (and a graph per set) alternate between steps, the copy in
    # of step i+1 runs on one copy stream while step i computes, and the copy
    # out of step i on another while step i+1 computes.  With a flush between
    # steps each step runs copy in -> step -> copy out on one stream.
    host_in = [in_pack.cpu().pin_memory(), in_pack.cpu().pin_memory()]   # the step inputs, packed
    host_out = [torch.empty_like(out_pack, device="cpu").pin_memory() for _ in range(2)]
    h2d = host_in[0].numel()
    d2h = host_out[0].numel()
    pipelined = graphs and not l2.enabled
    if pipelined:
        inp2, bufs2 = dict(inp), dict(bufs)
        in_pack2, in_views2 = pack_tensors({n: inp[n] for n in step_in}, "cuda")
        inp2.update(in_views2)
        out_pack2, out_views2 = pack_tensors({n: bufs[n] for n in ("O", "LSE")}, "cuda")
        bufs2.update(out_views2)
        step2 = make_parts(inp2, bufs2)[2]
        step2()
        torch.cuda.synchronize()
        g_step2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_step2):
            step2()
        packs_in, packs_out, runs = [in_pack, in_pack2], [out_pack, out_pack2], [run_step, g_step2.replay]
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def e2e_steps(nsteps):
            """nsteps pipelined steps; returns their device milliseconds (copy in of the first to copy out of the last)."""
            t_a, t_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t_a.record(stream)
            s_in.wait_event(t_a)
            s_out.wait_event(t_a)
            for i in range(nsteps):
                x = i & 1
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(ev_comp[x])        # step i-2 has read this input pack
                    packs_in[x].copy_(host_in[x], non_blocking=True)
                    ev_in[x].record(s_in)
                stream.wait_event(ev_in[x])
                if i >= 2:
                    stream.wait_event(ev_out[x])            # step i-2's outputs have left this pack
                runs[x]()
                ev_comp[x].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_comp[x])
                    host_out[x].copy_(packs_out[x], non_blocking=True)
                    ev_out[x].record(s_out)
            stream.wait_event(ev_out[(nsteps - 1) & 1])
            t_b.record(stream)
            torch.cuda.synchronize()
            return t_a.elapsed_time(t_b)

        e2e_steps(args.warmup)
        barrier(world)
        e2e_total = e2e_steps(K)
        barrier(world)
    else:
        def e2e_step():
            in_pack.copy_(host_in[0], non_blocking=True)
            run_step()
            host_out[0].copy_(out_pack, non_blocking=True)

        for _ in range(args.warmup):
            e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        e2e_total = l2.time(e2e_step, K, stream)
        barrier(world)
    e2e_ms = max_over_ranks(e2e_total, world)
    assert torch.equal(host_out[0], host_out[1]) or not pipelined, "the two output packs differ"

    peaks = load_peaks()
    achieved = alg["index_kernel"] / (idx_ms * 1e-3) / 1e9
    # profiles/index_decode_<workload without its "decode_" prefix>.txt
    short = wl.name[len("decode_"):] if wl.name.startswith("decode_") else wl.name
    traffic, traffic_src = read_profile_traffic(
        f"index_decode_{'shared_' if args.shared_index else ''}{short}.txt", DECODE_INDEX_FILES)
    tokens_per_step = wl.B * world
    step_ms = total_ms / K
    res = {
        "metric": METRIC, "value": tokens_per_step / (step_ms * 1e-3), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.B,
                   "context": wl.lengths[0] if len(set(wl.lengths)) == 1 else f"ragged {min(wl.lengths)}..{max(wl.lengths)}, total {sum(wl.lengths)}",
                   "Hq": wl.shape.Hq,
                   "Hkv": wl.shape.Hkv, "D": wl.shape.D, "HI": wl.shape.HI, "dI": wl.shape.dI, "Bk": wl.shape.Bk,
                   "k": wl.shape.k, "pages": "128-token, shuffled",
                   "index_keys": "one pool shared by the KV groups" if args.shared_index else "per KV group",
                   "cuda_graphs": graphs,
                   "scratch": "zero-filled once; calls skip the counter clears (scratch_zeroed) and leave them zero",
                   "l2": (f"flushed before every timed step ({alg['step'] / 1e6:.0f} MB read per step)" if l2.enabled
                          else f"no flush: inputs larger than L2 ({alg['step'] / 1e6:.0f} MB read per step)"),
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "kernel": "index_decode_kernel (with fused selection)", "achieved": achieved,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "peak_src": peaks["src"], "traffic": traffic, "traffic_src": traffic_src,
                     "algorithmic_bytes_per_launch": alg["index_kernel"], "launch_ms": idx_ms,
                     "step_algorithmic_bytes": alg["step"],
                     "step_frac": alg["step"] / (step_ms * 1e-3) / 1e9 / peaks["hbm_gbs"]},
        "breakdown_ms": {"index_score+topk+page_table": idx_ms, "attention+merge": rest_ms,
                         "per_call_graphs": per_call},
        "e2e": {"value": tokens_per_step / (e2e_ms / K * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "copies": ("pipelined: copy in and copy out on two streams, overlapping the neighbouring steps"
                           if pipelined else "serial: copy in, step, copy out on one stream")},
        "gpu_launches": 2 * K,
        "clocks": clocks,
    }
    return res, host_in[0], inp


def oracle_decode_step(h, sh):
    import oracle
    C = oracle.decode_scores(h["q_idx"], h["w"], h["kidx_pool"], h["seq_pt"], h["seq_len"])
    own = oracle.own_blocks_decode(h["seq_len"], sh.Bk)
    sel, cnt, _, _ = oracle.select(C, own[:, None], sh.k)
    return oracle.decode_attend(h["Q"], h["K_pool"], h["V_pool"], h["seq_pt"], h["seq_len"], sel, cnt,
                                1.0 / math.sqrt(sh.D))


def one_thread(fn):
    """Runs fn() with the oracle on one host thread; returns its result."""
    import oracle
    n = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        return fn()
    finally:
        oracle.set_num_threads(n)


def cpu_decode_baseline(wl, inp_host, budget_s: float, min_steps: int = 1):
    """Oracle decode steps on the host cores until the time budget is used;
    then one step on a single thread."""
    import oracle
    oracle.build()
    t0 = time.perf_counter()
    steps = 0
    while steps < min_steps or time.perf_counter() - t0 < budget_s:
        oracle_decode_step(inp_host, wl.shape)
        steps += 1
    dt = time.perf_counter() - t0

    def single():
        t1 = time.perf_counter()
        oracle_decode_step(inp_host, wl.shape)
        return time.perf_counter() - t1
    dt1 = one_thread(single)
    return {"value": wl.B * steps / dt, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{steps} full decode step(s) of {wl.name} (B={wl.B}) in {dt:.1f} s",
            "value_1_thread": wl.B / dt1, "sample_1_thread": f"one full decode step in {dt1:.1f} s"}


def cpu_prefill_baseline(wl, inp_host, budget_s: float, seed: int = 0):
    """The oracle's prefill layer (scores, selection, attention) on query rows
    drawn uniformly from the layer, 16 at a time, until the time budget is
    used: tokens/s = rows / time (a uniform sample has the layer's mean cost
    per query)."""
    import numpy as np
    import oracle
    oracle.build()
    sh = wl.shape
    rng = np.random.default_rng(seed)
    t0 = time.perf_counter()
    n = 0
    while n == 0 or time.perf_counter() - t0 < budget_s:
        rows = np.sort(rng.integers(0, wl.B * wl.S, 16)).astype(np.int64)
        C = oracle.prefill_scores(inp_host["q_idx"], inp_host["k_idx"], inp_host["w"], sh.Bk, rows)
        own = np.repeat(oracle.own_blocks_prefill(wl.S, sh.Bk, rows), sh.Hkv).reshape(-1, sh.Hkv)
        sel, cnt, _, _ = oracle.select(C, own, sh.k)
        oracle.prefill_attend(inp_host["Q"], inp_host["K"], inp_host["V"], sel, cnt, sh.Bk, 1.0 / math.sqrt(sh.D),
                              rows)
        n += len(rows)
    dt = time.perf_counter() - t0

    def single():
        r = np.sort(rng.integers(0, wl.B * wl.S, 16)).astype(np.int64)
        t1 = time.perf_counter()
        C1 = oracle.prefill_scores(inp_host["q_idx"], inp_host["k_idx"], inp_host["w"], sh.Bk, r)
        o1 = np.repeat(oracle.own_blocks_prefill(wl.S, sh.Bk, r), sh.Hkv).reshape(-1, sh.Hkv)
        s1, c1, _, _ = oracle.select(C1, o1, sh.k)
        oracle.prefill_attend(inp_host["Q"], inp_host["K"], inp_host["V"], s1, c1, sh.Bk, 1.0 / math.sqrt(sh.D), r)
        return time.perf_counter() - t1
    dt1 = one_thread(single)
    return {"value": n / dt, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} query rows of {wl.name} drawn uniformly (all heads and groups) in {dt:.1f} s",
            "extrapolated": True,
            "full_layer_s_extrapolated": wl.B * wl.S / (n / dt),
            "value_1_thread": 16 / dt1, "sample_1_thread": f"16 uniformly drawn query rows in {dt1:.1f} s"}


def cpu_chunk_baseline(wl, inp_host, budget_s: float):
    """The oracle's chunk layer on the chunk's first query offsets (every
    sequence, one offset at a time) until the time budget is used."""
    import oracle
    oracle.build()
    sh = wl.shape
    t0 = time.perf_counter()
    n = 0
    while n < wl.S and (n == 0 or time.perf_counter() - t0 < budget_s):
        part = {x: inp_host[x][:, n:n + 1] for x in ("Q", "q_idx", "w")}
        oracle.chunk_layer(part["Q"], part["q_idx"], part["w"], inp_host["K_pool"], inp_host["V_pool"],
                           inp_host["kidx_pool"], inp_host["seq_pt"], inp_host["q_pos"] + n, sh.k,
                           1.0 / math.sqrt(sh.D), sh.Bk)
        n += 1
    dt = time.perf_counter() - t0
    return {"value": wl.B * n / dt, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"the first {n} of {wl.S} query offsets of {wl.name} (B={wl.B}) in {dt:.1f} s"}


# ---------------------------------------------------------------------------
# prefill workload (optional)
# ---------------------------------------------------------------------------

def prefill_attention_flops(sel, count, S, Bk, G, D, q_pos=None):
    """4*D*G FLOPs per (query, group, key) over the unmasked selected keys
    (count from the selection); queries sit at q_pos[b] + i (0 without q_pos)."""
    import torch
    i = torch.arange(S, device=sel.device).view(1, S, 1, 1)
    if q_pos is not None:
        i = i + q_pos.long().view(-1, 1, 1, 1)
    s = sel.long()
    keys = torch.where(s < 0, torch.zeros_like(s),
                       torch.clamp(i + 1 - s * Bk, min=0, max=Bk))
    return float(keys.sum().item()) * 4 * D * G


def run_prefill_ours(args, wl, world, rank):
    import torch
    import block_sparse_attention_02_gb300 as msa
    from workloads import prefill_inputs
    sh = wl.shape
    inp = prefill_inputs(wl, device="cuda")
    ws_q = min(wl.S, args.prefill_chunk) * wl.B
    sel_probe = torch.empty(1, 1, 1, sh.k, dtype=torch.int32)
    ws_bytes = msa.msa_sparse_attn_prefill_workspace_size(inp["Q"], inp["K"], sel_probe, ws_q)
    bufs = msa.prefill_buffers(wl.B, wl.S, sh.Hq, sh.Hkv, sh.k, "cuda", ws_bytes)
    stream = torch.cuda.current_stream()
    e = bufs["dev_err"]

    def parts():
        return [
            lambda: msa.msa_index_score(msa.MSA_MODE_PREFILL, inp["q_idx"], inp["w"], inp["k_idx"], bufs["C"],
                                        dev_err=e),
            lambda: msa.msa_topk_blocks(msa.MSA_MODE_PREFILL, bufs["C"], sh.k, bufs["sel"], bufs["count"], dev_err=e),
            lambda: msa.msa_sparse_attn_prefill(inp["Q"], inp["K"], inp["V"], bufs["sel"], bufs["count"], bufs["O"],
                                                bufs["LSE"], bufs["ws"], dev_err=e),
        ]
    fns = parts()
    for _ in range(max(1, args.warmup)):
        for f in fns:
            f()
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(K):
        for j, f in enumerate(fns):
            ev[i][j].record(stream)
            f()
        ev[i][3].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    total_ms = max_over_ranks(start.elapsed_time(end), world)
    part_ms = [statistics.mean(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(K)) for j in range(3)]
    flops = prefill_attention_flops(bufs["sel"], bufs["count"], wl.S, sh.Bk, sh.G, sh.D)
    idx_flops = 2.0 * sh.HI * sh.dI * sh.Hkv * wl.B * sum(sh.Bk * (i // sh.Bk) for i in range(wl.S))
    peaks = load_peaks()
    tc = flops / (part_ms[2] * 1e-3) / 1e12
    step_ms = total_ms / K
    # DRAM bytes of the whole stage (CSR, attention, merge) of one layer
    traffic, traffic_src = read_profile_traffic(f"attn_stage_{wl.name}.txt", PREFILL_ATTN_FILES)
    res = {
        "metric": METRIC, "value": wl.B * wl.S * world / (step_ms * 1e-3), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.B, "seq_len": wl.S, "Hq": sh.Hq, "Hkv": sh.Hkv, "D": sh.D,
                   "HI": sh.HI, "dI": sh.dI, "Bk": sh.Bk, "k": sh.k, "query_chunk": ws_q,
                   "l2": "no flush: inputs larger than L2", "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "kernel": "sparse attention (a4+a6)", "achieved": tc,
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": tc / peaks["bf16_tflops"],
                     "peak_src": peaks["src"], "traffic": traffic, "traffic_src": traffic_src,
                     "traffic_gbs": None if traffic is None else traffic / (part_ms[2] * 1e-3) / 1e9,
                     "algorithmic_flops_per_launch": flops, "launch_ms": part_ms[2],
                     "index_tflops": idx_flops / (part_ms[0] * 1e-3) / 1e12,
                     "index_frac": idx_flops / (part_ms[0] * 1e-3) / 1e12 / peaks["bf16_tflops"]},
        "breakdown_ms": {"index_score": part_ms[0], "topk": part_ms[1], "sparse_attention": part_ms[2]},
        "gpu_launches": K * (2 + 5 * ((wl.B * wl.S + ws_q - 1) // ws_q)),
        "clocks": clocks,
    }
    return res, None, inp


# ---------------------------------------------------------------------------
# chunk over a paged cache (chunked prefill, multi-token decode)
# ---------------------------------------------------------------------------

def run_chunk_ours(args, wl, world, rank):
    """One MSA layer over a chunk of S queries per sequence after a cached
    prefix: tokens/s = B*S per step.  The roofline is that of the dominant
    kernel: the index score (HBM- or tensor-bound, whichever bound is higher)
    or the sparse attention (tensor)."""
    import torch
    import block_sparse_attention_02_gb300 as msa
    from workloads import chunk_inputs
    sh = wl.shape
    inp = chunk_inputs(wl, device="cuda")
    ws_q = min(wl.S, args.prefill_chunk) * wl.B
    sel_probe = torch.empty(1, 1, 1, sh.k, dtype=torch.int32)
    ws_bytes = msa.msa_sparse_attn_prefill_workspace_size(inp["Q"], inp["K_pool"], sel_probe, ws_q,
                                                          max_pages=wl.max_pages)
    bufs = msa.chunk_buffers(wl.B, wl.S, sh.Hq, sh.Hkv, sh.k, wl.max_pages, "cuda", ws_bytes)
    stream = torch.cuda.current_stream()
    e = bufs["dev_err"]
    fns = [
        lambda: msa.msa_index_score(msa.MSA_MODE_CHUNK, inp["q_idx"], inp["w"], inp["kidx_pool"], bufs["C"],
                                    seq_pt=inp["seq_pt"], q_pos=inp["q_pos"], dev_err=e),
        lambda: msa.msa_topk_blocks(msa.MSA_MODE_CHUNK, bufs["C"], sh.k, bufs["sel"], bufs["count"],
                                    q_pos=inp["q_pos"], dev_err=e),
        lambda: msa.msa_sparse_attn_prefill(inp["Q"], inp["K_pool"], inp["V_pool"], bufs["sel"], bufs["count"],
                                            bufs["O"], bufs["LSE"], bufs["ws"], dev_err=e, seq_pt=inp["seq_pt"],
                                            q_pos=inp["q_pos"]),
    ]
    for _ in range(max(1, args.warmup)):
        for f in fns:
            f()
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(K):
        for j, f in enumerate(fns):
            ev[i][j].record(stream)
            f()
        ev[i][3].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    assert int(e.item()) == 0, "device error during the timed steps"
    total_ms = max_over_ranks(start.elapsed_time(end), world)
    part_ms = [statistics.mean(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(K)) for j in range(3)]
    peaks = load_peaks()
    # algorithmic work: attention over the unmasked selected keys; index
    # scores of every earlier block of every query, and its HBM bytes (index
    # keys of each scored (b, g) block once, q_idx and w read, C written)
    att_flops = prefill_attention_flops(bufs["sel"], bufs["count"], wl.S, sh.Bk, sh.G, sh.D, inp["q_pos"])
    own = [[(p + s) // sh.Bk for s in range(wl.S)] for p in wl.prefix]
    idx_flops = 2.0 * sh.HI * sh.dI * sh.Hkv * sh.Bk * sum(sum(o) for o in own)
    idx_bytes = (sum(max(o) for o in own) * sh.Hkv * sh.Bk * sh.dI * 2
                 + wl.B * wl.S * sh.Hkv * (sh.HI * sh.dI * 2 + sh.HI * 4 + wl.max_pages * 4))
    idx_ms, att_ms = part_ms[0], part_ms[2]
    t_hbm = idx_bytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = idx_flops / (peaks["bf16_tflops"] * 1e12)
    if idx_ms >= att_ms and t_hbm >= t_tc:
        ach = idx_bytes / (idx_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "kernel": "index score (a1)", "achieved": ach, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": ach / peaks["hbm_gbs"], "algorithmic_bytes_per_launch": idx_bytes,
                "launch_ms": idx_ms}
    elif idx_ms >= att_ms:
        ach = idx_flops / (idx_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "kernel": "index score (a1)", "achieved": ach, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"], "algorithmic_flops_per_launch": idx_flops,
                "launch_ms": idx_ms}
    else:
        ach = att_flops / (att_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "kernel": "sparse attention (a4+a6)", "achieved": ach,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"],
                "algorithmic_flops_per_launch": att_flops, "launch_ms": att_ms}
    roof.update({"peak_src": peaks["src"], "traffic": None,
                 "index_hbm_frac": idx_bytes / (idx_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                 "index_tc_frac": idx_flops / (idx_ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
                 "attention_tc_frac": att_flops / (att_ms * 1e-3) / 1e12 / peaks["bf16_tflops"]})
    step_ms = total_ms / K
    step_bytes = idx_bytes + 2 * wl.B * wl.S * sh.Hq * sh.D * 2
    res = {
        "metric": METRIC, "value": wl.B * wl.S * world / (step_ms * 1e-3), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.B, "chunk": wl.S,
                   "cached_prefix": wl.prefix[0] if len(set(wl.prefix)) == 1 else list(wl.prefix),
                   "Hq": sh.Hq, "Hkv": sh.Hkv, "D": sh.D, "HI": sh.HI, "dI": sh.dI, "Bk": sh.Bk, "k": sh.k,
                   "pages": "128-token, shuffled", "query_chunk": ws_q,
                   "l2": f"no flush: a step moves more than twice the L2 (>= {step_bytes / 1e6:.0f} MB)",
                   "parallelism": f"replicas x{world}"},
        "roofline": roof,
        "breakdown_ms": {"index_score": part_ms[0], "topk": part_ms[1], "sparse_attention": part_ms[2]},
        # a few queries per sequence: page table + decode attention (2 launches); else 5 per query chunk
        "gpu_launches": K * (2 + (2 if wl.S <= 8 else 5 * ((wl.B * wl.S + ws_q - 1) // ws_q))),
        "clocks": clocks,
    }
    return res, None, inp


# ---------------------------------------------------------------------------
# dense comparator (attention over every token, no index branch)
# ---------------------------------------------------------------------------

def dense_decode_bytes(wl):
    """Algorithmic HBM bytes of a dense decode step: every cached K and V token once, Q read, O written."""
    sh = wl.shape
    return sum(wl.lengths) * sh.Hkv * sh.D * 2 * 2 + wl.B * sh.Hq * sh.D * 2 * 2


def dense_prefill_flops(wl):
    """4*D FLOPs per (query head, visible key) of a causal prefill: sum_i (i + 1) keys per head."""
    sh = wl.shape
    return 4.0 * sh.D * sh.Hq * wl.B * (wl.S * (wl.S + 1) / 2)


def run_dense_ours(args, wl, world, rank):
    """Times the dense comparator on a workload's inputs: a decode step (HBM
    roofline) or a prefill layer (tensor-core roofline)."""
    import torch
    import block_sparse_attention_02_gb300 as msa
    from workloads import DecodeWorkload, decode_inputs, prefill_inputs
    peaks = load_peaks()
    stream = torch.cuda.current_stream()
    decode = isinstance(wl, DecodeWorkload)
    if decode:
        inp = decode_inputs(wl, device="cuda")
        bufs = msa.dense_decode_buffers(wl.B, wl.shape.Hq, wl.shape.Hkv, inp["seq_pt"].shape[1], "cuda")
        fn = lambda: msa.dense_decode_step(inp, bufs, scratch_zeroed=True)
    else:
        inp = prefill_inputs(wl, device="cuda")
        bufs = None
        out = msa.dense_prefill_layer(inp)
        fn = lambda: msa.dense_prefill_layer(inp, out)
        bufs = out
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    assert int(bufs["dev_err"].item()) == 0, "device error during the dense warm-up"
    K = args.steps
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    work = dense_decode_bytes(wl) if decode else dense_prefill_flops(wl)
    l2 = L2Flush(decode and work < 2 * L2_BYTES)
    total = l2.time(fn, K, stream)
    barrier(world)
    clocks = sampler.stop()
    assert int(bufs["dev_err"].item()) == 0, "device error during the dense steps"
    step_ms = max_over_ranks(total, world) / K
    tokens = wl.B if decode else wl.B * wl.S
    if decode:
        ach = work / (step_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "kernel": "dense_decode_kernel", "achieved": ach, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": ach / peaks["hbm_gbs"], "algorithmic_bytes_per_launch": work}
    else:
        ach = work / (step_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "kernel": "dense_prefill_kernel", "achieved": ach, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"], "algorithmic_flops_per_launch": work}
    kind = "decode" if decode else "prefill"
    short = wl.name[len("decode_"):] if decode else wl.name[len("prefill_"):]
    traffic, traffic_src = read_profile_traffic(f"dense_{kind}_{short}_dram.txt", DENSE_FILES[kind])
    roof.update({"peak_src": peaks["src"], "traffic": traffic, "traffic_src": traffic_src, "launch_ms": step_ms})
    res = {"value": tokens * world / (step_ms * 1e-3), "unit": UNIT, "ms_per_step": step_ms, "steps": K,
           "warmup": args.warmup,
           "config": {"workload": wl.name, "comparator": "dense attention over every token (no index branch)",
                      "l2": "flushed before every timed step" if l2.enabled else "no flush: inputs larger than L2"},
           "roofline": roof, "gpu_launches": K, "clocks": clocks, "cpu_baseline": None}
    del inp, bufs
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


DEFAULT_WORKLOAD = "decode_b8_l60001"
# the other full-size workloads of the metric (prefill, the 1M-token decode,
# the ragged decode batch), timed after the headline one in the default run,
# then the dense comparator on the same inputs ("dense:" + workload)
EXTRA_WORKLOADS = ("prefill_s131072", "decode_b1_l1048576", "decode_ragged_b64", "dense:decode_b8_l60001",
                   "dense:decode_b1_l1048576", "dense:prefill_s131072")
SUB_KEYS = ("value", "unit", "ms_per_step", "steps", "warmup", "config", "roofline", "breakdown_ms", "e2e",
            "gpu_launches", "clocks", "cpu_baseline")


def run_workload(args, wl, world, rank):
    """Times one workload; returns its JSON record (with cpu_baseline on rank 0 at N = 1)."""
    import torch
    from workloads import ChunkWorkload, DecodeWorkload
    if isinstance(wl, DecodeWorkload):
        res, host_in, inp = run_decode_ours(args, wl, world, rank)
    elif isinstance(wl, ChunkWorkload):
        res, host_in, inp = run_chunk_ours(args, wl, world, rank)
    else:
        res, host_in, inp = run_prefill_ours(args, wl, world, rank)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        h = {n: t.cpu() for n, t in inp.items()}
        if isinstance(wl, DecodeWorkload):
            res["cpu_baseline"] = cpu_decode_baseline(wl, h, args.cpu_budget_s)
        elif isinstance(wl, ChunkWorkload):
            res["cpu_baseline"] = cpu_chunk_baseline(wl, h, args.cpu_budget_s)
        else:
            res["cpu_baseline"] = cpu_prefill_baseline(wl, h, args.cpu_budget_s)
        del h
    elif rank == 0:
        res["cpu_baseline"] = None
    del inp, host_in
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--also", default=",".join(EXTRA_WORKLOADS),
                    help="with the default workload: further workloads timed in the same run and reported as "
                         "sub-records under 'workloads' (empty: none)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    # queries per chunk of the prefill attention (CSR, attention, merge per
    # chunk): fewer, larger chunks cost fewer launches; 65,536 queries need
    # ~13 GB of bf16 partials in the workspace
    ap.add_argument("--prefill-chunk", type=int, default=65536)
    ap.add_argument("--shared-index", action="store_true",
                    help="decode with one index-key pool for all KV groups (k_idx group stride 0)")
    ap.add_argument("--seq", type=int, default=None, help="override the prefill sequence length (profiling)")
    ap.add_argument("--dense", action="store_true",
                    help="time only the dense comparator on the workload's inputs (profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    import torch
    from workloads import workload
    wl = workload(args.workload)
    if args.seq is not None and hasattr(wl, "S"):
        from dataclasses import replace
        wl = replace(wl, name=f"{wl.name}_s{args.seq}", S=args.seq)
    world, rank, _ = dist_setup()

    from workloads import ChunkWorkload, DecodeWorkload
    if args.impl == "reference":
        if rank != 0:
            return
        import oracle
        oracle.build()
        if isinstance(wl, DecodeWorkload):
            from workloads import decode_inputs
            h = decode_inputs(wl, device="cpu")
            for _ in range(args.warmup):
                oracle_decode_step(h, wl.shape)
            t0 = time.perf_counter()
            for _ in range(args.steps):
                oracle_decode_step(h, wl.shape)
            dt = time.perf_counter() - t0
            val = wl.B * args.steps / dt
            cfg = {"workload": wl.name, "batch": wl.B, "context": wl.lengths[0]}
            base = {"value": val, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                    "sample": f"{args.steps} full decode steps of {wl.name}"}
            ms = dt / args.steps * 1e3
        else:
            # prefill and chunk layers: each step is a bounded sample of the layer
            budget = args.cpu_budget_s / max(1, args.steps + args.warmup)
            if isinstance(wl, ChunkWorkload):
                from workloads import chunk_inputs
                h = chunk_inputs(wl, device="cpu")
                run = lambda: cpu_chunk_baseline(wl, h, budget)
                cfg = {"workload": wl.name, "batch": wl.B, "chunk": wl.S, "cached_prefix": wl.prefix[0]}
            else:
                from workloads import prefill_inputs
                h = prefill_inputs(wl, device="cpu")
                run = lambda: cpu_prefill_baseline(wl, h, budget)
                cfg = {"workload": wl.name, "batch": wl.B, "seq_len": wl.S}
            for _ in range(args.warmup):
                run()
            samples = [run() for _ in range(args.steps)]
            val = statistics.mean(x["value"] for x in samples)
            base = dict(samples[-1], value=val)
            base["sample"] = f"{args.steps} steps, each: " + samples[-1]["sample"]
            ms = wl.B * wl.S / val * 1e3
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
            "cpu_baseline": base,
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }))
        return

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device for --impl ours")
    from block_sparse_attention_02_gb300 import build as b
    b.build()
    if args.dense:
        res = run_dense_ours(args, wl, world, rank)
        res.update({"metric": METRIC, "n_gpus": world, "higher_is_better": True, "scaling": "weak",
                    "vs_baseline": None, "dtype": "bf16", "data": "synthetic"})
        if rank == 0:
            print(json.dumps(res))
        return
    res = run_workload(args, wl, world, rank)
    extra = [x for x in args.also.split(",") if x] if args.workload == DEFAULT_WORKLOAD and args.seq is None else []
    if extra:
        subs = {}
        for name in extra:
            if name.startswith("dense:"):
                sub = run_dense_ours(args, workload(name[len("dense:"):]), world, rank)
            else:
                sub = run_workload(args, workload(name), world, rank)
            subs[name] = {k: sub[k] for k in SUB_KEYS if k in sub}
        res["workloads"] = subs
        # the same-box speedup of MSA over the dense comparator, per workload
        msa_values = dict(subs, **{args.workload: res})
        res["msa_vs_dense"] = {n[len("dense:"):]: msa_values[n[len("dense:"):]]["value"] / subs[n]["value"]
                               for n in subs if n.startswith("dense:") and n[len("dense:"):] in msa_values}
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
