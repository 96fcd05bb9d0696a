"""Seeded synthetic inputs for the MiniMax Sparse Attention (MSA) hot path.

This module is shared by the tests, ``bench.py`` and the oracle's callers.  It
draws random tensors with the shapes, value distributions and structure of the
workloads the MSA pages describe and holds none of the method's arithmetic: no
scoring, selection, attention or merging happens here.

Recipes (all seeded):

* Q, K, V ~ N(0, 1)/sqrt(D) and q_idx, k_idx ~ N(0, 1)/sqrt(d_I), drawn in fp32
  and rounded to bf16; index-head weights w ~ U(0, 1) in fp32.
* Long prefill: a fraction of the key blocks (5 %) is shifted by +2 along one
  seeded unit direction per KV group (u_I in R^d_I for k_idx, u in R^D for K),
  so that block selection is not uniform.  The shifted block indices are the
  same for every group.
* Paged decode: every sequence b holds L_b tokens (the current token, at
  position L_b - 1, is already in the cache) in ceil(L_b / Bk) pages of Bk
  tokens.  Physical page ids are a seeded random permutation of the pool, so
  pages are shuffled.  Ragged batches draw L_b = floor(exp(U(ln lo, ln hi))).
* Chunk over a paged cache: sequence b has a cached prefix of q_pos[b] tokens
  and a chunk of S new tokens at positions q_pos[b] .. q_pos[b] + S - 1, all
  q_pos[b] + S tokens already in shuffled pages as in decode; the chunk's
  queries are drawn like prefill queries.

Big pools may be drawn directly on a CUDA device with a seeded CUDA generator;
the oracle then reads host copies of exactly those tensors.  Values therefore
depend on the device the generator ran on, never on which side consumes them.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import Dict, Optional, Sequence, Tuple

import torch

__all__ = [
    "MSAShape", "PrefillWorkload", "DecodeWorkload", "ChunkWorkload", "WORKLOADS",
    "prefill_inputs", "decode_inputs", "chunk_inputs", "ragged_lengths", "workload",
]


@dataclass(frozen=True)
class MSAShape:
    """Head layout of one MSA layer.

    Hq query heads share Hkv KV heads (GQA ratio G = Hq / Hkv).  The index
    branch has HI heads of width dI per KV group.  Keys are cut into blocks of
    Bk tokens and every (query, KV group) keeps k blocks, its own included.
    """
    Hq: int = 48
    Hkv: int = 8
    D: int = 128
    HI: int = 4
    dI: int = 64
    Bk: int = 128
    k: int = 16

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv


@dataclass(frozen=True)
class PrefillWorkload:
    name: str
    B: int
    S: int
    shape: MSAShape
    seed: int
    shift_frac: float = 0.0     # fraction of key blocks shifted (long prefill)
    shift_mag: float = 2.0

    @property
    def nb(self) -> int:
        return (self.S + self.shape.Bk - 1) // self.shape.Bk


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    lengths: Tuple[int, ...]     # L_b, current token included
    shape: MSAShape
    seed: int
    shuffle_pages: bool = True

    @property
    def B(self) -> int:
        return len(self.lengths)

    @property
    def pages_per_seq(self) -> Tuple[int, ...]:
        Bk = self.shape.Bk
        return tuple((L + Bk - 1) // Bk for L in self.lengths)

    @property
    def max_pages(self) -> int:
        return max(self.pages_per_seq)

    @property
    def num_pages(self) -> int:
        return sum(self.pages_per_seq)


@dataclass(frozen=True)
class ChunkWorkload:
    """S new tokens per sequence after a cached prefix of prefix[b] tokens."""
    name: str
    prefix: Tuple[int, ...]      # q_pos[b]: position of the chunk's first token
    S: int
    shape: MSAShape
    seed: int
    shuffle_pages: bool = True

    @property
    def B(self) -> int:
        return len(self.prefix)

    @property
    def lengths(self) -> Tuple[int, ...]:
        return tuple(p + self.S for p in self.prefix)

    @property
    def pages_per_seq(self) -> Tuple[int, ...]:
        Bk = self.shape.Bk
        return tuple((L + Bk - 1) // Bk for L in self.lengths)

    @property
    def max_pages(self) -> int:
        return max(self.pages_per_seq)

    @property
    def num_pages(self) -> int:
        return sum(self.pages_per_seq)


def ragged_lengths(B: int, lo: int, hi: int, seed: int) -> Tuple[int, ...]:
    """L_b = floor(exp(U(ln lo, ln hi))) for b < B, from a seeded CPU generator."""
    g = torch.Generator().manual_seed(seed)
    u = torch.rand(B, generator=g, dtype=torch.float64)
    ll = math.log(lo) + u * (math.log(hi) - math.log(lo))
    return tuple(int(math.floor(math.exp(float(x)))) for x in ll)


_SHAPE_TINY = MSAShape(Hq=4, Hkv=1, D=128, HI=2, dI=64, Bk=128, k=4)
_SHAPE_MSA = MSAShape()

# The five workloads of the MSA hot path.  Names say what they are.
WORKLOADS: Dict[str, object] = {
    # tiny causal prefill: 16 blocks, 1 KV group, 4 q heads, index 2 x 64, top-4
    "prefill_tiny_s2048": PrefillWorkload("prefill_tiny_s2048", B=1, S=2048, shape=_SHAPE_TINY, seed=0),
    # the same with k = 16, which covers every block and equals dense causal GQA
    "prefill_tiny_s2048_k16": PrefillWorkload(
        "prefill_tiny_s2048_k16", B=1, S=2048, shape=replace(_SHAPE_TINY, k=16), seed=0),
    # paged decode at concurrency 8 over a 60,000-token cached prefix
    "decode_b8_l60001": DecodeWorkload("decode_b8_l60001", lengths=(60001,) * 8, shape=_SHAPE_MSA, seed=1),
    # long causal prefill, 131,072 tokens, 5 % of key blocks shifted
    "prefill_s131072": PrefillWorkload("prefill_s131072", B=1, S=131072, shape=_SHAPE_MSA, seed=2,
                                       shift_frac=0.05),
    # 1M-token decode, batch 1
    "decode_b1_l1048576": DecodeWorkload("decode_b1_l1048576", lengths=(1048576,), shape=_SHAPE_MSA, seed=3),
    # ragged decode batch of 64 sequences, lengths log-uniform in [4096, 524288]
    "decode_ragged_b64": DecodeWorkload("decode_ragged_b64", lengths=ragged_lengths(64, 4096, 524288, 4),
                                        shape=_SHAPE_MSA, seed=4),
    # chunked prefill: an 8,192-token chunk after a 60,000-token cached prefix
    "chunk_b1_p60000_s8192": ChunkWorkload("chunk_b1_p60000_s8192", prefix=(60000,), S=8192, shape=_SHAPE_MSA,
                                           seed=5),
    # decode of 4 tokens per sequence (draft verification) at concurrency 8 after 60,000 cached tokens
    "verify_b8_p60000_s4": ChunkWorkload("verify_b8_p60000_s4", prefix=(60000,) * 8, S=4, shape=_SHAPE_MSA, seed=6),
}


def workload(name: str):
    return WORKLOADS[name]


# ---------------------------------------------------------------------------
# random tensor helpers
# ---------------------------------------------------------------------------

_CHUNK = 1 << 26  # elements per draw, bounds the fp32 temporary


def _gen(device: torch.device, seed: int) -> torch.Generator:
    return torch.Generator(device=device).manual_seed(seed)


def _randn_bf16(shape: Sequence[int], g: torch.Generator, scale: float,
                device: torch.device) -> torch.Tensor:
    """N(0, 1) * scale drawn in fp32, rounded to bf16, in chunks along dim 0."""
    out = torch.empty(tuple(shape), dtype=torch.bfloat16, device=device)
    if out.numel() == 0:
        return out
    flat = out.view(-1)
    for s in range(0, flat.numel(), _CHUNK):
        e = min(flat.numel(), s + _CHUNK)
        t = torch.randn(e - s, generator=g, device=device, dtype=torch.float32)
        flat[s:e] = (t * scale).to(torch.bfloat16)
    return out


def _rand_f32(shape: Sequence[int], g: torch.Generator, device: torch.device) -> torch.Tensor:
    return torch.rand(tuple(shape), generator=g, device=device, dtype=torch.float32)


def _unit(n: int, g: torch.Generator, device: torch.device) -> torch.Tensor:
    v = torch.randn(n, generator=g, device=device, dtype=torch.float32)
    return v / v.norm()


# ---------------------------------------------------------------------------
# prefill
# ---------------------------------------------------------------------------

def prefill_inputs(wl: PrefillWorkload, device="cpu") -> Dict[str, torch.Tensor]:
    """Row-major prefill tensors.

    Q [B,S,Hq,D], K and V [B,S,Hkv,D], q_idx [B,S,Hkv,HI,dI], k_idx [B,S,Hkv,dI]
    (all bf16) and w [B,S,Hkv,HI] fp32.  With ``shift_frac`` > 0 the key blocks
    listed in ``shifted_blocks`` carry the +shift_mag offset in k_idx and K.
    """
    device = torch.device(device)
    sh = wl.shape
    B, S = wl.B, wl.S
    g = _gen(device, wl.seed)
    out = {
        "Q": _randn_bf16((B, S, sh.Hq, sh.D), g, 1.0 / math.sqrt(sh.D), device),
        "K": _randn_bf16((B, S, sh.Hkv, sh.D), g, 1.0 / math.sqrt(sh.D), device),
        "V": _randn_bf16((B, S, sh.Hkv, sh.D), g, 1.0 / math.sqrt(sh.D), device),
        "q_idx": _randn_bf16((B, S, sh.Hkv, sh.HI, sh.dI), g, 1.0 / math.sqrt(sh.dI), device),
        "k_idx": _randn_bf16((B, S, sh.Hkv, sh.dI), g, 1.0 / math.sqrt(sh.dI), device),
        "w": _rand_f32((B, S, sh.Hkv, sh.HI), g, device),
    }
    if wl.shift_frac > 0:
        cg = torch.Generator().manual_seed(wl.seed + 2000)
        nshift = int(round(wl.shift_frac * wl.nb))
        blocks = torch.randperm(wl.nb, generator=cg)[:nshift].sort().values
        uI = torch.stack([_unit(sh.dI, cg, torch.device("cpu")) for _ in range(sh.Hkv)]).to(device)
        u = torch.stack([_unit(sh.D, cg, torch.device("cpu")) for _ in range(sh.Hkv)]).to(device)
        for j in blocks.tolist():
            t0, t1 = j * sh.Bk, min(S, (j + 1) * sh.Bk)
            ks = out["k_idx"][:, t0:t1].float() + wl.shift_mag * uI
            out["k_idx"][:, t0:t1] = ks.to(torch.bfloat16)
            kk = out["K"][:, t0:t1].float() + wl.shift_mag * u
            out["K"][:, t0:t1] = kk.to(torch.bfloat16)
        out["shifted_blocks"] = blocks.to(torch.int32)
    return out


# ---------------------------------------------------------------------------
# paged decode
# ---------------------------------------------------------------------------

def decode_inputs(wl: DecodeWorkload, device="cpu", pool_pages: Optional[int] = None
                  ) -> Dict[str, torch.Tensor]:
    """Paged decode tensors.

    Q [B,Hq,D], q_idx [B,Hkv,HI,dI] (bf16), w [B,Hkv,HI] fp32, and page pools
    K_pool, V_pool [P,Hkv,Bk,D], kidx_pool [P,Hkv,Bk,dI] (bf16).  The sequence
    page table seq_pt [B,max_pages] int32 maps logical block j of sequence b to
    its physical page (-1 past the end); seq_len [B] int32 holds L_b.
    """
    device = torch.device(device)
    sh = wl.shape
    P = wl.num_pages if pool_pages is None else pool_pages
    assert P >= wl.num_pages
    g = _gen(device, wl.seed)
    out = {
        "Q": _randn_bf16((wl.B, sh.Hq, sh.D), g, 1.0 / math.sqrt(sh.D), device),
        "q_idx": _randn_bf16((wl.B, sh.Hkv, sh.HI, sh.dI), g, 1.0 / math.sqrt(sh.dI), device),
        "w": _rand_f32((wl.B, sh.Hkv, sh.HI), g, device),
        "kidx_pool": _randn_bf16((P, sh.Hkv, sh.Bk, sh.dI), g, 1.0 / math.sqrt(sh.dI), device),
        "K_pool": _randn_bf16((P, sh.Hkv, sh.Bk, sh.D), g, 1.0 / math.sqrt(sh.D), device),
        "V_pool": _randn_bf16((P, sh.Hkv, sh.Bk, sh.D), g, 1.0 / math.sqrt(sh.D), device),
    }
    cg = torch.Generator().manual_seed(wl.seed + 1000)
    perm = torch.randperm(P, generator=cg) if wl.shuffle_pages else torch.arange(P)
    seq_pt = torch.full((wl.B, wl.max_pages), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(wl.pages_per_seq):
        seq_pt[b, :n] = perm[off:off + n].to(torch.int32)
        off += n
    out["seq_pt"] = seq_pt.to(device)
    out["seq_len"] = torch.tensor(wl.lengths, dtype=torch.int32).to(device)
    return out


def chunk_inputs(wl: ChunkWorkload, device="cpu", pool_pages: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """Tensors of one chunk over a paged cache.

    Q [B,S,Hq,D], q_idx [B,S,Hkv,HI,dI] (bf16) and w [B,S,Hkv,HI] fp32 for the
    chunk's queries; page pools K_pool, V_pool [P,Hkv,Bk,D], kidx_pool
    [P,Hkv,Bk,dI] (bf16) holding every sequence's q_pos[b] + S tokens (the
    chunk's own keys included); seq_pt [B,max_pages] int32 (-1 past the end),
    q_pos [B] int32 and seq_len = q_pos + S [B] int32.
    """
    device = torch.device(device)
    sh = wl.shape
    P = wl.num_pages if pool_pages is None else pool_pages
    assert P >= wl.num_pages
    g = _gen(device, wl.seed)
    out = {
        "Q": _randn_bf16((wl.B, wl.S, sh.Hq, sh.D), g, 1.0 / math.sqrt(sh.D), device),
        "q_idx": _randn_bf16((wl.B, wl.S, sh.Hkv, sh.HI, sh.dI), g, 1.0 / math.sqrt(sh.dI), device),
        "w": _rand_f32((wl.B, wl.S, sh.Hkv, sh.HI), g, device),
        "kidx_pool": _randn_bf16((P, sh.Hkv, sh.Bk, sh.dI), g, 1.0 / math.sqrt(sh.dI), device),
        "K_pool": _randn_bf16((P, sh.Hkv, sh.Bk, sh.D), g, 1.0 / math.sqrt(sh.D), device),
        "V_pool": _randn_bf16((P, sh.Hkv, sh.Bk, sh.D), g, 1.0 / math.sqrt(sh.D), device),
    }
    cg = torch.Generator().manual_seed(wl.seed + 1000)
    perm = torch.randperm(P, generator=cg) if wl.shuffle_pages else torch.arange(P)
    seq_pt = torch.full((wl.B, wl.max_pages), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(wl.pages_per_seq):
        seq_pt[b, :n] = perm[off:off + n].to(torch.int32)
        off += n
    out["seq_pt"] = seq_pt.to(device)
    out["q_pos"] = torch.tensor(wl.prefix, dtype=torch.int32).to(device)
    out["seq_len"] = torch.tensor(wl.lengths, dtype=torch.int32).to(device)
    return out
