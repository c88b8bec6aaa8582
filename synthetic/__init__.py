"""Seeded synthetic inputs for block-sparse attention.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no mask rule, no softmax, no split logic).  Both the CUDA
library's tests/bench and the fp64 oracle take their inputs from here, so the
two sides see bit-identical data.

Workload shapes follow the five configurations the library is measured on:

  C1  prefill 1x2x512x64     fp16, top-3 block scores, tril, causal
  C2  prefill 2x8x4096x128   bf16, top-16, tril + dense last rows, causal
  C3  prefill 1x32x16384x128 bf16, threshold 0.9 (~10% density), tril + dense last, causal
  C4  prefill 4x16x8192x64   fp16, non-causal, threshold 0.75 (~25% density), Q/K/V ~ N(0, 0.5^2)
  C5  GQA varlen decode 8 seqs, 32 q-heads / 8 kv-heads, d=128 bf16,
      cache_seqlens uniform in [8192, 65536], 64 selected blocks per (b, kv-head)

Recipe (all on the CPU, torch.Generator, seed 0 unless a test says otherwise):
  * Q, K, V: one generator, randn fp32 in the order Q, K, V, times `std`,
    then rounded to the storage dtype (round-to-nearest-even by torch).
  * block scores: a separate generator, rand fp32 [B, H, nq, nk] (uniform [0,1)).
  * decode: a generator draws cache_seqlens = randint(lo, hi + 1, (B,)), then for
    every (b, kv-head), in that order, randperm(nb - 1) whose first nsel - 1
    entries plus the last block nb - 1 form the selection, sorted descending and
    padded with -1 to max_sel.  A second generator draws q, then K and V for the
    valid tokens of each sequence (b ascending); tokens at or past
    cache_seqlens[b] are set to `fill` (0 by default, NaN in poisoning tests).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

BLOCK = 64


@dataclass(frozen=True)
class PrefillConfig:
    name: str
    B: int
    H: int
    S: int
    d: int
    dtype: torch.dtype
    causal: bool
    rule: str            # "topk" or "threshold"
    param: float         # k for top-k, threshold value for threshold
    tril: bool
    dense_last: bool
    std: float = 1.0

    @property
    def nblk(self) -> int:
        return math.ceil(self.S / BLOCK)


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    dtype: torch.dtype
    seqlen_lo: int
    seqlen_hi: int       # inclusive
    Smax: int
    nsel: int            # selected blocks per (b, kv-head), last block included
    max_sel: int


PREFILL_CONFIGS = {
    "C1": PrefillConfig("C1", 1, 2, 512, 64, torch.float16, True, "topk", 3, True, False),
    "C2": PrefillConfig("C2", 2, 8, 4096, 128, torch.bfloat16, True, "topk", 16, True, True),
    "C3": PrefillConfig("C3", 1, 32, 16384, 128, torch.bfloat16, True, "threshold", 0.9, True, True),
    "C4": PrefillConfig("C4", 4, 16, 8192, 64, torch.float16, False, "threshold", 0.75, False, False,
                        std=0.5),
}

DECODE_CONFIGS = {
    "C5": DecodeConfig("C5", 8, 32, 8, 128, torch.bfloat16, 8192, 65536, 65536, 64, 64),
}


def qkv(B: int, H: int, Sq: int, Sk: int, d: int, dtype: torch.dtype, std: float = 1.0,
        seed: int = 0):
    """Q [B,H,Sq,d], K and V [B,H,Sk,d] (BHSD, contiguous), drawn N(0, std^2)."""
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, Sq, d, generator=g)
    k = torch.randn(B, H, Sk, d, generator=g)
    v = torch.randn(B, H, Sk, d, generator=g)
    if std != 1.0:
        q, k, v = q * std, k * std, v * std
    return q.to(dtype), k.to(dtype), v.to(dtype)


def block_scores(B: int, H: int, nq: int, nk: int, seed: int = 0) -> torch.Tensor:
    """Uniform [0,1) fp32 importance scores, one per (query block, key block)."""
    g = torch.Generator().manual_seed(seed)
    return torch.rand(B, H, nq, nk, generator=g)


def prefill_inputs(cfg: PrefillConfig, seed: int = 0):
    """(q, k, v, scores) for a prefill configuration."""
    q, k, v = qkv(cfg.B, cfg.H, cfg.S, cfg.S, cfg.d, cfg.dtype, cfg.std, seed)
    scores = block_scores(cfg.B, cfg.H, cfg.nblk, cfg.nblk, seed)
    return q, k, v, scores


def decode_selection(B: int, Hkv: int, seqlen_lo: int, seqlen_hi: int, nsel: int, max_sel: int,
                     seed: int = 0, block: int = BLOCK):
    """cache_seqlens int32 [B] and block_indices int32 [B, Hkv, max_sel].

    Each (b, kv-head) row lists min(nsel, nb) distinct valid blocks, always
    including the last one, in descending order, padded with -1.
    """
    g = torch.Generator().manual_seed(seed)
    seqlens = torch.randint(seqlen_lo, seqlen_hi + 1, (B,), generator=g)
    idx = torch.full((B, Hkv, max_sel), -1, dtype=torch.int32)
    for b in range(B):
        nb = (int(seqlens[b]) + block - 1) // block
        for h in range(Hkv):
            perm = torch.randperm(nb - 1, generator=g)[: max(0, min(nsel, nb) - 1)]
            sel = torch.cat([torch.tensor([nb - 1]), perm]).sort(descending=True).values
            idx[b, h, : sel.numel()] = sel.to(torch.int32)
    return seqlens.to(torch.int32), idx


def decode_qkv(B: int, Hq: int, Hkv: int, Smax: int, d: int, dtype: torch.dtype,
               seqlens: torch.Tensor, seed: int = 0, fill: float = 0.0):
    """q [B,Hq,d]; K, V [B,Smax,Hkv,d] (BSHD) with N(0,1) valid tokens."""
    g = torch.Generator().manual_seed(seed + 1)
    q = torch.randn(B, Hq, d, generator=g).to(dtype)
    k = torch.full((B, Smax, Hkv, d), fill, dtype=dtype)
    v = torch.full((B, Smax, Hkv, d), fill, dtype=dtype)
    for b in range(B):
        n = int(seqlens[b])
        k[b, :n] = torch.randn(n, Hkv, d, generator=g).to(dtype)
        v[b, :n] = torch.randn(n, Hkv, d, generator=g).to(dtype)
    return q, k, v


def decode_inputs(cfg: DecodeConfig, seed: int = 0, fill: float = 0.0):
    """(q, k, v, cache_seqlens, block_indices) for a decode configuration."""
    seqlens, idx = decode_selection(cfg.B, cfg.Hkv, cfg.seqlen_lo, cfg.seqlen_hi, cfg.nsel,
                                    cfg.max_sel, seed)
    q, k, v = decode_qkv(cfg.B, cfg.Hq, cfg.Hkv, cfg.Smax, cfg.d, cfg.dtype, seqlens, seed, fill)
    return q, k, v, seqlens, idx


def random_block_mask(B: int, H: int, nq: int, nk: int, density: float, seed: int = 0):
    """Bernoulli(density) uint8 block mask, for edge-case tests."""
    g = torch.Generator().manual_seed(seed + 7)
    return (torch.rand(B, H, nq, nk, generator=g) < density).to(torch.uint8)
