"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws inputs: lengths, cu_seqlens prefix sums, block tables
and bf16 values.  It holds none of the attention arithmetic, so the oracle and
the CUDA path can both be fed from it.

Recipe (identical bits on every machine for a given seed):
  * lengths and block-id permutations come from ``numpy.random.default_rng(seed)``;
  * values come from a CPU ``torch.Generator`` seeded with ``value_seed``:
    ``randn`` in fp32, times sigma, rounded to bf16 (round-to-nearest-even) on
    the CPU, drawn in the order q, k, v (decode: q, k_pool, v_pool).

Workloads (lengths per the plan's packed layout and cu_seqlens semantics):
  * tiny:      lengths [1, 7, 64, 129] for q and k, H=2, D=64, N(0, 1);
  * packed:    16 sequences, L ~ U{1..2048}, cu_q == cu_k, H=16, D=128, N(0, 1), causal;
  * longtail:  one 8192-token sequence, then floor(exp(U(ln 16, ln 8193))) lengths
               (the last one clipped) until the total is 32768, order shuffled;
               H=32, D=128, N(0, 0.5^2), causal;
  * cross:     32 sequences, Lq ~ U{1..512}, Lk ~ U{1..4096} independent, then
               Lk = 1 for 4 sequences picked without replacement; H=8, D=64 or 256,
               N(0, 1), non-causal;
  * decode:    64 sequences, context ~ U{128..8192} tokens, n_blocks = ceil(ctx/16),
               Hq=32, Hkv=8, D=128, block_size=16; the pool holds exactly
               sum(n_blocks) blocks and logical block j of sequence s sits at
               physical id perm[offset_s + j] for a seeded permutation perm;
               step t covers logical blocks [32 t, 32 t + 32);
  * decode-long: a few long contexts (the first 65536 tokens, the others
               U{49152..65536}), the decode workload's heads, dims, block
               size and block-id permutation, and one tile holding every
               block of a context (4096 blocks), so one step covers it.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch


def cu_seqlens(lengths) -> np.ndarray:
    """int32 [B+1]: 0, then running totals of the lengths."""
    out = np.zeros(len(lengths) + 1, dtype=np.int64)
    out[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    if out[-1] > np.iinfo(np.int32).max:
        raise ValueError("total length does not fit int32")
    return out.astype(np.int32)


def bf16_normal(shape, sigma: float, gen: torch.Generator) -> torch.Tensor:
    """randn(shape) * sigma in fp32, rounded to bf16, on the CPU."""
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if sigma != 1.0:
        x = x * sigma
    return x.to(torch.bfloat16)


@dataclass
class VarlenCase:
    name: str
    lengths_q: List[int]
    lengths_k: List[int]
    num_heads: int
    head_dim: int
    causal: bool
    softmax_scale: float
    q: torch.Tensor            # bf16 [Tq, H, D], CPU
    k: torch.Tensor            # bf16 [Tk, H, D], CPU
    v: torch.Tensor            # bf16 [Tk, H, D], CPU
    cu_seqlens_q: np.ndarray   # int32 [B+1]
    cu_seqlens_k: np.ndarray   # int32 [B+1]

    @property
    def batch(self) -> int:
        return len(self.lengths_q)

    @property
    def total_q(self) -> int:
        return int(self.cu_seqlens_q[-1])

    @property
    def total_k(self) -> int:
        return int(self.cu_seqlens_k[-1])

    @property
    def max_seqlen_q(self) -> int:
        return max(self.lengths_q) if self.lengths_q else 0

    @property
    def max_seqlen_k(self) -> int:
        return max(self.lengths_k) if self.lengths_k else 0


def make_varlen(name: str, lengths_q, lengths_k, num_heads: int, head_dim: int, causal: bool,
                sigma: float, value_seed: int, softmax_scale: Optional[float] = None) -> VarlenCase:
    lengths_q = [int(x) for x in lengths_q]
    lengths_k = [int(x) for x in lengths_k]
    if len(lengths_q) != len(lengths_k):
        raise ValueError("q and k need one length per sequence each")
    cq, ck = cu_seqlens(lengths_q), cu_seqlens(lengths_k)
    gen = torch.Generator(device="cpu").manual_seed(int(value_seed))
    q = bf16_normal((int(cq[-1]), num_heads, head_dim), sigma, gen)
    k = bf16_normal((int(ck[-1]), num_heads, head_dim), sigma, gen)
    v = bf16_normal((int(ck[-1]), num_heads, head_dim), sigma, gen)
    if softmax_scale is None:
        softmax_scale = float(np.float32(1.0 / math.sqrt(head_dim)))
    return VarlenCase(name, lengths_q, lengths_k, num_heads, head_dim, bool(causal),
                      float(softmax_scale), q, k, v, cq, ck)


# -- length recipes ----------------------------------------------------------

def tiny_lengths() -> List[int]:
    return [1, 7, 64, 129]


def packed_lengths(seed: int) -> List[int]:
    rng = np.random.default_rng(seed)
    return [int(x) for x in rng.integers(1, 2049, 16)]


def longtail_lengths(seed: int, total: int = 32768, longest: int = 8192,
                     lo: int = 16) -> List[int]:
    rng = np.random.default_rng(seed)
    lengths = [longest]
    acc = longest
    while acc < total:
        x = int(math.floor(math.exp(rng.uniform(math.log(lo), math.log(longest + 1)))))
        x = min(x, total - acc)
        lengths.append(x)
        acc += x
    order = rng.permutation(len(lengths))
    return [lengths[int(j)] for j in order]


def cross_lengths(seed: int):
    rng = np.random.default_rng(seed)
    lq = rng.integers(1, 513, 32)
    lk = rng.integers(1, 4097, 32)
    ones = rng.choice(32, 4, replace=False)
    lk[ones] = 1
    return [int(x) for x in lq], [int(x) for x in lk]


# -- the named workloads -------------------------------------------------------

def tiny(causal: bool, seed: int = 0) -> VarlenCase:
    L = tiny_lengths()
    return make_varlen("tiny" + ("-causal" if causal else ""), L, L, 2, 64, causal, 1.0,
                       value_seed=seed)


@dataclass
class Fp8Inputs:
    """FP8 E4M3 q and k codes (uint8, shaped like the case's q and k) with one descale each."""
    q8: torch.Tensor
    k8: torch.Tensor
    descale_q: float
    descale_k: float


def fp8_qk(case: VarlenCase, descale: float = 1.0 / 32.0) -> Fp8Inputs:
    """The case's q and k rounded to FP8 E4M3 codes of x / descale (a power of two, so
    descale * code is exact in bf16 too); seeded through the case's own values."""
    def enc(t):
        return (t.float() / descale).to(torch.float8_e4m3fn).view(torch.uint8).contiguous()
    return Fp8Inputs(enc(case.q), enc(case.k), descale, descale)


def upstream_grad(case: VarlenCase, seed: int) -> torch.Tensor:
    """Seeded upstream gradient dL/dout for the backward: N(0, 1) in bf16, shaped like q."""
    g = torch.Generator().manual_seed(1_000_003 + seed)
    return torch.randn(case.q.shape, generator=g).to(torch.bfloat16)


def packed(seed: int = 0) -> VarlenCase:
    L = packed_lengths(seed)
    return make_varlen("packed", L, L, 16, 128, True, 1.0, value_seed=seed)


def longtail(seed: int = 0) -> VarlenCase:
    L = longtail_lengths(seed)
    return make_varlen("longtail", L, L, 32, 128, True, 0.5, value_seed=seed)


def cross(head_dim: int, seed: int = 0) -> VarlenCase:
    lq, lk = cross_lengths(seed)
    # same lengths for both head dims, separate value draws
    return make_varlen(f"cross-d{head_dim}", lq, lk, 8, head_dim, False, 1.0,
                       value_seed=seed * 1000 + head_dim)


VARLEN_WORKLOADS = {
    "tiny": lambda seed=0: tiny(False, seed),
    "tiny-causal": lambda seed=0: tiny(True, seed),
    "packed": packed,
    "longtail": longtail,
    "cross-d64": lambda seed=0: cross(64, seed),
    "cross-d256": lambda seed=0: cross(256, seed),
}


@dataclass
class DecodeCase:
    name: str
    context_lengths: List[int]
    n_blocks: List[int]
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    tile_capacity: int
    q: torch.Tensor              # bf16 [S, Hq, D]
    k_pool: torch.Tensor         # bf16 [N_blk, block_size, Hkv, D]
    v_pool: torch.Tensor         # bf16 [N_blk, block_size, Hkv, D]
    block_table: List[np.ndarray] = field(default_factory=list)  # per sequence: physical ids

    @property
    def num_seqs(self) -> int:
        return len(self.n_blocks)

    @property
    def num_blocks(self) -> int:
        return int(self.k_pool.shape[0])

    @property
    def num_steps(self) -> int:
        cap = self.tile_capacity
        return max((n + cap - 1) // cap for n in self.n_blocks) if self.n_blocks else 0

    def tile(self, t: int):
        """Inputs of step t: (tile_blocks int32 [S, cap], tile_block_counts int32 [S])."""
        cap = self.tile_capacity
        tb = np.zeros((self.num_seqs, cap), dtype=np.int32)
        tc = np.zeros((self.num_seqs,), dtype=np.int32)
        for s, ids in enumerate(self.block_table):
            part = ids[t * cap:(t + 1) * cap]
            tc[s] = len(part)
            tb[s, :len(part)] = part
        return tb, tc

    def tile_tokens(self, t: int) -> np.ndarray:
        """Tokens of step t that lie inside each sequence's context: int32 [S],
        min(tile_block_counts * block_size, context_length - t * cap * block_size), >= 0."""
        tb, tc = self.tile(t)
        start = t * self.tile_capacity * self.block_size
        ctx = np.asarray(self.context_lengths, dtype=np.int64)
        return np.clip(ctx - start, 0, tc.astype(np.int64) * self.block_size).astype(np.int32)

    def kv_bytes(self) -> int:
        """Bytes of K and V the listed blocks hold (each read once)."""
        per_block = self.block_size * self.num_kv_heads * self.head_dim * 2
        return 2 * per_block * sum(self.n_blocks)


def make_decode(name: str, n_blocks, num_q_heads: int, num_kv_heads: int, head_dim: int,
                block_size: int, tile_capacity: int, perm: np.ndarray, value_seed: int,
                sigma: float = 1.0, context_lengths=None) -> DecodeCase:
    n_blocks = [int(x) for x in n_blocks]
    total = sum(n_blocks)
    table = []
    off = 0
    for n in n_blocks:
        table.append(np.asarray(perm[off:off + n], dtype=np.int32))
        off += n
    gen = torch.Generator(device="cpu").manual_seed(int(value_seed))
    S = len(n_blocks)
    q = bf16_normal((S, num_q_heads, head_dim), sigma, gen)
    k_pool = bf16_normal((total, block_size, num_kv_heads, head_dim), sigma, gen)
    v_pool = bf16_normal((total, block_size, num_kv_heads, head_dim), sigma, gen)
    if context_lengths is None:
        context_lengths = [n * block_size for n in n_blocks]
    return DecodeCase(name, [int(c) for c in context_lengths], n_blocks, num_q_heads,
                      num_kv_heads, head_dim, block_size, tile_capacity, q, k_pool, v_pool,
                      table)


def decode(seed: int = 0, num_seqs: int = 64, ctx_lo: int = 128, ctx_hi: int = 8192,
           num_q_heads: int = 32, num_kv_heads: int = 8, head_dim: int = 128,
           block_size: int = 16, tile_capacity: int = 32) -> DecodeCase:
    rng = np.random.default_rng(seed)
    ctx = rng.integers(ctx_lo, ctx_hi + 1, num_seqs)
    n_blocks = [int(-(-int(c) // block_size)) for c in ctx]
    perm = rng.permutation(sum(n_blocks)).astype(np.int32)
    return make_decode("decode", n_blocks, num_q_heads, num_kv_heads, head_dim, block_size,
                       tile_capacity, perm, value_seed=seed, context_lengths=[int(c) for c in ctx])


def decode_long(seed: int = 0, num_seqs: int = 4, longest: int = 65536, shortest: int = 49152,
                num_q_heads: int = 32, num_kv_heads: int = 8, head_dim: int = 128,
                block_size: int = 16) -> DecodeCase:
    """A few long contexts decoded in one tile step each (tile capacity = the
    longest context's blocks)."""
    rng = np.random.default_rng(seed)
    ctx = [longest] + [int(c) for c in rng.integers(shortest, longest + 1, num_seqs - 1)]
    n_blocks = [int(-(-c // block_size)) for c in ctx]
    perm = rng.permutation(sum(n_blocks)).astype(np.int32)
    return make_decode("decode-long", n_blocks, num_q_heads, num_kv_heads, head_dim, block_size,
                       max(n_blocks), perm, value_seed=seed + 500, context_lengths=ctx)
