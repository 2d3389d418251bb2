"""Seeded synthetic inputs for paged decode attention: shapes and random draws only.

This module serves both the oracle (tests) and the CUDA library (tests, bench, smoke).  It
holds none of the method's arithmetic: no attention, no slot addressing, no block tables.
It draws sequence lengths, the order in which a pool hands out its physical blocks, and
N(0,1) bf16 tensors.  The one size it computes is how many physical blocks a pool must
have, which fixes the shape of the input buffers.

Model shapes follow the attention layouts the pages quote: Llama-3-8B (32 q / 8 KV heads,
head_dim 128), Llama-3-70B (64 / 8), Qwen2.5-7B (28 / 4), all with 16-token blocks.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

BLOCK_SIZE = 16
BF16_NAN_BITS = 0x7FC0          # a quiet-NaN bf16 pattern used to poison unread slots


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    lengths: str                 # "list", "fixed", "uniform", "lognormal"
    fixed_len: int = 0
    len_list: tuple = ()
    max_len: int = 0
    pool: str = "exact"          # "exact", "double" (2x oversized), "fixed"
    fixed_blocks: int = 0
    prefix_blocks: int = 0       # shared leading blocks of every table
    k_gain: float = 1.0          # K drawn as k_gain * N(0,1)
    append: bool = True          # one kv_append per sequence before decode
    kv_dtype: str = "bf16"       # "bf16" or "fp8"
    layers: int = 1              # layers stacked in each cache (one table for all)
    seed: int = 159000

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def scale(self) -> float:
        """1/sqrt(head_dim) rounded to fp32 (the value both sides receive)."""
        return float(np.float32(1.0 / math.sqrt(self.head_dim)))


WORKLOADS = {
    "tiny": Workload("tiny", 2, 8, 2, 64, "list", len_list=(18, 33), pool="fixed",
                     fixed_blocks=8, seed=159000),
    "llama3_8b": Workload("llama3_8b", 64, 32, 8, 128, "fixed", fixed_len=2048, seed=159001),
    "ragged": Workload("ragged", 256, 32, 8, 128, "uniform", max_len=4096, pool="double",
                       k_gain=0.5, seed=159002),
    "llama3_70b_long": Workload("llama3_70b_long", 4, 64, 8, 128, "fixed", fixed_len=32768,
                                seed=159003),
    "qwen25_7b_prefix": Workload("qwen25_7b_prefix", 128, 28, 4, 128, "lognormal",
                                 max_len=8192, prefix_blocks=32, append=False, seed=159004),
    "qwen25_7b_prefix_fp8": Workload("qwen25_7b_prefix_fp8", 128, 28, 4, 128, "lognormal",
                                     max_len=8192, prefix_blocks=32, append=False,
                                     kv_dtype="fp8", seed=159004),
    # the prefix-sharing batch with appends: sequences whose newest position falls in a
    # shared block diverge and get a private copy first (copy-on-write)
    "qwen25_7b_prefix_cow": Workload("qwen25_7b_prefix_cow", 128, 28, 4, 128, "lognormal",
                                     max_len=8192, prefix_blocks=32, append=True, seed=159004),
    # every layer of a model in one step: caches [layers, NB, Hkv, 16, D]
    "tiny_layers": Workload("tiny_layers", 2, 8, 2, 64, "list", len_list=(18, 33), pool="fixed",
                            fixed_blocks=8, layers=3, seed=159005),
    "llama3_8b_32l": Workload("llama3_8b_32l", 64, 32, 8, 128, "fixed", fixed_len=2048,
                              layers=32, seed=159006),
}


def _blocks(n: int) -> int:
    return -(-int(n) // BLOCK_SIZE)


def draw_seq_lens(w: Workload) -> np.ndarray:
    """Sequence lengths, counting the token appended this step (int32 [B])."""
    rng = np.random.Generator(np.random.PCG64(w.seed))
    if w.lengths == "list":
        L = np.array(w.len_list, dtype=np.int64)
    elif w.lengths == "fixed":
        L = np.full(w.batch, w.fixed_len, dtype=np.int64)
    elif w.lengths == "uniform":
        L = rng.integers(1, w.max_len, size=w.batch, endpoint=True)
    elif w.lengths == "lognormal":
        # median 1500, log-sigma 0.6, clipped to [16, max_len]
        L = np.rint(np.exp(rng.normal(math.log(1500.0), 0.6, size=w.batch)))
        L = np.clip(L, 16, w.max_len).astype(np.int64)
    else:
        raise ValueError(w.lengths)
    assert len(L) == w.batch
    return L.astype(np.int32)


def max_blocks(w: Workload, seq_lens) -> int:
    """Width of the block table: enough entries for the longest sequence."""
    return max(_blocks(int(L)) for L in seq_lens)


def pool_blocks(w: Workload, seq_lens) -> int:
    need = sum(_blocks(int(L)) for L in seq_lens)
    if w.prefix_blocks:
        need = w.prefix_blocks + sum(max(0, _blocks(int(L)) - w.prefix_blocks)
                                     for L in seq_lens)
        if w.append:                       # room for one private copy per sequence
            need += len(seq_lens)
    if w.pool == "exact":
        return need
    if w.pool == "double":
        return 2 * need
    if w.pool == "fixed":
        assert w.fixed_blocks >= need
        return w.fixed_blocks
    raise ValueError(w.pool)


def draw_free_order(w: Workload, num_blocks: int) -> np.ndarray:
    """Seeded permutation of physical block ids: the order the free pool hands them out."""
    rng = np.random.Generator(np.random.PCG64(w.seed + 7919))
    return rng.permutation(num_blocks).astype(np.int32)


def randn_bf16(shape, seed: int, device="cpu", gain: float = 1.0,
               chunk_rows: int = 1 << 14) -> torch.Tensor:
    """gain * N(0,1) drawn in fp32 by a seeded torch generator, rounded to bf16.  Drawn in
    chunks along dim 0 so that multi-GB pools need no multi-GB fp32 temporary."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    rows = shape[0]
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        x = torch.randn((r1 - r0,) + tuple(shape[1:]), generator=g, device=device,
                        dtype=torch.float32)
        if gain != 1.0:
            x.mul_(gain)
        out[r0:r1].copy_(x)
    return out


@dataclasses.dataclass
class Draw:
    """One seeded instance of a workload (bf16 tensors on ``device``)."""
    w: Workload
    seq_lens: np.ndarray         # int32 [B]
    num_blocks: int
    max_blocks: int
    free_order: np.ndarray       # int32 [num_blocks]
    # with w.layers > 1 every tensor below gets a leading [layers] dimension
    q: torch.Tensor              # bf16 [B, Hq, D]
    key_cache: torch.Tensor      # bf16 [NB, Hkv, 16, D]  (history; source of an fp8 pool)
    value_cache: torch.Tensor    # bf16 [NB, Hkv, 16, D]
    k_new: torch.Tensor          # bf16 [B, Hkv, D]
    v_new: torch.Tensor          # bf16 [B, Hkv, D]


def draw(w: Workload, device="cpu", seq_lens=None) -> Draw:
    L = draw_seq_lens(w) if seq_lens is None else np.asarray(seq_lens, dtype=np.int32)
    nb = pool_blocks(w, L)
    mb = max_blocks(w, L)
    B, Hq, Hkv, D = len(L), w.num_q_heads, w.num_kv_heads, w.head_dim
    s = w.seed * 16
    nl = w.layers
    lead = (nl,) if nl > 1 else ()
    rows = max(1, (1 << 24) // (Hkv * BLOCK_SIZE * D))

    def pool(seed, gain=1.0):               # drawn as [layers * NB, ...], then viewed
        t = randn_bf16((nl * nb, Hkv, BLOCK_SIZE, D), seed, device, gain, chunk_rows=rows)
        return t.view(lead + (nb, Hkv, BLOCK_SIZE, D))

    return Draw(
        w=w, seq_lens=L, num_blocks=nb, max_blocks=mb, free_order=draw_free_order(w, nb),
        q=randn_bf16(lead + (B, Hq, D), s + 1, device),
        key_cache=pool(s + 2, w.k_gain),
        value_cache=pool(s + 3),
        k_new=randn_bf16(lead + (B, Hkv, D), s + 4, device, w.k_gain),
        v_new=randn_bf16(lead + (B, Hkv, D), s + 5, device),
    )


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Host uint16 view of a bf16 tensor's bit patterns."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------------------------------
# Prefill workloads: per sequence a context of C_b cached positions and a chunk of P_b new
# positions (C_b = 0: a whole prompt).  The pages' prefill example is a prompt of about
# 2000 tokens ("理解 KV Cache" §2.1); shapes are the Llama-3-8B layer's.
# ------------------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class PrefillWorkload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    chunk: int                   # P_b for every sequence, or the upper end of U{1..chunk}
    context: int = 0             # C_b = context for every sequence, or U{0..context}
    ragged: bool = False         # draw P_b and C_b uniformly instead
    seed: int = 159100
    chunk_list: tuple = ()       # explicit P_b per sequence (with context_list), overriding the above
    context_list: tuple = ()
    kv_dtype: str = "bf16"       # the pool: "bf16", or "fp8" (E4M3, per-tensor scales amax / 448)

    @property
    def scale(self) -> float:
        return float(np.float32(1.0 / math.sqrt(self.head_dim)))


PREFILL_WORKLOADS = {
    "prefill_tiny": PrefillWorkload("prefill_tiny", 3, 8, 2, 64, chunk=40, context=37,
                                    ragged=True, seed=159100),
    "prefill_llama3_8b": PrefillWorkload("prefill_llama3_8b", 8, 32, 8, 128, chunk=2048,
                                         seed=159101),
    "chunked_prefill_llama3_8b": PrefillWorkload("chunked_prefill_llama3_8b", 16, 32, 8, 128,
                                                 chunk=512, context=8192, ragged=False,
                                                 seed=159102),
    # the same chunked batch over an FP8 E4M3 pool
    "chunked_prefill_llama3_8b_fp8": PrefillWorkload("chunked_prefill_llama3_8b_fp8", 16, 32, 8, 128,
                                                     chunk=512, context=8192, ragged=False,
                                                     seed=159102, kv_dtype="fp8"),
}


@dataclasses.dataclass
class PrefillDraw:
    w: PrefillWorkload
    chunk_lens: np.ndarray       # int32 [B]  P_b
    seq_lens: np.ndarray         # int32 [B]  C_b + P_b
    cu_q: np.ndarray             # int32 [B+1]
    num_blocks: int
    max_blocks: int
    free_order: np.ndarray
    q: torch.Tensor              # bf16 [T, Hq, D]
    key_cache: torch.Tensor      # bf16 [NB, Hkv, 16, D]  (the context's history)
    value_cache: torch.Tensor
    k_chunk: torch.Tensor        # bf16 [T, Hkv, D]  (the chunk's rows, appended before attention)
    v_chunk: torch.Tensor


def draw_prefill(w: PrefillWorkload, device="cpu") -> PrefillDraw:
    rng = np.random.Generator(np.random.PCG64(w.seed))
    if w.chunk_list:
        assert len(w.chunk_list) == len(w.context_list) == w.batch
        P, C = np.array(w.chunk_list), np.array(w.context_list)
    elif w.ragged:
        P = rng.integers(1, w.chunk, size=w.batch, endpoint=True)
        C = rng.integers(0, w.context, size=w.batch, endpoint=True)
    else:
        P = np.full(w.batch, w.chunk)
        C = (rng.integers(0, w.context, size=w.batch, endpoint=True) if w.context
             else np.zeros(w.batch, dtype=np.int64))
    P, C = P.astype(np.int32), C.astype(np.int32)
    L = (C + P).astype(np.int32)
    cu = np.concatenate([[0], np.cumsum(P)]).astype(np.int32)
    nb = int(sum(_blocks(int(x)) for x in L))
    mb = int(max(_blocks(int(x)) for x in L))
    T, Hq, Hkv, D = int(cu[-1]), w.num_q_heads, w.num_kv_heads, w.head_dim
    s = w.seed * 16
    rows = max(1, (1 << 24) // (Hkv * BLOCK_SIZE * D))
    return PrefillDraw(
        w=w, chunk_lens=P, seq_lens=L, cu_q=cu, num_blocks=nb, max_blocks=mb,
        free_order=draw_free_order(Workload(w.name, 1, 1, 1, D, "fixed", seed=w.seed), nb),
        q=randn_bf16((T, Hq, D), s + 1, device),
        key_cache=randn_bf16((nb, Hkv, BLOCK_SIZE, D), s + 2, device, chunk_rows=rows),
        value_cache=randn_bf16((nb, Hkv, BLOCK_SIZE, D), s + 3, device, chunk_rows=rows),
        k_chunk=randn_bf16((T, Hkv, D), s + 4, device),
        v_chunk=randn_bf16((T, Hkv, D), s + 5, device),
    )
