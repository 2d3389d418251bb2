"""The oracle: a plain, slow, obviously-correct CPU statement of paged decode attention.

TEST INFRASTRUCTURE ONLY.  Only tests/, ``__graft_entry__.smoke()`` and bench.py's
cpu_baseline / reference leg may import this package.  It shares no code with the CUDA
library in ``paged_kv_cache_159_gb300`` and never imports it.

Pieces and the passage each follows (page title, section):

* ``kv_bytes`` -- bytes = 2 * layers * kv_heads * head_dim * elem_bytes * tokens * seqs.
  "KV Cache 与推理优化" (note.yj-dis.top), section "KV Cache 有多大：一张显存账单";
  "一个请求为什么越生成越占内存?" (learning-field-guides), section "按 K 与 V 的维度推导容量";
  "理解 KV Cache" (steinslab.io), §1.4.
* ``blocks_needed`` / ``block_capacity`` / ``empty_slots`` -- a sequence of n positions
  takes ceil(n / bs) fixed-size blocks; "一个请求为什么越生成越占内存?", section
  "分页改变分配方式，不改变独立 token 的表示" (18 positions -> 2 blocks, 14 empty).
* ``slot_of`` / ``slot_mapping`` -- "理解 KV Cache" (steinslab.io), §3.3 and the §3.4 example.
* ``BlockAllocator`` / ``build_block_tables`` -- block lifecycle (allocate from a free
  pool, use, return), "理解 KV Cache" §3.5; block tables mapping logical to physical
  blocks and shared prefix blocks referenced by many tables, "KV Cache 与推理优化",
  section "PagedAttention：把 KV Cache 当虚拟内存管".
* ``copy_on_write`` / ``copy_blocks`` -- a shared prefix block is stored once and referenced
  by many tables until a request diverges, when the diverging request gets its own copy
  before it writes ("KV Cache 与推理优化", section "PagedAttention：把 KV Cache 当虚拟内存管",
  its benefits table and summary tree: 分歧时写时复制).
* ``fnv1a_64`` / ``block_hashes`` / ``PrefixCache`` -- automatic prefix caching: a hash
  per full block, a new request reuses the cached physical blocks of its longest cached
  prefix, and the lookup stops at the first block that misses ("KV Cache 与推理优化",
  section "APC：连计算都省了"); reuse must match the token sequence, the positions and the
  model ("一个请求为什么越生成越占内存?", paging section, on prefix sharing), so each block's
  hash chains the previous block's hash and starts from a per-model salt.  The hash is
  64-bit FNV-1a (Fowler, Noll, Vo), written from its definition.
* ``paged_prefill`` -- a prompt (or a chunk of one) of P tokens after C cached positions:
  query i sits at position C + i and attends causally over positions 0 .. C + i ("理解 KV
  Cache" §1.2: position i aggregates only positions <= i; §2.1: prefill computes every
  prompt position at once; "KV Cache 与推理优化", pitfalls table: packed sequences need a
  per-sequence (block-diagonal) causal mask).  Each query is therefore a decode query whose
  sequence length is its position + 1, and ``paged_prefill`` is ``paged_decode`` over those
  per-query lengths.
* ``kv_append`` / ``paged_decode`` / FP8 codec -- C code in ``pkv_oracle.c`` (fp64).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

BF16 = 0
FP8E4M3 = 1

_lib = None


def lib():
    """Load (building first if needed) the C part of the oracle."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.oracle_e4m3_decode.restype = ctypes.c_double
        L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_encode.restype = ctypes.c_uint8
        L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        L.oracle_e4m3_quantize.restype = ctypes.c_uint8
        L.oracle_e4m3_quantize.argtypes = [ctypes.c_float, ctypes.c_float]
        L.oracle_kv_append.restype = ctypes.c_int
        L.oracle_kv_append.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_float,
            ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p]
        L.oracle_paged_decode.restype = ctypes.c_int
        L.oracle_paged_decode.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_float,
            ctypes.c_float, ctypes.c_float, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
            ctypes.c_void_p]
        L.oracle_max_threads.restype = ctypes.c_int
        L.oracle_max_threads.argtypes = []
        _lib = L
    return _lib


def max_threads() -> int:
    return int(lib().oracle_max_threads())


# ------------------------------------------------------------------------------------
# Capacity arithmetic (plain integers).
# ------------------------------------------------------------------------------------
def kv_bytes(layers: int, kv_heads: int, head_dim: int, elem_bytes: int,
             tokens: int = 1, seqs: int = 1) -> int:
    """K and V bytes: 2 (K and V) x layers x kv_heads x head_dim x elem_bytes x T x N."""
    return 2 * layers * kv_heads * head_dim * elem_bytes * tokens * seqs


def blocks_needed(positions: int, block_size: int) -> int:
    """Whole blocks a sequence of ``positions`` cached tokens occupies (ceil)."""
    if positions < 0 or block_size < 1:
        raise ValueError("positions >= 0 and block_size >= 1 required")
    return (positions + block_size - 1) // block_size


def block_capacity(positions: int, block_size: int) -> int:
    """Token positions the allocated blocks can hold."""
    return blocks_needed(positions, block_size) * block_size


def empty_slots(positions: int, block_size: int) -> int:
    """Unused positions in the last block (internal fragmentation, < one block)."""
    return block_capacity(positions, block_size) - positions


# ------------------------------------------------------------------------------------
# Slot addressing ("理解 KV Cache" §3.3): two-level lookup.
# ------------------------------------------------------------------------------------
def slot_of(block_table, i: int, block_size: int):
    """Return (logical_block, offset, physical_block, slot) for token position i."""
    logical = i // block_size
    offset = i % block_size
    physical = int(block_table[logical])
    return logical, offset, physical, physical * block_size + offset


def slot_mapping(block_tables, seq_lens, block_size: int = 16) -> np.ndarray:
    """Slot of each sequence's newest token, at position seq_len - 1 (int64 [B])."""
    out = np.empty(len(seq_lens), dtype=np.int64)
    for b, L in enumerate(seq_lens):
        out[b] = slot_of(block_tables[b], int(L) - 1, block_size)[3]
    return out


# ------------------------------------------------------------------------------------
# Block lifecycle ("理解 KV Cache" §3.5): a free pool handed out in a fixed order,
# reference counts for blocks that several tables share.
# ------------------------------------------------------------------------------------
class BlockAllocator:
    def __init__(self, num_blocks: int, free_order=None):
        order = list(range(num_blocks)) if free_order is None else [int(x) for x in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of 0..num_blocks-1")
        self.num_blocks = num_blocks
        self.free = list(order)          # front of the list is handed out first
        self.refcount = [0] * num_blocks

    def alloc(self, n: int):
        if n > len(self.free):
            raise MemoryError("pool exhausted")
        ids, self.free = self.free[:n], self.free[n:]
        for i in ids:
            self.refcount[i] = 1
        return ids

    def share(self, ids):
        for i in ids:
            if self.refcount[i] < 1:
                raise ValueError("cannot share a free block")
            self.refcount[i] += 1

    def release(self, ids):
        for i in ids:
            if self.refcount[i] < 1:
                raise ValueError("double free")
            self.refcount[i] -= 1
            if self.refcount[i] == 0:
                self.free.append(i)


def build_block_tables(allocator: BlockAllocator, seq_lens, max_blocks: int,
                       block_size: int = 16, prefix_ids=()) -> np.ndarray:
    """One table row per sequence: its first min(len(prefix_ids), nblk) entries are the
    shared prefix blocks (one more reference each), the rest fresh blocks from the free
    pool in order; unused entries are -1.  int32 [B, max_blocks]."""
    prefix_ids = [int(x) for x in prefix_ids]
    tables = np.full((len(seq_lens), max_blocks), -1, dtype=np.int32)
    for b, L in enumerate(seq_lens):
        nblk = blocks_needed(int(L), block_size)
        if nblk > max_blocks:
            raise ValueError("sequence longer than its block table")
        shared = prefix_ids[:nblk]
        allocator.share(shared)
        fresh = allocator.alloc(nblk - len(shared))
        tables[b, :nblk] = shared + fresh
    return tables


def copy_on_write(allocator: BlockAllocator, block_tables, seq_lens, block_size: int = 16):
    """Make the block each sequence is about to write private, in batch order.

    Sequence b writes its newest position L_b - 1, in logical block (L_b - 1) // block_size.
    If that physical block is referenced more than once, the sequence diverges from the
    others sharing it: it takes a fresh block from the free pool, gives up its reference to
    the shared one, and its table entry is pointed at the fresh block, whose content must be
    a copy of the shared block's before anything is written.  A block whose other holders
    have all diverged already has one reference left and is written in place.

    Returns (tables, pairs): a new int32 table array and int32 [n, 2] (shared, fresh) pairs
    in the order they were made.  On exhaustion the allocator is left as it was and
    MemoryError is raised."""
    tables = np.array(block_tables, dtype=np.int32, copy=True)
    saved_free, saved_ref = list(allocator.free), list(allocator.refcount)
    pairs = []
    try:
        for b, L in enumerate(seq_lens):
            L = int(L)
            if L < 1 or blocks_needed(L, block_size) > tables.shape[1]:
                raise ValueError("sequence length outside its table")
            j = (L - 1) // block_size
            shared = int(tables[b, j])
            if shared < 0 or shared >= allocator.num_blocks or allocator.refcount[shared] < 1:
                raise ValueError("table entry is not an allocated block")
            if allocator.refcount[shared] == 1:
                continue                                   # private already
            fresh = allocator.alloc(1)[0]
            allocator.release([shared])                    # stays > 0: others still hold it
            tables[b, j] = fresh
            pairs.append((shared, fresh))
    except Exception:
        allocator.free, allocator.refcount = saved_free, saved_ref
        raise
    return tables, np.array(pairs, dtype=np.int32).reshape(-1, 2)


def copy_blocks(key_cache: np.ndarray, value_cache: np.ndarray, pairs, layered: bool = False):
    """cache[dst] = cache[src] for each (src, dst) pair, K and V; with ``layered`` the caches
    are [layers, NB, ...] and every layer is copied.  In place."""
    for src, dst in np.asarray(pairs, dtype=np.int64).reshape(-1, 2):
        if layered:
            key_cache[:, dst] = key_cache[:, src]
            value_cache[:, dst] = value_cache[:, src]
        else:
            key_cache[dst] = key_cache[src]
            value_cache[dst] = value_cache[src]


# ------------------------------------------------------------------------------------
# Automatic prefix caching ("KV Cache 与推理优化", section "APC：连计算都省了").
# ------------------------------------------------------------------------------------
FNV64_OFFSET = 0xCBF29CE484222325
FNV64_PRIME = 0x100000001B3
_M64 = (1 << 64) - 1


def fnv1a_64(data: bytes, h: int = FNV64_OFFSET) -> int:
    """64-bit FNV-1a: for each byte, xor it into the state, then multiply by the prime."""
    for byte in data:
        h = ((h ^ byte) * FNV64_PRIME) & _M64
    return h


def block_hashes(tokens, salt: int = 0, block_size: int = 16):
    """Hash of every full block of a token sequence (a partial last block has none).
    Block i hashes the 8 little-endian bytes of the previous block's hash (the salt for
    block 0) followed by its tokens as 4 little-endian bytes each, so equal hashes mean an
    equal salt and equal tokens in every position up to the end of that block."""
    out, prev = [], int(salt) & _M64
    for i in range(len(tokens) // block_size):
        data = prev.to_bytes(8, "little") + b"".join(
            int(t & 0xFFFFFFFF).to_bytes(4, "little") for t in tokens[i * block_size:(i + 1) * block_size])
        prev = fnv1a_64(data)
        out.append(prev)
    return out


class PrefixCache:
    """Cached full blocks, each held by one reference of its own while it is cached.

    An entry is (hash, block, parent block or -1, salt, tokens).  A lookup walks a request's
    full blocks in order; block i hits an entry with its hash whose parent is the block hit
    for i-1, whose salt is the request's and whose tokens are block i's tokens (so a hash
    collision can never hand out the wrong block), and the walk stops at the first miss.
    Every hit or insert stamps its entry from a counter; eviction takes the entry with the
    smallest stamp among those with no cached child whose block no table holds."""

    def __init__(self, block_size: int = 16):
        self.bs = block_size
        self.entries = {}             # block -> dict
        self.clock = 0

    def _touch(self, e):
        self.clock += 1
        e["stamp"] = self.clock

    def _match(self, h, parent, salt, toks):
        for e in self.entries.values():
            if e["hash"] == h and e["parent"] == parent and e["salt"] == salt and e["tokens"] == toks:
                return e
        return None

    def _blocks(self, tokens):
        return [list(map(int, tokens[i * self.bs:(i + 1) * self.bs]))
                for i in range(len(tokens) // self.bs)]

    def lookup(self, tokens, salt: int = 0):
        """Physical blocks of the longest cached prefix (full blocks only)."""
        hits, parent = [], -1
        for h, toks in zip(block_hashes(tokens, salt, self.bs), self._blocks(tokens)):
            e = self._match(h, parent, salt, toks)
            if e is None:
                break
            self._touch(e)
            hits.append(e["block"])
            parent = e["block"]
        return hits

    def insert(self, allocator: BlockAllocator, tokens, salt: int, table_row):
        """Cache every full block of a request whose table row is ``table_row``; blocks
        already cached (by an equal chain) are only stamped.  Returns how many blocks were
        added.  A row block that is cached under another chain makes the call fail with
        nothing changed (ValueError)."""
        hs, blocks = block_hashes(tokens, salt, self.bs), self._blocks(tokens)
        if len(table_row) < len(hs):
            raise ValueError("table row shorter than the full blocks")
        plan, parent, planned = [], -1, set()       # validate before changing anything
        for i, (h, toks) in enumerate(zip(hs, blocks)):
            e = self._match(h, parent, salt, toks)
            if e is not None:
                plan.append(("hit", e))
                parent = e["block"]
                continue
            b = int(table_row[i])
            if (b < 0 or b >= allocator.num_blocks or allocator.refcount[b] < 1 or
                    b in self.entries or b in planned):
                raise ValueError("row block is not an allocated, uncached block")
            planned.add(b)
            plan.append(("new", (h, b, parent, toks)))
            parent = b
        added = 0
        for kind, x in plan:
            if kind == "hit":
                self._touch(x)
                continue
            h, b, par, toks = x
            e = {"hash": h, "block": b, "parent": par, "salt": int(salt), "tokens": toks,
                 "children": 0, "stamp": 0}
            self._touch(e)
            self.entries[b] = e
            if par >= 0:
                self.entries[par]["children"] += 1
            allocator.share([b])
            added += 1
        return added

    def _drop(self, allocator: BlockAllocator, e):
        del self.entries[e["block"]]
        if e["parent"] >= 0:
            self.entries[e["parent"]]["children"] -= 1
        allocator.release([e["block"]])

    def evict(self, allocator: BlockAllocator, n: int):
        """Free up to n cached blocks, least recently used first; returns their ids."""
        out = []
        while len(out) < n:
            cand = [e for e in self.entries.values()
                    if e["children"] == 0 and allocator.refcount[e["block"]] == 1]
            if not cand:
                break
            e = min(cand, key=lambda x: x["stamp"])
            self._drop(allocator, e)
            out.append(e["block"])
        return out

    def clear(self, allocator: BlockAllocator):
        """Drop every entry (children before parents: leaves by stamp, repeatedly)."""
        while self.entries:
            leaves = [e for e in self.entries.values() if e["children"] == 0]
            self._drop(allocator, min(leaves, key=lambda x: x["stamp"]))


def live_positions(block_tables, seq_lens, num_blocks: int, block_size: int = 16) -> np.ndarray:
    """bool [num_blocks, block_size]: True where some sequence's position maps (slot_of)."""
    live = np.zeros((num_blocks, block_size), dtype=bool)
    for b, L in enumerate(seq_lens):
        L = int(L)
        nblk = blocks_needed(L, block_size)
        phys = np.asarray(block_tables[b][:nblk], dtype=np.int64)
        live[phys[:-1], :] = True                          # full blocks
        last = L - (nblk - 1) * block_size                 # positions in the last block
        live[phys[-1], :last] = True
    return live


def all_slots(block_tables, seq_lens, block_size: int = 16) -> np.ndarray:
    """int64 slots of every position 0..L-1 of every sequence, sequence-major."""
    out = []
    for b, L in enumerate(seq_lens):
        i = np.arange(int(L), dtype=np.int64)
        phys = np.asarray(block_tables[b], dtype=np.int64)[i // block_size]
        out.append(phys * block_size + i % block_size)
    return np.concatenate(out) if out else np.zeros(0, np.int64)


def poison_unused(cache: np.ndarray, block_tables, seq_lens, block_size: int, fill_bits: int):
    """Overwrite every cache position that no sequence may read -- tail slots of each
    sequence's last block and blocks no table references -- with ``fill_bits`` (a bf16
    NaN pattern in the tests).  ``cache`` is [num_blocks, Hkv, bs, D] of uint16/uint8."""
    live = live_positions(block_tables, seq_lens, cache.shape[0], block_size)
    mask = ~live                                           # [NB, bs]
    cache[np.broadcast_to(mask[:, None, :, None], cache.shape)] = fill_bits
    return cache


# ------------------------------------------------------------------------------------
# FP8 E4M3 codec and the fp64 kernels (C).
# ------------------------------------------------------------------------------------
def e4m3_decode(code: int) -> float:
    return float(lib().oracle_e4m3_decode(int(code) & 0xFF))


def e4m3_encode(x: float) -> int:
    return int(lib().oracle_e4m3_encode(float(x)))


def e4m3_quantize(x: float, scale: float) -> int:
    return int(lib().oracle_e4m3_quantize(float(x), float(scale)))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def kv_append(k_bits, v_bits, slots, key_cache, value_cache, block_size=16,
              kv_dtype=BF16, k_scale=1.0, v_scale=1.0) -> int:
    """Scatter K/V rows (bf16 bit patterns, uint16 [T, Hkv, D]) into the caches in place."""
    k_bits = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v_bits = np.ascontiguousarray(v_bits, dtype=np.uint16)
    slots = np.ascontiguousarray(slots, dtype=np.int64)
    assert key_cache.flags.c_contiguous and value_cache.flags.c_contiguous
    T, Hkv, D = k_bits.shape
    return int(lib().oracle_kv_append(
        _ptr(k_bits), _ptr(v_bits), _ptr(slots), T, Hkv, D, block_size, key_cache.shape[0],
        kv_dtype, k_scale, v_scale, _ptr(key_cache), _ptr(value_cache)))


def paged_decode(q_bits, key_cache, value_cache, block_tables, seq_lens, scale: float,
                 num_kv_heads: int, block_size: int = 16, kv_dtype=BF16, k_scale=1.0,
                 v_scale=1.0, pairs=None, num_threads: int = 1):
    """fp64 paged decode attention.  q_bits: uint16 [B, Hq, D] (bf16 patterns).
    Returns (status, out float64 [B, Hq, D]); with ``pairs`` only those (b, hq) rows of
    ``out`` are computed (the rest stay zero)."""
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    block_tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    assert key_cache.flags.c_contiguous and value_cache.flags.c_contiguous
    B, Hq, D = q_bits.shape
    out = np.zeros((B, Hq, D), dtype=np.float64)
    if pairs is not None:
        pairs = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
        pptr, npairs = _ptr(pairs), pairs.shape[0]
    else:
        pptr, npairs = None, 0
    st = lib().oracle_paged_decode(
        _ptr(q_bits), _ptr(key_cache), _ptr(value_cache), _ptr(block_tables), _ptr(seq_lens),
        B, Hq, num_kv_heads, D, block_tables.shape[1], block_size, key_cache.shape[0],
        kv_dtype, k_scale, v_scale, scale, pptr, npairs, num_threads, _ptr(out))
    return int(st), out


def paged_prefill(q_bits, key_cache, value_cache, block_tables, seq_lens, cu_q, scale: float,
                  num_kv_heads: int, block_size: int = 16, kv_dtype=BF16, k_scale=1.0,
                  v_scale=1.0, num_threads: int = 1):
    """fp64 causal attention of packed prompt chunks over the paged cache.

    q_bits: uint16 [T, Hq, D] (bf16 patterns), rows cu_q[b] .. cu_q[b+1]-1 belonging to
    sequence b; seq_lens[b] counts the sequence's positions including the chunk (whose K/V
    are already in the cache).  Row cu_q[b] + i is position seq_lens[b] - P_b + i and sees
    positions 0 .. that position.  Returns (status, out float64 [T, Hq, D])."""
    cu_q = np.asarray(cu_q, dtype=np.int64)
    rows, lens = [], []
    for b in range(len(seq_lens)):
        P = int(cu_q[b + 1] - cu_q[b])
        first = int(seq_lens[b]) - P
        if P < 0 or first < 0:
            return 1, None
        for i in range(P):
            rows.append(b)
            lens.append(first + i + 1)
    tables = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32)[np.asarray(rows, dtype=np.int64)]
                                  if rows else np.zeros((0, np.asarray(block_tables).shape[1]), np.int32))
    return paged_decode(q_bits, key_cache, value_cache, tables, np.asarray(lens, dtype=np.int32),
                        scale, num_kv_heads, block_size, kv_dtype, k_scale, v_scale,
                        num_threads=num_threads)
