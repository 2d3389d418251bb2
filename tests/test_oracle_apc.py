"""Pins of the oracle's automatic prefix caching (CPU).

"KV Cache 与推理优化", section "APC：连计算都省了": every full block gets a hash; a new
request whose prefix equals a cached one reuses those physical blocks; the lookup walks
the request's blocks and stops at the first miss, after which nothing can hit.  "一个请求为
什么越生成越占内存?" (paging section): reuse must match the tokens, their positions and the
model -- hence chained hashes with a per-model salt."""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "fnv1a64.txt")


def _golden():
    rows = []
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if not line:
            continue
        text, hexval = line.rsplit(None, 1)
        rows.append((text.strip('"').encode(), int(hexval, 16)))
    return rows


def test_fnv1a_64_published_values():
    rows = _golden()
    assert len(rows) == 3
    for data, want in rows:
        assert oracle.fnv1a_64(data) == want


def test_block_hash_is_fnv_of_parent_and_tokens():
    """Block 0 hashes the salt's 8 bytes and its tokens' 4-byte little-endian words; block 1
    starts from block 0's hash.  Checked against byte strings built by hand."""
    toks = list(range(100, 132))
    h = oracle.block_hashes(toks, salt=7)
    b0 = bytes([7, 0, 0, 0, 0, 0, 0, 0]) + b"".join(bytes([t, 0, 0, 0]) for t in range(100, 116))
    assert h[0] == oracle.fnv1a_64(b0)
    b1 = h[0].to_bytes(8, "little") + b"".join(bytes([t, 0, 0, 0]) for t in range(116, 132))
    assert h[1] == oracle.fnv1a_64(b1)
    assert len(oracle.block_hashes(toks[:31])) == 1           # a partial block has no hash


def test_chain_and_salt():
    rng = np.random.Generator(np.random.PCG64(3))
    toks = rng.integers(0, 128000, size=160).tolist()
    base = oracle.block_hashes(toks)
    other = list(toks)
    other[37] += 1                                            # in block 2
    h2 = oracle.block_hashes(other)
    assert h2[:2] == base[:2] and all(a != b for a, b in zip(h2[2:], base[2:]))
    assert all(a != b for a, b in zip(oracle.block_hashes(toks, salt=1), base))


def _request(alloc, cache, toks, salt=0):
    """Serve one prompt: reuse the cached prefix blocks, allocate the rest, cache all."""
    hits = cache.lookup(toks, salt)
    L = len(toks)
    nblk = oracle.blocks_needed(L, 16)
    t = oracle.build_block_tables(alloc, [L], nblk, 16, hits)[0]
    cache.insert(alloc, toks, salt, t)
    return hits, t


def test_lookup_stops_at_the_first_miss():
    a, c = oracle.BlockAllocator(64), oracle.PrefixCache()
    rng = np.random.Generator(np.random.PCG64(4))
    sys_prompt = rng.integers(0, 1000, size=64).tolist()       # 4 full blocks
    A = sys_prompt + rng.integers(0, 1000, size=40).tolist()
    hits, ta = _request(a, c, A)
    assert hits == [] and len(c.entries) == 6                  # 104 tokens: 6 full blocks
    # same system prompt, then different tokens: exactly the 4 prompt blocks hit
    B = sys_prompt + rng.integers(0, 1000, size=50).tolist()
    hits, tb = _request(a, c, B)
    assert hits == list(ta[:4]) and list(tb[:4]) == hits
    # a request equal to A except one token of block 1: only block 0 hits, although its
    # blocks 2.. hold the same tokens as A's (the page: nothing after the first miss hits)
    C = list(A)
    C[20] ^= 1
    assert c.lookup(C) == [ta[0]]
    # the same tokens under another model (salt) hit nothing
    assert c.lookup(A, salt=99) == []
    # a partial block is never reused: a 70-token prefix of A hits its 4 full blocks only
    assert c.lookup(A[:70]) == list(ta[:4])


def test_reference_counts_and_eviction():
    a, c = oracle.BlockAllocator(16), oracle.PrefixCache()
    A = list(range(48))                                        # 3 blocks
    hits, ta = _request(a, c, A)
    assert [a.refcount[b] for b in ta] == [2, 2, 2]            # the request + the cache
    a.release(list(ta))                                        # the request finishes
    assert [a.refcount[b] for b in ta] == [1, 1, 1] and len(a.free) == 13
    B = list(range(32)) + [999] * 16                           # shares blocks 0-1 with A
    hits, tb = _request(a, c, B)
    assert hits == list(ta[:2])
    # leaves held only by the cache: A's block 2 (B's block 2 is still held by B).  LRU
    # among leaves, children before parents: A's block 2 goes first, then nothing else
    # (blocks 0-1 have a cached child, B's block 2, held by B)
    assert c.evict(a, 5) == [ta[2]]
    a.release(list(tb))                                        # B finishes
    assert c.evict(a, 5) == [tb[2], ta[1], ta[0]]
    assert len(a.free) == 16 and c.entries == {}


def test_a_hash_collision_is_not_a_hit():
    """Plant an entry whose hash equals a request's block hash but whose tokens differ (a
    collision): the lookup must not return it."""
    a, c = oracle.BlockAllocator(8), oracle.PrefixCache()
    toks = list(range(16))
    h = oracle.block_hashes(toks)[0]
    blk = a.alloc(1)[0]
    c.entries[blk] = {"hash": h, "block": blk, "parent": -1, "salt": 0,
                      "tokens": list(range(1, 17)), "children": 0, "stamp": 0}
    assert c.lookup(toks) == []


def test_insert_rejects_a_block_cached_under_another_chain():
    a, c = oracle.BlockAllocator(8), oracle.PrefixCache()
    _, ta = _request(a, c, list(range(16)))
    with pytest.raises(ValueError):
        c.insert(a, list(range(100, 116)), 0, ta)               # ta[0] is cached already
    assert len(c.entries) == 1 and a.refcount[ta[0]] == 2
