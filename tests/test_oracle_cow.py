"""Pins of the oracle's copy-on-write (CPU).

The pages fix what copy-on-write must achieve: a prefix block is stored once and referenced
by every request that shares it, and a request that diverges gets its own copy before it
writes ("KV Cache 与推理优化", PagedAttention section: 相同前缀的块只存一份 ... 分歧时写时复制).
Paging and sharing change where K/V live, never what a request sees ("一个请求为什么越生成
越占内存?", section "分页改变分配方式，不改变独立 token 的表示").  So the strongest pin is an
equivalence: share + copy-on-write + append + decode must give, bit for bit, what private
copies of every block + append + decode give.  Hand-worked examples pin the bookkeeping."""
import numpy as np
import pytest

import oracle
import workloads


def test_hand_worked_example():
    # 8 blocks handed out in id order; blocks 0 and 1 hold a shared 32-position prefix.
    a = oracle.BlockAllocator(8)
    prefix = a.alloc(2)                                     # [0, 1], held by the prefix owner
    lens = [20, 32, 40, 17]
    t = oracle.build_block_tables(a, lens, 3, 16, prefix)
    assert t.tolist() == [[0, 1, -1], [0, 1, -1], [0, 1, 2], [0, 1, -1]]
    assert a.refcount[:3] == [5, 5, 1]
    t2, pairs = oracle.copy_on_write(a, t, lens)
    # seq 0 writes position 19 (block 1, shared): copy to 3; seq 1 position 31 (block 1):
    # copy to 4; seq 2 position 39 is in its own block 2: in place; seq 3 position 16
    # (block 1): copy to 5.  Block 1 keeps the owner's and seq 2's references.
    assert t2.tolist() == [[0, 3, -1], [0, 4, -1], [0, 1, 2], [0, 5, -1]]
    assert pairs.tolist() == [[1, 3], [1, 4], [1, 5]]
    assert a.refcount == [5, 2, 1, 1, 1, 1, 0, 0]
    assert a.free == [6, 7]
    assert t.tolist()[0] == [0, 1, -1]                      # the input is not modified


def test_last_holder_writes_in_place():
    a = oracle.BlockAllocator(4)
    blk = a.alloc(1)
    a.share(blk + blk)                                      # three holders of block 0
    t = np.zeros((3, 1), np.int32)
    t2, pairs = oracle.copy_on_write(a, t, [5, 5, 5])
    assert pairs.tolist() == [[0, 1], [0, 2]]
    assert t2[:, 0].tolist() == [1, 2, 0]
    assert a.refcount == [1, 1, 1, 0]


def test_exhaustion_leaves_the_allocator_unchanged():
    a = oracle.BlockAllocator(2)
    blk = a.alloc(1)
    a.share(blk + blk)
    t = np.zeros((3, 1), np.int32)
    with pytest.raises(MemoryError):
        oracle.copy_on_write(a, t, [3, 3, 3])
    assert a.refcount == [3, 0] and a.free == [1]


def _random_shared_case(seed, nblocks=64, prefix_blocks=3, batch=6, D=16, Hkv=2):
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = rng.integers(1, 16 * prefix_blocks + 20, size=batch).astype(np.int32)
    a = oracle.BlockAllocator(nblocks, rng.permutation(nblocks))
    prefix = a.alloc(prefix_blocks)
    mb = int(max(oracle.blocks_needed(int(L), 16) for L in lens))
    t = oracle.build_block_tables(a, lens, mb, 16, prefix)
    kc = workloads.bf16_bits(workloads.randn_bf16((nblocks, Hkv, 16, D), seed + 1))
    vc = workloads.bf16_bits(workloads.randn_bf16((nblocks, Hkv, 16, D), seed + 2))
    q = workloads.bf16_bits(workloads.randn_bf16((batch, 2 * Hkv, D), seed + 3))
    kn = workloads.bf16_bits(workloads.randn_bf16((batch, Hkv, D), seed + 4))
    vn = workloads.bf16_bits(workloads.randn_bf16((batch, Hkv, D), seed + 5))
    return a, lens, t, kc, vc, q, kn, vn


def _private_reference(lens, t, kc, vc, q, kn, vn, scale, Hkv):
    """Every sequence owns distinct blocks holding the same content: no sharing at all."""
    nblk = [oracle.blocks_needed(int(L), 16) for L in lens]
    pk = np.zeros((sum(nblk),) + kc.shape[1:], kc.dtype)
    pv = np.zeros_like(pk)
    pt = np.full(t.shape, -1, np.int32)
    nxt = 0
    for b, n in enumerate(nblk):
        for j in range(n):
            pk[nxt], pv[nxt] = kc[t[b, j]], vc[t[b, j]]
            pt[b, j] = nxt
            nxt += 1
    assert oracle.kv_append(kn, vn, oracle.slot_mapping(pt, lens), pk, pv) == 0
    st, out = oracle.paged_decode(q, pk, pv, pt, lens, scale, Hkv)
    assert st == 0
    return out


@pytest.mark.parametrize("seed", range(8))
def test_share_then_copy_on_write_equals_private_copies(seed):
    Hkv, scale = 2, float(np.float32(0.25))
    a, lens, t, kc, vc, q, kn, vn = _random_shared_case(seed, Hkv=Hkv)
    ref = _private_reference(lens, t, kc, vc, q, kn, vn, scale, Hkv)

    t2, pairs = oracle.copy_on_write(a, t, lens)
    k2, v2 = kc.copy(), vc.copy()
    oracle.copy_blocks(k2, v2, pairs)
    slots = oracle.slot_mapping(t2, lens)
    # invariants: every written block is held once; references equal table entries
    for s in slots:
        assert a.refcount[int(s) // 16] == 1
    held = sum(oracle.blocks_needed(int(L), 16) for L in lens) + 3     # + the prefix owner
    assert sum(a.refcount) == held
    assert len(a.free) == a.num_blocks - sum(1 for r in a.refcount if r > 0)
    assert oracle.kv_append(kn, vn, slots, k2, v2) == 0
    st, out = oracle.paged_decode(q, k2, v2, t2, lens, scale, Hkv)
    assert st == 0
    np.testing.assert_array_equal(out, ref)


def test_skipping_copy_on_write_is_caught():
    """The equivalence has teeth: appending straight into shared blocks changes what the
    other holders see (the seed is chosen so that several sequences write shared blocks)."""
    Hkv, scale = 2, float(np.float32(0.25))
    a, lens, t, kc, vc, q, kn, vn = _random_shared_case(3, Hkv=Hkv)
    ref = _private_reference(lens, t, kc, vc, q, kn, vn, scale, Hkv)
    _, pairs = oracle.copy_on_write(a, t, lens)
    assert len(pairs) >= 2
    k2, v2 = kc.copy(), vc.copy()
    assert oracle.kv_append(kn, vn, oracle.slot_mapping(t, lens), k2, v2) == 0
    st, out = oracle.paged_decode(q, k2, v2, t, lens, scale, Hkv)
    assert st == 0
    assert not np.array_equal(out, ref)


def test_layered_copy_blocks():
    k = np.arange(2 * 5 * 3, dtype=np.uint16).reshape(2, 5, 3)
    v = k + 1000
    oracle.copy_blocks(k, v, [[1, 4], [0, 2]], layered=True)
    assert (k[:, 4] == k[:, 1]).all() and (k[:, 2] == k[:, 0]).all()
    assert (v[:, 4] == v[:, 1]).all() and k[0, 3].tolist() == [9, 10, 11]
