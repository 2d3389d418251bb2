"""CPU-only checks of the C-ABI library: it loads, exports every symbol include/pkv.h
declares, and its host allocator / block tables / slot mapping equal the oracle's bit for
bit.  No kernel is launched here."""
import os
import re

import numpy as np
import pytest

import oracle
import workloads

pkv = pytest.importorskip("paged_kv_cache_159_gb300")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(pkv.LIB_PATH):
        from paged_kv_cache_159_gb300 import build
        build.build()
    return pkv.lib()


def _declared():
    with open(os.path.join(ROOT, "include", "pkv.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(lib):
    declared = _declared()
    assert len(declared) >= 18
    for name in declared:
        assert hasattr(lib, name), name
    assert set(declared) == set(pkv.EXPORTED)


def test_status_strings(lib):
    assert pkv.status_string(0) == "ok"
    assert "invalid" in pkv.status_string(1)
    assert pkv.status_string(99) == "unknown status"


@pytest.mark.parametrize("name", list(workloads.WORKLOADS))
def test_block_tables_and_slots_equal_the_oracle(lib, name):
    w = workloads.WORKLOADS[name]
    L = workloads.draw_seq_lens(w)
    nb = workloads.pool_blocks(w, L)
    mb = workloads.max_blocks(w, L)
    order = workloads.draw_free_order(w, nb)

    a = oracle.BlockAllocator(nb, order)
    prefix = a.alloc(w.prefix_blocks) if w.prefix_blocks else []
    t_orc = oracle.build_block_tables(a, L, mb, 16, prefix)

    p = pkv.Pool(nb, w.num_kv_heads, w.head_dim, free_order=order)
    prefix_p = p.alloc(w.prefix_blocks) if w.prefix_blocks else None
    if w.prefix_blocks:
        assert list(prefix_p) == list(prefix)
    t_pkv = p.build_block_tables(L, mb, prefix_p)
    assert np.array_equal(t_orc, t_pkv)
    assert p.num_free() == len(a.free)
    assert np.array_equal(pkv.slot_mapping(t_pkv, L), oracle.slot_mapping(t_orc, L))
    assert np.array_equal(pkv.slot_mapping_all(t_pkv, L), oracle.all_slots(t_orc, L))
    for blk in {int(x) for x in t_orc.ravel() if x >= 0}:
        assert p.refcount(blk) == a.refcount[blk]
    # return everything: the free lists stay in lock-step
    for row in t_orc:
        ids = [int(x) for x in row if x >= 0]
        a.release(ids)
        p.free(ids)
    if w.prefix_blocks:
        a.release(prefix)
        p.free(prefix_p)
    assert p.num_free() == nb == len(a.free)
    assert np.array_equal(p.alloc(nb), np.array(a.alloc(nb), dtype=np.int32))


def test_slot_mapping_page_example_at_block_size_4(lib):
    # steinslab.io §3.4: table [7, 3, 12], block_size 4, token 6 -> slot 14
    slots = pkv.slot_mapping(np.array([[7, 3, 12]], np.int32), np.array([7], np.int32), block_size=4)
    assert slots.tolist() == [14]


def test_allocator_errors(lib):
    with pytest.raises(pkv.PkvError) as e:
        pkv.Pool(0, 8, 128)
    assert e.value.status == pkv.ERR_INVALID
    for bad in (dict(head_dim=96), dict(block_size=32), dict(kv_dtype=7),
                dict(kv_dtype=pkv.KV_FP8E4M3, k_scale=0.0)):
        kw = dict(num_blocks=4, num_kv_heads=2, head_dim=64)
        kw.update(bad)
        with pytest.raises(pkv.PkvError):
            pkv.Pool(**kw)
    with pytest.raises(pkv.PkvError):
        pkv.Pool(4, 2, 64, free_order=[0, 1, 1, 2])
    p = pkv.Pool(4, 2, 64, free_order=[3, 2, 1, 0])
    with pytest.raises(pkv.PkvError) as e:
        p.alloc(5)
    assert e.value.status == pkv.ERR_OOM and p.num_free() == 4
    ids = p.alloc(2)
    assert ids.tolist() == [3, 2]
    with pytest.raises(pkv.PkvError):
        p.free([3, 3])                      # second reference does not exist
    assert p.refcount(3) == 1               # nothing changed by the failed call
    with pytest.raises(pkv.PkvError):
        p.share([1])                        # free block
    with pytest.raises(pkv.PkvError):
        p.build_block_tables([0], 2)         # empty sequence
    with pytest.raises(pkv.PkvError):
        p.build_block_tables([33], 2)        # needs 3 entries
    with pytest.raises(pkv.PkvError) as e:
        p.build_block_tables([16, 16, 16], 1)
    assert e.value.status == pkv.ERR_OOM
    assert p.num_free() == 2                # the failed call returned what it took
    assert p.alloc(2).tolist() == [1, 0]
    with pytest.raises(pkv.PkvError):
        pkv.slot_mapping(np.array([[5, -1]], np.int32), np.array([20], np.int32))


def test_decode_workspace_bytes_follows_the_plan(lib):
    # with the grid fixed, no device query is needed: counters + two partials per CTA
    p = pkv.Pool(64, 8, 128)
    ws = pkv.decode_workspace_bytes(p, 64, 32, 128, {"grid_ctas": 300})
    rows = 300 * 2 * 4
    assert ws >= 64 * 8 * 4 + rows * 128 * 4 + rows * 2 * 4
    assert pkv.decode_workspace_bytes(p, 4, 60, 2048, {"grid_ctas": 8}) == 0      # Hq % Hkv != 0
    assert pkv.decode_workspace_bytes(p, 4, 8 * 17, 2048, {"grid_ctas": 8}) == 0  # group > 16
    assert pkv.decode_workspace_bytes(p, 5000, 32, 8, {"grid_ctas": 8}) == 0      # batch > 4096
    # the split's cost per unit: -1 (an even split of the blocks) .. 4096; it sizes nothing
    for uc in (-1, 0, 1, 16, 4096):
        assert pkv.decode_workspace_bytes(p, 64, 32, 128, {"grid_ctas": 300, "unit_cost": uc}) == ws
    for uc in (-2, 4097):
        assert pkv.decode_workspace_bytes(p, 64, 32, 128, {"grid_ctas": 300, "unit_cost": uc}) == 0
    # the shared-prefix pass adds a partial state per query row (variant 3, one head per copy)
    wsp = pkv.decode_workspace_bytes(p, 64, 32, 128, {"grid_ctas": 300, "shared_prefix_blocks": 8})
    assert wsp >= ws + 64 * 4 + 64 * 32 * 128 * 4 + 64 * 32 * 2 * 4
    assert pkv.decode_workspace_bytes(p, 64, 32, 128, {"grid_ctas": 300, "shared_prefix_blocks": 8,
                                                       "variant": 2}) == 0


def test_device_calls_need_an_attached_pool(lib):
    p = pkv.Pool(8, 2, 64)
    st = lib.pkv_kv_append(p.handle, None, None, None, 1, None, None, None)
    assert st == pkv.ERR_INVALID
    st = lib.pkv_paged_attention_decode(p.handle, None, None, None, None, None, 1, 8, 1, 0.125,
                                        None, None, 0, None)
    assert st == pkv.ERR_INVALID


def test_pool_layers_descriptor(lib):
    # num_layers 0 means one layer; the stored descriptor says so
    assert pkv.Pool(4, 2, 64, num_layers=0).get_desc().num_layers == 1
    assert pkv.Pool(4, 2, 64, num_layers=80).get_desc().num_layers == 80
    for bad in (-1, 4097):
        with pytest.raises(pkv.PkvError) as e:
            pkv.Pool(4, 2, 64, num_layers=bad)
        assert e.value.status == pkv.ERR_INVALID
    # the kernels' (layer, block, head) tile index must fit in int32
    with pytest.raises(pkv.PkvError):
        pkv.Pool(1 << 20, 8, 128, num_layers=256)
    pkv.Pool((1 << 20) - 1, 8, 128, num_layers=255)


@pytest.mark.parametrize("layers,kv_heads,head_dim,elem", [
    (32, 8, 128, 2),      # Llama-3-8B: 128 KiB per token
    (80, 8, 128, 2),      # Llama-2/3-70B: 320 KiB per token
    (40, 32, 128, 2),     # the ~7B MHA worked example
    (32, 8, 128, 1),      # the same cache in FP8: half
])
def test_pool_bytes_per_token_equal_the_byte_formula(lib, layers, kv_heads, head_dim, elem):
    """A pool of L stacked layers costs exactly the pages' per-token byte count: K and V, every
    layer, every KV head, head_dim elements ("KV Cache 与推理优化", byte table; pinned in
    tests/golden/capacity.txt through oracle.kv_bytes)."""
    nb = 7
    p = pkv.Pool(nb, kv_heads, head_dim, pkv.KV_FP8E4M3 if elem == 1 else pkv.KV_BF16,
                 num_layers=layers)
    per_token = 2 * layers * p.layer_bytes() / (nb * pkv.BLOCK_SIZE)
    assert per_token == oracle.kv_bytes(layers, kv_heads, head_dim, elem, 1, 1)


def test_layer_workspace_counts_every_layer(lib):
    one = pkv.decode_workspace_bytes(pkv.Pool(64, 8, 128), 64, 32, 128, {"grid_ctas": 300})
    many = pkv.decode_workspace_bytes(pkv.Pool(64, 8, 128, num_layers=32), 64, 32, 128,
                                      {"grid_ctas": 300})
    assert many - one == (32 - 1) * 64 * 8 * 4        # one int32 counter per (layer, seq, head)


def test_layer_calls_need_an_attached_pool(lib):
    p = pkv.Pool(8, 2, 64, num_layers=3)
    assert lib.pkv_kv_append_layers(p.handle, None, None, None, 1, None, None, None) == pkv.ERR_INVALID
    assert lib.pkv_decode_step_layers(p.handle, None, None, None, None, None, None, None, 1, 8, 1,
                                      0.125, None, None, 0, None, None) == pkv.ERR_INVALID


def _both_allocators(nb, order, prefix_n, lens, mb):
    a = oracle.BlockAllocator(nb, order)
    p = pkv.Pool(nb, 2, 64, free_order=order)
    pre_a = a.alloc(prefix_n) if prefix_n else []
    pre_p = p.alloc(prefix_n) if prefix_n else None
    ta = oracle.build_block_tables(a, lens, mb, 16, pre_a)
    tp = p.build_block_tables(lens, mb, pre_p)
    np.testing.assert_array_equal(ta, tp)
    return a, p, ta


def _same_state(a, p):
    assert [p.refcount(i) for i in range(a.num_blocks)] == a.refcount
    assert p.num_free() == len(a.free)
    if a.free:                                  # the free list's order: take them all
        q = p.alloc(len(a.free))
        assert q.tolist() == a.free
        p.free(q)


@pytest.mark.parametrize("name", ["qwen25_7b_prefix_cow", "seeded"])
def test_cow_prepare_equals_the_oracle(lib, name):
    if name == "seeded":
        rng = np.random.Generator(np.random.PCG64(5))
        lens = rng.integers(1, 80, size=40).astype(np.int32)
        nb, prefix_n = 400, 4
        order = rng.permutation(nb).astype(np.int32)
    else:
        w = workloads.WORKLOADS[name]
        lens = workloads.draw_seq_lens(w)
        nb = workloads.pool_blocks(w, lens)
        order, prefix_n = workloads.draw_free_order(w, nb), w.prefix_blocks
    mb = int(max(oracle.blocks_needed(int(L), 16) for L in lens))
    a, p, t = _both_allocators(nb, order, prefix_n, lens, mb)
    ta, pa = oracle.copy_on_write(a, t, lens)
    tp, pp = p.cow_prepare(t, lens)
    assert len(pa) > 0
    np.testing.assert_array_equal(tp, ta)
    np.testing.assert_array_equal(pp, pa)
    _same_state(a, p)


def test_cow_prepare_hand_example_and_errors(lib):
    p = pkv.Pool(8, 2, 64)
    pre = p.alloc(2)
    lens = np.array([20, 32, 40, 17], np.int32)
    t = p.build_block_tables(lens, 3, pre)
    t2, pairs = p.cow_prepare(t, lens)
    assert t2.tolist() == [[0, 3, -1], [0, 4, -1], [0, 1, 2], [0, 5, -1]]
    assert pairs.tolist() == [[1, 3], [1, 4], [1, 5]]
    assert [p.refcount(i) for i in range(8)] == [5, 2, 1, 1, 1, 1, 0, 0]
    # INVALID: nothing changes
    with pytest.raises(pkv.PkvError) as e:
        p.cow_prepare(t2, np.array([20, 32, 40, 49], np.int32))     # needs a 4th entry
    assert e.value.status == pkv.ERR_INVALID
    bad = t2.copy()
    bad[3, 1] = 7                                                   # a free block
    with pytest.raises(pkv.PkvError):
        p.cow_prepare(bad, lens)
    assert [p.refcount(i) for i in range(8)] == [5, 2, 1, 1, 1, 1, 0, 0]


def test_cow_prepare_exhaustion_restores_everything(lib):
    for lens in ([3, 3, 3], [3, 3, 3, 3]):
        p = pkv.Pool(3, 2, 64, free_order=[0, 1, 2])
        blk = p.alloc(1)
        for _ in range(len(lens) - 1):
            p.share(blk)
        t = np.zeros((len(lens), 1), np.int32)
        a = oracle.BlockAllocator(3, [0, 1, 2])
        a.alloc(1)
        a.share([0] * (len(lens) - 1))
        if len(lens) == 3:                      # two copies fit: 0 -> 1, 0 -> 2
            t2, pairs = p.cow_prepare(t, np.array(lens, np.int32))
            ta, pa = oracle.copy_on_write(a, t, lens)
            np.testing.assert_array_equal(t2, ta)
            np.testing.assert_array_equal(pairs, pa)
            continue
        tables = t.copy()                       # three copies needed, two blocks free
        src = np.empty(4, np.int32)
        dst = np.empty(4, np.int32)
        n = pkv.ctypes.c_int32()
        st = lib.pkv_cow_prepare(p.handle, pkv._np_ptr(tables), pkv._np_ptr(np.array(lens, np.int32)),
                                 len(lens), 1, pkv._np_ptr(src), pkv._np_ptr(dst), pkv.ctypes.byref(n))
        assert st == pkv.ERR_OOM and n.value == 0
        np.testing.assert_array_equal(tables, t)
        with pytest.raises(MemoryError):
            oracle.copy_on_write(a, t, lens)
        _same_state(a, p)


def test_block_hashes_equal_the_oracle(lib):
    rng = np.random.Generator(np.random.PCG64(11))
    for n, salt in ((0, 0), (15, 3), (16, 0), (100, 2**64 - 1), (2048, 12345)):
        toks = rng.integers(-2**31, 2**31, size=n, dtype=np.int64).astype(np.int32)
        got = pkv.block_hashes(toks, salt)
        assert [int(x) for x in got] == oracle.block_hashes(toks.tolist(), salt)


def test_prefix_cache_follows_the_oracle_through_a_serving_trace(lib):
    """Requests with shared system prompts arrive, look up their cached prefix, take the
    rest from the free list, cache their blocks, finish and release; the pool evicts under
    pressure.  Every return value and the whole allocator state match the oracle's."""
    rng = np.random.Generator(np.random.PCG64(12))
    nb = 32                  # small enough that the trace evicts (38 blocks) and hits (150)
    order = rng.permutation(nb).astype(np.int32)
    a, c = oracle.BlockAllocator(nb, order), oracle.PrefixCache()
    p = pkv.Pool(nb, 2, 64, free_order=order)
    prompts = [rng.integers(0, 50000, size=int(n)).tolist() for n in (48, 64, 32)]
    live, hits, evicted = [], 0, 0
    for step in range(120):
        if live and (rng.random() < 0.45 or len(live) > 5):
            row = live.pop(int(rng.integers(len(live))))
            a.release(list(row))
            p.free(row)
        else:
            sysp = prompts[int(rng.integers(len(prompts)))]
            toks = sysp + rng.integers(0, 50000, size=int(rng.integers(0, 40))).tolist()
            salt = int(rng.integers(2))
            ha = c.lookup(toks, salt)
            hp = p.prefix_lookup(toks, salt)
            assert hp.tolist() == ha
            hits += len(ha)
            nblk = oracle.blocks_needed(len(toks), 16)
            need = nblk - len(ha)
            if need > len(a.free):                           # make room
                ea = c.evict(a, need - len(a.free))
                ep = p.prefix_evict(need - p.num_free())
                assert ep.tolist() == ea
                evicted += len(ea)
                if need > len(a.free):
                    continue
            ta = oracle.build_block_tables(a, [len(toks)], nblk, 16, ha)[0]
            tp = p.build_block_tables([len(toks)], nblk, hp)[0]
            assert tp.tolist() == ta.tolist()
            assert p.prefix_insert(toks, salt, tp) == c.insert(a, toks, salt, ta)
            live.append(tp)
        assert p.prefix_cached_blocks() == len(c.entries)
        assert [p.refcount(i) for i in range(nb)] == a.refcount
    assert hits > 100 and evicted > 20
    for row in live:
        a.release(list(row))
        p.free(row)
    c.clear(a)
    p.prefix_clear()
    assert p.prefix_cached_blocks() == 0 and p.num_free() == nb
    assert p.alloc(nb).tolist() == a.free                  # the free list's order too


def test_prefix_insert_errors_change_nothing(lib):
    p = pkv.Pool(8, 2, 64)
    row = p.alloc(2)
    toks = list(range(32))
    assert p.prefix_insert(toks, 0, row) == 2
    with pytest.raises(pkv.PkvError):
        p.prefix_insert(list(range(100, 132)), 0, row)     # blocks cached under another chain
    other = p.alloc(1)
    with pytest.raises(pkv.PkvError):
        p.prefix_insert(list(range(200, 232)), 0, [other[0], other[0]])   # the same block twice
    with pytest.raises(pkv.PkvError):
        p.prefix_insert(list(range(300, 316)), 0, [7])                    # a free block
    assert p.prefix_cached_blocks() == 2 and p.refcount(int(other[0])) == 1
    assert p.prefix_lookup(toks + [5] * 3).tolist() == row.tolist()


def test_prefill_plan_argument_errors(lib):
    p = pkv.Pool(64, 8, 128)
    bad = [
        (np.array([0, 5, 3], np.int32), np.array([5, 9], np.int32), 32, 4),    # negative chunk
        (np.array([1, 5], np.int32), np.array([5], np.int32), 32, 4),          # cu_q[0] != 0
        (np.array([0, 6], np.int32), np.array([5], np.int32), 32, 4),          # chunk longer than the sequence
        (np.array([0, 5], np.int32), np.array([100], np.int32), 32, 4),        # needs 7 table entries
        (np.array([0, 5], np.int32), np.array([5], np.int32), 12, 4),          # Hq not a multiple of Hkv
    ]
    for cu, lens, hq, mb in bad:
        out = np.zeros(1 << 16, np.uint8)
        grid = pkv.ctypes.c_int32()
        st = lib.pkv_prefill_plan(p.handle, pkv._np_ptr(cu), pkv._np_ptr(lens), lens.size, hq, mb,
                                  pkv._np_ptr(out), out.size, pkv.ctypes.byref(grid))
        assert st == pkv.ERR_INVALID, (cu, lens, hq)
    assert lib.pkv_prefill_plan_bytes(p.handle, 2, 8 * 17, 100) == 0          # group > 16
