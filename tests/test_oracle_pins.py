"""Pins for the oracle: each test checks it against something other than itself -- numbers
the pages print (tests/golden), a library routine (torch's fp64 scaled_dot_product_attention,
torch's float8_e4m3fn conversion), closed forms, invariants, or brute force."""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import BF16, FP8E4M3

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
NAN16 = 0x7FC0


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split("|")[0].split()


# ------------------------------------------------------------------ capacity arithmetic
def test_kv_bytes_matches_printed_numbers():
    rows = list(_rows("capacity.txt"))
    assert len(rows) >= 20
    for r in rows:
        layers, kvh, d, e, t, n, expected = map(int, r)
        assert oracle.kv_bytes(layers, kvh, d, e, t, n) == expected, r


def test_gqa_ratios_printed_by_the_pages():
    # pyllm.pages.dev §1.2 conclusions: 32 q / 8 KV heads -> 1/4; 28 q / 4 KV heads -> 1/7
    assert oracle.kv_bytes(32, 32, 128, 2) == 4 * oracle.kv_bytes(32, 8, 128, 2)
    assert oracle.kv_bytes(28, 28, 128, 2) == 7 * oracle.kv_bytes(28, 4, 128, 2)
    # note.yj-dis.top: 64 -> 8 KV heads takes 2560 KiB to 320 KiB per token
    assert oracle.kv_bytes(80, 64, 128, 2) == 8 * oracle.kv_bytes(80, 8, 128, 2)
    # note.yj-dis.top byte formula: FP8 (1 byte) halves a 2-byte cache
    assert 2 * oracle.kv_bytes(32, 8, 128, 1) == oracle.kv_bytes(32, 8, 128, 2)


def test_capacity_counterexample():
    # learning-field-guides acceptance: 13.04 GiB weights + 8 GiB KV + 3 GiB = 24.04 > 22
    kv_gib = oracle.kv_bytes(32, 8, 128, 2, 8192, 8) / 2**30
    assert kv_gib == 8.0
    assert math.isclose(13.04 + kv_gib + 3.0, 24.04) and 13.04 + kv_gib + 3.0 > 22.0


def test_block_counts_printed_by_the_pages():
    for r in _rows("blocks.txt"):
        n, bs, blocks, cap, empty = map(int, r)
        assert oracle.blocks_needed(n, bs) == blocks
        assert oracle.block_capacity(n, bs) == cap
        assert oracle.empty_slots(n, bs) == empty


def test_block_counts_brute_force():
    # smallest number of bs-sized blocks covering n positions, by search
    for bs in (1, 4, 16):
        for n in range(0, 200):
            k = 0
            while k * bs < n:
                k += 1
            assert oracle.blocks_needed(n, bs) == k
            assert 0 <= oracle.empty_slots(n, bs) < bs


# ------------------------------------------------------------------ slot addressing
def test_slot_example_printed_by_the_page():
    (row,) = list(_rows("slot_example.txt"))
    bs, table, token = int(row[0]), [int(x) for x in row[1].split(",")], int(row[2])
    expected = tuple(map(int, row[3:]))
    assert oracle.slot_of(table, token, bs) == expected


def test_slot_mapping_is_a_bijection_onto_used_blocks():
    # every position of every sequence lands in a distinct slot of its own blocks
    rng = np.random.default_rng(1)
    lens = [1, 15, 16, 17, 40, 64]
    alloc = oracle.BlockAllocator(40, rng.permutation(40))
    tables = oracle.build_block_tables(alloc, lens, 4)
    seen = set()
    for b, L in enumerate(lens):
        for i in range(L):
            lg, off, phys, slot = oracle.slot_of(tables[b], i, 16)
            assert phys == tables[b][i // 16] and slot // 16 == phys and slot % 16 == i % 16
            assert slot not in seen
            seen.add(slot)
    sm = oracle.slot_mapping(tables, lens)
    for b, L in enumerate(lens):
        assert sm[b] == tables[b][(L - 1) // 16] * 16 + (L - 1) % 16


# ------------------------------------------------------------------ allocator
def test_allocator_hands_out_free_order_without_replacement():
    order = np.random.default_rng(3).permutation(64)
    a = oracle.BlockAllocator(64, order)
    lens = [18, 33, 1, 16, 17]
    t = oracle.build_block_tables(a, lens, 3)
    used = [int(x) for x in t.ravel() if x >= 0]
    assert used == [int(x) for x in order[:len(used)]]
    assert len(used) == sum(oracle.blocks_needed(L, 16) for L in lens) == 2 + 3 + 1 + 1 + 2
    assert (t[2, 1:] == -1).all() and (t[0, 2] == -1)
    with pytest.raises(MemoryError):
        a.alloc(64)
    a.release(t[1, :3])
    assert a.free[-3:] == [int(x) for x in t[1, :3]]
    with pytest.raises(ValueError):
        a.release([int(t[1, 0])])


def test_allocator_prefix_sharing_and_refcounts():
    a = oracle.BlockAllocator(16, np.arange(16)[::-1])
    prefix = a.alloc(2)                       # 15, 14
    t = oracle.build_block_tables(a, [8, 40, 20], 3, prefix_ids=prefix)
    assert list(t[0]) == [15, -1, -1]          # 8 positions need only the first shared block
    assert list(t[1][:2]) == [15, 14] and list(t[2][:2]) == [15, 14]
    assert a.refcount[15] == 4 and a.refcount[14] == 3
    for row in t:
        a.release([int(x) for x in row if x >= 0])
    assert a.refcount[15] == 1 and 15 not in a.free
    a.release(prefix)
    assert sorted(a.free) == list(range(16))


# ------------------------------------------------------------------ FP8 E4M3 codec
def test_e4m3_decode_table_matches_torch_and_closed_forms():
    lib_vals = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(
        torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        ours = oracle.e4m3_decode(c)
        if c & 0x7F == 0x7F:
            assert math.isnan(ours) and math.isnan(lib_vals[c])
        else:
            assert ours == lib_vals[c], hex(c)
    assert oracle.e4m3_decode(0x7E) == 448.0 and oracle.e4m3_decode(0xFE) == -448.0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9 and oracle.e4m3_decode(0x08) == 2.0 ** -6
    assert oracle.e4m3_decode(0x38) == 1.0 and oracle.e4m3_decode(0x80) == 0.0


def test_e4m3_encode_matches_torch_rne_on_every_bf16_in_range():
    bits = np.arange(65536, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    keep = np.isfinite(vals) & (np.abs(vals) <= 448.0)
    vals = vals[keep]
    lib_codes = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([oracle.e4m3_encode(float(v)) for v in vals], dtype=np.uint8)
    bad = np.nonzero(ours != lib_codes)[0]
    assert bad.size == 0, [(float(vals[i]), ours[i], lib_codes[i]) for i in bad[:5]]


def test_e4m3_encode_random_fp32_and_ties():
    rng = np.random.default_rng(5)
    vals = (rng.standard_normal(20000) * rng.choice([1e-3, 0.1, 1, 30, 200], 20000))
    vals = vals.astype(np.float32)
    vals = vals[np.abs(vals) <= 448]
    lib_codes = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([oracle.e4m3_encode(float(v)) for v in vals], dtype=np.uint8)
    assert (ours == lib_codes).all()
    # exact ties round to the even mantissa
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00          # 0.5 ulp above zero -> 0
    assert oracle.e4m3_encode(3 * 2.0 ** -10) == 0x02      # 1.5 ulp -> 2
    assert oracle.e4m3_encode(1.0 + 1 / 16) == 0x38        # 1 + half ulp -> 1.0
    assert oracle.e4m3_encode(1.0 + 3 / 16) == 0x3A        # 1.125 + half ulp -> 1.25


def test_e4m3_encode_saturates_finite_overflow():
    for v in (448.0, 449.0, 464.0, 470.0, 480.0, 1e4, 3.0e38, float("inf")):
        assert oracle.e4m3_encode(v) == 0x7E
        assert oracle.e4m3_encode(-v) == 0xFE
    assert oracle.e4m3_encode(float("nan")) == 0x7F


def test_e4m3_quantize_uses_fp32_product_with_reciprocal():
    s = np.float32(0.0123)
    inv = np.float32(1.0) / s
    for x in np.linspace(-5, 5, 101, dtype=np.float32):
        y = np.float32(x * inv)
        assert oracle.e4m3_quantize(float(x), float(s)) == oracle.e4m3_encode(float(y))


# ------------------------------------------------------------------ helpers for decode pins
def _place(contig, table, bs, num_blocks, fill=NAN16, dtype=np.uint16):
    """Lay one sequence's contiguous rows [L, Hkv, D] into a paged pool by reshaping:
    rows [b*bs, (b+1)*bs) become physical block table[b] in head-first order."""
    L, Hkv, D = contig.shape
    nblk = -(-L // bs)
    pad = np.full((nblk * bs, Hkv, D), fill, dtype=dtype)
    pad[:L] = contig
    return pad.reshape(nblk, bs, Hkv, D).transpose(0, 2, 1, 3), table[:nblk]


def _make_case(rng, lens, Hq, Hkv, D, bs=16, extra_blocks=3, gain_k=1.0):
    nblk = [-(-L // bs) for L in lens]
    NB = sum(nblk) + extra_blocks
    perm = rng.permutation(NB).astype(np.int32)
    MB = max(nblk)
    tables = np.full((len(lens), MB), -1, dtype=np.int32)
    kc = np.full((NB, Hkv, bs, D), NAN16, dtype=np.uint16)
    vc = np.full((NB, Hkv, bs, D), NAN16, dtype=np.uint16)
    ks, vs = [], []
    pos = 0
    for b, L in enumerate(lens):
        tables[b, :nblk[b]] = perm[pos:pos + nblk[b]]
        pos += nblk[b]
        k = (torch.randn(L, Hkv, D, dtype=torch.float32) * gain_k).to(torch.bfloat16)
        v = torch.randn(L, Hkv, D, dtype=torch.float32).to(torch.bfloat16)
        ks.append(k)
        vs.append(v)
        kb = k.view(torch.int16).numpy().view(np.uint16)
        vb = v.view(torch.int16).numpy().view(np.uint16)
        blocks, ids = _place(kb, tables[b], bs, NB)
        kc[ids] = blocks
        blocks, ids = _place(vb, tables[b], bs, NB)
        vc[ids] = blocks
    q = torch.randn(len(lens), Hq, D, dtype=torch.float32).to(torch.bfloat16)
    return dict(q=q, ks=ks, vs=vs, kc=kc, vc=vc, tables=tables, lens=np.array(lens, np.int32))


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _sdpa_last_row(q_last, k, v, scale, Hq, Hkv):
    """Library attention: torch fp64 SDPA with a causal mask over the whole sequence,
    query heads grouped contiguously onto KV heads; returns the last query row [Hq, D]."""
    L, _, D = k.shape
    g = Hq // Hkv
    Q = torch.randn(1, Hq, L, D, dtype=torch.float64)
    Q[0, :, L - 1, :] = q_last.to(torch.float64)
    K = k.to(torch.float64).permute(1, 0, 2).repeat_interleave(g, dim=0)[None]
    V = v.to(torch.float64).permute(1, 0, 2).repeat_interleave(g, dim=0)[None]
    O = torch.nn.functional.scaled_dot_product_attention(Q, K, V, is_causal=True, scale=scale)
    return O[0, :, L - 1, :].numpy()


# ------------------------------------------------------------------ decode pins
@pytest.mark.parametrize("lens,Hq,Hkv,D", [
    ([18, 33], 8, 2, 64),            # the tiny workload's shape
    ([1, 7, 16, 17, 40], 8, 2, 64),
    ([5, 31, 32, 33], 4, 4, 128),    # MHA (group 1)
    ([12, 49], 8, 1, 64),            # MQA (one KV head)
    ([3, 70], 6, 3, 64),             # group 2, three KV heads
    ([100], 64, 8, 128),             # Llama-3-70B heads
    ([29, 65], 28, 4, 128),          # Qwen2.5-7B heads (group 7)
])
def test_decode_equals_last_row_of_causal_sdpa(lens, Hq, Hkv, D):
    torch.manual_seed(sum(lens) + Hq)
    rng = np.random.default_rng(sum(lens))
    c = _make_case(rng, lens, Hq, Hkv, D)
    scale = float(np.float32(1.0 / math.sqrt(D)))
    st, out = oracle.paged_decode(_bits(c["q"]), c["kc"], c["vc"], c["tables"], c["lens"],
                                  scale, Hkv)
    assert st == 0 and np.isfinite(out).all()
    for b, L in enumerate(lens):
        ref = _sdpa_last_row(c["q"][b], c["ks"][b], c["vs"][b], scale, Hq, Hkv)
        np.testing.assert_allclose(out[b], ref, rtol=1e-11, atol=1e-12)


def test_decode_pin_detects_planted_mistakes():
    # the SDPA pin is sharp enough to catch a wrong scale, a wrong head grouping and an
    # off-by-one length (each planted here, on the CPU, in the oracle's inputs)
    torch.manual_seed(0)
    rng = np.random.default_rng(0)
    c = _make_case(rng, [18, 33], 8, 2, 64)
    scale = 0.125
    ref = _sdpa_last_row(c["q"][1], c["ks"][1], c["vs"][1], scale, 8, 2)
    _, good = oracle.paged_decode(_bits(c["q"]), c["kc"], c["vc"], c["tables"], c["lens"], scale, 2)
    np.testing.assert_allclose(good[1], ref, rtol=1e-11, atol=1e-12)
    _, wrong_scale = oracle.paged_decode(_bits(c["q"]), c["kc"], c["vc"], c["tables"], c["lens"],
                                         scale * 1.01, 2)
    assert np.abs(wrong_scale[1] - ref).max() > 1e-6
    q_swapped = c["q"].clone()
    q_swapped[:, [0, 4]] = q_swapped[:, [4, 0]]          # strided instead of contiguous groups
    _, sw = oracle.paged_decode(_bits(q_swapped), c["kc"], c["vc"], c["tables"], c["lens"], scale, 2)
    assert np.abs(sw[1, 4] - ref[4]).max() > 1e-3
    short = c["lens"].copy()
    short[1] -= 1
    kc2, vc2 = c["kc"].copy(), c["vc"].copy()
    _, sh = oracle.paged_decode(_bits(c["q"]), kc2, vc2, c["tables"], short, scale, 2)
    assert np.abs(sh[1] - ref).max() > 1e-6


def test_decode_all_placements_of_an_8_block_pool_are_identical():
    # brute force: the tiny workload's 5 live blocks under all 8! physical placements
    torch.manual_seed(11)
    rng = np.random.default_rng(11)
    c = _make_case(rng, [18, 33], 8, 2, 64, extra_blocks=3)
    assert c["kc"].shape[0] == 8
    qb = _bits(c["q"])
    _, ref = oracle.paged_decode(qb, c["kc"], c["vc"], c["tables"], c["lens"], 0.125, 2)
    count = 0
    for perm in itertools.permutations(range(8)):
        perm = np.array(perm, dtype=np.int32)
        kc = np.empty_like(c["kc"])
        vc = np.empty_like(c["vc"])
        kc[perm] = c["kc"]
        vc[perm] = c["vc"]
        tables = np.where(c["tables"] >= 0, perm[np.maximum(c["tables"], 0)], -1).astype(np.int32)
        _, out = oracle.paged_decode(qb, kc, vc, tables, c["lens"], 0.125, 2)
        assert np.array_equal(out, ref)
        count += 1
    assert count == 40320


def test_single_key_returns_its_value_exactly():
    torch.manual_seed(2)
    c = _make_case(np.random.default_rng(2), [1, 1], 8, 2, 64)
    _, out = oracle.paged_decode(_bits(c["q"]), c["kc"], c["vc"], c["tables"], c["lens"], 0.125, 2)
    for b in range(2):
        v0 = c["vs"][b][0].to(torch.float64).numpy()            # [Hkv, D]
        assert np.array_equal(out[b], np.repeat(v0, 4, axis=0))


def test_identical_keys_return_mean_of_values():
    torch.manual_seed(3)
    c = _make_case(np.random.default_rng(3), [37], 8, 2, 64)
    k0 = c["ks"][0][:1].expand(37, -1, -1).contiguous()
    blocks, ids = _place(_bits(k0), c["tables"][0], 16, c["kc"].shape[0])
    c["kc"][ids] = blocks
    _, out = oracle.paged_decode(_bits(c["q"]), c["kc"], c["vc"], c["tables"], c["lens"], 0.125, 2)
    mean_v = c["vs"][0].to(torch.float64).mean(dim=0).numpy()   # [Hkv, D]
    np.testing.assert_allclose(out[0], np.repeat(mean_v, 4, axis=0), rtol=0, atol=1e-14)


def test_decode_rejects_bad_lengths_and_ids():
    torch.manual_seed(4)
    c = _make_case(np.random.default_rng(4), [18, 33], 8, 2, 64)
    for lens in ([0, 33], [18, 49]):
        st, out = oracle.paged_decode(_bits(c["q"]), c["kc"], c["vc"], c["tables"],
                                      np.array(lens, np.int32), 0.125, 2)
        assert st == 1 and np.isnan(out).any()
    t = c["tables"].copy()
    t[1, 2] = 99
    st, _ = oracle.paged_decode(_bits(c["q"]), c["kc"], c["vc"], t, c["lens"], 0.125, 2)
    assert st == 1


def test_fp8_pool_decode_equals_sdpa_on_dequantised_values():
    torch.manual_seed(6)
    rng = np.random.default_rng(6)
    lens, Hq, Hkv, D = [21, 50], 14, 2, 128
    c = _make_case(rng, lens, Hq, Hkv, D)
    ks, vs = np.float32(0.0137), np.float32(0.0151)
    kc8 = np.zeros(c["kc"].shape, np.uint8)
    vc8 = np.zeros(c["vc"].shape, np.uint8)
    deq_k, deq_v = [], []
    for b, L in enumerate(lens):
        kq = np.array([[[oracle.e4m3_quantize(float(x), float(ks)) for x in row] for row in tok]
                       for tok in c["ks"][b].float().numpy()], dtype=np.uint8)
        vq = np.array([[[oracle.e4m3_quantize(float(x), float(vs)) for x in row] for row in tok]
                       for tok in c["vs"][b].float().numpy()], dtype=np.uint8)
        blocks, ids = _place(kq, c["tables"][b], 16, kc8.shape[0], fill=0x7F, dtype=np.uint8)
        kc8[ids] = blocks
        blocks, ids = _place(vq, c["tables"][b], 16, vc8.shape[0], fill=0x7F, dtype=np.uint8)
        vc8[ids] = blocks
        lut = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(
            torch.float8_e4m3fn).to(torch.float64)
        deq_k.append(lut[torch.from_numpy(kq).long()] * float(ks))
        deq_v.append(lut[torch.from_numpy(vq).long()] * float(vs))
    scale = float(np.float32(1 / math.sqrt(D)))
    st, out = oracle.paged_decode(_bits(c["q"]), kc8, vc8, c["tables"], c["lens"], scale, Hkv,
                                  kv_dtype=FP8E4M3, k_scale=float(ks), v_scale=float(vs))
    assert st == 0
    for b in range(2):
        ref = _sdpa_last_row(c["q"][b], deq_k[b], deq_v[b], scale, Hq, Hkv)
        np.testing.assert_allclose(out[b], ref, rtol=1e-11, atol=1e-12)


# ------------------------------------------------------------------ kv_append pins
def test_kv_append_writes_exactly_the_mapped_rows():
    rng = np.random.default_rng(7)
    NB, Hkv, D, T = 6, 2, 64, 5
    kc = rng.integers(0, 65536, (NB, Hkv, 16, D), dtype=np.uint16)
    vc = rng.integers(0, 65536, (NB, Hkv, 16, D), dtype=np.uint16)
    k = rng.integers(0, 65536, (T, Hkv, D), dtype=np.uint16)
    v = rng.integers(0, 65536, (T, Hkv, D), dtype=np.uint16)
    slots = np.array([17, 32, -1, 95, 0], dtype=np.int64)
    kc0, vc0 = kc.copy(), vc.copy()
    assert oracle.kv_append(k, v, slots, kc, vc) == 0
    flat_k = kc.transpose(0, 2, 1, 3).reshape(NB * 16, Hkv, D)      # slot-major view
    flat_v = vc.transpose(0, 2, 1, 3).reshape(NB * 16, Hkv, D)
    flat_k0 = kc0.transpose(0, 2, 1, 3).reshape(NB * 16, Hkv, D)
    for t, s in enumerate(slots):
        if s >= 0:
            assert np.array_equal(flat_k[s], k[t]) and np.array_equal(flat_v[s], v[t])
    untouched = np.setdiff1d(np.arange(NB * 16), slots[slots >= 0])
    assert np.array_equal(flat_k[untouched], flat_k0[untouched])
    assert np.array_equal(flat_v[untouched], vc0.transpose(0, 2, 1, 3).reshape(NB * 16, Hkv, D)[untouched])
    assert oracle.kv_append(k, v, np.array([96, -1, -1, -1, -1], np.int64), kc, vc) == 1


def test_append_then_decode_sees_the_new_token_last():
    # the tiny workload's appends land at positions 17 and 32; before the append those
    # slots hold NaN, afterwards decode equals SDPA with the new K/V as the last row
    torch.manual_seed(8)
    rng = np.random.default_rng(8)
    lens = [18, 33]
    c = _make_case(rng, lens, 8, 2, 64)
    sm = oracle.slot_mapping(c["tables"], lens)
    for b, L in enumerate(lens):
        phys, off = sm[b] // 16, sm[b] % 16
        assert off == (L - 1) % 16
        c["kc"][phys, :, off, :] = NAN16
        c["vc"][phys, :, off, :] = NAN16
    st, out = oracle.paged_decode(_bits(c["q"]), c["kc"], c["vc"], c["tables"], c["lens"], 0.125, 2)
    assert np.isnan(out).all(axis=(1, 2)).all()
    k_new = torch.stack([c["ks"][b][-1] for b in range(2)])
    v_new = torch.stack([c["vs"][b][-1] for b in range(2)])
    assert oracle.kv_append(_bits(k_new), _bits(v_new), sm, c["kc"], c["vc"]) == 0
    st, out = oracle.paged_decode(_bits(c["q"]), c["kc"], c["vc"], c["tables"], c["lens"], 0.125, 2)
    assert st == 0
    for b in range(2):
        ref = _sdpa_last_row(c["q"][b], c["ks"][b], c["vs"][b], 0.125, 8, 2)
        np.testing.assert_allclose(out[b], ref, rtol=1e-11, atol=1e-12)


def test_poison_unused_marks_only_unread_positions():
    a = oracle.BlockAllocator(6, [3, 0, 5, 1, 4, 2])
    lens = [18, 5]
    t = oracle.build_block_tables(a, lens, 2)
    kc = np.zeros((6, 1, 16, 4), np.uint16)
    oracle.poison_unused(kc, t, lens, 16, NAN16)
    live = {(int(t[0][0]), o) for o in range(16)} | {(int(t[0][1]), o) for o in range(2)} | \
           {(int(t[1][0]), o) for o in range(5)}
    for blk in range(6):
        for o in range(16):
            assert (kc[blk, 0, o] == 0).all() == ((blk, o) in live)
