"""GPU parity of paged prefill / chunked prefill (tcgen05) against the oracle.

Each case appends the chunks' K/V with kv_append at pkv_slot_mapping_chunks' slots (bit-exact
with the oracle's append), then runs the plan: every packed row must satisfy
|gpu - oracle| <= 1e-2 + 1e-2*|oracle| against the fp64 causal attention over its own
sequence ("理解 KV Cache" §1.2, §2.1), with NaN in every pool position no row may see and in
the chunks' slots before the append."""
import numpy as np
import pytest
import torch

import workloads
from tests import _cases as C

pkv = pytest.importorskip("paged_kv_cache_159_gb300")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    pkv.lib()
    torch.cuda.set_device(0)


def _run(name, overrides=None, rows=None, fp8=False):
    c = C.build_prefill(name, overrides=overrides, fp8=fp8)
    C.prefill_append(c)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(C.prefill_pool_bits(c, c.key_cache), c.key_host)
    np.testing.assert_array_equal(C.prefill_pool_bits(c, c.value_cache), c.value_host)
    out = C.gpu_prefill(c)
    ref = C.oracle_prefill_rows(c, rows)
    got = C.bf16_to_f64(out if rows is None else out[torch.as_tensor(rows)])
    return C.tol_check(got, ref)


def test_prefill_tiny():
    _run("prefill_tiny")


@pytest.mark.parametrize("Hq,Hkv,D", [(8, 2, 128), (4, 4, 64), (4, 4, 128), (28, 4, 128), (16, 2, 64),
                                      (32, 2, 128), (12, 4, 64)])
def test_prefill_heads_and_head_dims(Hq, Hkv, D):
    """GQA groups 1, 3, 4, 7 (rows padded to 126), 8 and 16 at both head sizes; chunks and
    contexts long enough for several query tiles and several KV tiles per unit."""
    _run("prefill_tiny", {"num_q_heads": Hq, "num_kv_heads": Hkv, "head_dim": D, "batch": 5,
                          "chunk": 300, "context": 420, "seed": 159110 + Hq + D})


@pytest.mark.parametrize("Hq,Hkv,D", [(8, 2, 128), (4, 4, 64), (28, 4, 128), (16, 2, 64), (32, 2, 128)])
def test_prefill_fp8_pool(Hq, Hkv, D):
    """An E4M3 pool ("KV Cache 与推理优化", KV 量化: the cache stored in FP8, the arithmetic in
    higher precision): the tiles are converted to bf16 on the chip, the scales applied to the
    scores and the output.  The oracle decodes its own E4M3 copy of the pool."""
    _run("prefill_tiny", {"num_q_heads": Hq, "num_kv_heads": Hkv, "head_dim": D, "batch": 5,
                          "chunk": 300, "context": 420, "seed": 159130 + Hq + D}, fp8=True)


@pytest.mark.parametrize("chunk,context", [(1, 0), (129, 0), (16, 16), (257, 1), (64, 700)])
def test_prefill_fp8_edge_lengths(chunk, context):
    _run("prefill_tiny", {"ragged": False, "chunk": chunk, "context": context, "batch": 4,
                          "head_dim": 128, "seed": 159140 + chunk + context}, fp8=True)


@pytest.mark.parametrize("chunk,context", [(1, 0), (1, 700), (16, 16), (129, 0), (128, 128), (257, 1)])
def test_prefill_edge_lengths(chunk, context):
    """Single-row chunks, chunks and contexts at tile and block boundaries."""
    _run("prefill_tiny", {"ragged": False, "chunk": chunk, "context": context, "batch": 4,
                          "head_dim": 128, "seed": 159120 + chunk + context})


@pytest.mark.parametrize("D", [64, 128])
def test_prefill_sequences_without_new_rows(D):
    """Sequences whose chunk is empty this step (P_b = 0, context only) sit between others:
    they get no units and no rows, and the rows around them are unchanged."""
    _run("prefill_tiny", {"batch": 5, "head_dim": D, "num_q_heads": 8, "num_kv_heads": 2,
                          "chunk_list": (40, 0, 129, 0, 1), "context_list": (37, 50, 0, 300, 16),
                          "seed": 159130 + D})


def test_prefill_llama3_8b_full_size_sampled():
    """8 prompts of 2048 positions, Llama-3-8B layer shape: rows at the edges of blocks, query
    tiles and KV tiles of every sequence, checked against the oracle one by one."""
    pos = np.array([0, 1, 15, 16, 31, 32, 127, 128, 129, 1000, 2046, 2047])
    rows = np.concatenate([b * 2048 + pos for b in range(8)])
    _run("prefill_llama3_8b", rows=rows)


def test_chunked_prefill_llama3_8b_full_size_sampled():
    w = workloads.PREFILL_WORKLOADS["chunked_prefill_llama3_8b"]
    pos = np.array([0, 1, 31, 32, 255, 256, 510, 511])
    rows = np.concatenate([b * 512 + pos for b in range(w.batch)])
    _run("chunked_prefill_llama3_8b", rows=rows)


def test_chunked_prefill_llama3_8b_fp8_full_size_sampled():
    """The chunked workload over an E4M3 pool: contexts up to 8192 cached positions, so every
    unit streams many converted tiles."""
    w = workloads.PREFILL_WORKLOADS["chunked_prefill_llama3_8b"]
    pos = np.array([0, 1, 255, 256, 511])
    rows = np.concatenate([b * 512 + pos for b in range(w.batch)])
    _run("chunked_prefill_llama3_8b", rows=rows, fp8=True)


@pytest.mark.parametrize("D", [64, 128])
def test_prefill_fp8_sequences_without_new_rows(D):
    _run("prefill_tiny", {"batch": 5, "head_dim": D, "num_q_heads": 8, "num_kv_heads": 2,
                          "chunk_list": (40, 0, 129, 0, 1), "context_list": (37, 50, 0, 300, 16),
                          "seed": 159150 + D}, fp8=True)


def _plan_units(buf, grid):
    """Decode a plan (layout of pkv_prefill_plan): header, per-CTA ranges, units."""
    hdr = np.frombuffer(buf[:32].tobytes(), dtype=np.int32)
    off = np.frombuffer(buf[32:32 + 4 * (grid + 1)].tobytes(), dtype=np.int32)
    start = (32 + 4 * (grid + 1) + 31) // 32 * 32
    n = int(hdr[1])
    units = np.frombuffer(buf[start:start + 32 * n].tobytes(), dtype=np.int32).reshape(n, 8)
    return hdr, off, units


@pytest.mark.parametrize("name", ["prefill_tiny", "chunked_prefill_llama3_8b"])
def test_prefill_plan_covers_every_row_once_and_balances(name):
    """Every (sequence, KV head, query row) is in exactly one unit; each unit's key range is
    its rows' causal range; longest-first assignment keeps every CTA within one unit (plus
    its overhead) of the ideal share."""
    w = workloads.PREFILL_WORKLOADS[name]
    d = workloads.draw_prefill(w, "cpu")
    pool = pkv.Pool(d.num_blocks, w.num_kv_heads, w.head_dim)
    plan, grid = pkv.prefill_plan(pool, d.cu_q, d.seq_lens, w.num_q_heads, d.max_blocks)
    hdr, off, units = _plan_units(plan, grid)
    g = w.num_q_heads // w.num_kv_heads
    assert hdr[2] == grid and hdr[3] == g and hdr[4] == 256 // g
    assert off[0] == 0 and off[-1] == len(units) and np.all(np.diff(off) >= 1)
    seen = np.zeros((int(d.cu_q[-1]), w.num_kv_heads), np.int32)
    for b, h, row0, pos0, npos, nkv, kmax, _ in units:
        assert 1 <= npos <= 256 // g
        C = int(d.seq_lens[b] - d.chunk_lens[b])
        assert pos0 == C + (row0 - d.cu_q[b]) and kmax == pos0 + npos - 1 and nkv == kmax // 64 + 1
        seen[row0:row0 + npos, h] += 1
    assert np.all(seen == 1)
    load = np.array([sum(int(units[i, 5]) + 2 for i in range(off[c], off[c + 1])) for c in range(grid)])
    assert load.max() <= load.sum() / grid + units[:, 5].max() + 2


def test_prefill_flags_a_mismatched_plan_and_a_bad_table_entry():
    c = C.build_prefill("prefill_tiny")
    C.prefill_append(c)
    torch.cuda.synchronize()
    plan, grid = pkv.prefill_plan(c.pool, c.d.cu_q, c.d.seq_lens, c.w.num_q_heads, c.tables.shape[1])
    out = torch.full_like(c.d.q, 7.0)
    bt = torch.from_numpy(c.tables).cuda()
    # a plan made for another head count: nothing runs, the plan bit is set
    other, g2 = pkv.prefill_plan(c.pool, c.d.cu_q, c.d.seq_lens, 2 * c.w.num_q_heads, c.tables.shape[1])
    q2 = torch.zeros((c.d.q.shape[0], 2 * c.w.num_q_heads, c.w.head_dim), dtype=torch.bfloat16, device="cuda")
    o2 = torch.full_like(q2, 7.0)
    pkv.paged_prefill(c.pool, q2, c.key_cache, c.value_cache, bt, c.w.scale, torch.from_numpy(plan).cuda(), grid, o2)
    st, bits = c.pool.get_device_error()
    assert st == pkv.ERR_DEVICE and bits == pkv.DEVERR_PLAN
    assert bool((o2 == 7.0).all())
    # a table entry outside the pool is flagged (the kernel skips that block and finishes)
    bad = bt.clone()
    bad[0, 0] = c.d.num_blocks + 3
    pkv.paged_prefill(c.pool, c.d.q, c.key_cache, c.value_cache, bad, c.w.scale, torch.from_numpy(plan).cuda(), grid, out)
    st, bits = c.pool.get_device_error()
    assert st == pkv.ERR_DEVICE and bits & pkv.DEVERR_BLOCK_ID and not bits & pkv.DEVERR_TIMEOUT
    # the context is still usable: a correct run afterwards matches the oracle
    out = C.gpu_prefill(c)
    C.tol_check(C.bf16_to_f64(out), C.oracle_prefill_rows(c, threads=1))
