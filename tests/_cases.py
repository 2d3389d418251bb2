"""Build GPU parity cases: seeded inputs (workloads), block tables and slots from the
oracle's allocator, unread positions poisoned with NaN, and the oracle's own results."""
import dataclasses

import numpy as np
import torch

import oracle
import workloads
import paged_kv_cache_159_gb300 as pkv

NAN16 = workloads.BF16_NAN_BITS
FP8_NAN = 0x7F


def tol_check(gpu: np.ndarray, ref: np.ndarray, atol=1e-2, rtol=1e-2):
    """Elementwise |gpu - ref| <= atol + rtol*|ref| (the stated decode tolerance).
    Returns (max_abs_err, max_rel_err over |ref| > 1e-3)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    assert np.isfinite(gpu).all(), "non-finite output"
    err = np.abs(gpu - ref)
    bad = err > atol + rtol * np.abs(ref)
    assert not bad.any(), "%d elements out of tolerance; worst abs %.3g" % (bad.sum(), err.max())
    big = np.abs(ref) > 1e-3
    rel = (err[big] / np.abs(ref[big])).max() if big.any() else 0.0
    return float(err.max()), float(rel)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


@dataclasses.dataclass
class Case:
    w: workloads.Workload
    seq_lens: np.ndarray
    tables: np.ndarray
    slots: np.ndarray            # int64 [B] newest-token slots (append workloads)
    pool: "pkv.Pool"
    key_cache: torch.Tensor      # device pool (bf16 or uint8 codes)
    value_cache: torch.Tensor
    q: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    k_scale: float
    v_scale: float
    kv_dtype: int
    # oracle-side pools (host), before any append
    key_host: np.ndarray
    value_host: np.ndarray
    alloc: "oracle.BlockAllocator" = None    # the oracle's allocator after the tables


def build(name: str, device="cuda", seq_lens=None, overrides=None, free_order=None) -> Case:
    w = workloads.WORKLOADS[name]
    if overrides:
        w = dataclasses.replace(w, **overrides)
    d = workloads.draw(w, device, seq_lens)
    order = d.free_order if free_order is None else np.asarray(free_order, np.int32)
    alloc = oracle.BlockAllocator(d.num_blocks, order)
    prefix = alloc.alloc(w.prefix_blocks) if w.prefix_blocks else []
    tables = oracle.build_block_tables(alloc, d.seq_lens, d.max_blocks, 16, prefix)
    slots = oracle.slot_mapping(tables, d.seq_lens)
    live = torch.from_numpy(oracle.live_positions(tables, d.seq_lens, d.num_blocks)).to(device)
    dead = ~live                                               # [NB, 16]
    kc, vc = d.key_cache, d.value_cache
    nan = torch.tensor(NAN16, dtype=torch.int16, device=device).view(torch.bfloat16)
    kc[dead[:, None, :, None].expand_as(kc)] = nan
    vc[dead[:, None, :, None].expand_as(vc)] = nan
    # the new token's slot starts as NaN, unless it lies in a block other sequences share (and
    # read): there the sequence must diverge by copy-on-write before it writes
    private = np.array([alloc.refcount[int(s) // 16] == 1 for s in slots], dtype=bool)
    slots_dev = torch.from_numpy(slots[private]).to(device)
    if w.append and w.kv_dtype != "fp8":
        blk, off = slots_dev // 16, slots_dev % 16
        kc[blk, :, off, :] = nan
        vc[blk, :, off, :] = nan
    k_scale = v_scale = 1.0
    kv_dtype = pkv.KV_BF16
    if w.kv_dtype == "fp8":
        # The FP8 pool is written through kv_append from the bf16 history of every live
        # position; the per-tensor scales are amax / 448 in fp32.
        kv_dtype = pkv.KV_FP8E4M3
        all_slots = torch.from_numpy(oracle.all_slots(tables, d.seq_lens)).to(device)
        blk, off = all_slots // 16, all_slots % 16
        k_src = kc[blk, :, off, :].contiguous()                # [T, Hkv, D]
        v_src = vc[blk, :, off, :].contiguous()
        kmax = max(k_src.float().abs().max().item(), d.k_new.float().abs().max().item())
        vmax = max(v_src.float().abs().max().item(), d.v_new.float().abs().max().item())
        k_scale = float(np.float32(kmax) / np.float32(448.0))
        v_scale = float(np.float32(vmax) / np.float32(448.0))
        pool = pkv.Pool(d.num_blocks, w.num_kv_heads, w.head_dim, kv_dtype, k_scale, v_scale, order)
        pool.attach_device(torch.cuda.current_device())
        k8 = torch.full(kc.shape, FP8_NAN, dtype=torch.uint8, device=device)
        v8 = torch.full(vc.shape, FP8_NAN, dtype=torch.uint8, device=device)
        # host copies of the source rows for the oracle's own encode
        key_host = np.full(kc.shape, FP8_NAN, dtype=np.uint8)
        value_host = np.full(vc.shape, FP8_NAN, dtype=np.uint8)
        ks_host, vs_host = workloads.bf16_bits(k_src), workloads.bf16_bits(v_src)
        sl_host = all_slots.cpu().numpy()
        assert oracle.kv_append(ks_host, vs_host, sl_host, key_host, value_host, 16,
                                oracle.FP8E4M3, k_scale, v_scale) == 0
        pkv.kv_append(pool, k_src, v_src, all_slots, k8, v8)
        torch.cuda.synchronize()
        if w.append:                                           # the new token's slot starts as NaN
            blk, off = slots_dev // 16, slots_dev % 16
            k8[blk, :, off, :] = FP8_NAN
            v8[blk, :, off, :] = FP8_NAN
            for sl in slots[private]:
                key_host[sl // 16, :, sl % 16, :] = FP8_NAN
                value_host[sl // 16, :, sl % 16, :] = FP8_NAN
        kc, vc = k8, v8
    else:
        pool = pkv.Pool(d.num_blocks, w.num_kv_heads, w.head_dim, free_order=order)
        pool.attach_device(torch.cuda.current_device())
        key_host = workloads.bf16_bits(kc)
        value_host = workloads.bf16_bits(vc)
    return Case(w, d.seq_lens, tables, slots, pool, kc, vc, d.q, d.k_new, d.v_new, k_scale,
                v_scale, kv_dtype, key_host, value_host, alloc)


def oracle_append(c: Case):
    """The oracle's kv_append of each sequence's new token on its own host pools (in place)."""
    fp8 = c.kv_dtype == pkv.KV_FP8E4M3
    st = oracle.kv_append(workloads.bf16_bits(c.k_new), workloads.bf16_bits(c.v_new), c.slots,
                          c.key_host, c.value_host, 16, oracle.FP8E4M3 if fp8 else oracle.BF16,
                          c.k_scale, c.v_scale)
    assert st == 0


def oracle_decode(c: Case, pairs=None, threads=None):
    st, out = oracle.paged_decode(
        workloads.bf16_bits(c.q), c.key_host, c.value_host, c.tables, c.seq_lens, c.w.scale,
        c.w.num_kv_heads, 16, oracle.FP8E4M3 if c.kv_dtype == pkv.KV_FP8E4M3 else oracle.BF16,
        c.k_scale, c.v_scale, pairs=pairs, num_threads=threads or oracle.max_threads())
    assert st == 0
    return out


def device_tables(c: Case, device="cuda"):
    return (torch.from_numpy(c.tables).to(device), torch.from_numpy(c.seq_lens).to(device),
            torch.from_numpy(c.slots).to(device))


def gpu_step(c: Case, opts=None, append=True):
    """kv_append (if the workload appends) then decode; returns the bf16 output."""
    bt, sl, slots = device_tables(c)
    if append and c.w.append:
        pkv.kv_append(c.pool, c.k_new, c.v_new, slots, c.key_cache, c.value_cache)
    B, Hq, D = c.q.shape
    out = torch.empty_like(c.q)
    nbytes = pkv.decode_workspace_bytes(c.pool, B, Hq, bt.shape[1], opts)
    assert nbytes > 0
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=c.q.device)
    pkv.paged_attention_decode(c.pool, c.q, c.key_cache, c.value_cache, bt, sl, c.w.scale, out,
                               ws, opts)
    st, bits = c.pool.get_device_error()
    assert st == pkv.OK and bits == 0, (st, bits)
    counters = ws[:B * c.w.num_kv_heads * 4].view(torch.int32)
    assert int(torch.count_nonzero(counters)) == 0, "split counters not returned to zero"
    return out


# ------------------------------------------------------------------------------------
# Multi-layer cases: caches stacked [layers, NB, Hkv, 16, D], one table for every layer.
# The oracle has no layer dimension: each layer is a pool of its own, decoded and appended
# by the single-layer oracle functions.
# ------------------------------------------------------------------------------------
@dataclasses.dataclass
class LayerCase:
    w: workloads.Workload
    seq_lens: np.ndarray
    tables: np.ndarray
    slots: np.ndarray
    pool: "pkv.Pool"
    key_cache: torch.Tensor      # [layers, NB, Hkv, 16, D] (bf16 or uint8 codes)
    value_cache: torch.Tensor
    q: torch.Tensor              # bf16 [layers, B, Hq, D]
    k_new: torch.Tensor          # bf16 [layers, B, Hkv, D]
    v_new: torch.Tensor
    k_scale: float
    v_scale: float
    kv_dtype: int
    key_host: list               # per layer: the oracle's host pool before any append
    value_host: list


def build_layers(name: str, device="cuda", overrides=None, host_layers=None) -> LayerCase:
    """host_layers: the layers given host copies for the oracle (default: all)."""
    w = workloads.WORKLOADS[name]
    if overrides:
        w = dataclasses.replace(w, **overrides)
    d = workloads.draw(w, device)
    nl = w.layers
    assert nl > 1
    host_layers = range(nl) if host_layers is None else host_layers
    alloc = oracle.BlockAllocator(d.num_blocks, d.free_order)
    prefix = alloc.alloc(w.prefix_blocks) if w.prefix_blocks else []
    tables = oracle.build_block_tables(alloc, d.seq_lens, d.max_blocks, 16, prefix)
    slots = oracle.slot_mapping(tables, d.seq_lens)
    live = torch.from_numpy(oracle.live_positions(tables, d.seq_lens, d.num_blocks)).to(device)
    dead = ~live
    kc, vc = d.key_cache, d.value_cache
    nan = torch.tensor(NAN16, dtype=torch.int16, device=device).view(torch.bfloat16)
    for l in range(nl):                                        # unread positions are NaN
        kc[l][dead[:, None, :, None].expand_as(kc[l])] = nan
        vc[l][dead[:, None, :, None].expand_as(vc[l])] = nan
    slots_dev = torch.from_numpy(slots).to(device)
    blk, off = slots_dev // 16, slots_dev % 16
    fp8 = w.kv_dtype == "fp8"
    k_scale = v_scale = 1.0
    if fp8:
        all_slots = torch.from_numpy(oracle.all_slots(tables, d.seq_lens)).to(device)
        ab, ao = all_slots // 16, all_slots % 16
        k_src = torch.stack([kc[l][ab, :, ao, :] for l in range(nl)])   # [layers, T, Hkv, D]
        v_src = torch.stack([vc[l][ab, :, ao, :] for l in range(nl)])
        kmax = max(k_src.float().abs().max().item(), d.k_new.float().abs().max().item())
        vmax = max(v_src.float().abs().max().item(), d.v_new.float().abs().max().item())
        k_scale = float(np.float32(kmax) / np.float32(448.0))
        v_scale = float(np.float32(vmax) / np.float32(448.0))
        pool = pkv.Pool(d.num_blocks, w.num_kv_heads, w.head_dim, pkv.KV_FP8E4M3, k_scale, v_scale,
                        d.free_order, num_layers=nl)
        pool.attach_device(torch.cuda.current_device())
        k8 = torch.full(kc.shape, FP8_NAN, dtype=torch.uint8, device=device)
        v8 = torch.full(vc.shape, FP8_NAN, dtype=torch.uint8, device=device)
        pkv.kv_append_layers(pool, k_src, v_src, all_slots, k8, v8)
        torch.cuda.synchronize()
        key_host, value_host = [], []
        sl_host = all_slots.cpu().numpy()
        for l in host_layers:
            kh = np.full(kc.shape[1:], FP8_NAN, dtype=np.uint8)
            vh = np.full(vc.shape[1:], FP8_NAN, dtype=np.uint8)
            assert oracle.kv_append(workloads.bf16_bits(k_src[l]), workloads.bf16_bits(v_src[l]),
                                    sl_host, kh, vh, 16, oracle.FP8E4M3, k_scale, v_scale) == 0
            key_host.append(kh)
            value_host.append(vh)
        if w.append:                                           # new token's slot starts as NaN
            k8[:, blk, :, off, :] = FP8_NAN
            v8[:, blk, :, off, :] = FP8_NAN
            for kh, vh in zip(key_host, value_host):
                for sl in slots:
                    kh[sl // 16, :, sl % 16, :] = FP8_NAN
                    vh[sl // 16, :, sl % 16, :] = FP8_NAN
        kc, vc = k8, v8
        kv_dtype = pkv.KV_FP8E4M3
    else:
        if w.append:
            kc[:, blk, :, off, :] = nan
            vc[:, blk, :, off, :] = nan
        pool = pkv.Pool(d.num_blocks, w.num_kv_heads, w.head_dim, free_order=d.free_order,
                        num_layers=nl)
        pool.attach_device(torch.cuda.current_device())
        key_host = [workloads.bf16_bits(kc[l]) for l in host_layers]
        value_host = [workloads.bf16_bits(vc[l]) for l in host_layers]
        kv_dtype = pkv.KV_BF16
    return LayerCase(w, d.seq_lens, tables, slots, pool, kc, vc, d.q, d.k_new, d.v_new, k_scale,
                     v_scale, kv_dtype, key_host, value_host)


def oracle_layer(c: LayerCase, l: int, i: int, append: bool, threads=None):
    """The single-layer oracle on layer l (host copy i): append (optionally), then decode."""
    fp8 = c.kv_dtype == pkv.KV_FP8E4M3
    dt = oracle.FP8E4M3 if fp8 else oracle.BF16
    kh, vh = c.key_host[i].copy(), c.value_host[i].copy()
    if append:
        assert oracle.kv_append(workloads.bf16_bits(c.k_new[l]), workloads.bf16_bits(c.v_new[l]),
                                c.slots, kh, vh, 16, dt, c.k_scale, c.v_scale) == 0
    st, out = oracle.paged_decode(workloads.bf16_bits(c.q[l]), kh, vh, c.tables, c.seq_lens,
                                  c.w.scale, c.w.num_kv_heads, 16, dt, c.k_scale, c.v_scale,
                                  num_threads=threads or oracle.max_threads())
    assert st == 0
    return out, kh, vh


def gpu_layers(c: LayerCase, append: bool, opts=None):
    """decode_step_layers (with or without the fused append); returns out [layers, B, Hq, D]."""
    bt, sl, _ = device_tables(c)
    nl, B, Hq, D = c.q.shape
    out = torch.empty_like(c.q)
    nbytes = pkv.decode_workspace_bytes(c.pool, B, Hq, bt.shape[1], opts)
    assert nbytes > 0
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=c.q.device)
    pkv.decode_step_layers(c.pool, c.q, c.k_new if append else None, c.v_new if append else None,
                           c.key_cache, c.value_cache, bt, sl, c.w.scale, out, ws, opts)
    st, bits = c.pool.get_device_error()
    assert st == pkv.OK and bits == 0, (st, bits)
    counters = ws[:nl * B * c.w.num_kv_heads * 4].view(torch.int32)
    assert int(torch.count_nonzero(counters)) == 0, "split counters not returned to zero"
    return out


# ------------------------------------------------------------------------------------
# Prefill cases: each sequence's context history already in the pool, its chunk's K/V
# appended by kv_append at the chunk's slots, then causal attention of the chunk's rows.
# ------------------------------------------------------------------------------------
@dataclasses.dataclass
class PrefillCase:
    w: "workloads.PrefillWorkload"
    d: "workloads.PrefillDraw"
    tables: np.ndarray
    slots: np.ndarray            # int64 [T] chunk slots (oracle's addressing)
    pool: "pkv.Pool"
    key_cache: torch.Tensor
    value_cache: torch.Tensor
    key_host: np.ndarray
    value_host: np.ndarray
    kv_dtype: int = 0            # pkv.KV_BF16, or pkv.KV_FP8E4M3
    k_scale: float = 1.0
    v_scale: float = 1.0

    @property
    def fp8(self) -> bool:
        return self.kv_dtype == pkv.KV_FP8E4M3


def build_prefill(name: str, device="cuda", overrides=None, fp8=False) -> PrefillCase:
    w = workloads.PREFILL_WORKLOADS[name]
    if overrides:
        w = dataclasses.replace(w, **overrides)
    d = workloads.draw_prefill(w, device)
    alloc = oracle.BlockAllocator(d.num_blocks, d.free_order)
    tables = oracle.build_block_tables(alloc, d.seq_lens, d.max_blocks, 16)
    slots = np.array([oracle.slot_of(tables[b], pos, 16)[3]
                      for b in range(w.batch)
                      for pos in range(int(d.seq_lens[b] - d.chunk_lens[b]), int(d.seq_lens[b]))],
                     dtype=np.int64)
    live = torch.from_numpy(oracle.live_positions(tables, d.seq_lens, d.num_blocks)).to(device)
    kc, vc = d.key_cache, d.value_cache
    nan = torch.tensor(NAN16, dtype=torch.int16, device=device).view(torch.bfloat16)
    dead = ~live
    kc[dead[:, None, :, None].expand_as(kc)] = nan
    vc[dead[:, None, :, None].expand_as(vc)] = nan
    sd = torch.from_numpy(slots).to(device)                    # the chunk's slots start as NaN
    kc[sd // 16, :, sd % 16, :] = nan
    vc[sd // 16, :, sd % 16, :] = nan
    if not fp8:
        pool = pkv.Pool(d.num_blocks, w.num_kv_heads, w.head_dim, free_order=d.free_order)
        pool.attach_device(torch.cuda.current_device())
        return PrefillCase(w, d, tables, slots, pool, kc, vc, workloads.bf16_bits(kc), workloads.bf16_bits(vc))
    # An E4M3 pool: the history positions (every position but the chunks') written through
    # kv_append from their bf16 rows, the oracle encoding its own host copy; per-tensor scales
    # amax / 448 over the history and the chunks, in fp32.  Every other byte starts as NaN.
    hist = np.setdiff1d(oracle.all_slots(tables, d.seq_lens), slots)
    hs = torch.from_numpy(hist).to(device)
    k_src = kc[hs // 16, :, hs % 16, :].contiguous()
    v_src = vc[hs // 16, :, hs % 16, :].contiguous()
    kmax = max(k_src.float().abs().max().item() if len(hist) else 0.0, d.k_chunk.float().abs().max().item())
    vmax = max(v_src.float().abs().max().item() if len(hist) else 0.0, d.v_chunk.float().abs().max().item())
    k_scale = float(np.float32(kmax) / np.float32(448.0))
    v_scale = float(np.float32(vmax) / np.float32(448.0))
    pool = pkv.Pool(d.num_blocks, w.num_kv_heads, w.head_dim, pkv.KV_FP8E4M3, k_scale, v_scale, d.free_order)
    pool.attach_device(torch.cuda.current_device())
    k8 = torch.full(kc.shape, FP8_NAN, dtype=torch.uint8, device=device)
    v8 = torch.full(vc.shape, FP8_NAN, dtype=torch.uint8, device=device)
    key_host = np.full(kc.shape, FP8_NAN, dtype=np.uint8)
    value_host = np.full(vc.shape, FP8_NAN, dtype=np.uint8)
    if len(hist):
        assert oracle.kv_append(workloads.bf16_bits(k_src), workloads.bf16_bits(v_src), hist, key_host, value_host,
                                16, oracle.FP8E4M3, k_scale, v_scale) == 0
        pkv.kv_append(pool, k_src, v_src, hs, k8, v8)
        torch.cuda.synchronize()
    return PrefillCase(w, d, tables, slots, pool, k8, v8, key_host, value_host, pkv.KV_FP8E4M3, k_scale, v_scale)


def prefill_append(c: PrefillCase):
    """The chunk's K/V into the pools: the library on the GPU, the oracle on its host copy."""
    slots = pkv.slot_mapping_chunks(c.tables, c.d.seq_lens, c.d.cu_q)
    np.testing.assert_array_equal(slots, c.slots)
    pkv.kv_append(c.pool, c.d.k_chunk, c.d.v_chunk, torch.from_numpy(slots).cuda(), c.key_cache, c.value_cache)
    assert oracle.kv_append(workloads.bf16_bits(c.d.k_chunk), workloads.bf16_bits(c.d.v_chunk), c.slots,
                            c.key_host, c.value_host, 16, oracle.FP8E4M3 if c.fp8 else oracle.BF16,
                            c.k_scale, c.v_scale) == 0


def prefill_pool_bits(c: PrefillCase, t: torch.Tensor) -> np.ndarray:
    """A pool tensor as the host copies hold it (bf16 bit patterns, or E4M3 bytes)."""
    return t.cpu().numpy() if c.fp8 else workloads.bf16_bits(t)


def gpu_prefill(c: PrefillCase):
    plan, grid = pkv.prefill_plan(c.pool, c.d.cu_q, c.d.seq_lens, c.w.num_q_heads, c.tables.shape[1])
    out = torch.full_like(c.d.q, float("nan"))
    pkv.paged_prefill(c.pool, c.d.q, c.key_cache, c.value_cache, torch.from_numpy(c.tables).cuda(),
                      c.w.scale, torch.from_numpy(plan).cuda(), grid, out)
    st, bits = c.pool.get_device_error()
    assert st == pkv.OK and bits == 0, (st, bits)
    return out


def oracle_prefill_rows(c: PrefillCase, rows=None, threads=None):
    """The oracle's causal attention for packed rows (all rows by default): row cu_q[b] + i
    is position L_b - P_b + i, i.e. a decode query of length position + 1."""
    if rows is None:
        st, out = oracle.paged_prefill(workloads.bf16_bits(c.d.q), c.key_host, c.value_host, c.tables,
                                       c.d.seq_lens, c.d.cu_q, c.w.scale, c.w.num_kv_heads, 16,
                                       oracle.FP8E4M3 if c.fp8 else oracle.BF16, c.k_scale, c.v_scale,
                                       num_threads=threads or oracle.max_threads())
        assert st == 0
        return out
    rows = np.asarray(rows, dtype=np.int64)
    seq = np.searchsorted(c.d.cu_q, rows, side="right") - 1
    lens = (c.d.seq_lens[seq] - c.d.chunk_lens[seq] + (rows - c.d.cu_q[seq]) + 1).astype(np.int32)
    st, out = oracle.paged_decode(workloads.bf16_bits(c.d.q)[rows], c.key_host, c.value_host,
                                  np.ascontiguousarray(c.tables[seq]), lens, c.w.scale, c.w.num_kv_heads, 16,
                                  oracle.FP8E4M3 if c.fp8 else oracle.BF16, c.k_scale, c.v_scale,
                                  num_threads=threads or oracle.max_threads())
    assert st == 0
    return out
