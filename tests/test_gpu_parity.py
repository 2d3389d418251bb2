"""GPU parity: the CUDA library (through the C ABI) against the fp64 oracle.

kv_append must be bit-exact over the whole pool; decode must satisfy
|gpu - oracle| <= 1e-2 + 1e-2*|oracle| elementwise, at every size from the tiny workload
to the full benchmark workloads, for both contraction variants and every compiled
pipeline shape, with NaN in every position no sequence may read."""
import numpy as np
import pytest
import torch

import oracle
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


def _append_bit_exact(c: C.Case):
    C.oracle_append(c)
    torch.cuda.synchronize()
    assert np.array_equal(workloads.bf16_bits(c.key_cache), c.key_host)
    assert np.array_equal(workloads.bf16_bits(c.value_cache), c.value_host)


# ------------------------------------------------------------------ the five workloads
def test_tiny_workload():
    c = C.build("tiny")
    out = C.gpu_step(c)
    _append_bit_exact(c)                    # appends land at positions 17 and 32
    assert c.slots.tolist() == [int(c.tables[0][1]) * 16 + 1, int(c.tables[1][2]) * 16 + 0]
    ref = C.oracle_decode(c)
    C.tol_check(C.bf16_to_f64(out), ref)


@pytest.mark.parametrize("name", ["llama3_8b", "ragged", "llama3_70b_long",
                                  "qwen25_7b_prefix", "qwen25_7b_prefix_fp8"])
def test_full_size_workload(name):
    c = C.build(name)
    out = C.gpu_step(c)                     # the launch configuration the benchmark times
    if c.w.append:
        _append_bit_exact(c)
    ref = C.oracle_decode(c)
    mx, rel = C.tol_check(C.bf16_to_f64(out), ref)
    print("%s: max abs err %.3g, max rel err %.3g" % (name, mx, rel))


@pytest.mark.parametrize("name,overrides", [
    ("tiny", None),
    ("llama3_8b", None),
    ("ragged", None),
    ("tiny", dict(batch=4, num_q_heads=28, num_kv_heads=4, head_dim=128, lengths="list",
                  len_list=(1, 16, 17, 700), pool="double", kv_dtype="fp8", append=True, seed=5)),
    ("tiny", dict(batch=3, num_q_heads=16, num_kv_heads=2, head_dim=64, lengths="list",
                  len_list=(31, 32, 33), pool="double", kv_dtype="fp8", append=True, seed=6)),
], ids=["tiny", "llama3_8b", "ragged", "fp8-d128", "fp8-d64"])
def test_decode_step_equals_append_then_decode(name, overrides):
    # one launch (append inside the decode kernel) == kv_append + decode, bit for bit, and
    # the oracle agrees within tolerance
    c = C.build(name, overrides=overrides)
    bt, sl, slots = C.device_tables(c)
    kc2, vc2 = c.key_cache.clone(), c.value_cache.clone()
    out_two = C.gpu_step(c, dict(grid_ctas=0), append=True)          # kv_append + decode
    B, Hq, _ = c.q.shape
    ws = torch.zeros(pkv.decode_workspace_bytes(c.pool, B, Hq, bt.shape[1]), dtype=torch.uint8,
                     device="cuda")
    out_one = torch.empty_like(c.q)
    pkv.decode_step(c.pool, c.q, c.k_new, c.v_new, kc2, vc2, bt, sl, c.w.scale, out_one, ws)
    assert c.pool.get_device_error() == (pkv.OK, 0)
    assert torch.equal(kc2.view(torch.uint8), c.key_cache.view(torch.uint8))
    assert torch.equal(vc2.view(torch.uint8), c.value_cache.view(torch.uint8))
    assert torch.equal(out_one, out_two)
    C.oracle_append(c)
    if c.kv_dtype == pkv.KV_BF16:
        assert np.array_equal(workloads.bf16_bits(kc2), c.key_host)
    else:
        assert np.array_equal(kc2.cpu().numpy(), c.key_host)
        assert np.array_equal(vc2.cpu().numpy(), c.value_host)
    C.tol_check(C.bf16_to_f64(out_one), C.oracle_decode(c))


def test_fp8_append_matches_oracle_encoder_bit_for_bit():
    # every finite bf16 value, as K and V rows, through the GPU encoder and the oracle's
    D, Hkv = 128, 4
    bits = np.arange(65536, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    fin = bits[np.isfinite(vals)].astype(np.uint16)
    rows = -(-fin.size // (Hkv * D))
    padded = np.resize(fin, rows * Hkv * D).reshape(rows, Hkv, D)
    k = torch.from_numpy(padded.view(np.int16)).view(torch.bfloat16).cuda()
    v = torch.flip(k, dims=[2]).contiguous()
    for ks, vs in ((1.0, 1.0), (0.0137, 3.5), (2.0 ** -7, 1e-3)):
        nb = -(-rows // 16)
        pool = pkv.Pool(nb, Hkv, D, pkv.KV_FP8E4M3, ks, vs)
        pool.attach_device(0)
        kc = torch.zeros((nb, Hkv, 16, D), dtype=torch.uint8, device="cuda")
        vc = torch.zeros_like(kc)
        slots = torch.arange(rows, dtype=torch.int64, device="cuda")
        pkv.kv_append(pool, k, v, slots, kc, vc)
        assert pool.get_device_error()[0] == pkv.OK
        kh = np.zeros(kc.shape, np.uint8)
        vh = np.zeros(vc.shape, np.uint8)
        oracle.kv_append(padded, workloads.bf16_bits(v), np.arange(rows, dtype=np.int64), kh, vh,
                         16, oracle.FP8E4M3, ks, vs)
        assert np.array_equal(kc.cpu().numpy(), kh)
        assert np.array_equal(vc.cpu().numpy(), vh)


# ------------------------------------------------------------------ shapes and variants
SHAPES = [
    # (seq_lens, Hq, Hkv, D, kv)
    ((1, 7, 16, 17, 40, 100, 250), 8, 2, 64, "bf16"),
    ((5, 31, 32, 33, 300), 4, 4, 128, "bf16"),          # MHA
    ((12, 49, 130), 8, 1, 64, "bf16"),                  # MQA
    ((3, 70, 129), 6, 3, 64, "bf16"),                   # group 2
    ((100, 513, 1000), 64, 8, 128, "bf16"),             # group 8
    ((29, 65, 700), 28, 4, 128, "bf16"),                # group 7
    ((47, 200), 48, 3, 128, "bf16"),                    # group 16
    ((47, 300), 64, 4, 128, "bf16"),                    # group 16 over 4 KV heads (copies of 2, 4 heads)
    ((21, 50, 333), 28, 4, 128, "fp8"),
    ((9, 64, 257), 16, 2, 64, "fp8"),
    ((18, 33, 49, 600), 40, 4, 128, "fp8"),             # group 10 (16-row mma path)
]


def _custom(lens, Hq, Hkv, D, kv, seed=7):
    ov = dict(batch=len(lens), num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, lengths="list",
              len_list=tuple(lens), pool="double", kv_dtype=kv, append=(kv == "bf16"),
              seed=seed)
    return C.build("tiny", overrides=ov)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "%s-g%d-D%d-%s" % (len(s[0]), s[1] // s[2], s[3], s[4]))
def test_shapes_both_variants_and_grids(shape):
    lens, Hq, Hkv, D, kv = shape
    c = _custom(lens, Hq, Hkv, D, kv)
    bt, sl, slots = C.device_tables(c)
    if c.w.append:
        pkv.kv_append(c.pool, c.k_new, c.v_new, slots, c.key_cache, c.value_cache)
        _append_bit_exact(c)
    ref = C.oracle_decode(c)
    variants = [3, 2] + ([1] if Hq // Hkv <= 8 else [])
    for variant in variants:
        # grid 1: every unit whole in one CTA; small grids: units cut across CTAs
        for grid in (0, 1, 2, 3, 7, 64, 1000):
            out = C.gpu_step(c, dict(variant=variant, grid_ctas=grid), append=False)
            C.tol_check(C.bf16_to_f64(out), ref)
    for hp in (1, 2, 4):                        # KV heads per copy (variant 3)
        if Hkv % hp:
            continue
        for grid in (0, 1, 3, 64):
            out = C.gpu_step(c, dict(variant=3, heads_per_copy=hp, grid_ctas=grid), append=False)
            C.tol_check(C.bf16_to_f64(out), ref)
    # the split's cost per unit: an even split of the blocks, small and large costs (with a
    # cost far above the blocks, most CTAs get no task and leave)
    for uc in (-1, 1, 16, 64, 4096):
        for grid in (0, 3, 64):
            out = C.gpu_step(c, dict(unit_cost=uc, grid_ctas=grid), append=False)
            C.tol_check(C.bf16_to_f64(out), ref)
    for variant in (3, 2):
        for nw, ns in ((4, 2), (4, 4), (8, 2), (8, 3)):
            for grid in (0, 5):
                opts = dict(variant=variant, warps_per_cta=nw, stages=ns, grid_ctas=grid)
                if pkv.decode_workspace_bytes(c.pool, len(lens), Hq, bt.shape[1], opts) == 0:
                    continue                        # this ring does not fit in shared memory
                out = C.gpu_step(c, opts, append=False)
                C.tol_check(C.bf16_to_f64(out), ref)
    # the same call twice gives the same bits
    a = C.gpu_step(c, dict(grid_ctas=7), append=False)
    b = C.gpu_step(c, dict(grid_ctas=7), append=False)
    assert torch.equal(a, b)


def test_physical_placement_does_not_change_a_single_bit():
    # the same logical K/V under three physical placements: pool blocks permuted and the
    # tables rewritten to match
    lens = (1, 15, 16, 17, 200, 777)
    ov = dict(batch=len(lens), num_q_heads=32, num_kv_heads=8, head_dim=128, lengths="list",
              len_list=lens, pool="double", append=False, seed=9)
    c = C.build("tiny", overrides=ov)
    kc0, vc0, t0 = c.key_cache.clone(), c.value_cache.clone(), c.tables.copy()
    nb = kc0.shape[0]
    by_opts = {}
    for k in range(3):
        perm = np.random.default_rng(100 + k).permutation(nb) if k else np.arange(nb)
        pt = torch.from_numpy(perm).cuda()
        c.key_cache[pt] = kc0
        c.value_cache[pt] = vc0
        c.tables = np.where(t0 >= 0, perm[np.maximum(t0, 0)], -1).astype(np.int32)
        for opts in (None, dict(grid_ctas=3), dict(grid_ctas=11), dict(variant=1), dict(variant=2),
                     dict(warps_per_cta=8), dict(heads_per_copy=1), dict(heads_per_copy=2),
                     dict(unit_cost=-1), dict(unit_cost=200, grid_ctas=9)):
            by_opts.setdefault(repr(opts), []).append(C.gpu_step(c, opts, append=False))
    for o, lst in by_opts.items():
        assert np.isfinite(lst[0].float().cpu().numpy()).all()
        for out in lst[1:]:
            assert torch.equal(out, lst[0]), o


def test_single_position_returns_its_value_exactly():
    c = _custom((1, 1, 1), 8, 2, 128, "bf16")
    out = C.gpu_step(c, append=True)
    v_new = c.v_new.repeat_interleave(4, dim=1)            # [B, Hq, D]
    assert torch.equal(out, v_new)


def test_identical_keys_give_the_mean_of_values():
    c = _custom((37, 160), 8, 2, 64, "bf16")
    bt, sl, slots = C.device_tables(c)
    pkv.kv_append(c.pool, c.k_new, c.v_new, slots, c.key_cache, c.value_cache)
    live = oracle.all_slots(c.tables, c.seq_lens)
    s = torch.from_numpy(live).cuda()
    c.key_cache[s // 16, :, s % 16, :] = c.key_cache[s[:1] // 16, :, s[:1] % 16, :]
    out = C.gpu_step(c, append=False)
    vals = c.value_cache[s // 16, :, s % 16, :].float()      # [T, Hkv, D]
    off = 0
    for b, L in enumerate(c.seq_lens):
        mean = vals[off:off + L].mean(dim=0).repeat_interleave(4, dim=0)
        off += L
        torch.testing.assert_close(out[b].float(), mean, atol=1e-2, rtol=1e-2)


# ------------------------------------------------------------------ device error reporting
def test_device_errors_are_flagged_not_trapped():
    c = _custom((18, 33), 8, 2, 64, "bf16")
    bt, sl, slots = C.device_tables(c)
    out = torch.empty_like(c.q)
    ws = torch.zeros(pkv.decode_workspace_bytes(c.pool, 2, 8, 3), dtype=torch.uint8, device="cuda")
    bad = bt.clone()
    bad[1, 2] = c.pool.desc.num_blocks + 5
    pkv.paged_attention_decode(c.pool, c.q, c.key_cache, c.value_cache, bad, sl, 0.125, out, ws)
    st, bits = c.pool.get_device_error()
    assert st == pkv.ERR_DEVICE and bits & pkv.DEVERR_BLOCK_ID
    for L in (0, 3 * 16 + 1):
        sl2 = sl.clone()
        sl2[0] = L
        ws.zero_()
        pkv.paged_attention_decode(c.pool, c.q, c.key_cache, c.value_cache, bt, sl2, 0.125, out, ws)
        st, bits = c.pool.get_device_error()
        assert st == pkv.ERR_DEVICE and bits == pkv.DEVERR_SEQ_LEN
        assert torch.count_nonzero(out[0]) == 0
    bad_slots = slots.clone()
    bad_slots[0] = c.pool.desc.num_blocks * 16
    before = c.key_cache.clone()
    pkv.kv_append(c.pool, c.k_new, c.v_new, bad_slots, c.key_cache, c.value_cache)
    st, bits = c.pool.get_device_error()
    assert st == pkv.ERR_DEVICE and bits == pkv.DEVERR_SLOT
    changed = (c.key_cache.view(torch.int16) != before.view(torch.int16)).any(dim=(1, 3))
    assert changed.sum() == 1                              # only sequence 1's slot was written
    assert pool_ok(c)


def pool_ok(c):
    st, bits = c.pool.get_device_error()
    return st == pkv.OK and bits == 0


def test_host_side_argument_errors():
    c = _custom((18, 33), 8, 2, 64, "bf16")
    bt, sl, slots = C.device_tables(c)
    out = torch.empty_like(c.q)
    ws0 = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkv.PkvError):                        # misaligned q
        q2 = torch.empty(c.q.numel() + 1, dtype=torch.bfloat16, device="cuda")[1:].view_as(c.q)
        pkv.paged_attention_decode(c.pool, q2, c.key_cache, c.value_cache, bt, sl, 0.125, out, ws0)
    with pytest.raises(pkv.PkvError):                        # Hq not a multiple of Hkv
        q3 = torch.zeros(2, 7, 64, dtype=torch.bfloat16, device="cuda")
        pkv.paged_attention_decode(c.pool, q3, c.key_cache, c.value_cache, bt, sl, 0.125,
                                   torch.empty_like(q3), ws0)
    with pytest.raises(pkv.PkvError):                        # no workspace
        pkv.paged_attention_decode(c.pool, c.q, c.key_cache, c.value_cache, bt, sl, 0.125, out,
                                   None)
    ws = torch.zeros(pkv.decode_workspace_bytes(c.pool, 2, 8, 3), dtype=torch.uint8, device="cuda")
    with pytest.raises(pkv.PkvError):                        # workspace too small
        pkv.paged_attention_decode(c.pool, c.q, c.key_cache, c.value_cache, bt, sl, 0.125, out,
                                   ws[:256])
    with pytest.raises(pkv.PkvError):                        # CUDA-core variant is group <= 8
        q4 = torch.zeros(2, 32, 64, dtype=torch.bfloat16, device="cuda")
        pkv.paged_attention_decode(c.pool, q4, c.key_cache, c.value_cache, bt, sl, 0.125,
                                   torch.empty_like(q4), ws0, dict(variant=1))
    assert pool_ok(c)


def test_probe_copy():
    src = torch.randint(0, 255, (3 << 20,), dtype=torch.uint8, device="cuda")
    dst = torch.zeros_like(src)
    pkv.probe_copy(dst, src)
    torch.cuda.synchronize()
    assert torch.equal(src, dst)


def test_prepared_host_step_reads_the_refilled_host_buffers():
    """A DecodeStepHost is built once for a set of buffers; each run() uploads what the host
    buffers hold at that time (a serving loop refills them every step).  Two runs with
    different queries give the device-buffer decode of each, bit for bit."""
    c = C.build("qwen25_7b_prefix")
    assert not c.w.append
    bt, sl, _ = C.device_tables(c)
    B, Hq, _ = c.q.shape
    ws = torch.zeros(pkv.decode_workspace_bytes(c.pool, B, Hq, bt.shape[1]), dtype=torch.uint8, device="cuda")
    pin = lambda t: t.detach().cpu().pin_memory()
    host = {"q": pin(c.q), "block_tables": pin(bt), "seq_lens": pin(sl),
            "out": torch.empty(c.q.shape, dtype=c.q.dtype).pin_memory()}
    dev = {"q": torch.empty_like(c.q), "block_tables": torch.empty_like(bt), "seq_lens": torch.empty_like(sl),
           "out": torch.empty_like(c.q)}
    stream = torch.cuda.current_stream()
    step = pkv.DecodeStepHost(c.pool, host, dev, c.key_cache, c.value_cache, c.w.scale, ws, stream=stream)
    for q in (c.q, (c.q.float() * -0.5).to(torch.bfloat16)):
        host["q"].copy_(q.cpu())
        step.run()
        stream.synchronize()
        ref = torch.empty_like(c.q)
        pkv.paged_attention_decode(c.pool, q, c.key_cache, c.value_cache, bt, sl, c.w.scale, ref, ws)
        torch.cuda.synchronize()
        st, bits = c.pool.get_device_error()
        assert st == pkv.OK and bits == 0
        assert torch.equal(host["out"].view(torch.int16), ref.cpu().view(torch.int16))


@pytest.mark.parametrize("contiguous,prepared", [(False, False), (True, False), (True, True)])
@pytest.mark.parametrize("name", ["tiny", "llama3_8b", "qwen25_7b_prefix"])
def test_decode_step_from_host_memory_equals_the_device_step(name, contiguous, prepared):
    """pkv_decode_step_host (copies in, one-launch step, copy out, all from one call) gives
    the same bits as pkv_decode_step on device buffers: output and pool.  `prepared` runs it
    through DecodeStepHost (pointer structures built once, one C call per step)."""
    a = C.build(name)
    b = C.build(name)
    bt, sl, _ = C.device_tables(a)
    B, Hq, _ = a.q.shape
    ws_a = torch.zeros(pkv.decode_workspace_bytes(a.pool, B, Hq, bt.shape[1]), dtype=torch.uint8, device="cuda")
    ws_b = torch.zeros_like(ws_a)
    out_a = torch.empty_like(a.q)
    if a.w.append:
        pkv.decode_step(a.pool, a.q, a.k_new, a.v_new, a.key_cache, a.value_cache, bt, sl, a.w.scale, out_a, ws_a)
    else:
        pkv.paged_attention_decode(a.pool, a.q, a.key_cache, a.value_cache, bt, sl, a.w.scale, out_a, ws_a)
    pin = lambda t: t.detach().cpu().pin_memory()
    host = {"q": pin(b.q), "block_tables": pin(bt), "seq_lens": pin(sl),
            "out": torch.empty(b.q.shape, dtype=b.q.dtype).pin_memory()}
    dev = {"q": torch.empty_like(b.q), "block_tables": torch.empty_like(bt), "seq_lens": torch.empty_like(sl),
           "out": torch.empty_like(b.q)}
    if b.w.append:
        host.update(k_new=pin(b.k_new), v_new=pin(b.v_new))
        dev.update(k_new=torch.empty_like(b.k_new), v_new=torch.empty_like(b.v_new))
    if contiguous:                  # the inputs as views of one host and one device buffer
        names = [k for k in ("q", "k_new", "v_new", "block_tables", "seq_lens") if k in host]
        sizes = [host[k].numel() * host[k].element_size() for k in names]
        hbuf = torch.empty(sum(sizes), dtype=torch.uint8).pin_memory()
        dbuf = torch.empty(sum(sizes), dtype=torch.uint8, device="cuda")
        off = 0
        for k, n in zip(names, sizes):
            t = host[k]
            host[k] = hbuf[off:off + n].view(t.dtype).view(t.shape)
            host[k].copy_(t)
            dev[k] = dbuf[off:off + n].view(t.dtype).view(t.shape)
            off += n
        host["contiguous"] = True
    stream = torch.cuda.current_stream()
    if prepared:
        pkv.DecodeStepHost(b.pool, host, dev, b.key_cache, b.value_cache, b.w.scale, ws_b, stream=stream).run()
    else:
        pkv.decode_step_host(b.pool, host, dev, b.key_cache, b.value_cache, b.w.scale, ws_b, stream=stream)
    stream.synchronize()
    for c in (a, b):
        st, bits = c.pool.get_device_error()
        assert st == pkv.OK and bits == 0
    assert torch.equal(host["out"].view(torch.int16), out_a.cpu().view(torch.int16))
    assert torch.equal(a.key_cache.view(torch.int16), b.key_cache.view(torch.int16))
    assert torch.equal(a.value_cache.view(torch.int16), b.value_cache.view(torch.int16))
