"""GPU parity of copy-on-write: pkv_copy_blocks against the oracle's block copy (bit-exact),
and the whole step on the prefix-sharing batch with appends -- pkv_cow_prepare, then
pkv_copy_blocks, then the one-launch decode step -- against the oracle's copy_on_write,
copy_blocks, kv_append and decode ("KV Cache 与推理优化", PagedAttention section: shared
prefix blocks are stored once and copied when a request diverges)."""
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


@pytest.mark.parametrize("kv,layers,D,Hkv", [("bf16", 1, 128, 8), ("fp8", 3, 64, 2),
                                             ("bf16", 4, 64, 1)])
def test_copy_blocks_is_bit_exact(kv, layers, D, Hkv):
    nb = 96
    fp8 = kv == "fp8"
    pool = pkv.Pool(nb, Hkv, D, pkv.KV_FP8E4M3 if fp8 else pkv.KV_BF16, 1.0, 1.0,
                    num_layers=layers)
    pool.attach_device(0)
    g = torch.Generator(device="cuda").manual_seed(159100 + layers)
    shape = (layers, nb, Hkv, 16, D * (1 if fp8 else 2))
    kc = torch.randint(0, 256, shape, generator=g, device="cuda", dtype=torch.uint8)
    vc = torch.randint(0, 256, shape, generator=g, device="cuda", dtype=torch.uint8)
    rng = np.random.Generator(np.random.PCG64(159101))
    ids = rng.permutation(nb)
    src, dst = ids[:30].astype(np.int32), ids[30:60].astype(np.int32)
    src[5] = src[7]                                   # a source may be copied twice
    kh, vh = kc.cpu().numpy(), vc.cpu().numpy()
    oracle.copy_blocks(kh, vh, np.stack([src, dst], 1), layered=True)
    pkv.copy_blocks(pool, kc, vc, torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda())
    st, bits = pool.get_device_error()
    assert st == pkv.OK and bits == 0
    np.testing.assert_array_equal(kc.cpu().numpy(), kh)
    np.testing.assert_array_equal(vc.cpu().numpy(), vh)


def test_copy_blocks_flags_an_id_outside_the_pool():
    pool = pkv.Pool(8, 2, 64, num_layers=2)
    pool.attach_device(0)
    kc = torch.arange(2 * 8 * 2 * 16 * 64, device="cuda", dtype=torch.int32).view(2, 8, 2, 16, 64).to(torch.bfloat16)
    vc = kc.clone()
    before = kc.clone()
    pkv.copy_blocks(pool, kc, vc, torch.tensor([1, 8], dtype=torch.int32, device="cuda"),
                    torch.tensor([2, 3], dtype=torch.int32, device="cuda"))
    st, bits = pool.get_device_error()
    assert st == pkv.ERR_DEVICE and bits == pkv.DEVERR_BLOCK_ID
    assert torch.equal(kc[:, 2], before[:, 1])        # the valid pair was copied
    assert torch.equal(kc[:, 3], before[:, 3])        # the invalid one was skipped


def test_copy_on_write_step_on_the_prefix_sharing_batch():
    c = C.build("qwen25_7b_prefix_cow")
    lens = c.seq_lens
    mb = c.tables.shape[1]
    # the library's allocator in the same state as the oracle's
    pre = c.pool.alloc(c.w.prefix_blocks)
    t_lib = c.pool.build_block_tables(lens, mb, pre)
    np.testing.assert_array_equal(t_lib, c.tables)
    # host bookkeeping: bit-exact with the oracle
    t2, pairs = c.pool.cow_prepare(t_lib, lens)
    t2_o, pairs_o = oracle.copy_on_write(c.alloc, c.tables, lens)
    np.testing.assert_array_equal(t2, t2_o)
    np.testing.assert_array_equal(pairs, pairs_o)
    assert len(pairs) == 3
    # oracle: copy, append at the new slots, decode
    oracle.copy_blocks(c.key_host, c.value_host, pairs_o)
    c.tables, c.slots = t2_o, oracle.slot_mapping(t2_o, lens)
    C.oracle_append(c)
    ref = C.oracle_decode(c)
    # GPU: copy, then the one-launch append + decode
    pkv.copy_blocks(c.pool, c.key_cache, c.value_cache, torch.from_numpy(pairs[:, 0].copy()).cuda(),
                    torch.from_numpy(pairs[:, 1].copy()).cuda())
    bt, sl, _ = C.device_tables(c)
    out = torch.empty_like(c.q)
    ws = torch.zeros(pkv.decode_workspace_bytes(c.pool, len(lens), c.w.num_q_heads, mb),
                     dtype=torch.uint8, device="cuda")
    pkv.decode_step(c.pool, c.q, c.k_new, c.v_new, c.key_cache, c.value_cache, bt, sl, c.w.scale,
                    out, ws)
    st, bits = c.pool.get_device_error()
    assert st == pkv.OK and bits == 0
    np.testing.assert_array_equal(workloads.bf16_bits(c.key_cache), c.key_host)
    np.testing.assert_array_equal(workloads.bf16_bits(c.value_cache), c.value_host)
    C.tol_check(C.bf16_to_f64(out), ref)
