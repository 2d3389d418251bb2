"""Automatic prefix caching feeding the decode path, on the GPU.

Request A's prompt starts with a system prompt; its blocks are cached.  Request B starts
with the same system prompt: the lookup returns A's physical blocks for it ("KV Cache 与推理
优化", section "APC：连计算都省了"), B's table starts with them, only B's own positions are
appended, and B decodes over the shared blocks.  The premise of prefix caching is that equal
tokens at equal positions under one model give equal K/V, so B's private K/V for the
system prompt are A's rows; the oracle decodes B on such a private, unshared pool, and the
GPU must match it (and leave A's result unchanged)."""
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


def test_cached_system_prompt_is_reused_by_the_next_request():
    NB, Hkv, Hq, D = 32, 8, 32, 128
    scale = float(np.float32(1.0 / np.sqrt(D)))
    rng = np.random.Generator(np.random.PCG64(159200))
    sys_prompt = rng.integers(0, 128000, size=64).tolist()            # 4 full blocks
    tok_a = sys_prompt + rng.integers(0, 128000, size=40).tolist()    # 104 positions
    tok_b = sys_prompt + rng.integers(0, 128000, size=57).tolist()    # 121 positions
    La, Lb = len(tok_a), len(tok_b)
    kA = workloads.randn_bf16((La, Hkv, D), 159201, "cuda")
    vA = workloads.randn_bf16((La, Hkv, D), 159202, "cuda")
    kB = workloads.randn_bf16((Lb, Hkv, D), 159203, "cuda")
    vB = workloads.randn_bf16((Lb, Hkv, D), 159204, "cuda")
    kB[:64], vB[:64] = kA[:64], vA[:64]          # same tokens, same positions: same K/V
    q = workloads.randn_bf16((2, Hq, D), 159205, "cuda")

    pool = pkv.Pool(NB, Hkv, D, free_order=rng.permutation(NB).astype(np.int32))
    pool.attach_device(0)
    nan = torch.tensor(C.NAN16, dtype=torch.int16).view(torch.bfloat16).item()
    kc = torch.full((NB, Hkv, 16, D), nan, dtype=torch.bfloat16, device="cuda")
    vc = kc.clone()
    MB = 8
    # request A: nothing cached yet; prefill all its positions, then cache its blocks
    assert pool.prefix_lookup(tok_a).size == 0
    ta = pool.build_block_tables([La], MB)[0]
    sa = torch.from_numpy(pkv.slot_mapping_all(ta[None], [La])).cuda()
    pkv.kv_append(pool, kA, vA, sa, kc, vc)
    assert pool.prefix_insert(tok_a, 0, ta) == 6                      # 104 tokens: 6 full blocks
    # request B: its system prompt hits A's first 4 blocks; only positions 64.. are written
    hits = pool.prefix_lookup(tok_b)
    assert hits.tolist() == ta[:4].tolist()
    tb = pool.build_block_tables([Lb], MB, hits)[0]
    assert tb[:4].tolist() == ta[:4].tolist() and len(set(tb[4:8]) & set(ta)) == 0
    sb = torch.from_numpy(pkv.slot_mapping_all(tb[None], [Lb])[64:]).cuda()
    pkv.kv_append(pool, kB[64:].contiguous(), vB[64:].contiguous(), sb, kc, vc)
    assert pool.refcount(int(ta[0])) == 3                             # A, B and the cache

    tables = np.stack([ta, tb]).astype(np.int32)
    lens = np.array([La, Lb], np.int32)
    out = torch.empty_like(q)
    ws = torch.zeros(pkv.decode_workspace_bytes(pool, 2, Hq, MB), dtype=torch.uint8, device="cuda")
    pkv.paged_attention_decode(pool, q, kc, vc, torch.from_numpy(tables).cuda(),
                               torch.from_numpy(lens).cuda(), scale, out, ws)
    st, bits = pool.get_device_error()
    assert st == pkv.OK and bits == 0

    # oracle: each request on a private pool of its own rows, positions in order
    qb = workloads.bf16_bits(q)
    for r, (k, v, L) in enumerate(((kA, vA, La), (kB, vB, Lb))):
        nblk = oracle.blocks_needed(L, 16)
        pk = np.full((nblk, Hkv, 16, D), C.NAN16, np.uint16)
        pv = pk.copy()
        t = np.arange(nblk, dtype=np.int32)[None]
        assert oracle.kv_append(workloads.bf16_bits(k), workloads.bf16_bits(v),
                                oracle.all_slots(t, [L]), pk, pv) == 0
        st, ref = oracle.paged_decode(qb[r:r + 1], pk, pv, t, np.array([L], np.int32), scale, Hkv)
        assert st == 0
        C.tol_check(C.bf16_to_f64(out[r:r + 1]), ref)
