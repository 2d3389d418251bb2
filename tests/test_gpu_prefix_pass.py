"""GPU parity of the shared-prefix pass (pkv_decode_opts.shared_prefix_blocks).

Blocks that many sequences' tables share are stored once ("KV Cache 与推理优化",
PagedAttention section).  With the option set, a pass before the decode reads each such block
once per KV head for up to 64 query rows and leaves a partial softmax state per row, which the
decode merges with the blocks it streams itself.  The attention is the same for any tables, so
every case below must match the fp64 oracle within the decode tolerance: prefix-sharing batches
at several shared counts (including sequences that lie entirely inside the shared prefix, and a
count larger than the tables share), tables that share nothing, an FP8 pool, a step that
appends after copy-on-write, and a multi-layer launch."""
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


PREFIX_CASES = {
    # lengths below, at and past the 8 shared blocks (128 positions)
    "g7-d128-bf16": dict(batch=9, num_q_heads=28, num_kv_heads=4, head_dim=128, lengths="list",
                         len_list=(1, 5, 127, 128, 129, 400, 700, 1500, 3000), prefix_blocks=8,
                         pool="exact", append=False, seed=51),
    "g4-d64-bf16": dict(batch=20, num_q_heads=8, num_kv_heads=2, head_dim=64, lengths="list",
                        len_list=tuple(int(x) for x in np.random.Generator(np.random.PCG64(52)).integers(1, 900, 20)),
                        prefix_blocks=8, pool="exact", append=False, seed=52),
    "g16-d128-bf16": dict(batch=6, num_q_heads=32, num_kv_heads=2, head_dim=128, lengths="list",
                          len_list=(50, 140, 260, 700, 999, 1200), prefix_blocks=8, pool="exact",
                          append=False, seed=53),
    "g7-d128-fp8": dict(batch=9, num_q_heads=28, num_kv_heads=4, head_dim=128, lengths="list",
                        len_list=(1, 5, 127, 128, 129, 400, 700, 1500, 3000), prefix_blocks=8,
                        pool="exact", append=False, kv_dtype="fp8", seed=54),
    "g2-d64-fp8": dict(batch=7, num_q_heads=4, num_kv_heads=2, head_dim=64, lengths="list",
                       len_list=(16, 17, 100, 128, 300, 301, 640), prefix_blocks=8, pool="exact",
                       append=False, kv_dtype="fp8", seed=55),
}


@pytest.mark.parametrize("name", sorted(PREFIX_CASES))
def test_prefix_pass_matches_the_oracle(name):
    c = C.build("tiny", overrides=PREFIX_CASES[name])
    ref = C.oracle_decode(c)
    plain = C.gpu_step(c, dict(variant=3), append=False)
    C.tol_check(C.bf16_to_f64(plain), ref)
    for sp in (1, 4, 8, 64):                  # fewer than shared, exactly, more than shared
        for grid in (0, 3):
            out = C.gpu_step(c, dict(shared_prefix_blocks=sp, grid_ctas=grid), append=False)
            C.tol_check(C.bf16_to_f64(out), ref)
    # the same call twice gives the same bits
    a = C.gpu_step(c, dict(shared_prefix_blocks=8), append=False)
    b = C.gpu_step(c, dict(shared_prefix_blocks=8), append=False)
    assert torch.equal(a, b)


def test_prefix_pass_on_tables_that_share_nothing():
    # only the reference table itself is covered; every other sequence is streamed whole
    ov = dict(batch=5, num_q_heads=16, num_kv_heads=4, head_dim=128, lengths="list",
              len_list=(3, 90, 400, 1000, 77), pool="double", append=False, seed=56)
    c = C.build("tiny", overrides=ov)
    ref = C.oracle_decode(c)
    for sp in (2, 100):
        out = C.gpu_step(c, dict(shared_prefix_blocks=sp), append=False)
        C.tol_check(C.bf16_to_f64(out), ref)


def test_prefix_pass_full_size_prefix_sharing_workload():
    c = C.build("qwen25_7b_prefix")
    out = C.gpu_step(c, dict(shared_prefix_blocks=c.w.prefix_blocks), append=False)
    C.tol_check(C.bf16_to_f64(out), C.oracle_decode(c))


def test_prefix_pass_in_an_appending_step_after_copy_on_write():
    # sequences whose newest position lies in a shared block diverge first; the block that
    # receives the new token is never covered by the pass, so the step writes it first
    ov = dict(batch=10, num_q_heads=28, num_kv_heads=4, head_dim=128, lengths="lognormal",
              max_len=3000, prefix_blocks=64, append=True, seed=59)
    c = C.build("qwen25_7b_prefix_cow", overrides=ov)
    lens, mb = c.seq_lens, c.tables.shape[1]
    pre = c.pool.alloc(c.w.prefix_blocks)
    t_lib = c.pool.build_block_tables(lens, mb, pre)
    t2, pairs = c.pool.cow_prepare(t_lib, lens)
    t2_o, pairs_o = oracle.copy_on_write(c.alloc, c.tables, lens)
    np.testing.assert_array_equal(t2, t2_o)
    assert len(pairs) >= 2                         # some sequences diverge inside the prefix
    oracle.copy_blocks(c.key_host, c.value_host, pairs_o)
    c.tables, c.slots = t2_o, oracle.slot_mapping(t2_o, lens)
    C.oracle_append(c)
    ref = C.oracle_decode(c)
    if len(pairs):
        pkv.copy_blocks(c.pool, c.key_cache, c.value_cache, torch.from_numpy(pairs[:, 0].copy()).cuda(),
                        torch.from_numpy(pairs[:, 1].copy()).cuda())
    bt, sl, _ = C.device_tables(c)
    opts = dict(shared_prefix_blocks=c.w.prefix_blocks)
    out = torch.empty_like(c.q)
    ws = torch.zeros(pkv.decode_workspace_bytes(c.pool, len(lens), c.w.num_q_heads, mb, opts),
                     dtype=torch.uint8, device="cuda")
    pkv.decode_step(c.pool, c.q, c.k_new, c.v_new, c.key_cache, c.value_cache, bt, sl, c.w.scale, out, ws,
                    opts=opts)
    assert c.pool.get_device_error() == (pkv.OK, 0)
    np.testing.assert_array_equal(workloads.bf16_bits(c.key_cache), c.key_host)
    np.testing.assert_array_equal(workloads.bf16_bits(c.value_cache), c.value_host)
    C.tol_check(C.bf16_to_f64(out), ref)


@pytest.mark.parametrize("append", [False, True])
def test_prefix_pass_over_every_layer(append):
    # two shared blocks; with the append every new token lands past them, in a private block
    lens = (40, 33, 47, 64) if append else (18, 33, 40, 7)
    c = C.build_layers("tiny_layers", overrides=dict(batch=4, len_list=lens, pool="double", fixed_blocks=0,
                                                     prefix_blocks=2, append=append, seed=58))
    out = C.gpu_layers(c, append, dict(shared_prefix_blocks=4))
    for l in range(c.w.layers):
        ref, _, _ = C.oracle_layer(c, l, l, append)
        C.tol_check(C.bf16_to_f64(out[l]), ref)


def test_prefix_pass_needs_the_token_rows_variant():
    c = C.build("tiny")
    B, Hq, _ = c.q.shape
    mb = c.tables.shape[1]
    assert pkv.decode_workspace_bytes(c.pool, B, Hq, mb, dict(shared_prefix_blocks=4, variant=2)) == 0
    assert pkv.decode_workspace_bytes(c.pool, B, Hq, mb, dict(shared_prefix_blocks=4, heads_per_copy=2)) == 0
    assert pkv.decode_workspace_bytes(c.pool, B, Hq, mb, dict(shared_prefix_blocks=-1)) == 0
    assert pkv.decode_workspace_bytes(c.pool, B, Hq, mb, dict(shared_prefix_blocks=4)) > \
        pkv.decode_workspace_bytes(c.pool, B, Hq, mb)
