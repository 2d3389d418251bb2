"""Failure path of the kernels' bounded waits, without a GPU fault.

pkv_test_expire_waits() makes one role of every decode (or prefill) launch wait on an
mbarrier that nothing completes.  The wait must run out within its bound, the kernel must
report PKV_DEVERR_TIMEOUT through the pool's error word (pkv_get_device_error returns
PKV_ERR_TIMEOUT), copies already in flight must be waited for before the CTAs leave, and the
context must stay usable: the next normal call on the same pool, buffers and workspace must
match the oracle.  The decode workspace's split counters must also be back at zero."""
import time

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


@pytest.fixture(autouse=True)
def _hook_off():
    yield
    pkv.test_expire_waits(pkv.TEST_EXPIRE_NONE)


def test_hook_rejects_unknown_targets():
    with pytest.raises(pkv.PkvError):
        pkv.test_expire_waits(3)


@pytest.mark.parametrize("name,overrides", [
    ("llama3_8b", None),
    # units cut across CTAs: the cross-CTA merge still runs after the timeout
    ("tiny", dict(batch=3, num_q_heads=28, num_kv_heads=4, head_dim=128, lengths="list",
                  len_list=(40, 900, 3000), pool="double", append=False, seed=41)),
], ids=["llama3_8b", "split-units"])
def test_decode_wait_runs_out_then_the_context_is_usable(name, overrides):
    c = C.build(name, overrides=overrides)
    bt, sl, slots = C.device_tables(c)
    B, Hq, _ = c.q.shape
    nbytes = pkv.decode_workspace_bytes(c.pool, B, Hq, bt.shape[1])
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(c.q)
    pkv.test_expire_waits(pkv.TEST_EXPIRE_DECODE)
    t0 = time.perf_counter()
    pkv.paged_attention_decode(c.pool, c.q, c.key_cache, c.value_cache, bt, sl, c.w.scale, out, ws)
    st, bits = c.pool.get_device_error()
    elapsed = time.perf_counter() - t0
    assert st == pkv.ERR_TIMEOUT and bits & pkv.DEVERR_TIMEOUT, (st, bits)
    assert elapsed < 30.0
    counters = ws[:B * c.w.num_kv_heads * 4].view(torch.int32)
    assert int(torch.count_nonzero(counters)) == 0
    pkv.test_expire_waits(pkv.TEST_EXPIRE_NONE)
    # the same pool, buffers and workspace, now a normal step: kv_append + decode
    if c.w.append:
        pkv.kv_append(c.pool, c.k_new, c.v_new, slots, c.key_cache, c.value_cache)
        C.oracle_append(c)
    out.fill_(float("nan"))
    pkv.paged_attention_decode(c.pool, c.q, c.key_cache, c.value_cache, bt, sl, c.w.scale, out, ws)
    assert c.pool.get_device_error() == (pkv.OK, 0)
    C.tol_check(C.bf16_to_f64(out), C.oracle_decode(c))


def test_decode_step_wait_runs_out_then_the_step_reruns():
    # the one-launch step (append inside the decode kernel) with the wait run out, then the
    # same step again normally: the append is idempotent, so pools and output match the oracle
    c = C.build("ragged", overrides=dict(batch=16))
    bt, sl, _ = C.device_tables(c)
    B, Hq, _ = c.q.shape
    ws = torch.zeros(pkv.decode_workspace_bytes(c.pool, B, Hq, bt.shape[1]), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(c.q)
    pkv.test_expire_waits(pkv.TEST_EXPIRE_DECODE)
    pkv.decode_step(c.pool, c.q, c.k_new, c.v_new, c.key_cache, c.value_cache, bt, sl, c.w.scale, out, ws)
    st, bits = c.pool.get_device_error()
    assert st == pkv.ERR_TIMEOUT and bits & pkv.DEVERR_TIMEOUT
    pkv.test_expire_waits(pkv.TEST_EXPIRE_NONE)
    out.fill_(float("nan"))
    pkv.decode_step(c.pool, c.q, c.k_new, c.v_new, c.key_cache, c.value_cache, bt, sl, c.w.scale, out, ws)
    assert c.pool.get_device_error() == (pkv.OK, 0)
    C.oracle_append(c)
    torch.cuda.synchronize()
    assert np.array_equal(workloads.bf16_bits(c.key_cache), c.key_host)
    assert np.array_equal(workloads.bf16_bits(c.value_cache), c.value_host)
    C.tol_check(C.bf16_to_f64(out), C.oracle_decode(c))


@pytest.mark.parametrize("fp8", [False, True], ids=["bf16", "fp8"])
def test_prefill_wait_runs_out_then_the_context_is_usable(fp8):
    c = C.build_prefill("prefill_tiny", overrides={"head_dim": 128, "num_q_heads": 8, "num_kv_heads": 2}, fp8=fp8)
    C.prefill_append(c)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(C.prefill_pool_bits(c, c.key_cache), c.key_host)
    plan, grid = pkv.prefill_plan(c.pool, c.d.cu_q, c.d.seq_lens, c.w.num_q_heads, c.tables.shape[1])
    plan_d = torch.from_numpy(plan).cuda()
    bt = torch.from_numpy(c.tables).cuda()
    out = torch.empty_like(c.d.q)
    pkv.test_expire_waits(pkv.TEST_EXPIRE_PREFILL)
    t0 = time.perf_counter()
    pkv.paged_prefill(c.pool, c.d.q, c.key_cache, c.value_cache, bt, c.w.scale, plan_d, grid, out)
    st, bits = c.pool.get_device_error()
    elapsed = time.perf_counter() - t0
    assert st == pkv.ERR_TIMEOUT and bits & pkv.DEVERR_TIMEOUT, (st, bits)
    assert elapsed < 30.0
    pkv.test_expire_waits(pkv.TEST_EXPIRE_NONE)
    out.fill_(float("nan"))
    pkv.paged_prefill(c.pool, c.d.q, c.key_cache, c.value_cache, bt, c.w.scale, plan_d, grid, out)
    assert c.pool.get_device_error() == (pkv.OK, 0)
    C.tol_check(C.bf16_to_f64(out), C.oracle_prefill_rows(c))
