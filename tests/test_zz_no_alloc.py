"""The decode entry point that allocates nothing (pkv_paged_attention_decode_noalloc).

It serves hosts that cannot allocate device memory while they run, so its scratch is a
fixed array inside libpkv.so instead of a caller-provided workspace.  Here it is called
through the C ABI twice in a row and must match the regular entry point within the decode
tolerance each time; a shape that needs more scratch than the array holds is refused.
This file is collected last so that a failure here stops a -x run only after every other
test has run."""
import ctypes

import numpy as np
import pytest
import torch

from tests import _cases as C

pkv = pytest.importorskip("paged_kv_cache_159_gb300")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    torch.cuda.set_device(0)


def _noalloc(c, bt, sl, out):
    L = pkv.lib()
    return L.pkv_paged_attention_decode_noalloc(
        c.pool.handle, ctypes.c_void_p(c.q.data_ptr()), ctypes.c_void_p(c.key_cache.data_ptr()),
        ctypes.c_void_p(c.value_cache.data_ptr()), ctypes.c_void_p(bt.data_ptr()),
        ctypes.c_void_p(sl.data_ptr()), c.q.shape[0], c.q.shape[1], bt.shape[1],
        ctypes.c_float(c.w.scale), ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("name,overrides", [
    ("llama3_8b", None),
    ("tiny", dict(batch=5, num_q_heads=28, num_kv_heads=4, head_dim=128, lengths="list",
                  len_list=(1, 17, 300, 1000, 2500), pool="double", append=False, seed=31)),
])
def test_noalloc_decode_matches_the_workspace_entry_point(name, overrides):
    c = C.build(name, overrides=overrides)
    bt, sl, slots = C.device_tables(c)
    if c.w.append:
        pkv.kv_append(c.pool, c.k_new, c.v_new, slots, c.key_cache, c.value_cache)
    ref = C.gpu_step(c, append=False)                       # regular entry point
    ref64 = C.bf16_to_f64(ref)
    for _ in range(2):                                      # two calls in a row
        out = torch.full_like(c.q, float("nan"))
        assert _noalloc(c, bt, sl, out) == pkv.OK
        st, bits = c.pool.get_device_error()
        assert st == pkv.OK and bits == 0
        C.tol_check(C.bf16_to_f64(out), ref64)


def test_noalloc_refuses_shapes_beyond_its_scratch():
    # 4096 sequences x 512 KV heads need 8 MiB of counters alone: more than the array
    pool = pkv.Pool(16, 512, 64)
    pool.attach_device(0)
    assert pkv.decode_workspace_bytes(pool, 4096, 512, 1) > (8 << 20)
    q = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    st = pkv.lib().pkv_paged_attention_decode_noalloc(
        pool.handle, ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(q.data_ptr()),
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(q.data_ptr()),
        4096, 512, 1, ctypes.c_float(0.125), ctypes.c_void_p(q.data_ptr()), None)
    assert st == pkv.ERR_INVALID
    assert pool.get_device_error() == (pkv.OK, 0)
