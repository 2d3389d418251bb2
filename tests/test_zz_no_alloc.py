"""The decode entry point that allocates nothing (pkv_paged_attention_decode_noalloc).

Some callers cannot allocate device memory while they run: a serving process whose memory
manager owns every device byte, or a loop that cannot afford an allocation's implicit
synchronisation.  This entry point takes no workspace; its scratch is a fixed array inside
libpkv.so.  It runs the same kernel with the same launch plan as the workspace entry point,
so, called through the C ABI twice in a row, it must give the same bits, and it must agree
with the oracle within the decode tolerance.  One case cuts (sequence, KV head) units across
CTAs, so the split counters and partial states in the array are used; a shape needing more
scratch than the array holds is refused before anything is queued.  This file is collected
last so that a failure here stops a -x run only after every other test has run."""
import ctypes

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


CASES = [
    ("llama3_8b", None),                                   # every unit whole in one CTA
    ("tiny", dict(batch=5, num_q_heads=28, num_kv_heads=4, head_dim=128, lengths="list",
                  len_list=(1, 17, 300, 1000, 2500), pool="double", append=False, seed=31)),
    # 32 long units on a grid of hundreds of CTAs: every unit is cut across CTAs and merged
    ("tiny", dict(batch=4, num_q_heads=64, num_kv_heads=8, head_dim=128, lengths="fixed",
                  fixed_len=4096, pool="exact", append=False, seed=32)),
]


@pytest.mark.parametrize("name,overrides", CASES, ids=["whole-units", "ragged", "split-units"])
def test_noalloc_decode_matches_the_workspace_entry_point(name, overrides):
    c = C.build(name, overrides=overrides)
    bt, sl, slots = C.device_tables(c)
    if c.w.append:
        pkv.kv_append(c.pool, c.k_new, c.v_new, slots, c.key_cache, c.value_cache)
        C.oracle_append(c)
    ref = C.gpu_step(c, append=False)                       # the workspace entry point
    C.tol_check(C.bf16_to_f64(ref), C.oracle_decode(c))
    for _ in range(2):                                      # two calls in a row, same bits
        out = torch.full_like(c.q, float("nan"))
        assert _noalloc(c, bt, sl, out) == pkv.OK
        assert c.pool.get_device_error() == (pkv.OK, 0)
        assert torch.equal(out, ref)


def test_noalloc_python_wrapper():
    c = C.build("tiny")
    bt, sl, slots = C.device_tables(c)
    pkv.kv_append(c.pool, c.k_new, c.v_new, slots, c.key_cache, c.value_cache)
    C.oracle_append(c)
    out = torch.full_like(c.q, float("nan"))
    pkv.paged_attention_decode_noalloc(c.pool, c.q, c.key_cache, c.value_cache, bt, sl, c.w.scale, out)
    assert c.pool.get_device_error() == (pkv.OK, 0)
    C.tol_check(C.bf16_to_f64(out), C.oracle_decode(c))


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


def test_noalloc_invalid_arguments_queue_nothing():
    # a shape that fits but a bad argument (NULL output, non-finite scale): every check is
    # made before the counters' memset would be queued, and the call is refused
    c = C.build("tiny")
    bt, sl, _ = C.device_tables(c)
    L = pkv.lib()
    args = [c.pool.handle, ctypes.c_void_p(c.q.data_ptr()), ctypes.c_void_p(c.key_cache.data_ptr()),
            ctypes.c_void_p(c.value_cache.data_ptr()), ctypes.c_void_p(bt.data_ptr()),
            ctypes.c_void_p(sl.data_ptr()), c.q.shape[0], c.q.shape[1], bt.shape[1]]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.pkv_paged_attention_decode_noalloc(*args, ctypes.c_float(c.w.scale), None, stream) == pkv.ERR_INVALID
    out = torch.empty_like(c.q)
    assert L.pkv_paged_attention_decode_noalloc(*args, ctypes.c_float(float("inf")),
                                                ctypes.c_void_p(out.data_ptr()), stream) == pkv.ERR_INVALID
    assert c.pool.get_device_error() == (pkv.OK, 0)
