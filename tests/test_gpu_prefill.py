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


def _run(name, overrides=None, rows=None):
    c = C.build_prefill(name, overrides=overrides)
    C.prefill_append(c)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(workloads.bf16_bits(c.key_cache), c.key_host)
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


@pytest.mark.parametrize("chunk,context", [(1, 0), (1, 700), (16, 16), (129, 0), (128, 128), (257, 1)])
def test_prefill_edge_lengths(chunk, context):
    """Single-row chunks, chunks and contexts at tile and block boundaries."""
    _run("prefill_tiny", {"ragged": False, "chunk": chunk, "context": context, "batch": 4,
                          "head_dim": 128, "seed": 159120 + chunk + context})


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
