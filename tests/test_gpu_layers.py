"""GPU parity of the multi-layer entry points (pkv_kv_append_layers, pkv_decode_step_layers)
against the single-layer oracle applied to each layer.

A pool of L layers stacks each cache as [L, NB, Hkv, 16, D] and shares one block table
across layers ("KV Cache 与推理优化", byte table: every layer keeps K and V for every token;
"理解 KV Cache" §3.2: the per-block layout).  Nothing couples the layers, so layer l of the
result must be what the oracle computes on layer l alone."""
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


def _layer_pool_bits(t: torch.Tensor, l: int, fp8: bool) -> np.ndarray:
    x = t[l].contiguous()
    return x.cpu().numpy() if fp8 else workloads.bf16_bits(x)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_kv_append_layers_is_bit_exact(kv):
    c = C.build_layers("tiny_layers", overrides={"kv_dtype": kv})
    fp8 = kv == "fp8"
    _, _, slots = C.device_tables(c)
    pkv.kv_append_layers(c.pool, c.k_new, c.v_new, slots, c.key_cache, c.value_cache)
    st, bits = c.pool.get_device_error()
    assert st == pkv.OK and bits == 0
    dt = oracle.FP8E4M3 if fp8 else oracle.BF16
    for l in range(c.w.layers):
        kh, vh = c.key_host[l].copy(), c.value_host[l].copy()
        assert oracle.kv_append(workloads.bf16_bits(c.k_new[l]), workloads.bf16_bits(c.v_new[l]),
                                c.slots, kh, vh, 16, dt, c.k_scale, c.v_scale) == 0
        np.testing.assert_array_equal(_layer_pool_bits(c.key_cache, l, fp8), kh)
        np.testing.assert_array_equal(_layer_pool_bits(c.value_cache, l, fp8), vh)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("grid", [0, 1, 3, 7, 64])
@pytest.mark.parametrize("append", [True, False])
def test_decode_step_layers_tiny(kv, grid, append):
    # without the append, position L-1 already holds history (it is not poisoned)
    c = C.build_layers("tiny_layers", overrides={"kv_dtype": kv, "append": append})
    fp8 = kv == "fp8"
    opts = {"grid_ctas": grid} if grid else None
    out = C.gpu_layers(c, append, opts)
    for l in range(c.w.layers):
        ref, kh, vh = C.oracle_layer(c, l, l, append)
        C.tol_check(C.bf16_to_f64(out[l]), ref)
        # the fused append leaves every layer's pool exactly as the oracle's append does
        np.testing.assert_array_equal(_layer_pool_bits(c.key_cache, l, fp8), kh)
        np.testing.assert_array_equal(_layer_pool_bits(c.value_cache, l, fp8), vh)


def test_layers_with_ragged_lengths_and_a_cut_grid():
    """Several layers, ragged lengths (including 1 and multiples of 16) and grids that cut
    units across layer boundaries.  Re-running the fused append writes the same rows again,
    so one pool serves every grid."""
    lens = (1, 16, 17, 95, 160, 3, 33, 64)
    c = C.build_layers("tiny_layers", overrides={
        "batch": len(lens), "len_list": lens, "fixed_blocks": 40, "num_q_heads": 16,
        "num_kv_heads": 2, "head_dim": 128, "layers": 5})
    refs = [C.oracle_layer(c, l, l, True)[0] for l in range(c.w.layers)]
    for grid in (0, 5, 13, 29):
        out = C.gpu_layers(c, True, {"grid_ctas": grid} if grid else None)
        for l in range(c.w.layers):
            C.tol_check(C.bf16_to_f64(out[l]), refs[l])


def test_llama3_8b_all_32_layers_full_size():
    """The whole Llama-3-8B decode step: 32 layers x 64 sequences x 2048 positions (16 GiB of
    K/V) appended and decoded in one launch.  The oracle checks three sampled layers in full;
    every layer's new rows are checked in the pool."""
    sample = (0, 13, 31)
    c = C.build_layers("llama3_8b_32l", host_layers=sample)
    out = C.gpu_layers(c, True)
    assert torch.isfinite(out.float()).all()
    for i, l in enumerate(sample):
        ref, _, _ = C.oracle_layer(c, l, i, True)
        C.tol_check(C.bf16_to_f64(out[l]), ref)
    # the new token's K/V rows landed in every layer (bit copies for a bf16 pool)
    slots = torch.from_numpy(c.slots).cuda()
    blk, off = slots // 16, slots % 16
    for l in range(c.w.layers):
        got_k = c.key_cache[l][blk, :, off, :]                     # [B, Hkv, D]
        got_v = c.value_cache[l][blk, :, off, :]
        assert torch.equal(got_k.view(torch.int16), c.k_new[l].view(torch.int16))
        assert torch.equal(got_v.view(torch.int16), c.v_new[l].view(torch.int16))
