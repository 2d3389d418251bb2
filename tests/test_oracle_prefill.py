"""Pins of the oracle's paged prefill (CPU).

The definition ("理解 KV Cache" §1.2): Attention(Q, K, V) = softmax(Q K^T / sqrt(d_k) + M) V
with the causal mask M (-inf above the diagonal) over the whole n x n score matrix; prefill
computes all prompt rows at once (§2.1); GQA query heads share KV head h = hq // g ("KV Cache
与推理优化").  The oracle instead runs one decode query per prompt row over the paged cache,
so these tests compare it with the dense masked formula written out in numpy fp64, with torch's
own causal SDPA, and with itself across chunk boundaries."""
import numpy as np
import pytest
import torch

import oracle
import workloads


def _case(lens_ctx, chunks, Hq=8, Hkv=2, D=32, seed=0, nb_extra=5):
    """Paged pools holding each sequence's context + chunk, in shuffled blocks."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = [c + p for c, p in zip(lens_ctx, chunks)]
    nblk = sum(oracle.blocks_needed(L, 16) for L in lens)
    nb = nblk + nb_extra
    a = oracle.BlockAllocator(nb, rng.permutation(nb))
    mb = max(oracle.blocks_needed(L, 16) for L in lens)
    t = oracle.build_block_tables(a, lens, mb)
    kc = np.full((nb, Hkv, 16, D), 0x7FC0, np.uint16)
    vc = kc.copy()
    K = [workloads.bf16_bits(workloads.randn_bf16((L, Hkv, D), seed * 10 + b + 1)) for b, L in enumerate(lens)]
    V = [workloads.bf16_bits(workloads.randn_bf16((L, Hkv, D), seed * 10 + b + 101)) for b, L in enumerate(lens)]
    for b, L in enumerate(lens):
        assert oracle.kv_append(K[b], V[b], oracle.all_slots(t[b:b + 1], [L]), kc, vc) == 0
    cu = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    q = workloads.bf16_bits(workloads.randn_bf16((int(cu[-1]), Hq, D), seed * 10 + 999))
    return dict(t=t, kc=kc, vc=vc, K=K, V=V, q=q, cu=cu, lens=np.array(lens, np.int32),
                ctx=lens_ctx, chunks=chunks, Hq=Hq, Hkv=Hkv, D=D)


def _f64(bits):
    return bits.astype(np.uint32).__lshift__(16).view(np.float32).astype(np.float64)


def _dense(c, scale):
    """softmax(Q K^T * scale + M) V per sequence and head, the full masked matrix."""
    out = np.zeros(c["q"].shape, np.float64)
    g = c["Hq"] // c["Hkv"]
    for b, (C, P) in enumerate(zip(c["ctx"], c["chunks"])):
        L = C + P
        Q = _f64(c["q"][c["cu"][b]:c["cu"][b + 1]])          # [P, Hq, D]
        K, V = _f64(c["K"][b]), _f64(c["V"][b])              # [L, Hkv, D]
        # row i of the chunk is position C + i; M[i, j] = -inf for j > C + i
        M = np.where(np.arange(L)[None, :] > (C + np.arange(P))[:, None], -np.inf, 0.0)
        for hq in range(c["Hq"]):
            S = Q[:, hq, :] @ K[:, hq // g, :].T * scale + M
            W = np.exp(S - S.max(axis=1, keepdims=True))
            W /= W.sum(axis=1, keepdims=True)
            out[c["cu"][b]:c["cu"][b + 1], hq, :] = W @ V[:, hq // g, :]
    return out


@pytest.mark.parametrize("ctx,chunks", [([0], [37]), ([0, 0, 0], [16, 1, 50]),
                                        ([20, 0, 71], [33, 64, 5]), ([128], [1])])
def test_prefill_equals_the_dense_masked_softmax(ctx, chunks):
    c = _case(ctx, chunks, seed=len(ctx) + sum(chunks))
    scale = float(np.float32(1 / np.sqrt(c["D"])))
    st, out = oracle.paged_prefill(c["q"], c["kc"], c["vc"], c["t"], c["lens"], c["cu"], scale, c["Hkv"])
    assert st == 0
    np.testing.assert_allclose(out, _dense(c, scale), rtol=1e-12, atol=1e-12)


def test_prefill_equals_torch_causal_sdpa():
    c = _case([0, 0], [40, 23], Hq=12, Hkv=3, seed=7)
    scale = float(np.float32(1 / np.sqrt(c["D"])))
    st, out = oracle.paged_prefill(c["q"], c["kc"], c["vc"], c["t"], c["lens"], c["cu"], scale, c["Hkv"])
    assert st == 0
    g = c["Hq"] // c["Hkv"]
    for b in range(2):
        Q = torch.from_numpy(_f64(c["q"][c["cu"][b]:c["cu"][b + 1]])).permute(1, 0, 2)   # [Hq, P, D]
        K = torch.from_numpy(_f64(c["K"][b])).permute(1, 0, 2).repeat_interleave(g, 0)
        V = torch.from_numpy(_f64(c["V"][b])).permute(1, 0, 2).repeat_interleave(g, 0)
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, is_causal=True, scale=scale)
        np.testing.assert_allclose(out[c["cu"][b]:c["cu"][b + 1]], ref.permute(1, 0, 2).numpy(),
                                   rtol=1e-10, atol=1e-10)


def test_chunked_prefill_equals_the_whole_prompt():
    """Prefill of a chunk after C cached positions gives exactly rows C.. of the prefill of
    the whole prompt (same pool, same q rows)."""
    c = _case([0], [90], seed=3)
    scale = float(np.float32(1 / np.sqrt(c["D"])))
    st, whole = oracle.paged_prefill(c["q"], c["kc"], c["vc"], c["t"], c["lens"], c["cu"], scale, c["Hkv"])
    assert st == 0
    for C in (1, 16, 47, 89):
        st, part = oracle.paged_prefill(c["q"][C:], c["kc"], c["vc"], c["t"], c["lens"],
                                        np.array([0, 90 - C], np.int32), scale, c["Hkv"])
        assert st == 0
        np.testing.assert_array_equal(part, whole[C:])


def test_a_dropped_mask_is_caught():
    """Planted mistake: attending over the whole prompt (no causal mask) differs."""
    c = _case([0], [24], seed=5)
    scale = float(np.float32(1 / np.sqrt(c["D"])))
    st, out = oracle.paged_prefill(c["q"], c["kc"], c["vc"], c["t"], c["lens"], c["cu"], scale, c["Hkv"])
    st2, nomask = oracle.paged_decode(c["q"], c["kc"], c["vc"], np.repeat(c["t"], 24, 0),
                                      np.full(24, 24, np.int32), scale, c["Hkv"])
    assert not np.allclose(out[:-1], nomask[:-1])
    np.testing.assert_array_equal(out[-1], nomask[-1])       # the last row sees everything
