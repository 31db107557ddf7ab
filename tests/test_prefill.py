"""Chunked-context (prefill) attention over the paged pool: oracle pins on the CPU, then the
CUDA kernel against the oracle on the GPU."""
import math

import numpy as np
import pytest

import oracle


def _bf16_bits(x):
    import torch
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _build(rng, lens, bs, Hkv, D, fp8=False, K=None, V=None):
    """Oracle pool holding one sequence per entry of lens (random bf16 K/V unless given)."""
    nb = sum(-(-L // bs) for L in lens) + 3
    a, pool = oracle.Allocator(nb, bs), oracle.Pool(nb, bs, Hkv, D, fp8)
    a.set_free_order(rng.permutation(nb).astype(np.int32))
    Ks, Vs = [], []
    for b, L in enumerate(lens):
        assert a.reserve(b, L) == 0
        k = K[b] if K is not None else _bf16_bits(rng.standard_normal((L, Hkv, D)))
        v = V[b] if V is not None else _bf16_bits(rng.standard_normal((L, Hkv, D)))
        pool.append(k, v, a.slot_mapping([b] * L, np.arange(L)))
        Ks.append(oracle.bf16_bits_to_f64(k))
        Vs.append(oracle.bf16_bits_to_f64(v))
    mb = max(-(-L // bs) for L in lens)
    return a, pool, a.block_tables(list(range(len(lens))), mb), Ks, Vs


def test_prefill_matches_torch_sdpa_with_causal_mask():
    """Chunks at the start of a sequence, in its middle and at its end, GQA 4:1, against torch
    scaled_dot_product_attention in fp64 with the mask 'key position <= query position'."""
    import torch
    rng = np.random.default_rng(1)
    bs, Hkv, G, D = 16, 2, 4, 64
    Hq = Hkv * G
    ctx = [40, 77, 33]
    qn = [40, 20, 1]  # whole prompt, a middle chunk's view (chunk ends at ctx), one token
    a, pool, tables, Ks, Vs = _build(rng, ctx, bs, Hkv, D)
    cu = np.concatenate([[0], np.cumsum(qn)]).astype(np.int32)
    q = _bf16_bits(rng.standard_normal((int(cu[-1]), Hq, D)))
    out = pool.prefill_attention(q, cu, tables, np.array(ctx, np.int32), Hq, 0.125)
    qd = oracle.bf16_bits_to_f64(q)
    for b in range(3):
        L, n = ctx[b], qn[b]
        qb = torch.from_numpy(qd[cu[b]:cu[b + 1]]).permute(1, 0, 2)  # [Hq][n][D]
        kb = torch.from_numpy(Ks[b]).permute(1, 0, 2).repeat_interleave(G, 0)
        vb = torch.from_numpy(Vs[b]).permute(1, 0, 2).repeat_interleave(G, 0)
        qpos = torch.arange(L - n, L)[:, None]
        mask = torch.arange(L)[None, :] <= qpos
        ref = torch.nn.functional.scaled_dot_product_attention(qb, kb, vb, attn_mask=mask, scale=0.125)
        np.testing.assert_allclose(out[cu[b]:cu[b + 1]], ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-13)


def test_prefill_equal_keys_gives_prefix_means():
    """All keys equal: the softmax is uniform over the attended tokens, so query i of a chunk
    returns the mean of V over positions 0..p (p its position) — catches an off-by-one in the
    causal bound or the chunk offset."""
    rng = np.random.default_rng(2)
    bs, Hkv, D, L, n = 16, 1, 64, 50, 23
    krow = _bf16_bits(rng.standard_normal((1, Hkv, D)))
    K = [np.repeat(krow, L, axis=0)]
    a, pool, tables, Ks, Vs = _build(rng, [L], bs, Hkv, D, K=K)
    q = _bf16_bits(rng.standard_normal((n, 2, D)))
    out = pool.prefill_attention(q, np.array([0, n], np.int32), tables, np.array([L], np.int32), 2, 0.3)
    for i in range(n):
        p = L - n + i
        want = Vs[0][:p + 1, 0].mean(0)
        np.testing.assert_allclose(out[i, 0], want, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(out[i, 1], want, rtol=1e-12, atol=1e-13)


def test_prefill_brute_force_tiny():
    """Pure-Python softmax over explicit loops (block 4, D 8, GQA 2:1)."""
    rng = np.random.default_rng(3)
    bs, Hkv, G, D = 4, 1, 2, 8
    L, n = 11, 5
    nb = 4
    a, pool = oracle.Allocator(nb, bs), oracle.Pool(nb, bs, Hkv, D, False)
    assert a.reserve(0, L) == 0
    k = _bf16_bits(rng.standard_normal((L, Hkv, D)))
    v = _bf16_bits(rng.standard_normal((L, Hkv, D)))
    pool.append(k, v, a.slot_mapping([0] * L, np.arange(L)))
    q = _bf16_bits(rng.standard_normal((n, G, D)))
    out = pool.prefill_attention(q, np.array([0, n], np.int32), a.block_tables([0], 3), np.array([L], np.int32), G, 0.5)
    kf, vf, qf = (oracle.bf16_bits_to_f64(x) for x in (k, v, q))
    for i in range(n):
        p = L - n + i
        for j in range(G):
            s = [0.5 * sum(qf[i, j, d] * kf[t, 0, d] for d in range(D)) for t in range(p + 1)]
            m = max(s)
            w = [math.exp(x - m) for x in s]
            tot = sum(w)
            for d in range(D):
                want = sum(w[t] * vf[t, 0, d] for t in range(p + 1)) / tot
                assert abs(out[i, j, d] - want) <= 1e-12 * max(1.0, abs(want))


def test_prefill_rows_equal_decode_and_chunks_compose():
    """Every prefill row equals decode attention over a context ending at its position, and a
    prompt processed as chunks (each attending to everything before it) gives the rows of the
    single whole-prompt prefill."""
    rng = np.random.default_rng(4)
    bs, Hkv, G, D, L = 16, 2, 2, 64, 90
    Hq = Hkv * G
    a, pool, tables, _, _ = _build(rng, [L], bs, Hkv, D)
    q = _bf16_bits(rng.standard_normal((L, Hq, D)))
    whole = pool.prefill_attention(q, np.array([0, L], np.int32), tables, np.array([L], np.int32), Hq, 0.125)
    for i in (0, 1, 15, 16, 17, 63, 64, 89):
        dec = pool.attention(q[i:i + 1], tables, np.array([i + 1], np.int32), Hq, 0.125)
        assert np.array_equal(dec[0], whole[i])
    for c0, c1 in ((0, 30), (30, 64), (64, 65), (65, 90)):
        part = pool.prefill_attention(q[c0:c1], np.array([0, c1 - c0], np.int32), tables, np.array([c1], np.int32),
                                      Hq, 0.125)
        assert np.array_equal(part, whole[c0:c1])


def test_prefill_rejects_chunk_longer_than_context():
    rng = np.random.default_rng(5)
    a, pool, tables, _, _ = _build(rng, [10], 16, 1, 64)
    q = _bf16_bits(rng.standard_normal((11, 1, 64)))
    with pytest.raises(RuntimeError):
        pool.prefill_attention(q, np.array([0, 11], np.int32), tables, np.array([10], np.int32), 1, 0.1)
