"""Chunked-context (prefill) attention over the paged pool: oracle pins on the CPU, then the
CUDA kernel against the oracle on the GPU."""
import math

import numpy as np
import pytest

import oracle


KV_CODE = {"bf16": 0, "fp8_e4m3": 1, "int8": 2}  # the oracle pool's element code


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


@pytest.mark.parametrize("code", [1, 2])
def test_prefill_rows_equal_decode_on_one_byte_pools(code):
    """On FP8 and INT8 pools too, a prefill row is the decode definition over the context ending
    at its position: the same dequantised K/V (code x the (block, head) scale) and the same
    softmax, so the two oracle paths give identical values."""
    rng = np.random.default_rng(40 + code)
    bs, Hkv, G, D, L = 16, 2, 4, 64, 70
    Hq = Hkv * G
    a, pool, tables, _, _ = _build(rng, [L], bs, Hkv, D, fp8=code)
    assert np.any(pool.scales != 0) and np.any(pool.scales != 1)
    q = _bf16_bits(rng.standard_normal((L, Hq, D)))
    whole = pool.prefill_attention(q, np.array([0, L], np.int32), tables, np.array([L], np.int32), Hq, 0.125)
    for i in (0, 15, 16, 47, 69):
        dec = pool.attention(q[i:i + 1], tables, np.array([i + 1], np.int32), Hq, 0.125)
        assert np.array_equal(dec[0], whole[i])


def test_prefill_rejects_chunk_longer_than_context():
    rng = np.random.default_rng(5)
    a, pool, tables, _, _ = _build(rng, [10], 16, 1, 64)
    q = _bf16_bits(rng.standard_normal((11, 1, 64)))
    with pytest.raises(RuntimeError):
        pool.prefill_attention(q, np.array([0, 11], np.int32), tables, np.array([10], np.int32), 1, 0.1)


# ----------------------------------------------------------------------------- GPU parity
def _gpu():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_266_gb300 import build
    build.build()
    import paged_kv_cache_266_gb300 as pkv
    return torch, pkv


def _oracle_replay(sc, threads=8):
    """The oracle's pool after the same appends, the tables, and the prefill outputs."""
    a = oracle.Allocator(sc.num_blocks, sc.block_size)
    a.set_free_order(sc.free_order)
    pool = oracle.Pool(sc.num_blocks, sc.block_size, sc.Hkv, sc.D, KV_CODE[sc.kv_dtype])
    for b in range(sc.B):
        assert a.reserve(b, int(sc.ctx[b])) == 0
    for b in range(sc.B):
        if sc.past[b]:
            k, v = sc.kv(b, 0, int(sc.past[b]))
            pool.append(k, v, a.slot_mapping([b] * int(sc.past[b]), np.arange(int(sc.past[b]))))
    seqs, pos = sc.chunk_slots_positions()
    k, v = sc.chunk_kv()
    pool.append(k, v, a.slot_mapping(seqs, pos))
    tables = a.block_tables(list(range(sc.B)), sc.max_blocks)
    out = pool.prefill_attention(sc.query(), sc.cu_q, tables, sc.ctx, sc.Hq, 1 / math.sqrt(sc.D), threads=threads)
    return pool, tables, out


def _check_close(got_bits, ref):
    got = oracle.bf16_bits_to_f64(got_bits)
    err = np.abs(got - ref)
    assert err.max() <= 1e-2, err.max()
    assert err.mean() <= 1e-3, err.mean()


def _check_close_one_byte(got_bits, ref):
    """One-byte pools: a row led by one key returns code x scale, generally not a bf16 value, so
    the output's own rounding (half a bf16 ulp, <= 2^-8 relative) is part of the bound; the
    arithmetic adds the widened K/V and P, each rounded once to f16 (<= 2^-12 relative), which
    for these values (|V| < 5) stays below 4e-3."""
    got = oracle.bf16_bits_to_f64(got_bits)
    err = np.abs(got - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 4e-3
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), (float(err[worst]), float(ref[worst]), float(got[worst]))
    assert err.mean() <= 1e-3, err.mean()


@pytest.mark.gpu
@pytest.mark.parametrize("bs,G,D", [(16, 4, 128), (64, 4, 128), (64, 1, 128), (16, 8, 128), (128, 2, 128),
                                    (32, 16, 128), (16, 4, 64), (64, 1, 64), (64, 8, 64), (32, 16, 64),
                                    (128, 2, 64)])
def test_prefill_matches_oracle(bs, G, D):
    """Chunks at the start of a prompt, of one token, ending on a block boundary, spanning
    several KV tiles and query tiles with ragged ends; pool bytes bit-exact after the append.
    Head dims 128 and 64 (7B/8B/70B layers use 128; 64 is the other size the pool supports)."""
    torch, pkv = _gpu()
    import pkv_workloads as W
    from paged_kv_cache_266_gb300.runner import PrefillStep, _wrap_device
    sc = W.make_prefill_script(71 + bs + G + D, Hq=2 * G, Hkv=2, D=D, block_size=bs,
                               past=[0, 5, 64, 100, 250, 31, 0], chunk=[37, 1, 64, 150, 3, 200, 129])
    st = PrefillStep(sc)
    st.step()
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_error(st.pool.handle) == pkv.PKV_OK
    opool, tables, ref = _oracle_replay(sc)
    assert np.array_equal(st.tables_host, tables)
    kv_ptr, kv_bytes, _, _ = pkv.pkv_pool_raw(st.pool.handle)
    assert np.array_equal(_wrap_device(kv_ptr, kv_bytes).cpu().numpy(), opool.data)
    _check_close(st.out_host(), ref)
    st.close()


@pytest.mark.gpu
@pytest.mark.parametrize("kv", ["fp8_e4m3", "int8"])
@pytest.mark.parametrize("bs,G,D", [(16, 4, 128), (64, 4, 128), (128, 1, 128), (32, 16, 128), (16, 8, 64),
                                    (64, 2, 64)])
def test_prefill_one_byte_pools_match_oracle(kv, bs, G, D):
    """FP8 and INT8 pools: the codes are widened on chip (code x scale, to f16 with a power of two
    per sequence and head), q goes to f16 exactly and P is f16.  Pool bytes and scales bit-exact
    after the append; outputs within the one-byte bound of the oracle's exact dequantisation."""
    torch, pkv = _gpu()
    import pkv_workloads as W
    from paged_kv_cache_266_gb300.runner import PrefillStep, _wrap_device
    sc = W.make_prefill_script(171 + bs + G + D, Hq=2 * G, Hkv=2, D=D, block_size=bs, kv_dtype=kv,
                               past=[0, 5, 64, 100, 250, 31, 0], chunk=[37, 1, 64, 150, 3, 200, 129])
    st = PrefillStep(sc)
    st.step()
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_error(st.pool.handle) == pkv.PKV_OK
    opool, tables, ref = _oracle_replay(sc)
    assert np.array_equal(st.tables_host, tables)
    kv_ptr, kv_bytes, sc_ptr, sc_bytes = pkv.pkv_pool_raw(st.pool.handle)
    assert np.array_equal(_wrap_device(kv_ptr, kv_bytes).cpu().numpy(), opool.data)
    assert np.array_equal(_wrap_device(sc_ptr, sc_bytes).cpu().numpy().view(np.float32), opool.scales)
    _check_close_one_byte(st.out_host(), ref)
    st.close()


@pytest.mark.gpu
@pytest.mark.parametrize("kv", ["fp8_e4m3", "int8"])
def test_prefill_one_byte_pools_wide_range(kv):
    """Blocks whose K reach 2^17 and V 2^18 (past the f16 range, so the widened tiles must be
    rescaled by the sequence's power of two) beside blocks at 2^-10, with queries at 2^-17 (so q
    itself needs its own power of two to reach the f16 range): every output within 1e-2 (max)
    and 1e-3 (mean) of the largest |V| of its head, against the oracle."""
    torch, pkv = _gpu()
    rng = np.random.default_rng(7 if kv == "int8" else 8)
    bs, Hkv, G, D = 16, 2, 4, 128
    Hq = Hkv * G
    lens, chunk = [150, 61], [40, 61]
    nb = sum(-(-L // bs) for L in lens) + 2
    code = KV_CODE[kv]
    pool = pkv.KVPool(nb, bs, Hkv, D, {1: pkv.PKV_KV_FP8_E4M3, 2: pkv.PKV_KV_INT8}[code])
    a = pool.allocator
    order = rng.permutation(nb).astype(np.int32)
    pkv.pkv_allocator_set_free_order(a, order)
    oa, op = oracle.Allocator(nb, bs), oracle.Pool(nb, bs, Hkv, D, code)
    oa.set_free_order(order)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    vmax = np.zeros((len(lens), Hkv))
    for b, L in enumerate(lens):
        pkv.pkv_seq_reserve(a, b, L)
        oa.reserve(b, L)
        kexp = rng.choice([-10, 0, 17], size=-(-L // bs))
        vexp = rng.choice([-10, 0, 18], size=-(-L // bs))
        tok_blk = np.arange(L) // bs
        kf = rng.standard_normal((L, Hkv, D)) * np.exp2(kexp[tok_blk])[:, None, None]
        vf = rng.standard_normal((L, Hkv, D)) * np.exp2(vexp[tok_blk])[:, None, None]
        k, v = _bf16_bits(kf), _bf16_bits(vf)
        vmax[b] = np.abs(oracle.bf16_bits_to_f64(v)).max(axis=(0, 2))
        slots = pkv.pkv_slot_mapping(a, [b] * L, np.arange(L))
        pkv.pkv_append(pool.handle, dev(k), dev(v), torch.from_numpy(slots).cuda())
        op.append(k, v, slots)
    cu = np.concatenate([[0], np.cumsum(chunk)]).astype(np.int32)
    q = _bf16_bits(rng.standard_normal((int(cu[-1]), Hq, D)) * 2.0 ** -17)
    mb = max(-(-L // bs) for L in lens)
    tables = pkv.pkv_get_block_tables(a, np.arange(len(lens)), mb)
    out = torch.zeros(int(cu[-1]), Hq, D, dtype=torch.bfloat16, device="cuda")
    pkv.pkv_prefill_attention(pool.handle, dev(q), torch.from_numpy(cu).cuda(), max(chunk),
                              torch.from_numpy(tables).cuda(), torch.tensor(lens, dtype=torch.int32).cuda(),
                              1 / math.sqrt(D), out)
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_error(pool.handle) == pkv.PKV_OK
    ref = op.prefill_attention(q, cu, oa.block_tables(list(range(len(lens))), mb), np.array(lens, np.int32), Hq,
                               1 / math.sqrt(D))
    got = oracle.bf16_bits_to_f64(out.view(torch.int16).cpu().numpy().view(np.uint16))
    assert np.all(np.isfinite(got))
    for b in range(len(lens)):
        for h in range(Hkv):
            err = np.abs(got[cu[b]:cu[b + 1], h * G:(h + 1) * G] - ref[cu[b]:cu[b + 1], h * G:(h + 1) * G])
            assert err.max() <= 1e-2 * vmax[b, h] and err.mean() <= 1e-3 * vmax[b, h], (b, h, err.max(), vmax[b, h])
    pool.close()


@pytest.mark.gpu
@pytest.mark.parametrize("B", [512, 600])
def test_prefill_many_sequences_matches_oracle(B):
    """Many small chunks in one call: 512 sequences (the largest batch the kernel dispatches in
    order of causal work) and 600 (beyond it: index order); chunks of 1-3 tokens over pasts of
    0-79 tokens, every output against the oracle."""
    torch, pkv = _gpu()
    import pkv_workloads as W
    from paged_kv_cache_266_gb300.runner import PrefillStep
    rng = np.random.default_rng(B)
    sc = W.make_prefill_script(90 + B, Hq=8, Hkv=2, D=128, block_size=16,
                               past=rng.integers(0, 80, B).tolist(), chunk=rng.integers(1, 4, B).tolist())
    st = PrefillStep(sc)
    st.step()
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_error(st.pool.handle) == pkv.PKV_OK
    _, tables, ref = _oracle_replay(sc)
    assert np.array_equal(st.tables_host, tables)
    _check_close(st.out_host(), ref)
    st.close()


@pytest.mark.gpu
def test_prefill_fused_step_equals_separate_calls():
    torch, pkv = _gpu()
    import pkv_workloads as W
    from paged_kv_cache_266_gb300.runner import PrefillStep
    sc = W.make_prefill_script(80, B=4, Hq=16, Hkv=4, block_size=64, past_hi=700, chunk_lo=1, chunk_hi=300)
    st = PrefillStep(sc)
    st.step()
    torch.cuda.synchronize()
    fused = st.out_host()
    st.out.zero_()
    st.append()
    st.attention()
    torch.cuda.synchronize()
    assert np.array_equal(st.out_host(), fused)
    # deterministic: the same call again gives the same bits
    st.attention()
    torch.cuda.synchronize()
    assert np.array_equal(st.out_host(), fused)
    st.close()


@pytest.mark.gpu
def test_prefill_full_size_sampled():
    """8 sequences at seeded points of 32K prompts, 512-token chunks, Llama-3-8B layer shapes,
    block 64 (the measured configuration): sampled query rows against dense attention over the
    regenerated K/V of their sequence."""
    torch, pkv = _gpu()
    import pkv_workloads as W
    from paged_kv_cache_266_gb300.runner import PrefillStep
    sc = W.make_prefill_script()
    st = PrefillStep(sc)
    st.step()
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_error(st.pool.handle) == pkv.PKV_OK
    got = st.out_host()
    scale = 1 / math.sqrt(sc.D)
    for b in range(sc.B):
        P = int(sc.past[b])
        k, v = sc.kv(b, 0, int(sc.ctx[b]))
        K, V = oracle.bf16_bits_to_f64(k), oracle.bf16_bits_to_f64(v)
        for i in (0, 1, 130, int(sc.chunk[b]) - 1):
            row = int(sc.cu_q[b]) + i
            q = oracle.bf16_bits_to_f64(sc.query(row, row + 1)[0])
            for h in (0, sc.Hkv - 1):
                ref = oracle.dense_attention(q[h * sc.G:(h + 1) * sc.G], K[:P + i + 1, h], V[:P + i + 1, h], scale)
                err = np.abs(oracle.bf16_bits_to_f64(got[row, h * sc.G:(h + 1) * sc.G]) - ref)
                assert err.max() <= 1e-2 and err.mean() <= 1e-3, (b, i, h, err.max())
    st.close()


@pytest.mark.gpu
def test_prefill_rejects_unsupported_and_flags_bounds():
    torch, pkv = _gpu()
    dev = "cuda"
    q = torch.zeros(4, 6, 128, dtype=torch.bfloat16, device=dev)
    out = torch.zeros_like(q)
    cu = torch.tensor([0, 4], dtype=torch.int32, device=dev)
    tables = torch.zeros(1, 1, dtype=torch.int32, device=dev)
    ctx = torch.tensor([4], dtype=torch.int32, device=dev)
    pool = pkv.KVPool(4, 16, 2, 128, pkv.PKV_KV_BF16)
    with pytest.raises(pkv.PKVError):  # 6 query heads over 2 KV heads: 3 per group
        pkv.pkv_prefill_attention(pool.handle, q, cu, 4, tables, ctx, 0.1, out)
    q8 = torch.zeros(4, 8, 128, dtype=torch.bfloat16, device=dev)
    out8 = torch.zeros_like(q8)
    long_ctx = torch.tensor([40], dtype=torch.int32, device=dev)  # beyond 1 block of 16
    pkv.pkv_prefill_attention(pool.handle, q8, cu, 4, tables, long_ctx, 0.1, out8)
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_error(pool.handle) == pkv.PKV_ERR_BOUNDS
    short_ctx = torch.tensor([3], dtype=torch.int32, device=dev)  # chunk of 4 in a context of 3
    pkv.pkv_prefill_attention(pool.handle, q8, cu, 4, tables, short_ctx, 0.1, out8)
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_error(pool.handle) == pkv.PKV_ERR_BOUNDS
    bad_tab = torch.tensor([[7]], dtype=torch.int32, device=dev)  # block id outside a 4-block pool
    pkv.pkv_prefill_attention(pool.handle, q8, cu, 4, bad_tab, ctx, 0.1, out8)
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_error(pool.handle) == pkv.PKV_ERR_BOUNDS
    pkv.pkv_prefill_attention(pool.handle, q8, cu, 0, tables, ctx, 0.1, out8)  # max_q_len 0: nothing launched
    pool.close()
    fp8 = pkv.KVPool(4, 16, 2, 128, pkv.PKV_KV_FP8_E4M3)  # the one-byte path flags a bad block id too
    pkv.pkv_prefill_attention(fp8.handle, q8, cu, 4, bad_tab, ctx, 0.1, out8)
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_error(fp8.handle) == pkv.PKV_ERR_BOUNDS
    fp8.close()


@pytest.mark.gpu
def test_chunked_prefill_with_rope_matches_oracle():
    """A chunk's K and queries rotated by pkv_append_rope at their positions (which also appends
    the chunk's K/V), then the prefill attention: against the oracle's rotate-then-attend."""
    torch, pkv = _gpu()
    import pkv_workloads as W
    sc = W.make_prefill_script(90, Hq=8, Hkv=2, D=128, block_size=16, past=[33, 0, 100], chunk=[20, 65, 1])
    base = 10000.0
    pool = pkv.KVPool(sc.num_blocks, sc.block_size, sc.Hkv, sc.D)
    a = pool.allocator
    pkv.pkv_allocator_set_free_order(a, sc.free_order)
    oa = oracle.Allocator(sc.num_blocks, sc.block_size)
    oa.set_free_order(sc.free_order)
    op = oracle.Pool(sc.num_blocks, sc.block_size, sc.Hkv, sc.D, False)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    for b in range(sc.B):
        pkv.pkv_seq_reserve(a, b, int(sc.ctx[b]))
        oa.reserve(b, int(sc.ctx[b]))
    # the past, already rotated (as a previous chunk's append would have left it)
    for b in range(sc.B):
        P = int(sc.past[b])
        if P:
            k, v = sc.kv(b, 0, P)
            kr = oracle.rope(k, np.arange(P), base)
            slots = pkv.pkv_slot_mapping(a, [b] * P, np.arange(P))
            pkv.pkv_append(pool.handle, dev(kr), dev(v), torch.from_numpy(slots).cuda())
            op.append(kr, v, slots)
    seqs, pos = sc.chunk_slots_positions()
    k, v = sc.chunk_kv()
    q = sc.query()
    slots = pkv.pkv_slot_mapping(a, seqs, pos)
    kd, qd = dev(k), dev(q)
    pkv.pkv_append_rope(pool.handle, kd, dev(v), torch.from_numpy(slots).cuda(), torch.from_numpy(pos).cuda(), base,
                        q=qd)
    tables = pkv.pkv_get_block_tables(a, list(range(sc.B)), sc.max_blocks)
    out = torch.empty(int(sc.cu_q[-1]), sc.Hq, sc.D, dtype=torch.bfloat16, device="cuda")
    pkv.pkv_prefill_attention(pool.handle, qd, torch.from_numpy(sc.cu_q).cuda(), int(sc.chunk.max()),
                              torch.from_numpy(tables).cuda(), torch.from_numpy(sc.ctx).cuda(), 1 / math.sqrt(sc.D), out)
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_error(pool.handle) == pkv.PKV_OK
    kr, qr = oracle.rope(k, pos, base), oracle.rope(q, pos, base)
    assert np.array_equal(kd.view(torch.int16).cpu().numpy().view(np.uint16), kr)
    op.append(kr, v, slots)
    ref = op.prefill_attention(qr, sc.cu_q, tables, sc.ctx, sc.Hq, 1 / math.sqrt(sc.D))
    _check_close(out.view(torch.int16).cpu().numpy().view(np.uint16), ref)
    pool.close()


@pytest.mark.gpu
@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3", "int8"])
def test_prefill_bounded_waits_report_timeout_and_leave_the_context_usable(stall_hooks, kv):
    """Every mbarrier wait in the prefill kernel is bounded. With the test hooks each K/V stage
    (each code stage on one-byte pools) expects bytes no copy delivers and the waits give up after
    20 ms: the call reports PKV_ERR_TIMEOUT without a fault, tensor memory is released, and the next
    normal call gives the same bits as before."""
    torch, pkv = _gpu()
    import pkv_workloads as W
    from paged_kv_cache_266_gb300.runner import PrefillStep
    sc = W.make_prefill_script(91, B=3, Hq=8, Hkv=2, block_size=64, past=[300, 0, 40], chunk=[200, 90, 17],
                               kv_dtype=kv)
    st = PrefillStep(sc)
    st.step()
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_error(st.pool.handle) == pkv.PKV_OK
    good = st.out_host().copy()
    stall_hooks[0]()
    st.attention()
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_error(st.pool.handle) == pkv.PKV_ERR_TIMEOUT
    stall_hooks[1]()
    st.out.zero_()
    st.attention()
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_error(st.pool.handle) == pkv.PKV_OK
    assert np.array_equal(st.out_host(), good)
    st.close()
