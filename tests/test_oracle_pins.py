"""Pins for the CPU oracle: each check ties it to something other than itself —
worked values printed on the pages, the OCP E4M3 table, library routines
(torch's CPU float8 conversion and scaled_dot_product_attention in fp64),
closed forms, special cases and invariants."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import oracle.drive as odrive
import pkv_workloads as W
from boundary_rows import near_boundary_rows

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _bf16_bits(x):
    """float -> bf16 bit patterns via torch (round to nearest even)."""
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# ----------------------------------------------------------------------------- KV memory formula
def test_m_kv_worked_values():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "kv_memory.txt")) if l.strip() and not l.startswith("#")]
    for r in rows:
        *args, expected = r
        assert oracle.m_kv(*[float(a) for a in args]) == float(expected)


def test_m_kv_capacity_reading():
    # ~30 GB holds ~1e5 tokens (FP16) / ~2e5 (FP8) at 327680 / 163840 bytes per token: the GiB reading
    # gives 98304 / 196608 tokens, within 2% of the round numbers the page prints.
    per_tok16 = oracle.m_kv(80, 8, 128, 1, 1, 2)
    per_tok8 = oracle.m_kv(80, 8, 128, 1, 1, 1)
    assert 30 * 2**30 / per_tok16 == 98304
    assert 30 * 2**30 / per_tok8 == 196608
    assert abs(98304 - 1e5) / 1e5 < 0.02 and abs(196608 - 2e5) / 2e5 < 0.02


def test_m_kv_is_linear_in_each_factor():
    base = oracle.m_kv(2, 4, 64, 100, 3, 2)
    assert oracle.m_kv(4, 4, 64, 100, 3, 2) == 2 * base
    assert oracle.m_kv(2, 4, 64, 300, 3, 2) == 3 * base
    assert oracle.m_kv(2, 4, 64, 100, 3, 1) * 2 == base


# ----------------------------------------------------------------------------- E4M3 codec
def _golden_e4m3():
    out = []
    for line in open(os.path.join(GOLDEN, "e4m3_points.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        v, code, kind = line.split()
        out.append((float(eval(v, {"__builtins__": {}})), int(code, 16), kind))
    return out


def test_e4m3_golden_points():
    for v, code, kind in _golden_e4m3():
        if kind == "decode":
            assert oracle.e4m3_decode(code) == v, (v, hex(code))
            assert oracle.e4m3_encode(v) == code
        else:
            assert oracle.e4m3_encode(v) == code, (v, hex(code), hex(oracle.e4m3_encode(v)))
            assert oracle.e4m3_encode_array(np.array([v]), exhaustive=True)[0] == code
    assert math.isnan(oracle.e4m3_decode(0x7F)) and math.isnan(oracle.e4m3_decode(0xFF))


def test_e4m3_decode_matches_torch_float8_for_all_codes():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([oracle.e4m3_decode(c) for c in range(256)])
    assert np.array_equal(np.isnan(ref), np.isnan(mine))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], mine[ok])


def test_e4m3_grid_invariants():
    vals = np.array([oracle.e4m3_decode(c) for c in range(0x7F)])
    assert np.all(np.diff(vals) > 0)  # codes 0..126 increase strictly
    assert vals[-1] == 448.0 and vals[1] == 2.0 ** -9
    # spacing is constant inside a binade and doubles from one binade to the next
    for e in range(1, 15):
        seg = vals[8 * e: 8 * e + 9] if 8 * e + 9 <= len(vals) else vals[8 * e:]
        assert len(set(np.diff(seg[:8]))) == 1
    assert len(set(np.diff(vals[:9]))) == 1  # subnormals share the first normal binade's spacing


def test_e4m3_encode_matches_torch_in_range_and_exhaustive_search():
    rng = _rng(1)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 50,
        rng.standard_normal(5000).astype(np.float32) * 1e-3,
        (rng.uniform(-447.9, 447.9, 5000)).astype(np.float32),
    ])
    # exact midpoints between all neighbouring finite codes (ties)
    vals = np.array([oracle.e4m3_decode(c) for c in range(0x7F)])
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids, vals.astype(np.float32)])
    x = x[np.abs(x) < 448]
    ref = torch.tensor(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    fast = oracle.e4m3_encode_array(x)
    brute = oracle.e4m3_encode_array(x, exhaustive=True)
    assert np.array_equal(fast, brute)
    assert np.array_equal(fast, ref)


def test_e4m3_saturates_instead_of_overflowing():
    x = np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e6, 3e38, -500.0], dtype=np.float32)
    assert list(oracle.e4m3_encode_array(x)) == [0x7E] * 7 + [0xFE]


# ----------------------------------------------------------------------------- allocator
def test_allocator_golden_trace():
    lines = [l.rstrip("\n") for l in open(os.path.join(GOLDEN, "allocator_trace.txt")) if not l.startswith("#")]
    lines = [l for l in lines if l.strip()]
    a = oracle.Allocator(8, 16)
    ids = {}
    sid = lambda s: ids.setdefault(s, len(ids) + 100)
    for line in lines:
        lhs, rhs = [p.strip() for p in line.split("->")]
        parts = lhs.split()
        fields = [f.strip() for f in rhs.split("|")]
        if parts[0] == "reserve":
            rc = a.reserve(sid(parts[1]), int(parts[2]))
            assert rc == {"ok": 0, "oom": 2}[fields[0]], line
        elif parts[0] == "release":
            assert a.release(sid(parts[1])) == 0, line
        elif parts[0] == "slot":
            s = sid(parts[1])
            if fields[0] == "noseq":
                assert a.num_pages(s) == -1
            else:
                assert a.slot_mapping([s], [int(parts[2])])[0] == int(fields[0]), line
            continue
        if len(fields) > 1 and fields[1]:
            name, pages = fields[1].split(":")
            assert a.block_tables([sid(name.strip())], a.num_pages(sid(name.strip()))).tolist() == [
                [int(p) for p in pages.split()]], line
        assert a.free_list().tolist() == [int(p) for p in fields[2].split(":")[1].split()], line


def test_allocator_oom_is_atomic_and_conserves_blocks():
    a = oracle.Allocator(10, 16)
    assert a.reserve(1, 100) == 0  # 7 blocks
    before = a.free_list().tolist()
    assert a.reserve(2, 4 * 16 + 1) == 2  # needs 5, 3 free
    assert a.free_list().tolist() == before and a.num_pages(2) == -1
    assert a.reserve(1, 7 * 16 + 49) == 2  # 4 more blocks, 3 free: growth is refused too
    assert a.num_pages(1) == 7 and a.free_list().tolist() == before
    assert a.reserve(1, 7 * 16) == 0 and a.num_pages(1) == 7  # already has the capacity
    assert a.release(1) == 0 and a.num_free() == 10
    assert a.release(1) == 3


def test_allocator_churn_conserves_blocks():
    w = W.make_workload("c4")
    a = oracle.Allocator(w.num_blocks, w.block_size)
    assert a.set_free_order(w.free_order) == 0
    live = set()
    for i, op in enumerate(w.alloc_ops):
        if op[0] == "reserve":
            assert a.reserve(op[1], op[2]) == 0
            live.add(op[1])
        else:
            assert a.release(op[1]) == 0
            live.discard(op[1])
        if i % 97 == 0:
            held = sum(a.num_pages(s) for s in live)
            assert held + a.num_free() == w.num_blocks
    tables = a.block_tables(w.seq_ids, w.max_blocks())
    used = tables[tables >= 0]
    assert len(np.unique(used)) == len(used)  # no block handed out twice
    for b in range(w.B):
        assert (tables[b] >= 0).sum() == -(-int(w.attend_lens[b]) // w.block_size)


def test_slot_mapping_definition():
    a = oracle.Allocator(6, 4)
    a.set_free_order([5, 4, 3, 2, 1, 0])
    a.reserve(7, 10)  # pops 0, 1, 2
    assert a.block_tables([7], 3).tolist() == [[0, 1, 2]]
    pos = np.arange(10)
    assert a.slot_mapping([7] * 10, pos).tolist() == list(range(10))
    assert a.slot_mapping([7], [-1]).tolist() == [-1]


# ----------------------------------------------------------------------------- dense attention
def _sdpa(q, K, V, scale):
    """torch scaled_dot_product_attention in fp64 on the CPU: q [G][D], K/V [L][D]."""
    qt = torch.tensor(q)[None, :, None, :]  # [1, G, 1, D]
    Kt = torch.tensor(K)[None, None].expand(1, q.shape[0], *K.shape)
    Vt = torch.tensor(V)[None, None].expand(1, q.shape[0], *V.shape)
    return torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, scale=scale)[0, :, 0, :].numpy()


@pytest.mark.parametrize("L,G,D", [(1, 1, 8), (3, 2, 16), (40, 4, 64), (257, 8, 128)])
def test_dense_attention_matches_torch_sdpa(L, G, D):
    rng = _rng(L * 10 + G)
    q, K, V = rng.standard_normal((G, D)), rng.standard_normal((L, D)), rng.standard_normal((L, D))
    scale = 1 / math.sqrt(D)
    np.testing.assert_allclose(oracle.dense_attention(q, K, V, scale), _sdpa(q, K, V, scale), rtol=1e-12,
                               atol=1e-13)


def test_dense_attention_special_cases():
    rng = _rng(5)
    D = 16
    V = rng.standard_normal((9, D))
    q = rng.standard_normal((2, D))
    # one token: softmax of one element is 1
    assert np.array_equal(oracle.dense_attention(q, rng.standard_normal((1, D)), V[:1], 0.3), np.stack([V[0]] * 2))
    # identical keys: uniform weights, the mean of V
    K = np.tile(rng.standard_normal(D), (9, 1))
    np.testing.assert_allclose(oracle.dense_attention(q, K, V, 0.7), np.stack([V.mean(0)] * 2), rtol=1e-13,
                               atol=1e-14)
    # one-hot query with a huge scale selects the value of the key with the largest component
    K = rng.standard_normal((9, D))
    qh = np.zeros((1, D))
    qh[0, 3] = 1.0
    np.testing.assert_allclose(oracle.dense_attention(qh, K, V, 1e4)[0], V[np.argmax(K[:, 3])], atol=1e-12)
    # empty context gives zeros
    assert np.array_equal(oracle.dense_attention(q, np.zeros((0, D)), np.zeros((0, D)), 1.0), np.zeros((2, D)))


# ----------------------------------------------------------------------------- paged pool
def _paged_case(bs, Hkv, D, G, lens, order_seed, fp8=False, seed=0):
    """Build a pool through the oracle allocator + append; return (pool, tables, dense K/V, q)."""
    rng = _rng(seed)
    B = len(lens)
    need = sum(-(-L // bs) for L in lens)
    nb = need + 3
    alloc = oracle.Allocator(nb, bs)
    alloc.set_free_order(_rng(order_seed).permutation(nb).astype(np.int32))
    for b, L in enumerate(lens):
        alloc.reserve(b, L)
    max_blocks = max(1, max(-(-L // bs) for L in lens))
    tables = alloc.block_tables(np.arange(B), max_blocks)
    pool = oracle.Pool(nb, bs, Hkv, D, fp8)
    Ks, Vs = [], []
    for b, L in enumerate(lens):
        k = _bf16_bits(rng.standard_normal((L, Hkv, D)))
        v = _bf16_bits(rng.standard_normal((L, Hkv, D)))
        slots = alloc.slot_mapping([b] * L, np.arange(L))
        assert pool.append(k, v, slots) == 0
        Ks.append(k)
        Vs.append(v)
    q = _bf16_bits(rng.standard_normal((B, Hkv * G, D)))
    return pool, tables, Ks, Vs, q


@pytest.mark.parametrize("bs,G", [(16, 2), (64, 1), (16, 8)])
def test_paged_attention_equals_dense_over_unpaged_inputs(bs, G):
    lens = [1, 5, 16, 17, 70, 0]
    Hkv, D = 2, 64
    pool, tables, Ks, Vs, q = _paged_case(bs, Hkv, D, G, lens, order_seed=3)
    out = pool.attention(q, tables, np.array(lens), Hkv * G, 0.125)
    qd = oracle.bf16_bits_to_f64(q)
    for b, L in enumerate(lens):
        for h in range(Hkv):
            K = oracle.bf16_bits_to_f64(Ks[b][:, h, :])
            V = oracle.bf16_bits_to_f64(Vs[b][:, h, :])
            qq = qd[b, h * G:(h + 1) * G]  # contiguous grouping: query head j reads KV head j // G
            ref = _sdpa(qq, K, V, 0.125) if L else np.zeros((G, D))
            np.testing.assert_allclose(out[b, h * G:(h + 1) * G], ref, rtol=1e-12, atol=1e-13)


def test_paged_attention_invariant_to_block_ids_and_block_size():
    lens = [3, 33, 64, 100]
    outs = []
    for bs, order_seed in [(16, 1), (16, 2), (64, 1), (32, 9)]:
        pool, tables, _, _, q = _paged_case(bs, 2, 64, 2, lens, order_seed=order_seed, seed=11)
        outs.append(pool.attention(q, tables, np.array(lens), 4, 0.125))
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])  # same gathered values, same arithmetic: bit-identical


@pytest.mark.parametrize("chunk", [1, 2, 7, 64, 1000])
def test_split_merge_equals_unsplit(chunk):
    lens = [1, 9, 64, 130, 0]
    pool, tables, _, _, q = _paged_case(16, 2, 64, 4, lens, order_seed=4, seed=2)
    full = pool.attention(q, tables, np.array(lens), 8, 0.2)
    split = pool.attention_split(q, tables, np.array(lens), 8, 0.2, chunk)
    np.testing.assert_allclose(split, full, rtol=1e-12, atol=1e-13)


def test_threads_do_not_change_results():
    lens = [5, 80, 33]
    pool, tables, _, _, q = _paged_case(16, 4, 64, 2, lens, order_seed=5)
    a = pool.attention(q, tables, np.array(lens), 8, 0.1, threads=1)
    b = pool.attention(q, tables, np.array(lens), 8, 0.1, threads=5)
    assert np.array_equal(a, b)


def test_bf16_append_then_read_returns_the_bytes():
    lens = [7, 20]
    pool, tables, Ks, Vs, _ = _paged_case(16, 2, 64, 1, lens, order_seed=6)
    for b, L in enumerate(lens):
        for t in range(L):
            blk = tables[b, t // 16]
            for h in range(2):
                for d in (0, 17, 63):
                    for kv, src in ((0, Ks), (1, Vs)):
                        off = pool.elem_byte(blk, kv, h, t % 16, d)
                        assert pool.data[off:off + 2].view(np.uint16)[0] == src[b][t, h, d]


# ----------------------------------------------------------------------------- FP8 append + attention
def test_fp8_scale_is_block_amax_over_448_and_fixed_by_first_write():
    bs, Hkv, D = 16, 1, 128
    pool = oracle.Pool(2, bs, Hkv, D, True)
    rng = _rng(8)
    x = rng.standard_normal((3, 1, D)) * 2
    k, v = _bf16_bits(x), _bf16_bits(-x)
    assert pool.append(k, v, np.array([16, 17, 18])) == 0  # block 1, offsets 0..2
    kf = oracle.bf16_bits_to_f64(k)
    amax = np.float32(np.abs(kf).max())
    assert pool.scales[4 * 1 + 0] == np.float32(amax / np.float32(448))
    assert pool.scales[0] == 0  # block 0 untouched
    # the element with the largest magnitude lands on +-448
    i, _, d = np.unravel_index(np.argmax(np.abs(kf)), kf.shape)
    code = pool.data[pool.elem_byte(1, 0, 0, i, d)]
    assert code & 0x7F == 0x7E
    # a later append into the same block keeps the scale and saturates
    big = _bf16_bits(np.full((1, 1, D), 1e3))
    assert pool.append(big, big, np.array([19])) == 0
    assert pool.scales[4] == np.float32(amax / np.float32(448))
    assert pool.data[pool.elem_byte(1, 0, 0, 3, 5)] == 0x7E
    # writing offset 0 again re-derives the scale from this call's tokens
    assert pool.append(big, big, np.array([16])) == 0
    assert pool.scales[4] == np.float32(1000.0) / np.float32(448)  # bf16(1e3) is exactly 1000


def test_fp8_zero_block_gets_unit_scale():
    pool = oracle.Pool(1, 16, 1, 64, True)
    z = np.zeros((1, 1, 64), dtype=np.uint16)
    pool.append(z, z, np.array([0]))
    assert pool.scales[0] == 1.0 and pool.scales[1] == 1.0


def test_fp8_attention_equals_dense_over_torch_decoded_codes():
    lens = [1, 17, 40]
    bs, Hkv, D, G = 16, 2, 128, 4
    pool, tables, _, _, q = _paged_case(bs, Hkv, D, G, lens, order_seed=7, fp8=True, seed=9)
    out = pool.attention(q, tables, np.array(lens), Hkv * G, 1 / math.sqrt(D))
    codes = torch.tensor(pool.data).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    qd = oracle.bf16_bits_to_f64(q)
    for b, L in enumerate(lens):
        for h in range(Hkv):
            K = np.zeros((L, D))
            V = np.zeros((L, D))
            for t in range(L):
                blk = tables[b, t // bs]
                for kv, M in ((0, K), (1, V)):
                    s = pool.scales[(blk * Hkv + h) * 4 + kv]
                    for d in range(D):
                        M[t, d] = codes[pool.elem_byte(blk, kv, h, t % bs, d)] * s
            ref = _sdpa(qd[b, h * G:(h + 1) * G], K, V, 1 / math.sqrt(D))
            np.testing.assert_allclose(out[b, h * G:(h + 1) * G], ref, rtol=1e-11, atol=1e-12)


def test_fp8_quantisation_error_within_half_step():
    # |decode(encode(x/s))*s - x| <= half a grid step at x/s (relative 2^-4 for normals)
    pool = oracle.Pool(1, 16, 1, 128, True)
    rng = _rng(12)
    x = _bf16_bits(rng.standard_normal((16, 1, 128)))
    pool.append(x, x, np.arange(16))
    s = pool.scales[0]
    xf = oracle.bf16_bits_to_f64(x)[:, 0, :]
    for t in range(16):
        for d in range(0, 128, 7):
            back = oracle.e4m3_decode(int(pool.data[pool.elem_byte(0, 0, 0, t, d)])) * s
            assert abs(back - xf[t, d]) <= max(abs(xf[t, d]) * 2 ** -4, 2 ** -10 * s) + 1e-12


@pytest.mark.parametrize("dtype", ["fp8_e4m3", "int8"])
def test_oracle_quantisation_at_rounding_boundaries(dtype):
    """CPU pin of the oracle's append quantisation on the rounding-boundary rows of the GPU test
    below: every block's scale is numpy's IEEE fp32 amax / 448 (int8: / 127), and every stored K
    code is torch's float8_e4m3fn conversion (round to nearest even; |q| < 464 here) of numpy's
    fp32 quotient x / s, or for int8 its nearest-even integer clipped to +-127.  On the int8 rows
    a quotient taken in fp64 instead of fp32 changes codes; on both, rounding ties away from zero
    instead of to even does."""
    import torch
    D, n = 128, 300
    i8 = dtype == "int8"
    rows = near_boundary_rows(i8, n, D, seed=21 if i8 else 22)
    pool = oracle.Pool(n, 16, 1, D, odrive.KV_CODE[dtype])
    slots = np.arange(n, dtype=np.int64) * 16
    assert pool.append(rows, rows, slots) == 0
    x = (rows[:, 0, :].astype(np.uint32) << 16).view(np.float32)
    amax = np.abs(x).max(axis=1)
    sc = (amax / np.float32(127.0 if i8 else 448.0)).astype(np.float32)
    assert np.array_equal(pool.scales.reshape(n, 1, 4)[:, 0, 0], sc)
    assert np.array_equal(pool.scales.reshape(n, 1, 4)[:, 0, 1], sc)
    q = (x / sc[:, None]).astype(np.float32)
    if i8:
        want = np.clip(np.rint(q.astype(np.float64)), -127, 127).astype(np.int8).view(np.uint8)
    else:
        # below 464, the midpoint above the largest code, nearest-even needs no saturation rule
        # (the amax element's own quotient can exceed 448 by the rounding of s)
        assert np.abs(q).max() < 464.0
        want = torch.tensor(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    k_codes = pool.data.reshape(n, 2, 1, 16, D)[:, 0, 0, 0, :]  # K row of offset 0 of each block
    assert np.array_equal(k_codes, want)
