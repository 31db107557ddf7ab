"""RoPE fused into the append: oracle pins on the CPU; the GPU kernel against the oracle."""
import math
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle


def _bf16_of_bits(b: int) -> Fraction:
    """Exact value of a finite bf16 bit pattern."""
    f = struct.unpack("<f", struct.pack("<I", (b & 0xFFFF) << 16))[0]
    return Fraction(f)


def _nearest_bf16_bits(x: float) -> int:
    """Brute-force round-to-nearest-even of a double to bf16: compare the exact distances to
    every bf16 neighbour (walking the ordered magnitudes)."""
    if math.isnan(x):
        return 0x7FC0
    sign = 0x8000 if math.copysign(1.0, x) < 0 else 0
    if math.isinf(x):
        return sign | 0x7F80
    a = Fraction(abs(x))
    if a >= Fraction(2) ** 128:
        return sign | 0x7F80
    # largest magnitude pattern <= a (patterns 0..0x7F7F order like their values)
    lo, hi = 0, 0x7F7F
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if _bf16_of_bits(mid) <= a:
            lo = mid
        else:
            hi = mid - 1
    below = lo
    above = below + 1  # 0x7F80 is +inf
    vb = _bf16_of_bits(below)
    va = Fraction(2) ** 128 if above == 0x7F80 else _bf16_of_bits(above)
    db, da = a - vb, va - a
    if db < da or (db == da and below % 2 == 0):
        return sign | below
    return sign | above


def test_f64_to_bf16_matches_brute_force_rounding():
    rng = np.random.default_rng(1)
    xs = [0.0, -0.0, 1.0, -1.0, 3.0e38, 3.4e38, 3.3895313892515355e38, 3.3961775292304547e38, 1e-40, -1e-39,
          9.183549615799121e-41, 2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -135, 1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8,
          1 + 2.0 ** -8 + 2.0 ** -40, 65504.0, float("inf"), float("-inf")]
    xs += list(rng.standard_normal(300) * 10.0 ** rng.uniform(-45, 38, 300))
    xs += [float(np.float64(np.frombuffer(struct.pack("<Q", int(b)), dtype=np.float64)[0]))
           for b in rng.integers(0, 2 ** 63, 200, dtype=np.uint64) if np.isfinite(
               np.frombuffer(struct.pack("<Q", int(b)), dtype=np.float64)[0])]
    for x in xs:
        assert oracle.f64_to_bf16_bits(x) == _nearest_bf16_bits(x), x


def _bits(x):
    import torch
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_rope_position_zero_is_identity_and_single_pair_closed_form():
    rng = np.random.default_rng(2)
    x = _bits(rng.standard_normal((5, 3, 128)))
    assert np.array_equal(oracle.rope(x, np.zeros(5, np.int64), 10000.0), x)
    # D = 2: one pair turning by the angle p (base^0 = 1)
    x2 = _bits(rng.standard_normal((7, 1, 2)))
    pos = np.array([0, 1, 2, 17, 1000, 32767, 131071], np.int64)
    got = oracle.rope(x2, pos, 500000.0)
    xf = oracle.bf16_bits_to_f64(x2)
    for i, p in enumerate(pos):
        c, s = math.cos(p), math.sin(p)
        a, b = xf[i, 0]
        assert got[i, 0, 0] == _nearest_bf16_bits(a * c - b * s)
        assert got[i, 0, 1] == _nearest_bf16_bits(b * c + a * s)


def test_rope_preserves_pair_norms_and_depends_on_relative_position():
    rng = np.random.default_rng(3)
    D = 64
    q = rng.standard_normal((6, 2, D))
    k = rng.standard_normal((6, 2, D))
    p = rng.integers(0, 40000, 6)
    pk = rng.integers(0, 40000, 6)
    yq = oracle.rope_f64(q, p, 10000.0)
    n_in = q[..., :D // 2] ** 2 + q[..., D // 2:] ** 2
    n_out = yq[..., :D // 2] ** 2 + yq[..., D // 2:] ** 2
    np.testing.assert_allclose(n_out, n_in, rtol=1e-12)
    for shift in (1, 777, 50000):
        a = np.einsum("nhd,nhd->nh", oracle.rope_f64(q, p + shift, 10000.0), oracle.rope_f64(k, pk + shift, 10000.0))
        b = np.einsum("nhd,nhd->nh", yq, oracle.rope_f64(k, pk, 10000.0))
        np.testing.assert_allclose(a, b, rtol=1e-8, atol=1e-9)


def test_rope_matches_torch_rotate_half_in_fp64():
    import torch
    rng = np.random.default_rng(4)
    N, H, D, base = 9, 4, 128, 500000.0
    x = _bits(rng.standard_normal((N, H, D)))
    pos = rng.integers(0, 131072, N).astype(np.int64)
    xt = torch.from_numpy(oracle.bf16_bits_to_f64(x))
    inv = torch.tensor([base ** (-2.0 * i / D) for i in range(D // 2)], dtype=torch.float64)
    ang = torch.from_numpy(pos.astype(np.float64))[:, None] * inv[None, :]
    cos = torch.cat([torch.cos(ang), torch.cos(ang)], -1)[:, None, :]
    sin = torch.cat([torch.sin(ang), torch.sin(ang)], -1)[:, None, :]
    rot = torch.cat([-xt[..., D // 2:], xt[..., :D // 2]], -1)
    ref = (xt * cos + rot * sin).numpy()
    got = oracle.bf16_bits_to_f64(oracle.rope(x, pos, base))
    # one bf16 rounding of the same fp64 values: within half a bf16 ulp, 2^(floor(log2|v|) - 8)
    _, e = np.frexp(ref)
    half_ulp = np.ldexp(1.0, e - 1 - 8)
    assert (np.abs(got - ref) <= half_ulp * (1 + 1e-9)).all()
    # and the rounded values agree with rounding torch's values, except on a rounding edge
    same = np.array([oracle.f64_to_bf16_bits(v) for v in ref.reshape(-1)]).reshape(ref.shape) == oracle.rope(x, pos, base)
    assert same.mean() > 0.9999


# ----------------------------------------------------------------------------- GPU
@pytest.mark.gpu
@pytest.mark.parametrize("kv_dtype,D,bs", [("bf16", 128, 16), ("bf16", 64, 64), ("fp8_e4m3", 128, 16)])
def test_append_rope_matches_oracle(kv_dtype, D, bs):
    """K and q rotated in place bit-exact against the oracle's fp64 rotation; the pool holds the
    rotated K (bf16 bit-exact; fp8: the oracle's quantisation of the oracle's rotated K); the
    decode attention over the rotated data within tolerance."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_266_gb300 import build
    build.build()
    import paged_kv_cache_266_gb300 as pkv
    from paged_kv_cache_266_gb300.runner import _wrap_device
    fp8 = kv_dtype == "fp8_e4m3"
    rng = np.random.default_rng(7)
    Hkv, G, nb, base = 2, 4, 40, 500000.0
    Hq = Hkv * G
    lens = [37, 1, 130, 64]
    pool = pkv.KVPool(nb, bs, Hkv, D, pkv.PKV_KV_FP8_E4M3 if fp8 else pkv.PKV_KV_BF16)
    a = pool.allocator
    oa, op = oracle.Allocator(nb, bs), oracle.Pool(nb, bs, Hkv, D, fp8)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    host = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
    for b, L in enumerate(lens):
        pkv.pkv_seq_reserve(a, b, L)
        oa.reserve(b, L)
    # the whole history appended through the RoPE path, in two calls (prompt, then the rest)
    seqs = np.concatenate([np.full(L, b) for b, L in enumerate(lens)])
    pos = np.concatenate([np.arange(L) for L in lens]).astype(np.int64)
    k = (rng.standard_normal((len(pos), Hkv, D)) * 2).astype(np.float32)
    v = rng.standard_normal((len(pos), Hkv, D)).astype(np.float32)
    kb, vb = _bits(k), _bits(v)
    cut = len(pos) // 2
    for lo, hi in ((0, cut), (cut, len(pos))):
        slots = pkv.pkv_slot_mapping(a, seqs[lo:hi], pos[lo:hi])
        assert np.array_equal(slots, oa.slot_mapping(seqs[lo:hi], pos[lo:hi]))
        kd = dev(kb[lo:hi])
        pkv.pkv_append_rope(pool.handle, kd, dev(vb[lo:hi]), torch.from_numpy(slots).cuda(),
                            torch.from_numpy(pos[lo:hi]).cuda(), base)
        torch.cuda.synchronize()
        kr = oracle.rope(kb[lo:hi], pos[lo:hi], base)
        assert np.array_equal(host(kd), kr)
        op.append(kr, vb[lo:hi], slots)
    assert pkv.pkv_check_device_error(pool.handle) == pkv.PKV_OK
    kv_ptr, kv_bytes, sc_ptr, sc_bytes = pkv.pkv_pool_raw(pool.handle)
    assert np.array_equal(_wrap_device(kv_ptr, kv_bytes).cpu().numpy(), op.data)
    if fp8:
        assert np.array_equal(_wrap_device(sc_ptr, sc_bytes).cpu().numpy().view(np.float32), op.scales)
    # a decode-style call: q rotated with the same kernel (no K/V rows: N = 0 appends nothing, so
    # rotate q alongside a one-token append at each sequence's last position)
    qb = _bits(rng.standard_normal((len(lens), Hq, D)))
    qd = dev(qb)
    last = np.array([L - 1 for L in lens], np.int64)
    slots_last = pkv.pkv_slot_mapping(a, np.arange(len(lens)), last)
    k_last = kb[np.cumsum(lens) - 1]
    v_last = vb[np.cumsum(lens) - 1]
    pkv.pkv_append_rope(pool.handle, dev(k_last), dev(v_last), torch.from_numpy(slots_last).cuda(),
                        torch.from_numpy(last).cuda(), base, q=qd)
    torch.cuda.synchronize()
    qr = oracle.rope(qb, last, base)
    assert np.array_equal(host(qd), qr)
    op.append(oracle.rope(k_last, last, base), v_last, slots_last)  # the same re-append on the oracle's pool
    assert np.array_equal(_wrap_device(kv_ptr, kv_bytes).cpu().numpy(), op.data)
    mb = max(-(-L // bs) for L in lens)
    tables = pkv.pkv_get_block_tables(a, list(range(len(lens))), mb)
    ctx = np.array(lens, np.int32)
    out = torch.empty(len(lens), Hq, D, dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(pkv.pkv_decode_workspace_bytes(pool.handle, len(lens), Hq, mb), dtype=torch.uint8, device="cuda")
    pkv.pkv_decode_attention(pool.handle, qd, torch.from_numpy(tables).cuda(), torch.from_numpy(ctx).cuda(),
                             1 / math.sqrt(D), out, ws)
    torch.cuda.synchronize()
    ref = op.attention(qr, tables, ctx, Hq, 1 / math.sqrt(D))
    err = np.abs(oracle.bf16_bits_to_f64(host(out)) - ref)
    assert err.max() <= (3e-2 if fp8 else 1e-2) and err.mean() <= 1e-3
    pool.close()


@pytest.mark.gpu
def test_append_rope_rejects_bad_arguments():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_266_gb300 import build
    build.build()
    import paged_kv_cache_266_gb300 as pkv
    pool = pkv.KVPool(4, 16, 1, 128)
    k = torch.zeros(1, 1, 128, dtype=torch.bfloat16, device="cuda")
    s = torch.zeros(1, dtype=torch.int64, device="cuda")
    for base in (0.0, 1.0, float("inf"), float("nan")):
        with pytest.raises(pkv.PKVError):
            pkv.pkv_append_rope(pool.handle, k, k.clone(), s, s, base)
    pool.close()


@pytest.mark.gpu
def test_decode_step_rope_equals_separate_calls_and_oracle():
    """pkv_decode_step_rope on a GQA batch: the same bits as pkv_append_rope followed by
    pkv_decode_attention, and within tolerance of the oracle's rotate-then-attend."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_266_gb300 import build
    build.build()
    import paged_kv_cache_266_gb300 as pkv
    import pkv_workloads as W
    from paged_kv_cache_266_gb300.runner import DecodeStep
    w = W.custom_workload(330, 6, 16, 4, 128, 16, [3, 40, 100, 17, 64, 250])
    base = 10000.0
    outs = []
    for fused in (True, False):
        st = DecodeStep(w)
        pos = torch.from_numpy(w.lens.astype(np.int64)).cuda()
        k, q = st.k_new.clone(), st.q.clone()
        if fused:
            pkv.pkv_decode_step_rope(st.pool.handle, k, st.v_new, st.slots_new, pos, base, q, st.tables, st.lens,
                                     st.scale, st.out, st.workspace)
        else:
            pkv.pkv_append_rope(st.pool.handle, k, st.v_new, st.slots_new, pos, base, q=q)
            pkv.pkv_decode_attention(st.pool.handle, q, st.tables, st.lens, st.scale, st.out, st.workspace)
        torch.cuda.synchronize()
        assert pkv.pkv_check_device_error(st.pool.handle) == pkv.PKV_OK
        outs.append(st.out_host())
        if fused:
            from oracle import drive as odrive
            opool, oalloc, tables = odrive.build(w, with_new_token=False)
            kr = oracle.rope(w.new_k(), w.lens.astype(np.int64), base)
            opool.append(kr, w.new_v(), oalloc.slot_mapping(w.seq_ids, w.lens))
            qr = oracle.rope(w.query(), w.lens.astype(np.int64), base)
            ref = opool.attention(qr, tables, w.attend_lens, w.Hq, st.scale)
            err = np.abs(oracle.bf16_bits_to_f64(outs[0]) - ref)
            assert err.max() <= 1e-2 and err.mean() <= 1e-3
        st.close()
    assert np.array_equal(outs[0], outs[1])
