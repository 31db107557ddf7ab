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
