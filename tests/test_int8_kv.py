"""INT8 KV cache: oracle pins on the CPU, then append and decode attention on the GPU."""
import math

import numpy as np
import pytest

import oracle


def _bits(x):
    import torch
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_int8_encode_is_clamped_round_half_even():
    """Against numpy's rint (nearest, ties to even) and clip, over ties, the clamp edges and a
    random sweep."""
    ties = np.arange(-130.5, 131.0, 1.0, dtype=np.float32)
    rng = np.random.default_rng(1)
    qs = np.concatenate([ties, ties + np.float32(1e-3), ties - np.float32(1e-3),
                         rng.uniform(-140, 140, 5000).astype(np.float32),
                         np.array([0.0, -0.0, 127.0, -127.0, 126.5, -126.5, 1e9, -1e9], np.float32)])
    want = np.clip(np.rint(qs.astype(np.float64)), -127, 127).astype(np.int8)
    assert np.array_equal(oracle.int8_encode_array(qs), want)


def test_int8_append_scales_and_error_bound():
    """A fresh block's scale is amax/127 over the call's tokens in it (per K|V and head); every
    stored value reads back within half a scale step of its input, and each amax element reads
    back as +-127 codes."""
    rng = np.random.default_rng(2)
    bs, Hkv, D, nb = 16, 2, 64, 4
    pool = oracle.Pool(nb, bs, Hkv, D, 2)
    a = oracle.Allocator(nb, bs)
    assert a.reserve(0, 40) == 0
    x = rng.standard_normal((40, Hkv, D)) * 3
    k, v = _bits(x), _bits(-x)
    slots = a.slot_mapping([0] * 40, np.arange(40))
    assert pool.append(k, v, slots) == 0
    kf, vf = oracle.bf16_bits_to_f64(k), oracle.bf16_bits_to_f64(v)
    for kv, src in ((0, kf), (1, vf)):
        for i, slot in enumerate(slots):
            blk, t = int(slot) // bs, int(slot) % bs
            toks = [j for j, s in enumerate(slots) if int(s) // bs == blk]
            for h in range(Hkv):
                amax = np.float32(np.abs(src[toks, h]).max())
                scale = pool.scales[(blk * Hkv + h) * 4 + kv]
                assert scale == np.float32(amax / np.float32(127.0))
                codes = np.array([pool.data[pool.elem_byte(blk, kv, h, t, d)] for d in range(D)], np.uint8).view(np.int8)
                back = codes.astype(np.float64) * float(scale)
                assert np.all(np.abs(back - src[i, h]) <= float(scale) / 2 * (1 + 1e-6))
                if abs(src[i, h]).max() == amax:
                    assert np.abs(codes).max() == 127


def test_int8_single_token_attention_is_the_dequantised_row():
    rng = np.random.default_rng(3)
    bs, Hkv, D = 16, 1, 64
    pool = oracle.Pool(2, bs, Hkv, D, 2)
    a = oracle.Allocator(2, bs)
    assert a.reserve(0, 1) == 0
    k, v = _bits(rng.standard_normal((1, 1, D))), _bits(rng.standard_normal((1, 1, D)))
    slots = a.slot_mapping([0], [0])
    pool.append(k, v, slots)
    q = _bits(rng.standard_normal((1, 2, D)))
    out = pool.attention(q, a.block_tables([0], 1), np.array([1], np.int32), 2, 0.3)
    blk = int(slots[0]) // bs
    scale = float(pool.scales[blk * Hkv * 4 + 1])
    codes = np.array([pool.data[pool.elem_byte(blk, 1, 0, 0, d)] for d in range(D)], np.uint8).view(np.int8)
    np.testing.assert_array_equal(out[0, 0], codes * scale)
    np.testing.assert_array_equal(out[0, 1], codes * scale)
