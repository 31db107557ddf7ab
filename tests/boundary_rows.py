"""Seeded input rows for quantisation at rounding boundaries (test inputs only: the expected
codes come from the oracle or from independent library conversions, never from here)."""
import numpy as np

import oracle


def near_boundary_rows(int8: bool, n_tok: int, D: int, seed: int) -> np.ndarray:
    """Token rows (one KV head) for quantisation at rounding boundaries.  Element 0 of a row is
    its amax, so a token opening its own block gets the scale s = amax/448 (amax/127 for int8);
    the other elements are bf16 values x whose fp32 quotient x / s lies within 16 fp32 steps of
    a code's rounding boundary (the midpoint of two adjacent E4M3 values; a half-integer for
    int8), found by trying every positive bf16 value up to amax, with random signs, and random
    bf16 values below amax where too few are that close.  The amax values: random ones, powers
    of two times the code's largest value (s a power of two: the boundaries are hit exactly) and
    the same times 1.125, 1.25 or 1.375 (exact boundary hits at a scale whose reciprocal is
    inexact)."""
    import torch
    rng = np.random.default_rng(seed)
    cmax = 127.0 if int8 else 448.0
    if int8:
        bounds = np.arange(0.5, 127.0, 1.0)
    else:
        vals = np.array([oracle.e4m3_decode(c) for c in range(0x7F)])
        bounds = (vals[:-1] + vals[1:]) / 2
    bounds = bounds.astype(np.float32)
    bound_bits = bounds.view(np.int32).astype(np.int64)
    pos_bits = np.arange(1, 0x7F80, dtype=np.uint32)
    allx = (pos_bits << 16).view(np.float32)

    def to_bf16(a):
        return torch.tensor(np.asarray(a, np.float32)).to(torch.bfloat16).float().numpy()

    rows = np.zeros((n_tok, 1, D), dtype=np.uint16)
    for t in range(n_tok):
        kind = t % 3
        if kind == 0:
            amax = to_bf16(rng.uniform(1.0, 2.0) * 2.0 ** rng.integers(-8, 9))
        else:
            f = 1.0 if kind == 1 else float(rng.choice([1.125, 1.25, 1.375]))
            amax = to_bf16(cmax * f * 2.0 ** rng.integers(-8, 9))
        amax = np.float32(amax)
        sc = np.float32(amax / np.float32(cmax))
        xs = allx[allx <= amax]
        q = (xs / sc).astype(np.float32)
        i = np.clip(np.searchsorted(bounds, q), 1, len(bounds) - 1)
        qb = q.view(np.int32).astype(np.int64)
        steps = np.minimum(np.abs(qb - bound_bits[i - 1]), np.abs(qb - bound_bits[i]))
        near = xs[steps <= 16]
        pick = rng.choice(near, size=min(len(near), D - 1), replace=False) if len(near) else near
        fill = rng.choice(xs, size=D - 1 - len(pick))
        x = np.concatenate([pick, fill]).astype(np.float32) * rng.choice([-1.0, 1.0], size=D - 1)
        row = np.concatenate([[amax], x]).astype(np.float32)
        rows[t, 0] = torch.tensor(row).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return rows
