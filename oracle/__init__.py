"""CPU oracle for paged decode attention — TEST INFRASTRUCTURE ONLY.

Only tests/, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import this package.  The product library never loads it, and
it shares no code with the CUDA path: ``pkv_oracle.cpp`` is a plain fp64
restatement of what the TensorRT-LLM pages describe (allocator, append, FP8
E4M3 codec, decode attention, split merge, block reuse, chunked-context prefill
attention, RoPE, KV-memory formula); see the header of
that file for the page and section each function follows.

Pins: every function here is checked in ``tests/test_oracle_*.py`` against
something other than itself (worked values from the pages, the OCP E4M3 table,
torch's CPU float8 conversion and scaled-dot-product attention, closed forms,
brute force and invariants).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None

OK, ERR_INVALID, ERR_OOM, ERR_NO_SEQ, ERR_BOUNDS, ERR_SLOT = 0, 1, 2, 3, 4, 5


def build_native(force: bool = False) -> str:
    """Compile the oracle (g++, no fast-math, no FMA contraction) into oracle/_build."""
    if os.path.exists(_LIB_PATH) and not force and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                           _SRC, "-o", tmp])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build_native())
    vp, i32, i64, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
    sig = {
        "oracle_alloc_new": (vp, [i32, i32]),
        "oracle_alloc_delete": (None, [vp]),
        "oracle_alloc_set_free_order": (i32, [vp, vp, i32]),
        "oracle_alloc_reserve": (i32, [vp, i64, i64]),
        "oracle_alloc_release": (i32, [vp, i64]),
        "oracle_alloc_num_free": (i32, [vp]),
        "oracle_alloc_num_pages": (i32, [vp, i64]),
        "oracle_alloc_free_list": (None, [vp, vp]),
        "oracle_alloc_block_tables": (i32, [vp, vp, i32, i32, vp]),
        "oracle_alloc_slot_mapping": (i32, [vp, vp, vp, i64, vp]),
        "oracle_alloc_share_prefix": (i32, [vp, i64, i64, i64, vp, vp]),
        "oracle_alloc_holders": (i32, [vp, i32]),
        "oracle_copy_block": (None, [vp, vp, i32, i32, i32, i32, i64, i64]),
        "oracle_m_kv": (f64, [f64] * 6),
        "oracle_e4m3_decode": (f64, [ctypes.c_uint8]),
        "oracle_e4m3_encode": (ctypes.c_uint8, [ctypes.c_float]),
        "oracle_e4m3_encode_exhaustive": (ctypes.c_uint8, [ctypes.c_float]),
        "oracle_e4m3_encode_array": (None, [vp, i64, vp, i32]),
        "oracle_append": (i32, [vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, i64]),
        "oracle_dense_attention": (None, [vp, vp, vp, i64, i32, i32, f64, vp]),
        "oracle_decode_attention": (i32, [vp, vp, i32, i32, i32, i32, i32, vp, vp, i32, vp, i32, i32, f64, vp, i32]),
        "oracle_decode_attention_split": (i32, [vp, vp, i32, i32, i32, i32, i32, vp, vp, i32, vp, i32, i32, f64, i32,
                                                vp]),
        "oracle_prefill_attention": (i32, [vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, i32, vp, i32, i32, f64, vp,
                                           i32]),
        "oracle_rope": (None, [vp, vp, i64, i32, i32, f64, vp]),
        "oracle_rope_f64": (None, [vp, vp, i64, i32, i32, f64, vp]),
        "oracle_f64_to_bf16_bits": (ctypes.c_uint16, [f64]),
        "oracle_int8_encode_array": (None, [vp, i64, vp]),
        "oracle_pool_bytes": (i64, [i32, i32, i32, i32, i32]),
        "oracle_scale_floats": (i64, [i32, i32]),
        "oracle_elem_byte": (i64, [i64, i32, i32, i32, i32, i32, i32, i32, i32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _p(a: np.ndarray):
    return a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ----------------------------------------------------------------------------- allocator
class Allocator:
    """Replica of the pages' block allocator (free list with pop() from the end)."""

    def __init__(self, num_blocks: int, block_size: int):
        self.num_blocks, self.block_size = num_blocks, block_size
        self._h = _L().oracle_alloc_new(num_blocks, block_size)

    def __del__(self):
        if getattr(self, "_h", None):
            _L().oracle_alloc_delete(self._h)
            self._h = None

    def set_free_order(self, order) -> int:
        o = _c(order, np.int32)
        return _L().oracle_alloc_set_free_order(self._h, _p(o), len(o))

    def reserve(self, seq: int, n_tokens: int) -> int:
        return _L().oracle_alloc_reserve(self._h, seq, n_tokens)

    def release(self, seq: int) -> int:
        return _L().oracle_alloc_release(self._h, seq)

    def num_free(self) -> int:
        return _L().oracle_alloc_num_free(self._h)

    def num_pages(self, seq: int) -> int:
        return _L().oracle_alloc_num_pages(self._h, seq)

    def free_list(self) -> np.ndarray:
        out = np.empty(self.num_free(), dtype=np.int32)
        _L().oracle_alloc_free_list(self._h, _p(out))
        return out

    def block_tables(self, seqs, max_blocks: int) -> np.ndarray:
        s = _c(seqs, np.int64)
        out = np.empty((len(s), max_blocks), dtype=np.int32)
        rc = _L().oracle_alloc_block_tables(self._h, _p(s), len(s), max_blocks, _p(out))
        if rc:
            raise RuntimeError(f"oracle block_tables rc={rc}")
        return out

    def slot_mapping(self, seqs, positions) -> np.ndarray:
        s, p = _c(seqs, np.int64), _c(positions, np.int64)
        out = np.empty(len(s), dtype=np.int64)
        rc = _L().oracle_alloc_slot_mapping(self._h, _p(s), _p(p), len(s), _p(out))
        if rc:
            raise RuntimeError(f"oracle slot_mapping rc={rc}")
        return out

    def share_prefix(self, src: int, dst: int, n_tokens: int):
        """(status, cow_src, cow_dst); see oracle_alloc_share_prefix."""
        cs, cd = ctypes.c_int32(), ctypes.c_int32()
        rc = _L().oracle_alloc_share_prefix(self._h, src, dst, n_tokens, ctypes.byref(cs), ctypes.byref(cd))
        return rc, cs.value, cd.value

    def holders(self, page: int) -> int:
        return _L().oracle_alloc_holders(self._h, page)

    def replay(self, ops) -> None:
        """Run an allocation script of ("reserve", seq, tokens) / ("release", seq) ops."""
        for op in ops:
            rc = self.reserve(op[1], op[2]) if op[0] == "reserve" else self.release(op[1])
            if rc:
                raise RuntimeError(f"oracle allocator op {op} rc={rc}")


# ----------------------------------------------------------------------------- formulas
def m_kv(n_layers, n_kv_heads, d_head, n_tokens, batch, bytes_per_elem) -> float:
    return _L().oracle_m_kv(n_layers, n_kv_heads, d_head, n_tokens, batch, bytes_per_elem)


def e4m3_decode(code: int) -> float:
    return _L().oracle_e4m3_decode(code)


def e4m3_encode(x: float) -> int:
    return _L().oracle_e4m3_encode(x)


def e4m3_encode_array(x, exhaustive: bool = False) -> np.ndarray:
    xs = _c(x, np.float32).ravel()
    out = np.empty(xs.shape, dtype=np.uint8)
    _L().oracle_e4m3_encode_array(_p(xs), xs.size, _p(out), 1 if exhaustive else 0)
    return out.reshape(np.shape(x))


def dense_attention(q, K, V, scale: float) -> np.ndarray:
    """softmax(scale q K^T) V for q [G][D], K/V [L][D] (fp64)."""
    q, K, V = _c(q, np.float64), _c(K, np.float64), _c(V, np.float64)
    G, D = q.shape
    L = K.shape[0]
    out = np.empty((G, D), dtype=np.float64)
    _L().oracle_dense_attention(_p(q), _p(K), _p(V), L, D, G, scale, _p(out))
    return out


# ----------------------------------------------------------------------------- pool replica
class Pool:
    """Host replica of the paged KV pool (same byte layout as the device pool)."""

    def __init__(self, num_blocks: int, block_size: int, n_kv_heads: int, head_dim: int, fp8):
        """fp8: the element code — False/0 bf16, True/1 fp8 e4m3, 2 int8."""
        self.num_blocks, self.bs, self.Hkv, self.D, self.fp8 = num_blocks, block_size, n_kv_heads, head_dim, int(fp8)
        self.data = np.zeros(_L().oracle_pool_bytes(num_blocks, block_size, n_kv_heads, head_dim, self.fp8),
                             dtype=np.uint8)
        self.scales = np.zeros(_L().oracle_scale_floats(num_blocks, n_kv_heads), dtype=np.float32)

    def copy_block(self, src: int, dst: int) -> None:
        _L().oracle_copy_block(_p(self.data), _p(self.scales), self.bs, self.Hkv, self.D, self.fp8, src, dst)

    def elem_byte(self, blk, kv, h, t, d) -> int:
        return _L().oracle_elem_byte(blk, kv, h, t, d, self.bs, self.Hkv, self.D, self.fp8)

    def append(self, k_new, v_new, slots) -> int:
        k, v, s = _c(k_new, np.uint16), _c(v_new, np.uint16), _c(slots, np.int64)
        return _L().oracle_append(_p(self.data), _p(self.scales), self.num_blocks, self.bs, self.Hkv, self.D,
                                  self.fp8, _p(k), _p(v), _p(s), len(s))

    def attention(self, q, tables, lens, n_q_heads: int, scale: float, threads: int = 1) -> np.ndarray:
        q, t, l = _c(q, np.uint16), _c(tables, np.int32), _c(lens, np.int32)
        B = len(l)
        out = np.zeros((B, n_q_heads, self.D), dtype=np.float64)
        rc = _L().oracle_decode_attention(_p(self.data), _p(self.scales), self.num_blocks, self.bs, self.Hkv, self.D,
                                          self.fp8, _p(q), _p(t), t.shape[1] if t.ndim == 2 else 0, _p(l), B,
                                          n_q_heads, scale, _p(out), threads)
        if rc:
            raise RuntimeError(f"oracle attention rc={rc}")
        return out

    def prefill_attention(self, q, cu_q, tables, ctx_lens, n_q_heads: int, scale: float,
                          threads: int = 1) -> np.ndarray:
        """Chunked-context attention: rows cu_q[b]..cu_q[b+1]-1 of q are the last queries of
        sequence b's ctx_lens[b] cached tokens, each attending causally (see the C source)."""
        q, c, t, l = _c(q, np.uint16), _c(cu_q, np.int32), _c(tables, np.int32), _c(ctx_lens, np.int32)
        B = len(l)
        out = np.zeros((int(c[-1]) if B else 0, n_q_heads, self.D), dtype=np.float64)
        rc = _L().oracle_prefill_attention(_p(self.data), _p(self.scales), self.num_blocks, self.bs, self.Hkv, self.D,
                                           self.fp8, _p(q), _p(c), _p(t), t.shape[1] if t.ndim == 2 else 0, _p(l), B,
                                           n_q_heads, scale, _p(out), threads)
        if rc:
            raise RuntimeError(f"oracle prefill attention rc={rc}")
        return out

    def attention_split(self, q, tables, lens, n_q_heads: int, scale: float, chunk: int) -> np.ndarray:
        q, t, l = _c(q, np.uint16), _c(tables, np.int32), _c(lens, np.int32)
        B = len(l)
        out = np.zeros((B, n_q_heads, self.D), dtype=np.float64)
        rc = _L().oracle_decode_attention_split(_p(self.data), _p(self.scales), self.num_blocks, self.bs, self.Hkv,
                                                self.D, self.fp8, _p(q), _p(t), t.shape[1], _p(l), B, n_q_heads,
                                                scale, chunk, _p(out))
        if rc:
            raise RuntimeError(f"oracle split attention rc={rc}")
        return out


def rope(x_bits, positions, base: float) -> np.ndarray:
    """RoPE ("rotate half") of bf16 rows [N][H][D] at the given positions, rounded to bf16 bits."""
    x = _c(x_bits, np.uint16)
    pos = _c(positions, np.int64)
    N, H, D = x.shape
    out = np.empty_like(x)
    _L().oracle_rope(_p(x), _p(pos), N, H, D, float(base), _p(out))
    return out


def rope_f64(x, positions, base: float) -> np.ndarray:
    """The same rotation in fp64 without rounding (x: float64 [N][H][D])."""
    x = _c(x, np.float64)
    pos = _c(positions, np.int64)
    N, H, D = x.shape
    out = np.empty_like(x)
    _L().oracle_rope_f64(_p(x), _p(pos), N, H, D, float(base), _p(out))
    return out


def f64_to_bf16_bits(x: float) -> int:
    return int(_L().oracle_f64_to_bf16_bits(float(x)))


def int8_encode_array(q) -> np.ndarray:
    """INT8 codes of fp32 quotients x / scale (nearest even, clamped to [-127, 127])."""
    qs = np.ascontiguousarray(np.asarray(q, dtype=np.float32)).reshape(-1)
    out = np.empty(qs.size, dtype=np.int8)
    _L().oracle_int8_encode_array(_p(qs), qs.size, _p(out))
    return out.reshape(np.shape(q))


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to fp64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)
