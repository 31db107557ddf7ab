"""Paged KV cache and decode attention for one GB300 — Python binding.

Argument marshalling only: every call goes straight to the C ABI declared in
``include/pkv.h`` (libpkv.so, built in-tree by ``build.py``).  Host arrays are
numpy; device buffers are torch CUDA tensors (torch provides device memory and
streams, nothing else).  There is no fallback: if libpkv.so is missing the
import of any entry point raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

__all__ = [
    "PKVError", "PKV_KV_BF16", "PKV_KV_FP8_E4M3", "PKV_KV_INT8", "KV_DTYPES", "library_path",
    "pkv_allocator_create", "pkv_allocator_destroy", "pkv_allocator_set_free_order",
    "pkv_allocator_shuffle_free_list", "pkv_seq_reserve",
    "pkv_seq_release", "pkv_seq_reserve_many", "pkv_seq_share_prefix", "pkv_block_refcount",
    "pkv_pool_copy_block", "pkv_append_rope", "pkv_decode_step_rope", "pkv_prefill_attention", "pkv_prefill_step", "pkv_seq_num_blocks", "pkv_num_free_blocks", "pkv_free_list", "pkv_get_block_tables",
    "pkv_slot_mapping", "pkv_stage_prefill", "pkv_stage_decode", "pkv_pool_create", "pkv_pool_destroy", "pkv_pool_allocator", "pkv_pool_raw",
    "pkv_check_device_error", "pkv_append", "pkv_decode_attention", "pkv_decode_step", "pkv_decode_workspace_bytes",
    "pkv_decode_workspace_init", "pkv_decode_attention_static", "PKV_STATIC_WORKSPACE_BYTES", "pkv_stage_copy", "pkv_kv_bytes",
    "pkv_status_str", "pkv_debug_reload_env", "KVPool",
]

PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_OOM, PKV_ERR_NO_SEQ, PKV_ERR_BOUNDS, PKV_ERR_CUDA, PKV_ERR_TIMEOUT = range(7)
PKV_KV_BF16, PKV_KV_FP8_E4M3, PKV_KV_INT8 = 0, 1, 2
KV_DTYPES = {"bf16": PKV_KV_BF16, "fp8_e4m3": PKV_KV_FP8_E4M3, "int8": PKV_KV_INT8}
PKV_STATIC_WORKSPACE_BYTES = 8 << 20  # include/pkv.h

_lib = None


def library_path() -> str:
    return _build.LIB


class PKVError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {pkv_status_str(status)} (status {status})")
        self.status = status


def _L():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        raise RuntimeError(f"libpkv.so is not built ({_build.LIB}); run __graft_entry__.build() or "
                           "python -m paged_kv_cache_266_gb300.build")
    lib = ctypes.CDLL(_build.LIB)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    P = ctypes.POINTER
    sig = {
        "pkv_allocator_create": (i32, [i32, i32, P(vp)]),
        "pkv_allocator_destroy": (i32, [vp]),
        "pkv_allocator_set_free_order": (i32, [vp, vp, i32]),
        "pkv_allocator_shuffle_free_list": (i32, [vp, ctypes.c_uint64]),
        "pkv_seq_reserve": (i32, [vp, i64, i64]),
        "pkv_seq_release": (i32, [vp, i64]),
        "pkv_seq_reserve_many": (i32, [vp, vp, vp, i64, P(i64)]),
        "pkv_seq_share_prefix": (i32, [vp, i64, i64, i64, P(ctypes.c_int32), P(ctypes.c_int32)]),
        "pkv_block_refcount": (i32, [vp, i32, P(i32)]),
        "pkv_pool_copy_block": (i32, [vp, i32, i32, vp]),
        "pkv_append_rope": (i32, [vp, vp, vp, vp, vp, i64, ctypes.c_double, vp, i32, vp]),
        "pkv_decode_step_rope": (i32, [vp, vp, vp, vp, vp, i64, ctypes.c_double, vp, vp, i32, vp, i32, i32,
                                       ctypes.c_float, vp, vp, ctypes.c_size_t, vp]),
        "pkv_prefill_attention": (i32, [vp, vp, vp, i32, vp, i32, vp, i32, i32, ctypes.c_float, vp, vp]),
        "pkv_prefill_step": (i32, [vp, vp, vp, vp, i64, vp, vp, i32, vp, i32, vp, i32, i32, ctypes.c_float, vp, vp]),
        "pkv_seq_num_blocks": (i32, [vp, i64, P(i32)]),
        "pkv_num_free_blocks": (i32, [vp, P(i32)]),
        "pkv_free_list": (i32, [vp, vp, i32, P(i32)]),
        "pkv_get_block_tables": (i32, [vp, vp, i32, i32, vp]),
        "pkv_slot_mapping": (i32, [vp, vp, vp, i64, vp]),
        "pkv_stage_prefill": (i32, [vp, vp, vp, vp, i32, i32, vp, vp, vp, vp]),
        "pkv_stage_decode": (i32, [vp, vp, vp, i32, i32, i32, vp, vp, vp]),
        "pkv_pool_create": (i32, [i32, i32, i32, i32, i32, P(vp)]),
        "pkv_pool_destroy": (i32, [vp]),
        "pkv_pool_allocator": (i32, [vp, P(vp)]),
        "pkv_pool_raw": (i32, [vp, P(vp), P(sz), P(vp), P(sz)]),
        "pkv_check_device_error": (i32, [vp]),
        "pkv_append": (i32, [vp, vp, vp, vp, i64, vp]),
        "pkv_decode_attention": (i32, [vp, vp, vp, i32, vp, i32, i32, ctypes.c_float, vp, vp, sz, vp]),
        "pkv_decode_workspace_bytes": (i32, [vp, i32, i32, i32, P(sz)]),
        "pkv_decode_step": (i32, [vp, vp, vp, vp, i64, vp, vp, i32, vp, i32, i32, ctypes.c_float, vp, vp, sz, vp]),
        "pkv_decode_workspace_init": (i32, [vp, sz, vp]),
        "pkv_decode_attention_static": (i32, [vp, vp, vp, i32, vp, i32, i32, ctypes.c_float, vp, vp]),
        "pkv_stage_copy": (i32, [vp, vp, sz, vp]),
        "pkv_debug_reload_env": (i32, []),
        "pkv_kv_bytes": (ctypes.c_uint64, [i64, i64, i64, i64, i64, ctypes.c_double]),
        "pkv_status_str": (ctypes.c_char_p, [i32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    _lib = lib
    return lib


def _check(rc: int, what: str):
    if rc != PKV_OK:
        raise PKVError(rc, what)


def _np(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _dev(t, dtype_name: str, what: str) -> int:
    """Device pointer of a contiguous torch CUDA tensor of the expected dtype."""
    import torch
    want = {"bf16": torch.bfloat16, "i32": torch.int32, "i64": torch.int64, "u8": torch.uint8}[dtype_name]
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{what}: expected a CUDA tensor")
    if t.dtype != want:
        raise TypeError(f"{what}: expected dtype {want}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{what}: tensor must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


# ----------------------------------------------------------------------------- allocator
def pkv_allocator_create(num_blocks: int, block_size: int) -> int:
    h = ctypes.c_void_p()
    _check(_L().pkv_allocator_create(num_blocks, block_size, ctypes.byref(h)), "pkv_allocator_create")
    return h.value


def pkv_allocator_destroy(a: int) -> None:
    _check(_L().pkv_allocator_destroy(a), "pkv_allocator_destroy")


def pkv_allocator_set_free_order(a: int, order) -> None:
    o = _np(order, np.int32)
    _check(_L().pkv_allocator_set_free_order(a, o.ctypes.data, len(o)), "pkv_allocator_set_free_order")


def pkv_allocator_shuffle_free_list(a: int, seed: int) -> None:
    _check(_L().pkv_allocator_shuffle_free_list(a, seed & ((1 << 64) - 1)), "pkv_allocator_shuffle_free_list")


def pkv_seq_reserve(a: int, seq_id: int, n_tokens: int) -> None:
    _check(_L().pkv_seq_reserve(a, seq_id, n_tokens), "pkv_seq_reserve")


def pkv_seq_reserve_many(a: int, seq_ids, n_tokens) -> None:
    s, n = _np(seq_ids, np.int64), _np(n_tokens, np.int64)
    if s.shape != n.shape:
        raise ValueError("seq_ids and n_tokens must have the same length")
    done = ctypes.c_int64()
    _check(_L().pkv_seq_reserve_many(a, s.ctypes.data, n.ctypes.data, len(s), ctypes.byref(done)),
           f"pkv_seq_reserve_many (after {done.value} reservations)")


def pkv_seq_share_prefix(a: int, src_seq: int, dst_seq: int, n_tokens: int):
    """New sequence dst starts with src's first n_tokens; returns (cow_src_block, cow_dst_block),
    both -1 when no block has to be copied."""
    cs, cd = ctypes.c_int32(), ctypes.c_int32()
    _check(_L().pkv_seq_share_prefix(a, src_seq, dst_seq, n_tokens, ctypes.byref(cs), ctypes.byref(cd)),
           "pkv_seq_share_prefix")
    return cs.value, cd.value


def pkv_block_refcount(a: int, block: int) -> int:
    n = ctypes.c_int()
    _check(_L().pkv_block_refcount(a, block, ctypes.byref(n)), "pkv_block_refcount")
    return n.value


def pkv_seq_release(a: int, seq_id: int) -> None:
    _check(_L().pkv_seq_release(a, seq_id), "pkv_seq_release")


def pkv_seq_num_blocks(a: int, seq_id: int) -> int:
    n = ctypes.c_int()
    _check(_L().pkv_seq_num_blocks(a, seq_id, ctypes.byref(n)), "pkv_seq_num_blocks")
    return n.value


def pkv_num_free_blocks(a: int) -> int:
    n = ctypes.c_int()
    _check(_L().pkv_num_free_blocks(a, ctypes.byref(n)), "pkv_num_free_blocks")
    return n.value


def pkv_free_list(a: int) -> np.ndarray:
    out = np.empty(pkv_num_free_blocks(a), dtype=np.int32)
    n = ctypes.c_int()
    _check(_L().pkv_free_list(a, out.ctypes.data, len(out), ctypes.byref(n)), "pkv_free_list")
    return out[:n.value]


def _out_array(out, shape, dtype):
    if out is None:
        return np.empty(shape, dtype=dtype)
    if out.shape != tuple(shape) or out.dtype != dtype or not out.flags["C_CONTIGUOUS"]:
        raise ValueError(f"out must be a contiguous {np.dtype(dtype).name} array of shape {tuple(shape)}")
    return out


def pkv_get_block_tables(a: int, seq_ids, max_blocks: int, out: np.ndarray | None = None) -> np.ndarray:
    s = _np(seq_ids, np.int64)
    out = _out_array(out, (len(s), max_blocks), np.int32)
    _check(_L().pkv_get_block_tables(a, s.ctypes.data, len(s), max_blocks, out.ctypes.data), "pkv_get_block_tables")
    return out


def pkv_slot_mapping(a: int, seq_ids, positions, out: np.ndarray | None = None) -> np.ndarray:
    s, p = _np(seq_ids, np.int64), _np(positions, np.int64)
    if s.shape != p.shape:
        raise ValueError("seq_ids and positions must have the same length")
    out = _out_array(out, (len(s),), np.int64)
    _check(_L().pkv_slot_mapping(a, s.ctypes.data, p.ctypes.data, len(s), out.ctypes.data), "pkv_slot_mapping")
    return out


def _out_flat(out, n: int, dtype, what: str) -> np.ndarray:
    """A contiguous array of `dtype` with room for n elements (new if out is None)."""
    if out is None:
        return np.empty(n, dtype=dtype)
    if out.dtype != dtype or not out.flags["C_CONTIGUOUS"] or out.size < n:
        raise ValueError(f"{what} must be a contiguous {np.dtype(dtype).name} array of at least {n} elements")
    return out


def pkv_stage_prefill(a: int, seq_ids, p0, p1, max_blocks: int, slots_out=None, cu_out=None, ctx_out=None,
                      tables_out=None):
    """Reserve and write one chunked prefill call's host inputs (see pkv.h); returns (slots
    [sum(p1 - p0)], cu [n + 1], ctx [n], tables [n][max_blocks]) as views of the outputs."""
    s, b, e = _np(seq_ids, np.int64), _np(p0, np.int64), _np(p1, np.int64)
    if not (s.shape == b.shape == e.shape) or s.ndim != 1:
        raise ValueError("seq_ids, p0 and p1 must be 1-D of the same length")
    n = len(s)
    total = int((e - b).sum()) if n else 0
    slots = _out_flat(slots_out, max(total, 0), np.int64, "slots_out")
    cu = _out_flat(cu_out, n + 1, np.int32, "cu_out")
    ctx = _out_flat(ctx_out, n, np.int32, "ctx_out")
    tables = _out_flat(tables_out, n * max_blocks, np.int32, "tables_out")
    _check(_L().pkv_stage_prefill(a, s.ctypes.data, b.ctypes.data, e.ctypes.data, n, max_blocks, slots.ctypes.data,
                                  cu.ctypes.data, ctx.ctypes.data, tables.ctypes.data), "pkv_stage_prefill")
    return (slots.reshape(-1)[:total], cu.reshape(-1)[:n + 1], ctx.reshape(-1)[:n],
            tables.reshape(-1)[:n * max_blocks].reshape(n, max_blocks))


def pkv_stage_decode(a: int, seq_ids, pos, n_pad: int, max_blocks: int, tables_out=None, slots_out=None,
                     lens_out=None):
    """Reserve and write one decode step's host inputs, padded to n_pad rows (see pkv.h);
    returns (tables [n_pad][max_blocks], slots [n_pad], lens [n_pad])."""
    s, p = _np(seq_ids, np.int64), _np(pos, np.int64)
    if s.shape != p.shape or s.ndim != 1:
        raise ValueError("seq_ids and pos must be 1-D of the same length")
    tables = _out_flat(tables_out, n_pad * max_blocks, np.int32, "tables_out")
    slots = _out_flat(slots_out, n_pad, np.int64, "slots_out")
    lens = _out_flat(lens_out, n_pad, np.int32, "lens_out")
    _check(_L().pkv_stage_decode(a, s.ctypes.data, p.ctypes.data, len(s), n_pad, max_blocks, tables.ctypes.data,
                                 slots.ctypes.data, lens.ctypes.data), "pkv_stage_decode")
    return (tables.reshape(-1)[:n_pad * max_blocks].reshape(n_pad, max_blocks), slots.reshape(-1)[:n_pad],
            lens.reshape(-1)[:n_pad])


# ----------------------------------------------------------------------------- pool
def pkv_pool_create(num_blocks: int, block_size: int, n_kv_heads: int, head_dim: int, kv_dtype: int) -> int:
    h = ctypes.c_void_p()
    _check(_L().pkv_pool_create(num_blocks, block_size, n_kv_heads, head_dim, kv_dtype, ctypes.byref(h)),
           "pkv_pool_create")
    return h.value


def pkv_pool_destroy(pool: int) -> None:
    _check(_L().pkv_pool_destroy(pool), "pkv_pool_destroy")


def pkv_pool_allocator(pool: int) -> int:
    h = ctypes.c_void_p()
    _check(_L().pkv_pool_allocator(pool, ctypes.byref(h)), "pkv_pool_allocator")
    return h.value


def pkv_pool_raw(pool: int):
    kv, kvb, sc, scb = ctypes.c_void_p(), ctypes.c_size_t(), ctypes.c_void_p(), ctypes.c_size_t()
    _check(_L().pkv_pool_raw(pool, ctypes.byref(kv), ctypes.byref(kvb), ctypes.byref(sc), ctypes.byref(scb)),
           "pkv_pool_raw")
    return kv.value, kvb.value, sc.value or 0, scb.value


def pkv_pool_copy_block(pool: int, src_block: int, dst_block: int, stream=None) -> None:
    _check(_L().pkv_pool_copy_block(pool, src_block, dst_block, _stream(stream)), "pkv_pool_copy_block")


def pkv_check_device_error(pool: int) -> int:
    """Status code of the pool's device error word (read and cleared)."""
    return _L().pkv_check_device_error(pool)


def pkv_append(pool: int, k_new, v_new, slot_mapping, stream=None) -> None:
    """k_new, v_new: bf16 CUDA tensors [N, Hkv, D]; slot_mapping: int64 CUDA tensor [N]."""
    N = slot_mapping.shape[0]
    _check(_L().pkv_append(pool, _dev(k_new, "bf16", "k_new"), _dev(v_new, "bf16", "v_new"),
                           _dev(slot_mapping, "i64", "slot_mapping"), N, _stream(stream)), "pkv_append")


def pkv_append_rope(pool: int, k_new, v_new, slot_mapping, positions, rope_base: float, q=None, stream=None) -> None:
    """k_new (and q, if given) are rotated in place at `positions` (int64 CUDA [N]), then K/V are
    appended like pkv_append."""
    N = slot_mapping.shape[0]
    _check(_L().pkv_append_rope(pool, _dev(k_new, "bf16", "k_new"), _dev(v_new, "bf16", "v_new"),
                                _dev(slot_mapping, "i64", "slot_mapping"), _dev(positions, "i64", "positions"), N,
                                float(rope_base), _dev(q, "bf16", "q") if q is not None else None,
                                q.shape[1] if q is not None else 0, _stream(stream)), "pkv_append_rope")


def pkv_decode_attention(pool: int, q, block_tables, context_lens, scale: float, out, workspace,
                         stream=None) -> None:
    """q/out: bf16 CUDA [B, Hq, D]; block_tables int32 [B, max_blocks]; context_lens int32 [B];
    workspace: uint8 CUDA tensor of pkv_decode_workspace_bytes() bytes, zeroed before first use."""
    B, Hq = q.shape[0], q.shape[1]
    _check(_L().pkv_decode_attention(pool, _dev(q, "bf16", "q"), _dev(block_tables, "i32", "block_tables"),
                                     block_tables.shape[1], _dev(context_lens, "i32", "context_lens"), B, Hq,
                                     float(scale), _dev(out, "bf16", "out"), _dev(workspace, "u8", "workspace"),
                                     workspace.numel(), _stream(stream)), "pkv_decode_attention")


def pkv_decode_step(pool: int, k_new, v_new, slot_mapping, q, block_tables, context_lens, scale: float, out, workspace,
                    stream=None) -> None:
    """pkv_append(k_new, v_new, slot_mapping) then pkv_decode_attention(...), launched back to back."""
    B, Hq = q.shape[0], q.shape[1]
    _check(_L().pkv_decode_step(pool, _dev(k_new, "bf16", "k_new"), _dev(v_new, "bf16", "v_new"),
                                _dev(slot_mapping, "i64", "slot_mapping"), slot_mapping.shape[0], _dev(q, "bf16", "q"),
                                _dev(block_tables, "i32", "block_tables"), block_tables.shape[1],
                                _dev(context_lens, "i32", "context_lens"), B, Hq, float(scale), _dev(out, "bf16", "out"),
                                _dev(workspace, "u8", "workspace"), workspace.numel(), _stream(stream)),
           "pkv_decode_step")


def pkv_prefill_attention(pool: int, q, cu_q_lens, max_q_len: int, block_tables, context_lens, scale: float, out,
                          stream=None) -> None:
    """q/out: bf16 CUDA [total_q, Hq, 128]; cu_q_lens int32 [B+1]; block_tables int32 [B, max_blocks];
    context_lens int32 [B] (the chunks' K/V already appended)."""
    B, Hq = context_lens.shape[0], q.shape[1]
    _check(_L().pkv_prefill_attention(pool, _dev(q, "bf16", "q"), _dev(cu_q_lens, "i32", "cu_q_lens"), int(max_q_len),
                                      _dev(block_tables, "i32", "block_tables"), block_tables.shape[1],
                                      _dev(context_lens, "i32", "context_lens"), B, Hq, float(scale),
                                      _dev(out, "bf16", "out"), _stream(stream)), "pkv_prefill_attention")


def pkv_prefill_step(pool: int, k_new, v_new, slot_mapping, q, cu_q_lens, max_q_len: int, block_tables, context_lens,
                     scale: float, out, stream=None) -> None:
    """pkv_append(k_new, v_new, slot_mapping) then pkv_prefill_attention(...), launched back to back."""
    B, Hq = context_lens.shape[0], q.shape[1]
    _check(_L().pkv_prefill_step(pool, _dev(k_new, "bf16", "k_new"), _dev(v_new, "bf16", "v_new"),
                                 _dev(slot_mapping, "i64", "slot_mapping"), slot_mapping.shape[0], _dev(q, "bf16", "q"),
                                 _dev(cu_q_lens, "i32", "cu_q_lens"), int(max_q_len),
                                 _dev(block_tables, "i32", "block_tables"), block_tables.shape[1],
                                 _dev(context_lens, "i32", "context_lens"), B, Hq, float(scale), _dev(out, "bf16", "out"),
                                 _stream(stream)), "pkv_prefill_step")


def pkv_decode_step_rope(pool: int, k_new, v_new, slot_mapping, positions, rope_base: float, q, block_tables,
                         context_lens, scale: float, out, workspace, stream=None) -> None:
    """pkv_append_rope(k_new, v_new, slot_mapping, positions, rope_base, q) then pkv_decode_attention(...)."""
    B, Hq = q.shape[0], q.shape[1]
    _check(_L().pkv_decode_step_rope(pool, _dev(k_new, "bf16", "k_new"), _dev(v_new, "bf16", "v_new"),
                                     _dev(slot_mapping, "i64", "slot_mapping"), _dev(positions, "i64", "positions"),
                                     slot_mapping.shape[0], float(rope_base), _dev(q, "bf16", "q"),
                                     _dev(block_tables, "i32", "block_tables"), block_tables.shape[1],
                                     _dev(context_lens, "i32", "context_lens"), B, Hq, float(scale),
                                     _dev(out, "bf16", "out"), _dev(workspace, "u8", "workspace"), workspace.numel(),
                                     _stream(stream)), "pkv_decode_step_rope")


def pkv_decode_workspace_bytes(pool: int, B: int, n_q_heads: int, max_blocks: int) -> int:
    n = ctypes.c_size_t()
    _check(_L().pkv_decode_workspace_bytes(pool, B, n_q_heads, max_blocks, ctypes.byref(n)),
           "pkv_decode_workspace_bytes")
    return n.value


def pkv_decode_workspace_init(workspace, stream=None) -> None:
    _check(_L().pkv_decode_workspace_init(_dev(workspace, "u8", "workspace"), workspace.numel(), _stream(stream)),
           "pkv_decode_workspace_init")


def pkv_decode_attention_static(pool: int, q, block_tables, context_lens, scale: float, out, stream=None) -> None:
    """pkv_decode_attention with the library's fixed device scratch instead of a caller workspace
    (for callers that cannot allocate device memory); no allocation happens in this call."""
    B, Hq = q.shape[0], q.shape[1]
    rc = _L().pkv_decode_attention_static(pool, _dev(q, "bf16", "q"), _dev(block_tables, "i32", "block_tables"),
                                          block_tables.shape[1], _dev(context_lens, "i32", "context_lens"), B, Hq,
                                          float(scale), _dev(out, "bf16", "out"), _stream(stream))
    if rc == PKV_ERR_INVALID_ARG:
        need = pkv_decode_workspace_bytes(pool, B, Hq, block_tables.shape[1])
        if need > PKV_STATIC_WORKSPACE_BYTES:
            raise PKVError(rc, f"pkv_decode_attention_static: needs {need} bytes of scratch, the fixed limit is "
                               f"{PKV_STATIC_WORKSPACE_BYTES}")
    _check(rc, "pkv_decode_attention_static")


def pkv_stage_copy(dst, src, nbytes: int | None = None, stream=None) -> None:
    """Kernel-driven copy between torch tensors: each one a CUDA tensor or a pinned CPU tensor,
    contiguous; nbytes defaults to the smaller of the two sizes (a multiple of 16)."""
    def ptr(t, what):
        import torch
        if not isinstance(t, torch.Tensor) or not t.is_contiguous():
            raise TypeError(f"{what}: expected a contiguous torch tensor")
        if not t.is_cuda and not t.is_pinned():
            raise ValueError(f"{what}: a CPU tensor must be pinned")
        return t.data_ptr(), t.numel() * t.element_size()
    d, dn = ptr(dst, "dst")
    s, sn = ptr(src, "src")
    n = min(dn, sn) if nbytes is None else int(nbytes)
    if n < 0 or n > dn or n > sn:
        raise ValueError(f"pkv_stage_copy: {n} bytes do not fit the buffers ({dn}, {sn})")
    _check(_L().pkv_stage_copy(d, s, n, _stream(stream)), "pkv_stage_copy")


def pkv_kv_bytes(n_layers: int, n_kv_heads: int, head_dim: int, n_tokens: int, batch: int,
                 bytes_per_elem: float) -> int:
    return _L().pkv_kv_bytes(n_layers, n_kv_heads, head_dim, n_tokens, batch, bytes_per_elem)


def pkv_status_str(s: int) -> str:
    try:
        return _L().pkv_status_str(s).decode()
    except Exception:  # library not loadable: still report the code
        return f"status {s}"


# ----------------------------------------------------------------------------- convenience
class KVPool:
    """Owns a pool handle (destroyed with the object) and remembers its geometry."""

    def __init__(self, num_blocks: int, block_size: int, n_kv_heads: int, head_dim: int,
                 kv_dtype: int = PKV_KV_BF16):
        self.handle = pkv_pool_create(num_blocks, block_size, n_kv_heads, head_dim, kv_dtype)
        self.allocator = pkv_pool_allocator(self.handle)
        self.num_blocks, self.block_size, self.n_kv_heads, self.head_dim = num_blocks, block_size, n_kv_heads, head_dim
        self.kv_dtype = kv_dtype

    def close(self):
        if getattr(self, "handle", None):
            pkv_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def pkv_debug_reload_env() -> None:
    """Re-read the library's PKV_TEST_* / PKV_ATTN_* environment settings (tests switching the
    bounded-wait hooks on and off)."""
    _check(_L().pkv_debug_reload_env(), "pkv_debug_reload_env")
