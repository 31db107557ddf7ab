"""One in-flight-batching decode step over a paged pool, driven through the C ABI.

``DecodeStep`` takes a workload description (batch, heads, block size, context
lengths, an allocation script and seeded inputs), builds the pool on the GPU,
replays the allocation script on the pool's allocator, writes every sequence's
history K/V with ``pkv_append`` and keeps the step's inputs resident.  ``step()``
is the hot path: append the new token of every sequence, then decode attention
over the grown contexts.  ``step_host()`` is the same step starting from the
caller's host arrays (q, new K/V and lengths copied into a pinned staging buffer,
block tables and slot mapping written there by the allocator, one copy to the
device, the output copied back).
"""
from __future__ import annotations

import math

import numpy as np

from . import _L, _check
from . import (KV_DTYPES, KVPool, pkv_allocator_set_free_order, pkv_append,
               pkv_decode_attention, pkv_decode_step, pkv_decode_workspace_bytes, pkv_get_block_tables,
               pkv_num_free_blocks, pkv_pool_copy_block, pkv_prefill_attention, pkv_prefill_step, pkv_seq_release,
               pkv_seq_reserve, pkv_seq_share_prefix, pkv_slot_mapping, pkv_stage_copy)

def replay(allocator: int, ops) -> None:
    for op in ops:
        if op[0] == "reserve":
            pkv_seq_reserve(allocator, op[1], op[2])
        else:
            pkv_seq_release(allocator, op[1])


def _bf16(torch, arr: np.ndarray, device):
    return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16).to(device)


class DecodeStep:
    def __init__(self, w, device: str = "cuda"):
        import torch
        self.torch, self.w, self.device = torch, w, device
        self.pool = KVPool(w.num_blocks, w.block_size, w.Hkv, w.D, KV_DTYPES[w.kv_dtype])
        a = self.pool.allocator
        pkv_allocator_set_free_order(a, w.free_order)
        replay(a, w.alloc_ops)
        self.max_blocks = max(1, w.max_blocks())
        self.tables_host = pkv_get_block_tables(a, w.seq_ids, self.max_blocks)
        self.scale = 1.0 / math.sqrt(w.D)
        for t0, t1 in w.hist_chunks():
            seqs, pos = w.hist_positions(t0, t1)
            slots = torch.from_numpy(pkv_slot_mapping(a, seqs, pos)).to(device)
            pkv_append(self.pool.handle, _bf16(torch, w.history_k(t0, t1), device),
                       _bf16(torch, w.history_v(t0, t1), device), slots)
        torch.cuda.synchronize()
        self.q = _bf16(torch, w.query(), device)
        self.k_new = _bf16(torch, w.new_k(), device)
        self.v_new = _bf16(torch, w.new_v(), device)
        self.slots_new_host = pkv_slot_mapping(a, w.seq_ids, w.lens) if w.append else np.zeros(0, np.int64)
        self.slots_new = torch.from_numpy(self.slots_new_host).to(device)
        self.tables = torch.from_numpy(self.tables_host).to(device)
        self.lens_host = w.attend_lens.astype(np.int32)
        self.lens = torch.from_numpy(self.lens_host).to(device)
        self.out = torch.empty(w.B, w.Hq, w.D, dtype=torch.bfloat16, device=device)
        self.ws_bytes = pkv_decode_workspace_bytes(self.pool.handle, w.B, w.Hq, self.max_blocks)
        self.workspace = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=device)
        self._host = None
        self.batch = w.B

    def limit_batch(self, n: int) -> None:
        """Run the step on the first n sequences only (same pool); used to size profiling runs."""
        torch, w = self.torch, self.w
        n = max(1, min(n, w.B))
        self.q, self.k_new, self.v_new = self.q[:n], self.k_new[:n], self.v_new[:n]
        self.slots_new = self.slots_new[:n] if w.append else self.slots_new
        self.slots_new_host = self.slots_new_host[:n] if w.append else self.slots_new_host
        self.tables, self.tables_host = self.tables[:n], self.tables_host[:n]
        self.lens, self.lens_host = self.lens[:n], self.lens_host[:n]
        self.out = self.out[:n]
        self.batch = n
        self._host = None  # host staging (and its captured graph) follows the batch

    def append(self, stream=None):
        if self.w.append:
            pkv_append(self.pool.handle, self.k_new, self.v_new, self.slots_new, stream)

    def attention(self, stream=None):
        pkv_decode_attention(self.pool.handle, self.q, self.tables, self.lens, self.scale, self.out, self.workspace,
                             stream)

    def step(self, stream=None, fused: bool = True):
        """Append the new tokens, then attend.  fused: one pkv_decode_step call (the attention
        kernel's set-up overlaps the append); otherwise pkv_append then pkv_decode_attention."""
        if fused and self.w.append:
            pkv_decode_step(self.pool.handle, self.k_new, self.v_new, self.slots_new, self.q, self.tables, self.lens,
                            self.scale, self.out, self.workspace, stream)
        else:
            self.append(stream)
            self.attention(stream)
        return self.out

    # --- end to end from host buffers
    def _prepare_host(self):
        """One pinned staging buffer holding every input of a step (q, new K/V, block tables,
        context lengths, slots) and a device buffer of the same layout whose slices are the
        kernel arguments, so a step needs one host-to-device copy and one copy back (both
        pkv_stage_copy: the SMs move these few hundred KB faster than a copy engine starts)."""
        torch, w = self.torch, self.w
        n = self.batch
        parts = [("q", (n, w.Hq, w.D), np.int16), ("k", (n, w.Hkv, w.D), np.int16),
                 ("v", (n, w.Hkv, w.D), np.int16), ("tables", (n, self.max_blocks), np.int32),
                 ("lens", (n,), np.int32), ("slots", (n if w.append else 0,), np.int64)]
        offs, total = {}, 0
        for name, shape, dt in parts:
            offs[name] = total
            total += (int(np.prod(shape)) * np.dtype(dt).itemsize + 255) // 256 * 256
        hbuf = torch.empty(total, dtype=torch.uint8).pin_memory()
        dbuf = torch.empty(total, dtype=torch.uint8, device=self.device)
        hnp = hbuf.numpy()
        H, Dv = {}, {}
        tdt = {np.int16: torch.int16, np.int32: torch.int32, np.int64: torch.int64}
        for name, shape, dt in parts:
            nbytes = int(np.prod(shape)) * np.dtype(dt).itemsize
            H[name] = hnp[offs[name]:offs[name] + nbytes].view(dt).reshape(shape)
            Dv[name] = dbuf[offs[name]:offs[name] + nbytes].view(tdt[dt]).view(shape)
        # the caller's inputs of the step, in ordinary (pageable) host memory: every host-driven
        # step copies them into the pinned staging buffer first
        src = {"q": np.ascontiguousarray(w.query()[:n]).view(np.int16),
               "k": np.ascontiguousarray(w.new_k()[:n]).view(np.int16),
               "v": np.ascontiguousarray(w.new_v()[:n]).view(np.int16),
               "lens": np.ascontiguousarray(self.lens_host[:n])}
        # the allocator writes tables and slots straight into the staging buffer; the sequence
        # ids and positions are fixed for the batch, so every host address is taken once here
        ids = np.ascontiguousarray(w.seq_ids[:n], dtype=np.int64)
        pos = np.ascontiguousarray(w.lens[:n], dtype=np.int64)
        ptrs = (ids.ctypes.data, pos.ctypes.data, H["tables"].ctypes.data, H["slots"].ctypes.data)
        self._host = {"hbuf": hbuf, "dbuf": dbuf, "H": H, "src": src, "ids": ids, "pos": pos, "ptrs": ptrs,
                      "q": Dv["q"].view(torch.bfloat16), "k": Dv["k"].view(torch.bfloat16),
                      "v": Dv["v"].view(torch.bfloat16), "tables": Dv["tables"], "lens": Dv["lens"],
                      "slots": Dv["slots"], "out": torch.empty(n, w.Hq, w.D, dtype=torch.int16).pin_memory()}

    def _issue_host_step(self, stream):
        """Copy-in, the step, copy-out, on `stream` (no synchronisation)."""
        torch, w, X = self.torch, self.w, self._host
        pkv_stage_copy(X["dbuf"], X["hbuf"], stream=stream)
        if w.append:
            pkv_decode_step(self.pool.handle, X["k"], X["v"], X["slots"], X["q"], X["tables"], X["lens"], self.scale,
                            self.out, self.workspace, stream)
        else:
            pkv_decode_attention(self.pool.handle, X["q"], X["tables"], X["lens"], self.scale, self.out,
                                 self.workspace, stream)
        pkv_stage_copy(X["out"], self.out, stream=stream)

    def step_host(self, stream=None, graph: bool = True):
        """Host-to-host step; returns (h2d_bytes, d2h_bytes).  The step's q / new K / new V are
        copied from the caller's host arrays into the pinned staging buffer, the allocator writes
        the block tables and the slot mapping next to them, one copy takes every input to the
        device, the fused step runs, and the output comes back.  With `graph` the copy-in, step
        and copy-out are captured once as a CUDA graph and replayed (the launch-bound part of a
        decode step, "TensorRT-LLM 推理加速实战" §7.1); the staging buffer is read at replay."""
        torch, w, a = self.torch, self.w, self.pool.allocator
        if self._host is None:
            self._prepare_host()
        X = self._host
        n = self.batch
        for name in ("q", "k", "v", "lens"):
            np.copyto(X["H"][name], X["src"][name])
        lib = _L()
        ids, pos, tables, slots = X["ptrs"]
        _check(lib.pkv_get_block_tables(a, ids, n, self.max_blocks, tables), "pkv_get_block_tables")
        if w.append:
            _check(lib.pkv_slot_mapping(a, ids, pos, n, slots), "pkv_slot_mapping")
        if not graph:
            self._issue_host_step(stream)
        else:
            if X.get("graph") is None:
                self._issue_host_step(None)  # warm-up outside capture (plans, modules)
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                side = torch.cuda.Stream()
                side.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(side):
                    with torch.cuda.graph(g, stream=side):
                        self._issue_host_step(side)
                torch.cuda.current_stream().wait_stream(side)
                X["graph"] = g
            X["graph"].replay()
        torch.cuda.current_stream().synchronize()
        return X["hbuf"].numel(), X["out"].numel() * 2

    def out_host(self) -> np.ndarray:
        return self.out.view(self.torch.int16).cpu().numpy().view(np.uint16)

    def pool_bytes_host(self):
        """Copy the device pool bytes (and fp8 scales) to host numpy arrays."""
        from . import pkv_pool_raw
        kv_ptr, kv_bytes, sc_ptr, sc_bytes = pkv_pool_raw(self.pool.handle)
        kv = _wrap_device(kv_ptr, kv_bytes).cpu().numpy()
        sc = _wrap_device(sc_ptr, sc_bytes).cpu().numpy().view(np.float32) if sc_bytes else np.zeros(0, np.float32)
        return kv, sc

    def close(self):
        self.pool.close()


class PrefixDecode:
    """A decode step over children that share one prompt prefix (block reuse).

    share=True: the parent sequence takes the prefix (reserve + pkv_append), every child is forked
    from it with pkv_seq_share_prefix (the whole prefix blocks are aliased; a partial last block is
    copied with pkv_pool_copy_block), appends its own suffix, and the parent is released.
    share=False: every child holds and writes its own copy of the prefix (the same logical
    contexts without reuse, for comparison).  step()/attention() are the same calls as for any
    other batch: the attention kernel does not know which blocks are shared."""

    def __init__(self, sc, share: bool = True, device: str = "cuda"):
        import torch
        self.torch, self.sc, self.share, self.device = torch, sc, share, device
        nb = sc.num_blocks if share else sc.blocks_unshared() + 4
        self.pool = KVPool(nb, sc.block_size, sc.Hkv, sc.D, KV_DTYPES[sc.kv_dtype])
        a = self.pool.allocator
        pk, pv = sc.prefix_kv()
        dpk, dpv = _bf16(torch, pk, device), _bf16(torch, pv, device)
        P = sc.P
        self.cow_copies = 0
        if share:
            pkv_seq_reserve(a, sc.parent, P)
            pkv_append(self.pool.handle, dpk, dpv,
                       torch.from_numpy(pkv_slot_mapping(a, [sc.parent] * P, np.arange(P))).to(device))
        for b in range(sc.B):
            total = P + int(sc.suffix_lens[b]) + 1
            if share:
                cs, cd = pkv_seq_share_prefix(a, sc.parent, b, P)
                if cs >= 0:
                    pkv_pool_copy_block(self.pool.handle, cs, cd)
                    self.cow_copies += 1
                pkv_seq_reserve(a, b, total)
            else:
                pkv_seq_reserve(a, b, total)
                pkv_append(self.pool.handle, dpk, dpv,
                           torch.from_numpy(pkv_slot_mapping(a, [b] * P, np.arange(P))).to(device))
            n = int(sc.suffix_lens[b])
            if n:
                sk, sv = sc.suffix_kv(b)
                slots = pkv_slot_mapping(a, [b] * n, np.arange(P, P + n))
                pkv_append(self.pool.handle, _bf16(torch, sk, device), _bf16(torch, sv, device),
                           torch.from_numpy(slots).to(device))
        if share:
            pkv_seq_release(a, sc.parent)
        torch.cuda.synchronize()
        self.blocks_held = nb - pkv_num_free_blocks(a)
        seqs = np.arange(sc.B)
        self.max_blocks = sc.max_blocks
        self.tables_host = pkv_get_block_tables(a, seqs, self.max_blocks)
        self.tables = torch.from_numpy(self.tables_host).to(device)
        self.lens_host = sc.attend_lens
        self.lens = torch.from_numpy(self.lens_host).to(device)
        self.slots_new = torch.from_numpy(pkv_slot_mapping(a, seqs, P + sc.suffix_lens)).to(device)
        k, v, q = sc.step_inputs()
        self.k_new, self.v_new, self.q = _bf16(torch, k, device), _bf16(torch, v, device), _bf16(torch, q, device)
        self.scale = 1.0 / math.sqrt(sc.D)
        self.out = torch.empty(sc.B, sc.Hq, sc.D, dtype=torch.bfloat16, device=device)
        ws = pkv_decode_workspace_bytes(self.pool.handle, sc.B, sc.Hq, self.max_blocks)
        self.workspace = torch.zeros(ws, dtype=torch.uint8, device=device)

    def step(self, stream=None):
        pkv_decode_step(self.pool.handle, self.k_new, self.v_new, self.slots_new, self.q, self.tables, self.lens,
                        self.scale, self.out, self.workspace, stream)
        return self.out

    def attention(self, stream=None):
        pkv_decode_attention(self.pool.handle, self.q, self.tables, self.lens, self.scale, self.out, self.workspace,
                             stream)

    def out_host(self) -> np.ndarray:
        return self.out.view(self.torch.int16).cpu().numpy().view(np.uint16)

    def close(self):
        self.pool.close()


class PrefillStep:
    """One chunked-context step through the C ABI: the pool holds every sequence's past tokens
    (appended at set-up); step() appends the chunks' K/V and runs the prefill attention
    (pkv_prefill_step), attention() runs the attention alone."""

    def __init__(self, sc, device: str = "cuda"):
        import torch
        self.torch, self.sc, self.device = torch, sc, device
        self.pool = KVPool(sc.num_blocks, sc.block_size, sc.Hkv, sc.D, KV_DTYPES[sc.kv_dtype])
        a = self.pool.allocator
        pkv_allocator_set_free_order(a, sc.free_order)
        for b in range(sc.B):
            pkv_seq_reserve(a, b, int(sc.ctx[b]))
        chunk_tokens = 1 << 16
        for b in range(sc.B):
            for t0 in range(0, int(sc.past[b]), chunk_tokens):
                t1 = min(int(sc.past[b]), t0 + chunk_tokens)
                k, v = sc.kv(b, t0, t1)
                slots = pkv_slot_mapping(a, [b] * (t1 - t0), np.arange(t0, t1))
                pkv_append(self.pool.handle, _bf16(torch, k, device), _bf16(torch, v, device),
                           torch.from_numpy(slots).to(device))
        torch.cuda.synchronize()
        seqs, pos = sc.chunk_slots_positions()
        self.slots = torch.from_numpy(pkv_slot_mapping(a, seqs, pos)).to(device)
        k, v = sc.chunk_kv()
        self.k_new, self.v_new = _bf16(torch, k, device), _bf16(torch, v, device)
        self.q = _bf16(torch, sc.query(), device)
        self.cu_q = torch.from_numpy(sc.cu_q).to(device)
        self.max_q = int(sc.chunk.max()) if sc.B else 0
        self.tables_host = pkv_get_block_tables(a, np.arange(sc.B), sc.max_blocks)
        self.tables = torch.from_numpy(self.tables_host).to(device)
        self.ctx = torch.from_numpy(sc.ctx).to(device)
        self.scale = 1.0 / math.sqrt(sc.D)
        self.out = torch.zeros(int(sc.cu_q[-1]), sc.Hq, sc.D, dtype=torch.bfloat16, device=device)

    def step(self, stream=None):
        pkv_prefill_step(self.pool.handle, self.k_new, self.v_new, self.slots, self.q, self.cu_q, self.max_q,
                         self.tables, self.ctx, self.scale, self.out, stream)
        return self.out

    def append(self, stream=None):
        pkv_append(self.pool.handle, self.k_new, self.v_new, self.slots, stream)

    def attention(self, stream=None):
        pkv_prefill_attention(self.pool.handle, self.q, self.cu_q, self.max_q, self.tables, self.ctx, self.scale,
                              self.out, stream)

    def out_host(self) -> np.ndarray:
        return self.out.view(self.torch.int16).cpu().numpy().view(np.uint16)

    def close(self):
        self.pool.close()


def _wrap_device(ptr: int, nbytes: int):
    """A torch uint8 CUDA tensor viewing [ptr, ptr + nbytes) (borrowed memory)."""
    import torch

    class _Arr:
        __cuda_array_interface__ = {"shape": (nbytes,), "typestr": "|u1", "data": (ptr, False), "version": 3,
                                    "strides": None}

    return torch.as_tensor(_Arr(), device="cuda")
