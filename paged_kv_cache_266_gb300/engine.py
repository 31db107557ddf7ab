"""In-flight batching decode loop for one attention layer over a paged pool.

"TensorRT-LLM 深度实战" (chenxutan.com), §3.2 (continuous / in-flight batching): every step
finished sequences leave and release their pages (§3.1 release), waiting ones join, and the
running batch takes one forward step.  "TensorRT-LLM 推理加速实战" (socake.github.io), §7.1:
decode steps are launch-bound at small batch and are replayed from CUDA graphs, one graph per
batch-size bucket because a graph is fixed to its shapes.

Each step here:
  1. releases the finished sequences' blocks (pkv_seq_release);
  2. admits joining sequences.  Without chunked context their prompt's K/V are written at once
     (pkv_seq_reserve + pkv_append, as a prefill would leave them).  With chunked context
     ("TensorRT-LLM 深度实战" §7.3) a joiner's prompt is prefilled `chunk` tokens per step: one
     pkv_prefill_step appends every prefilling sequence's next chunk and attends its queries
     causally (its slots, chunk offsets and tables written by one pkv_stage_prefill), and the
     sequence decodes from the step after its last chunk.  With a system
     prompt (prefix caching, "TensorRT-LLM 推理加速实战" §8 KV cache reuse) the shared prefix
     is cached once and every joiner forks it (pkv_seq_share_prefix) instead of prefilling it;
  3. gives every decoding sequence room for one more token and writes block tables, new-token
     slots and context lengths (padding rows included) straight into a pinned staging buffer,
     in one pkv_stage_decode call, next to the step's q / new K / new V;
  4. runs, on the decode batch padded to its bucket, one host-to-device copy, pkv_decode_step
     (append + attention) and the copy of the output back — captured once per bucket as a CUDA
     graph and replayed.  Padding rows have context length 0 and slot -1, so they write nothing
     and read nothing; their outputs are zeros.
"""
from __future__ import annotations

import math

import numpy as np

from . import _L, _check
from . import (KV_DTYPES, KVPool, pkv_append, pkv_decode_step, pkv_decode_workspace_bytes,
               pkv_pool_copy_block, pkv_prefill_step, pkv_seq_release, pkv_seq_reserve,
               pkv_seq_share_prefix, pkv_slot_mapping, pkv_stage_copy)

DEFAULT_BUCKETS = (8, 16, 32, 64, 128, 256, 512, 1024)


class ChunkedContextScheduler:
    """Chunked context ("TensorRT-LLM 深度实战" §7.3): a joining request's input is processed in
    pieces of at most `chunk` tokens, one piece per step, while the other requests decode; a
    request decodes from the step after its last piece.  Requests are kept in admission order.

    With a shared system prompt of `system` tokens every input starts with it; if the prompt is
    cached once and forked into each request (`reuse`, "TensorRT-LLM 推理加速实战" §8 KV cache
    reuse), a request's prefill starts after it.  Pure host bookkeeping, no device work."""

    def __init__(self, chunk: int, system: int = 0, reuse: bool = True):
        if chunk < 1:
            raise ValueError("chunk must be positive")
        self.chunk, self.system, self.reuse = chunk, system, reuse
        self._req: dict[int, list[int]] = {}  # seq -> [input tokens, prefilled, decoded], admission order

    def __len__(self) -> int:
        return len(self._req)

    def finish(self, seq: int) -> None:
        """A decoding request leaves (a request still prefilling cannot finish)."""
        n, done, _ = self._req[seq]
        if done < n:
            raise ValueError(f"sequence {seq} finished before its prompt was prefilled")
        del self._req[seq]

    def admit(self, seq: int, prompt_tokens: int) -> None:
        if seq in self._req:
            raise ValueError(f"sequence {seq} is already admitted")
        self._req[seq] = [self.system + prompt_tokens, self.system if self.reuse else 0, 0]

    def plan(self):
        """This step's work: ([(seq, p0, p1)] pieces prefilled now, positions p0..p1-1; [seq]
        decoding).  The pieces count as prefilled from here on."""
        prefill, decode = [], []
        for seq, r in self._req.items():
            if r[1] < r[0]:
                p1 = min(r[0], r[1] + self.chunk)
                prefill.append((seq, r[1], p1))
                r[1] = p1
            else:
                decode.append(seq)
        return prefill, decode

    def cached(self, seq: int) -> int:
        """Tokens `seq` holds before this step's decode token: its input and its decoded tokens."""
        r = self._req[seq]
        return r[0] + r[2]

    def mark_decoded(self, seqs) -> None:
        for seq in seqs:
            self._req[seq][2] += 1


class _Bucket:
    """Device buffers, pinned staging and (optionally) the captured graph for one batch size."""

    def __init__(self, torch, loop, Bp: int, device):
        sc = loop.script
        self.Bp = Bp
        parts = [("q", (Bp, sc.Hq, sc.D), np.int16), ("k", (Bp, sc.Hkv, sc.D), np.int16),
                 ("v", (Bp, sc.Hkv, sc.D), np.int16), ("tables", (Bp, loop.max_blocks), np.int32),
                 ("lens", (Bp,), np.int32), ("slots", (Bp,), np.int64)]
        offs, total = {}, 0
        for name, shape, dt in parts:
            offs[name] = total
            total += (int(np.prod(shape)) * np.dtype(dt).itemsize + 255) // 256 * 256
        self.hbuf = torch.empty(total, dtype=torch.uint8).pin_memory()
        self.dbuf = torch.empty(total, dtype=torch.uint8, device=device)
        tdt = {np.int16: torch.int16, np.int32: torch.int32, np.int64: torch.int64}
        hnp = self.hbuf.numpy()
        self.H, self.Dv = {}, {}
        for name, shape, dt in parts:
            nbytes = int(np.prod(shape)) * np.dtype(dt).itemsize
            self.H[name] = hnp[offs[name]:offs[name] + nbytes].view(dt).reshape(shape)
            self.Dv[name] = self.dbuf[offs[name]:offs[name] + nbytes].view(tdt[dt]).view(shape)
        self.q = self.Dv["q"].view(torch.bfloat16)
        self.k = self.Dv["k"].view(torch.bfloat16)
        self.v = self.Dv["v"].view(torch.bfloat16)
        self.out = torch.zeros(Bp, sc.Hq, sc.D, dtype=torch.bfloat16, device=device)
        self.out_host = torch.empty(Bp, sc.Hq, sc.D, dtype=torch.int16).pin_memory()
        self.out_np = self.out_host.numpy().view(np.uint16)  # the step's output as the caller sees it
        ws = pkv_decode_workspace_bytes(loop.pool.handle, Bp, sc.Hq, loop.max_blocks)
        self.workspace = torch.zeros(ws, dtype=torch.uint8, device=device)
        self.graphs = {}  # one captured graph per input mode (q/K/V staged on the host or on the device)
        self.out_ptrs = tuple(self.H[k].ctypes.data for k in ("tables", "slots", "lens"))
        self.qkv_bytes = offs["tables"]  # [q | k | v] lead the layout; tables, lens, slots follow

    def run(self, torch, loop, device_inputs: bool = False):
        """Copy the staged inputs in, run the fused step, copy the output out (no sync); both
        copies are pkv_stage_copy (SM-driven: faster than a copy engine at these sizes).  With
        device_inputs the step's q/K/V are already in the device buffer and only the tables,
        lengths and slots cross from the host."""
        if device_inputs:
            pkv_stage_copy(self.dbuf[self.qkv_bytes:], self.hbuf[self.qkv_bytes:])
        else:
            pkv_stage_copy(self.dbuf, self.hbuf)
        pkv_decode_step(loop.pool.handle, self.k, self.v, self.Dv["slots"], self.q, self.Dv["tables"],
                        self.Dv["lens"], loop.scale, self.out, self.workspace)
        pkv_stage_copy(self.out_host, self.out)


class _PrefillStaging:
    """Pinned and device buffers for the small inputs of one chunked prefill call (slots, chunk
    offsets, context lengths, block tables), sized for `tokens` chunk tokens and `seqs`
    sequences: the allocator writes into the pinned copy and one pkv_stage_copy moves it."""

    def __init__(self, torch, tokens: int, seqs: int, max_blocks: int, device):
        self.tokens, self.seqs = tokens, seqs
        parts = [("slots", (tokens,), np.int64), ("cu", (seqs + 1,), np.int32), ("ctx", (seqs,), np.int32),
                 ("tables", (seqs, max_blocks), np.int32)]
        offs, total = {}, 0
        for name, shape, dt in parts:
            offs[name] = total
            total += (int(np.prod(shape)) * np.dtype(dt).itemsize + 255) // 256 * 256
        self.hbuf = torch.empty(total, dtype=torch.uint8).pin_memory()
        self.dbuf = torch.empty(total, dtype=torch.uint8, device=device)
        tdt = {np.int32: torch.int32, np.int64: torch.int64}
        hnp = self.hbuf.numpy()
        self.H, self.D = {}, {}
        for name, shape, dt in parts:
            nbytes = int(np.prod(shape)) * np.dtype(dt).itemsize
            self.H[name] = hnp[offs[name]:offs[name] + nbytes].view(dt).reshape(shape)
            self.D[name] = self.dbuf[offs[name]:offs[name] + nbytes].view(tdt[dt]).view(shape)
        # host addresses the allocator writes to, and the copy's (fixed for the buffer's life)
        self.out_ptrs = tuple(self.H[k].ctypes.data for k in ("slots", "cu", "ctx", "tables"))
        self.copy = (self.dbuf.data_ptr(), self.hbuf.data_ptr(), total)


class DecodeLoop:
    def __init__(self, script, graphs: bool = True, buckets=DEFAULT_BUCKETS, device: str = "cuda",
                 prompts=None, system_seq: int | None = None):
        """prompts: optional {seq_id: (k, v)} of device bf16 tensors [n][Hkv][D] (a joining
        sequence's prompt K/V as its prefill produced them; with chunked context (a script with
        chunk > 0) (k, v, q), q [n][Hq][D] the prompt's queries, rows from the first position the
        request prefills: after the system prompt when it is cached); else drawn from the script.

        Chunked context (script.chunk > 0, "TensorRT-LLM 深度实战" §7.3): a joining sequence's
        prompt is prefilled `chunk` tokens per step (its chunk's K/V appended and its queries
        attending causally, one pkv_prefill_step for all prefilling sequences of the step) and
        the sequence decodes from the step after its last chunk.

        system_seq: the sequence id under which a script's shared system prompt is cached (any id
        no request uses; needed when the script has a system prompt)."""
        import torch
        self.prompts = prompts or {}
        self.torch, self.script, self.graphs, self.device = torch, script, graphs, device
        self.pool = KVPool(script.num_blocks, script.block_size, script.Hkv, script.D, KV_DTYPES[script.kv_dtype])
        self.alloc = self.pool.allocator
        self.max_blocks = -(-script.max_len // script.block_size)
        self.scale = 1.0 / math.sqrt(script.D)
        self.buckets = sorted(buckets)
        self._bk = {}
        # decoding sequences in admission order and the tokens each holds before this step's token
        self._ids = np.zeros(0, dtype=np.int64)
        self._pos = np.zeros(0, dtype=np.int64)
        self.attended_tokens = 0  # context tokens the last step's decode attention read (all sequences)
        self.t = 0
        self.timing = {"admit_s": 0.0, "prepare_s": 0.0, "device_s": 0.0}  # host wall time per phase
        self.scheduler = (ChunkedContextScheduler(script.chunk, script.system, script.reuse) if script.chunk
                          else None)
        self.system_seq = system_seq
        if script.chunk and script.system:
            # prefix caching ("TensorRT-LLM 推理加速实战" §8, KV cache reuse): the shared system
            # prompt is cached once under its own sequence and, with reuse, joiners fork it
            # (without reuse it stays cached, unused, so both schedules hold the same pool)
            if system_seq is None:
                raise ValueError("a script with a system prompt needs system_seq")
            k, v = script.system_kv()
            pkv_seq_reserve(self.alloc, system_seq, script.system)
            slots = pkv_slot_mapping(self.alloc, [system_seq] * script.system, np.arange(script.system))
            to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
            pkv_append(self.pool.handle, to_dev(k), to_dev(v), torch.from_numpy(slots).to(device))
        self.last_prefill = ([], None)  # chunked context: (chunks [(seq, p0, p1)], output bits)
        self._pf = None  # chunked context: staging of the prefill call's small inputs
        self._adm = None  # staging of the joiners' prompt slots

    @property
    def running(self) -> list:
        return self._ids.tolist()

    @property
    def lens(self) -> dict:
        """Tokens each decoding sequence holds before its next step's token."""
        return dict(zip(self._ids.tolist(), self._pos.tolist()))

    def _bucket(self, B: int) -> _Bucket:
        Bp = next((b for b in self.buckets if b >= B), None)
        if Bp is None:
            raise ValueError(f"batch {B} exceeds the largest bucket {self.buckets[-1]}")
        if Bp not in self._bk:
            self._bk[Bp] = _Bucket(self.torch, self, Bp, self.device)
        return self._bk[Bp]

    def _admit(self, joined):
        """Admit the step's joining sequences: every prompt reserved and its slots written by one
        pkv_stage_prefill (positions 0 .. n-1) into pinned staging, moved by one pkv_stage_copy,
        then each prompt's K/V appended from its slice of the staged slots."""
        torch = self.torch
        n = len(joined)
        rows = np.zeros((3, n), dtype=np.int64)  # seq ids, first position (0), prompt length
        rows[0] = [s for s, _ in joined]
        rows[2] = [m for _, m in joined]
        total = int(rows[2].sum())
        if self._adm is None or self._adm.tokens < total or self._adm.seqs < n:
            old = self._adm
            self._adm = _PrefillStaging(torch, max(total, 2 * old.tokens if old else total, 1),
                                        max(n, 2 * old.seqs if old else n), self.max_blocks, self.device)
        S = self._adm
        lib = _L()
        r = rows.ctypes.data
        _check(lib.pkv_stage_prefill(self.alloc, r, r + 8 * n, r + 16 * n, n, self.max_blocks, *S.out_ptrs),
               "pkv_stage_prefill")
        if total:
            _check(lib.pkv_stage_copy(*S.copy, torch.cuda.current_stream().cuda_stream), "pkv_stage_copy")
        off = 0
        for seq, m in joined:
            if m:
                if seq in self.prompts:
                    dk, dv = self.prompts[seq]
                else:
                    k, v = self.script.prompt_kv(seq, m)
                    dk = torch.from_numpy(np.ascontiguousarray(k).view(np.int16)).view(torch.bfloat16).to(self.device)
                    dv = torch.from_numpy(np.ascontiguousarray(v).view(np.int16)).view(torch.bfloat16).to(self.device)
                pkv_append(self.pool.handle, dk, dv, S.D["slots"][off:off + m])
                off += m
        self._ids = np.concatenate([self._ids, np.array([q for q, _ in joined], dtype=np.int64)])
        self._pos = np.concatenate([self._pos, np.array([m for _, m in joined], dtype=np.int64)])

    def _prefill_chunks(self, prefill):
        """One chunked-context prefill call for all of this step's prompt chunks: the chunks'
        rows gathered on the device, the allocator's slots and tables written into pinned
        staging and moved by one pkv_stage_copy."""
        torch, sc = self.torch, self.script
        n = len(prefill)
        rows = np.array(prefill, dtype=np.int64).reshape(n, 3).T.copy()  # seq ids, p0, p1
        counts = rows[2] - rows[1]
        total = int(counts.sum())
        ks, vs, qs = [], [], []
        base = sc.system if sc.reuse else 0  # staged rows start after a cached system prompt
        for s, p0, p1 in prefill:
            if s in self.prompts:
                dk, dv, dq = self.prompts[s]
                ks.append(dk[p0 - base:p1 - base])
                vs.append(dv[p0 - base:p1 - base])
                qs.append(dq[p0 - base:p1 - base])
            else:
                k, v, q = sc.prompt_rows(s, p0, p1)
                to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(
                    self.device)
                ks.append(to_dev(k))
                vs.append(to_dev(v))
                qs.append(to_dev(q))
        if self._pf is None or self._pf.tokens < total or self._pf.seqs < n:
            old = self._pf
            self._pf = _PrefillStaging(torch, max(total, 2 * old.tokens if old else total),
                                       max(n, 2 * old.seqs if old else n), self.max_blocks, self.device)
        S = self._pf
        lib = _L()
        r = rows.ctypes.data  # reserve, then slots / offsets / lengths / tables into the staging
        _check(lib.pkv_stage_prefill(self.alloc, r, r + 8 * n, r + 16 * n, n, self.max_blocks, *S.out_ptrs),
               "pkv_stage_prefill")
        _check(lib.pkv_stage_copy(*S.copy, torch.cuda.current_stream().cuda_stream), "pkv_stage_copy")
        out = torch.empty(total, sc.Hq, sc.D, dtype=torch.bfloat16, device=self.device)
        cat = (lambda xs: xs[0]) if n == 1 else torch.cat  # one sequence: its rows are contiguous already
        pkv_prefill_step(self.pool.handle, cat(ks), cat(vs), S.D["slots"][:total], cat(qs),
                         S.D["cu"][:n + 1], int(counts.max()), S.D["tables"][:n], S.D["ctx"][:n], self.scale, out)
        return out

    def device_input_region(self, B: int):
        """The device bytes a decode step of B sequences reads its q / new K / new V from when it
        runs with device_inputs=True: (region, q, k, v), region a uint8 tensor [q | k | v] of the
        batch's bucket and q [B][Hq][D], k and v [B][Hkv][D] bf16 views of its first rows.  A
        producer on the device (the layer's QKV projection) writes the step's rows there."""
        bk = self._bucket(B)
        return bk.dbuf[:bk.qkv_bytes], bk.q[:B], bk.k[:B], bk.v[:B]

    def step(self, inputs=None, device_inputs: bool = False):
        """Run the next scheduled step; returns (decoding sequence ids, output [B][Hq][D] bf16 bits: a
        view of the batch bucket's pinned output buffer, valid until that bucket's next step).
        inputs: optional host (k_new, v_new, q) for the decoding sequences (else drawn from the
        script).  device_inputs: the step's q/K/V are already on the device, in the region
        device_input_region() names (written there before this call, on the current stream).
        With chunked context the step's prefill chunks and their output are in self.last_prefill."""
        import time
        torch, sc = self.torch, self.script
        t0 = time.perf_counter()
        finished, joined = sc.steps[self.t]
        for s in finished:
            pkv_seq_release(self.alloc, s)
            if sc.chunk:
                self.scheduler.finish(s)
        if finished and not sc.chunk:
            keep = ~np.isin(self._ids, np.asarray(finished, dtype=np.int64))
            self._ids, self._pos = self._ids[keep], self._pos[keep]
        if sc.chunk:
            for s, m in joined:
                if sc.system and sc.reuse:  # the joiner forks the cached system prompt (partial block copied)
                    cs, cd = pkv_seq_share_prefix(self.alloc, self.system_seq, s, sc.system)
                    if cs >= 0:
                        pkv_pool_copy_block(self.pool.handle, cs, cd)
                self.scheduler.admit(s, m)
            prefill, decode = self.scheduler.plan()
            pre_out = self._prefill_chunks(prefill) if prefill else None
            self._ids = np.array(decode, dtype=np.int64)
            self._pos = np.array([self.scheduler.cached(s) for s in decode], dtype=np.int64)
            self.scheduler.mark_decoded(decode)
            self.last_prefill = (prefill, pre_out)
        elif joined:
            self._admit(joined)
        t1 = time.perf_counter()
        B = len(self._ids)
        if not B:
            self.t += 1
            self.attended_tokens = 0
            if sc.chunk and self.last_prefill[1] is not None:
                torch.cuda.current_stream().synchronize()
            return [], np.zeros((0, sc.Hq, sc.D), dtype=np.uint16)
        ids, pos = self._ids, self._pos
        run = ids.tolist()
        bk = self._bucket(B)
        # room for this step's token, then tables, slots and lengths (padding rows included)
        _check(_L().pkv_stage_decode(self.alloc, ids.ctypes.data, pos.ctypes.data, B, bk.Bp, self.max_blocks,
                                     *bk.out_ptrs), "pkv_stage_decode")
        if not device_inputs:
            H = bk.H
            k, v, q = inputs if inputs is not None else sc.step_inputs(self.t, run)
            H["q"][:B] = q.view(np.int16)
            H["k"][:B] = k.view(np.int16)
            H["v"][:B] = v.view(np.int16)
            H["q"][B:] = 0
            H["k"][B:] = 0
            H["v"][B:] = 0
        t2 = time.perf_counter()
        if self.graphs:
            g = bk.graphs.get(device_inputs)
            if g is None:
                bk.run(torch, self, device_inputs)  # warm-up outside capture (builds plans, loads modules)
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                side = torch.cuda.Stream()
                side.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(side):
                    with torch.cuda.graph(g, stream=side):
                        bk.run(torch, self, device_inputs)
                torch.cuda.current_stream().wait_stream(side)
                bk.graphs[device_inputs] = g
            g.replay()
        else:
            bk.run(torch, self, device_inputs)
        torch.cuda.current_stream().synchronize()
        t3 = time.perf_counter()
        self.timing["admit_s"] += t1 - t0
        self.timing["prepare_s"] += t2 - t1
        self.timing["device_s"] += t3 - t2
        self.attended_tokens = int(pos.sum()) + B
        if not sc.chunk:
            self._pos = pos + 1
        self.t += 1
        return run, bk.out_np[:B]

    def close(self):
        self.pool.close()
