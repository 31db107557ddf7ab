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
     causally, and the sequence decodes from the step after its last chunk.  With a system
     prompt (prefix caching, "TensorRT-LLM 推理加速实战" §8 KV cache reuse) the shared prefix
     is cached once and every joiner forks it (pkv_seq_share_prefix) instead of prefilling it;
  3. gives every decoding sequence room for one more token (pkv_seq_reserve_many grows by whole
     blocks), writes block tables, new-token slots and context lengths straight into a pinned
     staging buffer together with the step's q / new K / new V;
  4. runs, on the decode batch padded to its bucket, one host-to-device copy, pkv_decode_step
     (append + attention) and the copy of the output back — captured once per bucket as a CUDA
     graph and replayed.  Padding rows have context length 0 and slot -1, so they write nothing
     and read nothing; their outputs are zeros.
"""
from __future__ import annotations

import math

import numpy as np

from . import (KV_DTYPES, KVPool, pkv_append, pkv_decode_step, pkv_decode_workspace_bytes, pkv_get_block_tables,
               pkv_pool_copy_block, pkv_prefill_step, pkv_seq_release, pkv_seq_reserve, pkv_seq_reserve_many,
               pkv_seq_share_prefix, pkv_slot_mapping, pkv_stage_copy)

DEFAULT_BUCKETS = (8, 16, 32, 64, 128, 256, 512, 1024)


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
        ws = pkv_decode_workspace_bytes(loop.pool.handle, Bp, sc.Hq, loop.max_blocks)
        self.workspace = torch.zeros(ws, dtype=torch.uint8, device=device)
        self.graph = None

    def run(self, torch, loop):
        """Copy the staged inputs in, run the fused step, copy the output out (no sync); both
        copies are pkv_stage_copy (SM-driven: faster than a copy engine at these sizes)."""
        pkv_stage_copy(self.dbuf, self.hbuf)
        pkv_decode_step(loop.pool.handle, self.k, self.v, self.Dv["slots"], self.q, self.Dv["tables"],
                        self.Dv["lens"], loop.scale, self.out, self.workspace)
        pkv_stage_copy(self.out_host, self.out)


class DecodeLoop:
    def __init__(self, script, graphs: bool = True, buckets=DEFAULT_BUCKETS, device: str = "cuda",
                 prompts=None):
        """prompts: optional {seq_id: (k, v)} of device bf16 tensors [n][Hkv][D] (a joining
        sequence's prompt K/V as its prefill produced them; with chunked context (a script with
        chunk > 0) (k, v, q), q [n][Hq][D] the prompt's queries, rows from the first position the
        request prefills: after the system prompt when it is cached); else drawn from the script.

        Chunked context (script.chunk > 0, "TensorRT-LLM 深度实战" §7.3): a joining sequence's
        prompt is prefilled `chunk` tokens per step (its chunk's K/V appended and its queries
        attending causally, one pkv_prefill_step for all prefilling sequences of the step) and
        the sequence decodes from the step after its last chunk."""
        import torch
        self.prompts = prompts or {}
        self.torch, self.script, self.graphs, self.device = torch, script, graphs, device
        self.pool = KVPool(script.num_blocks, script.block_size, script.Hkv, script.D, KV_DTYPES[script.kv_dtype])
        self.alloc = self.pool.allocator
        self.max_blocks = -(-script.max_len // script.block_size)
        self.scale = 1.0 / math.sqrt(script.D)
        self.buckets = sorted(buckets)
        self._bk = {}
        self.lens: dict[int, int] = {}
        self.running: list[int] = []
        self.t = 0
        self.timing = {"admit_s": 0.0, "prepare_s": 0.0, "device_s": 0.0}  # host wall time per phase
        self.state: dict = {}  # chunked context: seq -> [prompt_len, prefilled, decoded]
        if script.chunk and script.system:
            # prefix caching ("TensorRT-LLM 推理加速实战" §8, KV cache reuse): the shared system
            # prompt is cached once under its own sequence; joiners fork it
            from pkv_workloads import SYSTEM_SEQ
            self.system_seq = SYSTEM_SEQ
            k, v = script.system_kv()
            pkv_seq_reserve(self.alloc, SYSTEM_SEQ, script.system)
            slots = pkv_slot_mapping(self.alloc, [SYSTEM_SEQ] * script.system, np.arange(script.system))
            to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
            pkv_append(self.pool.handle, to_dev(k), to_dev(v), torch.from_numpy(slots).to(device))
        self.last_prefill = ([], None)  # chunked context: (chunks [(seq, p0, p1)], output bits)

    def _bucket(self, B: int) -> _Bucket:
        Bp = next((b for b in self.buckets if b >= B), None)
        if Bp is None:
            raise ValueError(f"batch {B} exceeds the largest bucket {self.buckets[-1]}")
        if Bp not in self._bk:
            self._bk[Bp] = _Bucket(self.torch, self, Bp, self.device)
        return self._bk[Bp]

    def _admit(self, seq: int, n: int):
        torch = self.torch
        pkv_seq_reserve(self.alloc, seq, n)
        if n:
            slots = pkv_slot_mapping(self.alloc, [seq] * n, np.arange(n, dtype=np.int64))
            if seq in self.prompts:
                dk, dv = self.prompts[seq]
            else:
                k, v = self.script.prompt_kv(seq, n)
                dk = torch.from_numpy(np.ascontiguousarray(k).view(np.int16)).view(torch.bfloat16).to(self.device)
                dv = torch.from_numpy(np.ascontiguousarray(v).view(np.int16)).view(torch.bfloat16).to(self.device)
            pkv_append(self.pool.handle, dk, dv, torch.from_numpy(slots).to(self.device, non_blocking=True))
        self.lens[seq] = n
        self.running.append(seq)

    def _prefill_chunks(self, prefill):
        """One chunked-context prefill call for all of this step's prompt chunks."""
        torch, sc = self.torch, self.script
        ks, vs, qs, seqs, pos = [], [], [], [], []
        for s, p0, p1 in prefill:
            pkv_seq_reserve(self.alloc, s, p1)
            if s in self.prompts:  # staged rows from position `base` (after a cached system prompt)
                base = sc.system if sc.reuse else 0
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
            seqs += [s] * (p1 - p0)
            pos += list(range(p0, p1))
        ids = [s for s, _, _ in prefill]
        slots = pkv_slot_mapping(self.alloc, seqs, np.asarray(pos, dtype=np.int64))
        cu = np.concatenate([[0], np.cumsum([p1 - p0 for _, p0, p1 in prefill])]).astype(np.int32)
        ctx = np.array([p1 for _, _, p1 in prefill], dtype=np.int32)
        tables = pkv_get_block_tables(self.alloc, ids, self.max_blocks)
        dev = self.device
        out = torch.empty(int(cu[-1]), sc.Hq, sc.D, dtype=torch.bfloat16, device=dev)
        pkv_prefill_step(self.pool.handle, torch.cat(ks), torch.cat(vs), torch.from_numpy(slots).to(dev),
                         torch.cat(qs), torch.from_numpy(cu).to(dev), int(np.diff(cu).max()),
                         torch.from_numpy(tables).to(dev), torch.from_numpy(ctx).to(dev), self.scale, out)
        for s, p0, p1 in prefill:
            self.state[s][1] = p1
        return out

    def step(self, inputs=None):
        """Run the next scheduled step; returns (decoding sequence ids, output [B][Hq][D] bf16 bits).
        inputs: optional (k_new, v_new, q) for the decoding sequences (else drawn from the script).
        With chunked context the step's prefill chunks and their output are in self.last_prefill."""
        import time
        torch, sc = self.torch, self.script
        t0 = time.perf_counter()
        finished, joined = sc.steps[self.t]
        for s in finished:
            pkv_seq_release(self.alloc, s)
            if sc.chunk:
                continue
            self.running.remove(s)
            del self.lens[s]
        if sc.chunk:
            if sc.system and sc.reuse:  # joiners fork the cached system prompt (partial block copied)
                for s, _ in joined:
                    cs, cd = pkv_seq_share_prefix(self.alloc, self.system_seq, s, sc.system)
                    if cs >= 0:
                        pkv_pool_copy_block(self.pool.handle, cs, cd)
            prefill, decode = sc.plan_step(self.t, self.state)
            pre_out = self._prefill_chunks(prefill) if prefill else None
            self.running = decode
            self.lens = {s: self.state[s][0] + self.state[s][2] for s in decode}
            for s in decode:
                self.state[s][2] += 1
            self.last_prefill = (prefill, pre_out)
        else:
            for s, n in joined:
                self._admit(s, n)
        t1 = time.perf_counter()
        run = list(self.running)
        if not run:
            self.t += 1
            if sc.chunk and self.last_prefill[1] is not None:
                torch.cuda.current_stream().synchronize()
            return run, np.zeros((0, sc.Hq, sc.D), dtype=np.uint16)
        B = len(run)
        pos = np.array([self.lens[s] for s in run], dtype=np.int64)
        pkv_seq_reserve_many(self.alloc, run, pos + 1)  # room for this step's token
        bk = self._bucket(B)
        H = bk.H
        k, v, q = inputs if inputs is not None else sc.step_inputs(self.t, run)
        H["q"][:B] = q.view(np.int16)
        H["k"][:B] = k.view(np.int16)
        H["v"][:B] = v.view(np.int16)
        H["q"][B:] = 0
        H["k"][B:] = 0
        H["v"][B:] = 0
        pkv_get_block_tables(self.alloc, run, self.max_blocks, out=H["tables"][:B])
        H["tables"][B:] = -1
        pkv_slot_mapping(self.alloc, run, pos, out=H["slots"][:B])
        H["slots"][B:] = -1
        H["lens"][:B] = pos + 1
        H["lens"][B:] = 0
        t2 = time.perf_counter()
        if self.graphs:
            if bk.graph is None:
                bk.run(torch, self)  # warm-up outside capture (builds plans, loads modules)
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                side = torch.cuda.Stream()
                side.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(side):
                    with torch.cuda.graph(g, stream=side):
                        bk.run(torch, self)
                torch.cuda.current_stream().wait_stream(side)
                bk.graph = g
            bk.graph.replay()
        else:
            bk.run(torch, self)
        torch.cuda.current_stream().synchronize()
        t3 = time.perf_counter()
        self.timing["admit_s"] += t1 - t0
        self.timing["prepare_s"] += t2 - t1
        self.timing["device_s"] += t3 - t2
        if not sc.chunk:
            for s in run:
                self.lens[s] += 1
        self.t += 1
        return run, bk.out_host.numpy()[:B].view(np.uint16).copy()

    def close(self):
        self.pool.close()
