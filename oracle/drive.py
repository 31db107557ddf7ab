"""Run the oracle over a workload — TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Builds the oracle's own allocator replica and host pool from the workload's seeded
inputs (replaying the same allocation script and the same append calls as the
device path) and evaluates the decode step in fp64.
"""
from __future__ import annotations

import math
import os

import numpy as np

from . import Allocator, Pool

KV_CODE = {"bf16": 0, "fp8_e4m3": 1, "int8": 2}  # element codes of the oracle's pool


def build(w, with_new_token: bool = True):
    """(pool, allocator, block_tables) after the history and (optionally) the step's append."""
    alloc = Allocator(w.num_blocks, w.block_size)
    if alloc.set_free_order(w.free_order):
        raise RuntimeError("oracle: bad free order")
    alloc.replay(w.alloc_ops)
    tables = alloc.block_tables(w.seq_ids, max(1, w.max_blocks()))
    pool = Pool(w.num_blocks, w.block_size, w.Hkv, w.D, KV_CODE[w.kv_dtype])
    for t0, t1 in w.hist_chunks():
        seqs, pos = w.hist_positions(t0, t1)
        rc = pool.append(w.history_k(t0, t1), w.history_v(t0, t1), alloc.slot_mapping(seqs, pos))
        if rc:
            raise RuntimeError(f"oracle append rc={rc}")
    if w.append and with_new_token:
        rc = pool.append(w.new_k(), w.new_v(), alloc.slot_mapping(w.seq_ids, w.lens))
        if rc:
            raise RuntimeError(f"oracle append rc={rc}")
    return pool, alloc, tables


def attention(w, pool, tables, threads: int | None = None, seqs=None, q=None) -> np.ndarray:
    """fp64 decode attention of the step, [B, Hq, D]; `seqs` limits it to some sequences; `q` is
    the step's query (`w.query()`) when the caller has already drawn it."""
    q = w.query() if q is None else q
    lens = w.attend_lens
    if seqs is not None:
        seqs = np.asarray(seqs)
        q, tables, lens = q[seqs], tables[seqs], lens[seqs]
    return pool.attention(q, tables, lens, w.Hq, 1.0 / math.sqrt(w.D), threads=threads or os.cpu_count() or 1)


class ChunkedContextPlan:
    """The chunked-context schedule of "TensorRT-LLM 深度实战" §7.3 (ChunkedContextScheduler), as
    the oracle's own restatement: a request's input is cut into chunks of at most chunk_size
    tokens; every step, each admitted request in admission order either processes its next chunk
    (input[prefill_progress : prefill_progress + chunk_size], then the progress advances and the
    request stops prefilling once the progress reaches the input's length) or, once it has
    stopped prefilling, decodes one token.  So a request decodes from the step after its last
    chunk.  With a shared system prompt of `system` tokens every input starts with it; when the
    prompt is cached and forked (reuse), a request's progress starts at `system`."""

    def __init__(self, chunk_size: int, system: int = 0, reuse: bool = True):
        self.chunk_size, self.system, self.reuse = chunk_size, system, reuse
        self.requests = []  # admission order: dicts with id, input_len, prefill_progress, is_prefilling, decoded

    def step(self, finished, joined):
        """Apply the step's departures and arrivals, then schedule it: returns ([(id, p0, p1)]
        chunks, [decoding ids]), both in admission order."""
        gone = set(finished)
        for r in self.requests:
            if r["id"] in gone and r["is_prefilling"]:
                raise RuntimeError(f"request {r['id']} left while prefilling")
        self.requests = [r for r in self.requests if r["id"] not in gone]
        for rid, n in joined:
            start = self.system if (self.system and self.reuse) else 0
            self.requests.append({"id": rid, "input_len": self.system + n, "prefill_progress": start,
                                  "is_prefilling": start < self.system + n, "decoded": 0})
        chunks, decode = [], []
        for r in self.requests:
            if r["is_prefilling"]:
                p0 = r["prefill_progress"]
                p1 = min(r["input_len"], p0 + self.chunk_size)
                chunks.append((r["id"], p0, p1))
                r["prefill_progress"] = p1
                if p1 >= r["input_len"]:
                    r["is_prefilling"] = False
            else:
                decode.append(r["id"])
        return chunks, decode

    def cached(self, rid: int) -> int:
        """Tokens request `rid` holds before its decode token of this step: its input plus the
        tokens it decoded in earlier steps."""
        r = next(r for r in self.requests if r["id"] == rid)
        return r["input_len"] + r["decoded"]

    def decoded(self, ids) -> None:
        for r in self.requests:
            if r["id"] in ids:
                r["decoded"] += 1


def run_chunked_loop(script, n_steps: int | None = None, threads: int | None = None):
    """Replay a chunked-context decode loop ("TensorRT-LLM 深度实战" §7.3): each step, finished
    sequences release their pages; every prefilling sequence appends its next prompt chunk and
    its chunk's queries attend causally over its cache (one append call for all chunks of the
    step); every decoding sequence appends one token and attends.  Yields per step (decode ids,
    fp64 decode output [B][Hq][D], prefill chunks [(seq, p0, p1)], fp64 prefill output
    [sum(p1 - p0)][Hq][D]); the pool replica is returned last."""
    from . import Allocator, Pool
    sc = script
    alloc = Allocator(sc.num_blocks, sc.block_size)
    pool = Pool(sc.num_blocks, sc.block_size, sc.Hkv, sc.D, KV_CODE[sc.kv_dtype])
    max_blocks = -(-sc.max_len // sc.block_size)
    scale = 1.0 / math.sqrt(sc.D)
    nthreads = threads or os.cpu_count() or 1
    plan = ChunkedContextPlan(sc.chunk, sc.system, sc.reuse)
    outs = []
    if sc.system:  # the shared system prompt, cached once (prefix caching)
        from pkv_workloads import SYSTEM_SEQ
        if alloc.reserve(SYSTEM_SEQ, sc.system):
            raise RuntimeError("oracle loop: out of pages")
        k, v = sc.system_kv()
        pool.append(k, v, alloc.slot_mapping([SYSTEM_SEQ] * sc.system, np.arange(sc.system)))
    for t in range(len(sc.steps) if n_steps is None else n_steps):
        for s in sc.steps[t][0]:
            if alloc.release(s):
                raise RuntimeError("oracle loop: release failed")
        if sc.system and sc.reuse:  # joiners fork the cached system prompt
            for s, _ in sc.steps[t][1]:
                rc, cs, cd = alloc.share_prefix(SYSTEM_SEQ, s, sc.system)
                if rc:
                    raise RuntimeError(f"oracle loop: fork failed ({rc})")
                if cs >= 0:
                    pool.copy_block(cs, cd)
        prefill, decode = plan.step(sc.steps[t][0], sc.steps[t][1])
        out_pre = np.zeros((0, sc.Hq, sc.D))
        if prefill:
            ks, vs, qs, seqs, pos = [], [], [], [], []
            for s, p0, p1 in prefill:
                if alloc.reserve(s, p1):
                    raise RuntimeError("oracle loop: out of pages")
                k, v, q = sc.prompt_rows(s, p0, p1)
                ks.append(k)
                vs.append(v)
                qs.append(q)
                seqs += [s] * (p1 - p0)
                pos += list(range(p0, p1))
            pool.append(np.concatenate(ks), np.concatenate(vs), alloc.slot_mapping(seqs, pos))
            cu = np.concatenate([[0], np.cumsum([p1 - p0 for _, p0, p1 in prefill])]).astype(np.int32)
            ids = [s for s, _, _ in prefill]
            tables = alloc.block_tables(ids, max_blocks)
            ctx = np.array([p1 for _, _, p1 in prefill], dtype=np.int32)
            out_pre = pool.prefill_attention(np.concatenate(qs), cu, tables, ctx, sc.Hq, scale, threads=nthreads)
        out_dec = np.zeros((0, sc.Hq, sc.D))
        if decode:
            lens = np.array([plan.cached(s) for s in decode], dtype=np.int64)
            for s, L in zip(decode, lens):
                if alloc.reserve(s, int(L) + 1):
                    raise RuntimeError("oracle loop: out of pages")
            k, v, q = sc.step_inputs(t, decode)
            pool.append(k, v, alloc.slot_mapping(decode, lens))
            tables = alloc.block_tables(decode, max_blocks)
            out_dec = pool.attention(q, tables, (lens + 1).astype(np.int32), sc.Hq, scale, threads=nthreads)
            plan.decoded(set(decode))
        outs.append((list(decode), out_dec, list(prefill), out_pre))
    return outs, pool


def run_loop(script, n_steps: int | None = None, threads: int | None = None):
    """Replay a decode-loop schedule (finished sequences release their pages, joiners get their
    prompt appended, every running sequence appends one token and attends).  Yields, per step,
    (running sequence ids, fp64 output [B][Hq][D]); the pool replica is returned last."""
    from . import Allocator, Pool
    sc = script
    alloc = Allocator(sc.num_blocks, sc.block_size)
    pool = Pool(sc.num_blocks, sc.block_size, sc.Hkv, sc.D, KV_CODE[sc.kv_dtype])
    max_blocks = -(-sc.max_len // sc.block_size)
    lens, running = {}, []
    steps = sc.steps if n_steps is None else sc.steps[:n_steps]
    outs = []
    for t, (finished, joined) in enumerate(steps):
        for s in finished:
            if alloc.release(s):
                raise RuntimeError("oracle loop: release failed")
            running.remove(s)
            del lens[s]
        for s, n in joined:
            if alloc.reserve(s, n):
                raise RuntimeError("oracle loop: out of pages")
            if n:
                k, v = sc.prompt_kv(s, n)
                pool.append(k, v, alloc.slot_mapping([s] * n, np.arange(n)))
            lens[s] = n
            running.append(s)
        for s in running:
            if alloc.reserve(s, lens[s] + 1):
                raise RuntimeError("oracle loop: out of pages")
        k, v, q = sc.step_inputs(t, running)
        pos = np.array([lens[s] for s in running], dtype=np.int64)
        pool.append(k, v, alloc.slot_mapping(running, pos))
        tables = alloc.block_tables(running, max_blocks)
        out = pool.attention(q, tables, (pos + 1).astype(np.int32), sc.Hq, 1.0 / math.sqrt(sc.D),
                             threads=threads or os.cpu_count() or 1)
        for s in running:
            lens[s] += 1
        outs.append((list(running), out))
    return outs, pool
