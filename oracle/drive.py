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


def attention(w, pool, tables, threads: int | None = None, seqs=None) -> np.ndarray:
    """fp64 decode attention of the step, [B, Hq, D]; `seqs` limits it to some sequences."""
    q = w.query()
    lens = w.attend_lens
    if seqs is not None:
        seqs = np.asarray(seqs)
        q, tables, lens = q[seqs], tables[seqs], lens[seqs]
    return pool.attention(q, tables, lens, w.Hq, 1.0 / math.sqrt(w.D), threads=threads or os.cpu_count() or 1)


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
