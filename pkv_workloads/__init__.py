"""Seeded synthetic workloads for paged decode attention.

This package only draws random inputs and describes the five workloads; it holds
none of the method's arithmetic (no allocator, append, quantisation or attention
code).  Both the CUDA path and the CPU oracle consume what it produces, so the
two always see the same bytes.

Shapes follow the head shapes and batch mixes that the TensorRT-LLM pages use
("TensorRT-LLM 推理加速实战", §8 KV Cache 深入 / §8.1 KV Cache 显存估算: Llama-3.1-70B
with 8 KV heads and head_dim 128; "TensorRT-LLM 深度实战", §3.1 Paged KV Cache with
page_size 16; the 200-concurrent-request FP8 scenario of the aiqz.cc page,
KV缓存管理 section).  No dataset is involved; every input is drawn here.

Random numbers: splitmix64 (counter-based, see gen.c).  Each workload has a base
seed 266*1000 + index; each independent stream (context lengths, free-list
permutation, churn script, history K, history V, new K, new V, Q) uses as its
seed the tag-th output of the base stream.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libpkvgen.so")
_lib = None

TAG_LENS, TAG_PERM, TAG_CHURN, TAG_K_HIST, TAG_V_HIST, TAG_K_NEW, TAG_V_NEW, TAG_Q = range(1, 9)
TEMP_SEQ_BASE = 1_000_000
HIST_CHUNK_TOKENS = 65536
MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15


def build_native(force: bool = False) -> str:
    """Compile gen.c into an in-tree shared library (gcc, portable flags)."""
    if os.path.exists(_LIB_PATH) and not force:
        src_m = os.path.getmtime(os.path.join(_HERE, "gen.c"))
        if os.path.getmtime(_LIB_PATH) >= src_m:
            return _LIB_PATH
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off",
                           os.path.join(_HERE, "gen.c"), "-o", tmp, "-lm", "-lpthread"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _native():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build_native())
        lib.wl_splitmix64_at.restype = ctypes.c_uint64
        lib.wl_splitmix64_at.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.wl_normal_at.restype = ctypes.c_double
        lib.wl_normal_at.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.wl_normal_bf16.restype = None
        lib.wl_normal_bf16.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double,
                                       ctypes.c_double, ctypes.c_void_p, ctypes.c_int]
        _lib = lib
    return _lib


# ----------------------------------------------------------------------------- scalar draws
def splitmix64_at(seed: int, i: int) -> int:
    """i-th output (0-based) of the splitmix64 stream with initial state `seed` (pure Python)."""
    z = (seed + (i + 1) * GAMMA) & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def unit(seed: int, i: int) -> float:
    """Uniform in [0, 1) from the top 53 bits of draw i."""
    return (splitmix64_at(seed, i) >> 11) * (1.0 / (1 << 53))


def uniform_int(seed: int, i: int, lo: int, hi: int) -> int:
    """Uniform integer in [lo, hi] (multiply-shift on 53 random bits)."""
    n = hi - lo + 1
    return lo + (((splitmix64_at(seed, i) >> 11) * n) >> 53)


def normal(seed: int, i: int) -> float:
    """i-th standard normal of the stream (Box-Muller cosine branch), fp64."""
    return _native().wl_normal_at(seed & MASK64, i)


def stream_seed(base_seed: int, tag: int) -> int:
    return splitmix64_at(base_seed, tag)


def permutation(seed: int, n: int) -> np.ndarray:
    """Seeded Fisher-Yates (Durstenfeld) shuffle of 0..n-1; draw k picks the k-th swap partner."""
    a = list(range(n))
    k = 0
    for i in range(n - 1, 0, -1):
        j = uniform_int(seed, k, 0, i)
        k += 1
        a[i], a[j] = a[j], a[i]
    return np.asarray(a, dtype=np.int32)


def normal_bf16(seed: int, offset: int, n: int, threads: int | None = None) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(0,1) draws offset .. offset+n-1."""
    out = np.empty(n, dtype=np.uint16)
    if n:
        t = threads or min(64, os.cpu_count() or 1)
        _native().wl_normal_bf16(seed & MASK64, offset, n, 0.0, 1.0, out.ctypes.data, t)
    return out


# ----------------------------------------------------------------------------- workloads
@dataclass
class Workload:
    """One synthetic decode step over a paged KV pool.

    lens[b]      tokens already cached for sequence b before the step;
    append       whether the step writes one new token per sequence at position lens[b];
    attend_lens  context length the attention covers (lens + append);
    free_order   initial free-list order handed to the allocator (a permutation);
    alloc_ops    allocator script: ("reserve", seq_id, total_tokens) / ("release", seq_id);
    seq_ids      the batch's sequence ids, in batch order.
    """
    name: str
    index: int
    description: str
    B: int
    Hq: int
    Hkv: int
    D: int
    block_size: int
    kv_dtype: str  # "bf16" | "fp8_e4m3" | "int8"
    num_blocks: int
    lens: np.ndarray
    append: bool
    free_order: np.ndarray
    alloc_ops: list = field(default_factory=list)
    seq_ids: np.ndarray = None

    @property
    def seed(self) -> int:
        return 266 * 1000 + self.index

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def attend_lens(self) -> np.ndarray:
        return (self.lens + (1 if self.append else 0)).astype(np.int32)

    @property
    def n_hist(self) -> int:
        return int(self.lens.sum())

    @property
    def hist_offsets(self) -> np.ndarray:
        """Start of each sequence's tokens in the concatenated history stream."""
        return np.concatenate([[0], np.cumsum(self.lens)]).astype(np.int64)

    @property
    def elem_bytes(self) -> int:
        return 2 if self.kv_dtype == "bf16" else 1

    def kv_read_bytes(self) -> int:
        """K+V bytes one attention pass must read: 2*D*bytes per (token, kv head)."""
        return int(self.attend_lens.astype(np.int64).sum()) * self.Hkv * 2 * self.D * self.elem_bytes

    # --- tensors (bf16 bit patterns as uint16) ---
    def history_k(self, tok_begin: int = 0, tok_end: int | None = None) -> np.ndarray:
        return self._hist(TAG_K_HIST, tok_begin, tok_end)

    def history_v(self, tok_begin: int = 0, tok_end: int | None = None) -> np.ndarray:
        return self._hist(TAG_V_HIST, tok_begin, tok_end)

    def _hist(self, tag, tok_begin, tok_end):
        tok_end = self.n_hist if tok_end is None else tok_end
        row = self.Hkv * self.D
        flat = normal_bf16(stream_seed(self.seed, tag), tok_begin * row, (tok_end - tok_begin) * row)
        return flat.reshape(tok_end - tok_begin, self.Hkv, self.D)

    def new_k(self) -> np.ndarray:
        return normal_bf16(stream_seed(self.seed, TAG_K_NEW), 0, self.B * self.Hkv * self.D).reshape(
            self.B, self.Hkv, self.D)

    def new_v(self) -> np.ndarray:
        return normal_bf16(stream_seed(self.seed, TAG_V_NEW), 0, self.B * self.Hkv * self.D).reshape(
            self.B, self.Hkv, self.D)

    def query(self) -> np.ndarray:
        return normal_bf16(stream_seed(self.seed, TAG_Q), 0, self.B * self.Hq * self.D).reshape(
            self.B, self.Hq, self.D)

    def hist_positions(self, tok_begin: int = 0, tok_end: int | None = None):
        """(seq_ids, positions) of history tokens [tok_begin, tok_end) of the concatenated stream."""
        tok_end = self.n_hist if tok_end is None else tok_end
        off = self.hist_offsets
        t = np.arange(tok_begin, tok_end, dtype=np.int64)
        b = np.searchsorted(off, t, side="right") - 1
        return self.seq_ids[b], (t - off[b]).astype(np.int64)

    def hist_chunks(self, chunk: int = HIST_CHUNK_TOKENS):
        """Token ranges [t0, t1) of the concatenated history, one append call each (fp8 block
        scales are fixed by the call that writes a block's first slot, so both sides must use
        the same call boundaries)."""
        return [(t, min(self.n_hist, t + chunk)) for t in range(0, self.n_hist, chunk)]

    def max_blocks(self) -> int:
        return int(-(-int(self.attend_lens.max()) // self.block_size)) if self.B else 0


def _ceil_div(a, b):
    return -(-a // b)


def _simple_ops(lens, append):
    return [("reserve", b, int(lens[b]) + (1 if append else 0)) for b in range(len(lens))]


def make_workload(name: str) -> Workload:
    """The five workloads: c0 (tiny parity case) .. c4 (churned FP8 pool)."""
    idx = int(name[1:])
    seed = 266 * 1000 + idx
    s_lens = stream_seed(seed, TAG_LENS)
    s_perm = stream_seed(seed, TAG_PERM)
    if idx == 0:
        lens = np.array([5, 17, 33, 64], dtype=np.int64)
        w = Workload(name, 0, "tiny paged decode, GQA 2:1, head_dim 64, block 16, 32-block pool, permuted blocks",
                     4, 4, 2, 64, 16, "bf16", 32, lens, True, permutation(s_perm, 32))
    elif idx == 1:
        lens = np.array([uniform_int(s_lens, b, 128, 2048) for b in range(32)], dtype=np.int64)
        need = int(sum(_ceil_div(int(L) + 1, 64) for L in lens))
        nb = need + _ceil_div(need, 10)
        w = Workload(name, 1, "Llama-2-7B-shape MHA layer decode, batch 32, contexts U[128,2048], block 64",
                     32, 32, 32, 128, 64, "bf16", nb, lens, True, permutation(s_perm, nb))
    elif idx == 2:
        lens = np.array([min(4096, max(16, int(round(512.0 * math.exp(normal(s_lens, b)))))) for b in range(128)],
                        dtype=np.int64)
        nb = (2 * 1 * 8 * 128 * 4096 * 128 * 2) // (64 * 2 * 8 * 128 * 2)  # M_kv(128 seqs x 4096) / block bytes
        w = Workload(name, 2, "Llama-3-8B-shape GQA in-flight batch, batch 128, lognormal contexts, block 64",
                     128, 32, 8, 128, 64, "bf16", nb, lens, True, permutation(s_perm, nb))
    elif idx == 3:
        k = 1024
        lens = np.array([32 * k, 48 * k, 64 * k, 80 * k, 96 * k, 112 * k, 128 * k, 128 * k], dtype=np.int64)
        nb = int(sum(_ceil_div(int(L), 64) for L in lens))
        w = Workload(name, 3, "70B-shape long context, batch 8, 32k-128k contexts, GQA 8:1, block 64",
                     8, 64, 8, 128, 64, "bf16", nb, lens, False, permutation(s_perm, nb))
    elif idx == 4:
        lens = np.array([uniform_int(s_lens, b, 64, 8192) for b in range(200)], dtype=np.int64)
        nb = (200 * 8192) // 16
        w = Workload(name, 4, "200-request churned pool, FP8-e4m3 KV with per-(block,head) scales, block 16",
                     200, 32, 8, 128, 16, "fp8_e4m3", nb, lens, True, np.arange(nb, dtype=np.int32))
    else:
        raise ValueError(name)
    w.seq_ids = np.arange(w.B, dtype=np.int64)
    if idx == 4:
        w.alloc_ops = _churn_ops(w, stream_seed(seed, TAG_CHURN))
    else:
        w.alloc_ops = _simple_ops(w.lens, w.append)
    return w


def _churn_ops(w: Workload, s_churn: int):
    """1000 seeded create/release cycles of temporary sequences, their release, then round-robin
    growth of the batch block by block.  Temporary sequences hold whole blocks (k * block_size
    tokens), so the script can count held blocks without modelling the allocator."""
    ops, live, held, tid = [], [], 0, 0
    bs = w.block_size
    for i in range(1000):
        u = unit(s_churn, 3 * i)
        if u < 0.5 and w.num_blocks - held >= 64:
            k = uniform_int(s_churn, 3 * i + 1, 1, 64)
            seq = TEMP_SEQ_BASE + tid
            tid += 1
            ops.append(("reserve", seq, k * bs))
            live.append((seq, k))
            held += k
        elif live:
            j = uniform_int(s_churn, 3 * i + 2, 0, len(live) - 1)
            seq, k = live.pop(j)
            ops.append(("release", seq))
            held -= k
    for seq, _ in live:
        ops.append(("release", seq))
    total = [int(L) + (1 if w.append else 0) for L in w.lens]
    need = [_ceil_div(t, bs) for t in total]
    for r in range(max(need)):
        for b in range(w.B):
            if need[b] > r:
                ops.append(("reserve", b, min((r + 1) * bs, total[b])))
    return ops


WORKLOADS = ("c0", "c1", "c2", "c3", "c4")


def custom_workload(index: int, B: int, Hq: int, Hkv: int, D: int, block_size: int, lens, append: bool = True,
                    kv_dtype: str = "bf16", spare_blocks: int = 3, shuffle: bool = True) -> Workload:
    """A small workload for edge cases: explicit context lengths, pool sized to fit plus spares,
    a seeded shuffled free list, every sequence reserved in batch order."""
    lens = np.asarray(lens, dtype=np.int64)
    seed = 266 * 1000 + index
    total = [int(L) + (1 if append else 0) for L in lens]
    nb = sum(_ceil_div(t, block_size) for t in total) + spare_blocks
    order = permutation(stream_seed(seed, TAG_PERM), nb) if shuffle else np.arange(nb, dtype=np.int32)
    w = Workload(f"custom{index}", index, "edge case", B, Hq, Hkv, D, block_size, kv_dtype, nb, lens, append, order)
    w.seq_ids = np.arange(B, dtype=np.int64)
    w.alloc_ops = _simple_ops(lens, append)
    return w


def truncated(w: Workload, n: int) -> Workload:
    """The same workload seen through its first n sequences (for sizing measurements)."""
    import copy
    t = copy.copy(w)
    t.B = n
    t.lens = w.lens[:n]
    t.seq_ids = w.seq_ids[:n]
    t.name = f"{w.name}[:{n}]"
    return t


# ----------------------------------------------------------------------------- decode loop
TAG_LOOP_SCHED, TAG_LOOP_PROMPT_K, TAG_LOOP_PROMPT_V, TAG_LOOP_K, TAG_LOOP_V, TAG_LOOP_Q = range(20, 26)
TAG_LOOP_PROMPT_Q, TAG_LOOP_SYSTEM_K, TAG_LOOP_SYSTEM_V = 26, 27, 28
SYSTEM_SEQ = 1 << 40  # sequence id of the cached system prompt (prefix caching in the loop)


@dataclass
class LoopScript:
    """A seeded schedule of in-flight-batching decode steps ("TensorRT-LLM 深度实战", §3.2: each
    step removes finished sequences, admits waiting ones and runs one forward pass).

    steps[t] = (finished, joined): sequence ids leaving before step t and (seq_id, prompt_len)
    pairs admitted before step t.  Every running sequence then appends one token and attends.
    Tensors are drawn per (sequence, position) / (step, row) so both sides read the same bytes."""
    name: str
    seed: int
    Hq: int
    Hkv: int
    D: int
    block_size: int
    kv_dtype: str
    num_blocks: int
    max_batch: int
    steps: list
    max_len: int
    chunk: int = 0  # chunked context: prompt tokens prefilled per step (0: prompts appended at once)
    system: int = 0  # every prompt starts with this many shared system-prompt tokens
    reuse: bool = True  # prefix caching: joiners fork the cached system prompt (else they prefill it)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def system_kv(self):
        """K and V of the shared system prompt ([system][Hkv][D] bf16 bits), from their own streams."""
        n, row = self.system, self.Hkv * self.D
        k = normal_bf16(stream_seed(self.seed, TAG_LOOP_SYSTEM_K), 0, n * row).reshape(n, self.Hkv, self.D)
        v = normal_bf16(stream_seed(self.seed, TAG_LOOP_SYSTEM_V), 0, n * row).reshape(n, self.Hkv, self.D)
        return k, v

    def prompt_rows(self, seq_id: int, p0: int, p1: int):
        """K, V and queries of prompt tokens p0 .. p1-1 of a request: with a system prompt, the
        request's own tokens start at position `system` and are drawn from its own streams."""
        S = self.system
        ks, vs, qs = [], [], []
        if p0 < S:  # system-prompt rows (only without reuse): shared K/V, the request's own queries
            sk, sv = self.system_kv()
            ks.append(sk[p0:min(p1, S)])
            vs.append(sv[p0:min(p1, S)])
            qs.append(self.prompt_q(seq_id, self.max_len - S + p0, self.max_len - S + min(p1, S)))
        if p1 > S:
            lo = max(p0, S)
            k, v = self.prompt_kv(seq_id, p1 - S)
            ks.append(k[lo - S:])
            vs.append(v[lo - S:])
            qs.append(self.prompt_q(seq_id, lo - S, p1 - S))
        return np.concatenate(ks), np.concatenate(vs), np.concatenate(qs)

    def prompt_q(self, seq_id: int, p0: int, p1: int):
        """Queries of a joining sequence's prompt tokens p0 .. p1-1 ([p1-p0][Hq][D] bf16 bits), for
        the chunked prefill of its prompt."""
        row = self.Hq * self.D
        off = (seq_id * self.max_len + p0) * row
        return normal_bf16(stream_seed(self.seed, TAG_LOOP_PROMPT_Q), off, (p1 - p0) * row).reshape(p1 - p0, self.Hq,
                                                                                                      self.D)

    def prompt_kv(self, seq_id: int, n: int):
        """History K and V ([n][Hkv][D] bf16 bits) of a joining sequence's prompt."""
        row = self.Hkv * self.D
        off = seq_id * self.max_len * row
        k = normal_bf16(stream_seed(self.seed, TAG_LOOP_PROMPT_K), off, n * row).reshape(n, self.Hkv, self.D)
        v = normal_bf16(stream_seed(self.seed, TAG_LOOP_PROMPT_V), off, n * row).reshape(n, self.Hkv, self.D)
        return k, v

    def step_inputs(self, t: int, running):
        """(k_new, v_new, q) of step t for the running sequences, in their order (row i of step t
        is drawn from the block of the stream reserved for that step and row)."""
        n = len(running)
        row_kv, row_q = self.Hkv * self.D, self.Hq * self.D
        k = normal_bf16(stream_seed(self.seed, TAG_LOOP_K), t * self.max_batch * row_kv, n * row_kv)
        v = normal_bf16(stream_seed(self.seed, TAG_LOOP_V), t * self.max_batch * row_kv, n * row_kv)
        q = normal_bf16(stream_seed(self.seed, TAG_LOOP_Q), t * self.max_batch * row_q, n * row_q)
        return k.reshape(n, self.Hkv, self.D), v.reshape(n, self.Hkv, self.D), q.reshape(n, self.Hq, self.D)


def make_chunked_loop_script(index: int = 45, n_steps: int = 32, max_batch: int = 16, Hq: int = 8, Hkv: int = 2,
                             D: int = 128, block_size: int = 16, kv_dtype: str = "bf16", prompt_lo: int = 1,
                             prompt_hi: int = 300, p_finish: float = 0.12, chunk: int = 64, system: int = 0,
                             reuse: bool = True, num_blocks: int | None = None) -> LoopScript:
    """Seeded churn with chunked context: a joining sequence first prefills its prompt, `chunk`
    tokens per step, and decodes from the step after its last chunk; each step every decoding
    sequence finishes with probability p_finish, then new sequences (prompt lengths U[prompt_lo,
    prompt_hi]) fill the batch back to max_batch.  With `system` > 0 every prompt starts with the
    same `system` tokens, cached once (prefix caching, "TensorRT-LLM 推理加速实战" §8 KV cache
    reuse): a request forks them and prefills only its own prompt_lo..prompt_hi tokens."""
    seed = 266 * 1000 + index
    s = stream_seed(seed, TAG_LOOP_SCHED)
    draw = 0
    state: dict = {}
    steps, next_id, peak = [], 0, 0
    for t in range(n_steps):
        finished = []
        for sid in list(state):
            n, done, _ = state[sid]
            if done >= n:  # only decoding sequences finish
                if unit(s, draw) < p_finish:
                    finished.append(sid)
                    del state[sid]
                draw += 1
        joined = []
        while len(state) < max_batch:
            n = uniform_int(s, draw, prompt_lo, prompt_hi)
            draw += 1
            joined.append((next_id, n))
            state[next_id] = [system + n, system if reuse else 0, 0]
            next_id += 1
        steps.append((finished, joined))
        for sid, st in state.items():  # the step: a chunk for prefilling sequences, a token for decoders
            if st[1] < st[0]:
                st[1] = min(st[0], st[1] + chunk)
            else:
                st[2] += 1
        # blocks held: shared system blocks once, each request its own (and a copied partial one)
        shared = system // block_size if reuse else 0
        peak = max(peak, shared + (1 if system % block_size else 0) +
                   sum(_ceil_div(st[1] + st[2], block_size) - shared for st in state.values()))
    max_len = 2 * system + prompt_hi + n_steps + 1  # room for the system-prompt queries' stream rows
    nb = num_blocks or peak + 8 + (system // block_size + 1 if system else 0)
    name = f"chunkloop{index}" + (f"-sys{system}" + ("" if reuse else "-noreuse") if system else "")
    return LoopScript(name, seed, Hq, Hkv, D, block_size, kv_dtype, nb, max_batch, steps, max_len, chunk, system,
                      reuse)


def make_loop_script(index: int = 40, n_steps: int = 32, max_batch: int = 24, Hq: int = 8, Hkv: int = 2, D: int = 128,
                     block_size: int = 16, kv_dtype: str = "bf16", prompt_lo: int = 1, prompt_hi: int = 300,
                     p_finish: float = 0.12, num_blocks: int | None = None) -> LoopScript:
    """Seeded churn: each step every running sequence finishes with probability p_finish, then new
    sequences (prompt lengths U[prompt_lo, prompt_hi]) fill the batch back to max_batch.  The
    pool is sized so that the script never runs out of blocks."""
    seed = 266 * 1000 + index
    s = stream_seed(seed, TAG_LOOP_SCHED)
    draw = 0
    running, lens, steps, next_id, peak = [], {}, [], 0, 0
    for t in range(n_steps):
        finished = []
        for sid in list(running):
            if unit(s, draw) < p_finish:
                finished.append(sid)
                running.remove(sid)
                del lens[sid]
            draw += 1
        joined = []
        while len(running) < max_batch:
            n = uniform_int(s, draw, prompt_lo, prompt_hi)
            draw += 1
            joined.append((next_id, n))
            running.append(next_id)
            lens[next_id] = n
            next_id += 1
        steps.append((finished, joined))
        for sid in running:
            lens[sid] += 1
        peak = max(peak, sum(_ceil_div(L, block_size) for L in lens.values()))
    max_len = prompt_hi + n_steps + 1
    nb = num_blocks or peak + 8
    return LoopScript(f"loop{index}", seed, Hq, Hkv, D, block_size, kv_dtype, nb, max_batch, steps, max_len)


# ----------------------------------------------------------------------------- shared prefixes
TAG_PFX_LENS, TAG_PFX_K, TAG_PFX_V, TAG_SFX_K, TAG_SFX_V, TAG_PFX_Q, TAG_PFX_NEW_K, TAG_PFX_NEW_V = range(30, 38)


@dataclass
class PrefixScript:
    """B requests that share one P-token prompt prefix (a system prompt) and then diverge with
    suffixes of their own (block reuse: "TensorRT-LLM 推理加速实战", §8; enable_block_reuse in
    the pnsm.cn TensorRT-LLM page, §3.1).

    The parent sequence (id B) holds the prefix; child b (id b) is forked from it at P tokens,
    then holds suffix_lens[b] tokens of its own at positions P .. P + suffix_lens[b] - 1.  The
    step appends one new token per child at position P + suffix_lens[b] and attends over
    P + suffix_lens[b] + 1 tokens."""
    name: str
    seed: int
    B: int
    Hq: int
    Hkv: int
    D: int
    block_size: int
    kv_dtype: str
    P: int
    suffix_lens: np.ndarray
    num_blocks: int

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def parent(self) -> int:
        return self.B

    @property
    def max_suffix(self) -> int:
        return int(self.suffix_lens.max()) if self.B else 0

    @property
    def attend_lens(self) -> np.ndarray:
        return (self.P + self.suffix_lens + 1).astype(np.int32)

    @property
    def max_blocks(self) -> int:
        return _ceil_div(int(self.attend_lens.max()), self.block_size)

    def prefix_kv(self):
        row = self.Hkv * self.D
        k = normal_bf16(stream_seed(self.seed, TAG_PFX_K), 0, self.P * row).reshape(self.P, self.Hkv, self.D)
        v = normal_bf16(stream_seed(self.seed, TAG_PFX_V), 0, self.P * row).reshape(self.P, self.Hkv, self.D)
        return k, v

    def suffix_kv(self, b: int):
        row, n = self.Hkv * self.D, int(self.suffix_lens[b])
        off = b * self.max_suffix * row
        k = normal_bf16(stream_seed(self.seed, TAG_SFX_K), off, n * row).reshape(n, self.Hkv, self.D)
        v = normal_bf16(stream_seed(self.seed, TAG_SFX_V), off, n * row).reshape(n, self.Hkv, self.D)
        return k, v

    def step_inputs(self):
        """(k_new, v_new, q) of the decode step, one row per child."""
        rkv, rq = self.B * self.Hkv * self.D, self.B * self.Hq * self.D
        k = normal_bf16(stream_seed(self.seed, TAG_PFX_NEW_K), 0, rkv).reshape(self.B, self.Hkv, self.D)
        v = normal_bf16(stream_seed(self.seed, TAG_PFX_NEW_V), 0, rkv).reshape(self.B, self.Hkv, self.D)
        q = normal_bf16(stream_seed(self.seed, TAG_PFX_Q), 0, rq).reshape(self.B, self.Hq, self.D)
        return k, v, q

    def logical_kv(self, b: int):
        """Child b's whole history as one [P + suffix][Hkv][D] array (what it attends, minus the
        step's own token)."""
        pk, pv = self.prefix_kv()
        sk, sv = self.suffix_kv(b)
        return np.concatenate([pk, sk]), np.concatenate([pv, sv])

    def blocks_unshared(self) -> int:
        """Blocks the children would hold with no sharing (each its own copy of the prefix)."""
        return int(sum(_ceil_div(int(L), self.block_size) for L in self.attend_lens))

    def blocks_shared(self) -> int:
        """Blocks held with sharing: the prefix's whole blocks once, each child its own partial
        prefix block (copied) and suffix blocks."""
        full = self.P // self.block_size
        return full + int(sum(_ceil_div(int(L), self.block_size) - full for L in self.attend_lens))


def make_prefix_script(index: int = 60, B: int = 128, Hq: int = 32, Hkv: int = 8, D: int = 128, block_size: int = 64,
                       kv_dtype: str = "bf16", P: int = 2048, suffix_lo: int = 128,
                       suffix_hi: int = 2048) -> PrefixScript:
    seed = 266 * 1000 + index
    s = stream_seed(seed, TAG_PFX_LENS)
    suffix = np.array([uniform_int(s, b, suffix_lo, suffix_hi) for b in range(B)], dtype=np.int64)
    sc = PrefixScript(f"prefix{index}", seed, B, Hq, Hkv, D, block_size, kv_dtype, P, suffix, 0)
    # parent's partial block stays held until the parent is released; + spares
    sc.num_blocks = sc.blocks_shared() + (1 if P % block_size else 0) + 4
    return sc


# ----------------------------------------------------------------------------- chunked prefill
TAG_PF_LENS, TAG_PF_PERM, TAG_PF_K, TAG_PF_V, TAG_PF_Q = range(40, 45)


@dataclass
class PrefillScript:
    """One chunked-context step ("TensorRT-LLM 深度实战", §7.3): sequence b already caches
    past[b] tokens and now processes a chunk of chunk[b] prompt tokens — their K/V are appended
    and each of their queries attends to the past and, causally, to the chunk.

    K/V of sequence b at position t and the chunk's queries are drawn from counter streams at
    fixed offsets, so any subset can be regenerated."""
    name: str
    seed: int
    B: int
    Hq: int
    Hkv: int
    D: int
    block_size: int
    kv_dtype: str
    past: np.ndarray
    chunk: np.ndarray
    num_blocks: int
    free_order: np.ndarray

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def ctx(self) -> np.ndarray:
        return (self.past + self.chunk).astype(np.int32)

    @property
    def max_len(self) -> int:
        return int(self.ctx.max()) if self.B else 0

    @property
    def cu_q(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.chunk)]).astype(np.int32)

    @property
    def max_blocks(self) -> int:
        return max(1, _ceil_div(self.max_len, self.block_size))

    def kv(self, b: int, t0: int, t1: int):
        """K and V of sequence b, positions t0 .. t1-1, as [t1-t0][Hkv][D] bf16 bits."""
        row = self.Hkv * self.D
        off = (b * self.max_len + t0) * row
        n = (t1 - t0) * row
        k = normal_bf16(stream_seed(self.seed, TAG_PF_K), off, n).reshape(t1 - t0, self.Hkv, self.D)
        v = normal_bf16(stream_seed(self.seed, TAG_PF_V), off, n).reshape(t1 - t0, self.Hkv, self.D)
        return k, v

    def chunk_kv(self):
        """The chunks' K/V rows in cu_q order."""
        ks, vs = zip(*(self.kv(b, int(self.past[b]), int(self.ctx[b])) for b in range(self.B))) if self.B else ((), ())
        row = (0, self.Hkv, self.D)
        return (np.concatenate(ks) if ks else np.zeros(row, np.uint16),
                np.concatenate(vs) if vs else np.zeros(row, np.uint16))

    def query(self, r0: int = 0, r1: int | None = None) -> np.ndarray:
        """Query rows r0 .. r1-1 of the packed chunks ([rows][Hq][D] bf16 bits)."""
        r1 = int(self.cu_q[-1]) if r1 is None else r1
        row = self.Hq * self.D
        return normal_bf16(stream_seed(self.seed, TAG_PF_Q), r0 * row, (r1 - r0) * row).reshape(r1 - r0, self.Hq,
                                                                                                 self.D)

    def chunk_slots_positions(self):
        """(sequence, position) of every chunk row, in cu_q order."""
        seqs = np.concatenate([np.full(int(self.chunk[b]), b) for b in range(self.B)]) if self.B else np.zeros(0)
        pos = np.concatenate([np.arange(int(self.past[b]), int(self.ctx[b])) for b in range(self.B)]) if self.B \
            else np.zeros(0)
        return seqs.astype(np.int64), pos.astype(np.int64)

    def flops(self) -> int:
        """Causal attention FLOPs of the step: 4 * D per (query head, query, attended key)."""
        keys = sum(int(self.chunk[b]) * int(self.past[b]) + int(self.chunk[b]) * (int(self.chunk[b]) + 1) // 2
                   for b in range(self.B))
        return 4 * self.D * self.Hq * keys


def make_prefill_script(index: int = 70, B: int = 8, Hq: int = 32, Hkv: int = 8, D: int = 128, block_size: int = 64,
                        past=None, chunk=None, past_lo: int = 0, past_hi: int = 32256, chunk_lo: int = 512,
                        chunk_hi: int = 512, kv_dtype: str = "bf16", spare_blocks: int = 3) -> PrefillScript:
    """Default: 8 sequences of the long-context serving setting ("TensorRT-LLM 深度实战" §7.2-7.3:
    32K contexts, chunks of 512 tokens, 4096 tokens per step), each at a seeded point of its
    prompt (past U[0, 32256]), Llama-3-8B layer shapes, block 64."""
    seed = 266 * 1000 + index
    s = stream_seed(seed, TAG_PF_LENS)
    past = np.asarray(past if past is not None else [uniform_int(s, 2 * b, past_lo, past_hi) for b in range(B)],
                      dtype=np.int64)
    chunk = np.asarray(chunk if chunk is not None else [uniform_int(s, 2 * b + 1, chunk_lo, chunk_hi)
                                                        for b in range(B)], dtype=np.int64)
    nb = int(sum(_ceil_div(int(p + c), block_size) for p, c in zip(past, chunk))) + spare_blocks
    order = permutation(stream_seed(seed, TAG_PF_PERM), nb)
    return PrefillScript(f"prefill{index}", seed, len(past), Hq, Hkv, D, block_size, kv_dtype, past, chunk, nb, order)
