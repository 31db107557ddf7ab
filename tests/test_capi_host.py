"""Host-side checks of the C ABI (no GPU): the library loads, exports every entry point
declared in include/pkv.h, and its block allocator matches the oracle's replica bit for bit."""
import os
import re

import numpy as np
import pytest

import oracle
import pkv_workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_266_gb300 import build
    build.build()
    import paged_kv_cache_266_gb300 as m
    m._L()
    return m


def _declared():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(pkv_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol(pkv):
    import ctypes
    lib = ctypes.CDLL(pkv.library_path())
    names = _declared()
    assert len(names) >= 20
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol(pkv):
    missing = [n for n in _declared() if not hasattr(pkv, n)]
    assert not missing, missing


def test_kv_bytes_worked_values(pkv):
    assert pkv.pkv_kv_bytes(80, 8, 128, 1, 1, 2) == 327680
    assert pkv.pkv_kv_bytes(80, 8, 128, 1, 1, 1) == 163840
    assert pkv.pkv_kv_bytes(1, 8, 128, 4096, 128, 2) == 2 ** 31
    assert pkv.pkv_kv_bytes(80, 8, 128, 1, 1, 0.5) == 81920


def test_status_strings(pkv):
    for s in range(7):
        assert pkv.pkv_status_str(s)
    assert pkv.pkv_status_str(0) == "ok"


def test_invalid_arguments_are_rejected_without_device_work(pkv):
    L = pkv._L()
    import ctypes
    h = ctypes.c_void_p()
    assert L.pkv_pool_create(16, 16, 2, 96, 0, ctypes.byref(h)) == pkv.PKV_ERR_INVALID_ARG  # head_dim
    assert L.pkv_pool_create(16, 24, 2, 64, 0, ctypes.byref(h)) == pkv.PKV_ERR_INVALID_ARG  # block size
    assert L.pkv_pool_create(16, 16, 2, 64, 7, ctypes.byref(h)) == pkv.PKV_ERR_INVALID_ARG  # dtype
    assert L.pkv_pool_create(0, 16, 2, 64, 0, ctypes.byref(h)) == pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_append(None, None, None, None, 1, None) == pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_decode_attention(None, None, None, 1, None, 1, 1, 1.0, None, None, 0, None) == \
        pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_allocator_create(0, 16, ctypes.byref(h)) == pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_allocator_create(4, 48, ctypes.byref(h)) == pkv.PKV_ERR_INVALID_ARG
    # staging copy: checked before any CUDA call (these addresses are never dereferenced)
    assert L.pkv_stage_copy(None, None, 0, None) == pkv.PKV_OK  # nothing to copy
    assert L.pkv_stage_copy(None, 4096, 64, None) == pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_stage_copy(4096, 8192 + 8, 64, None) == pkv.PKV_ERR_INVALID_ARG  # misaligned
    assert L.pkv_stage_copy(4096, 8192, 40, None) == pkv.PKV_ERR_INVALID_ARG  # not a multiple of 16
    assert L.pkv_stage_copy(4096, 4096 + 32, 64, None) == pkv.PKV_ERR_INVALID_ARG  # overlapping ranges


def _both(pkv, nb, bs, order=None):
    a = pkv.pkv_allocator_create(nb, bs)
    o = oracle.Allocator(nb, bs)
    if order is not None:
        pkv.pkv_allocator_set_free_order(a, order)
        assert o.set_free_order(order) == 0
    return a, o


def _same_state(pkv, a, o, live):
    assert pkv.pkv_free_list(a).tolist() == o.free_list().tolist()
    for s in live:
        assert pkv.pkv_seq_num_blocks(a, s) == o.num_pages(s)
    if live:
        ids = sorted(live)
        mb = max(o.num_pages(s) for s in ids) + 2
        assert np.array_equal(pkv.pkv_get_block_tables(a, ids, mb), o.block_tables(ids, mb))


def test_allocator_matches_oracle_on_random_scripts(pkv):
    rng = np.random.default_rng(0)
    for trial in range(20):
        nb, bs = int(rng.integers(1, 200)), int(2 ** rng.integers(4, 9))
        a, o = _both(pkv, nb, bs, rng.permutation(nb).astype(np.int32) if trial % 2 else None)
        live = set()
        for _ in range(300):
            if rng.random() < 0.6 or not live:
                s = int(rng.integers(0, 40))
                n = int(rng.integers(0, 6 * bs))
                rc_o = o.reserve(s, n)
                try:
                    pkv.pkv_seq_reserve(a, s, n)
                    rc = 0
                except pkv.PKVError as e:
                    rc = e.status
                assert rc == {0: 0, 2: pkv.PKV_ERR_OOM}[rc_o]
                if rc == 0:
                    live.add(s)
            else:
                s = int(rng.choice(sorted(live)))
                assert o.release(s) == 0
                pkv.pkv_seq_release(a, s)
                live.discard(s)
            _same_state(pkv, a, o, live)
        # slot mapping over every held position, plus padding
        for s in live:
            n = o.num_pages(s) * bs
            pos = np.arange(-1, n)
            assert np.array_equal(pkv.pkv_slot_mapping(a, [s] * len(pos), pos), o.slot_mapping([s] * len(pos), pos))
        pkv.pkv_allocator_destroy(a)


def test_allocator_matches_oracle_on_churned_workload(pkv):
    w = W.make_workload("c4")
    a, o = _both(pkv, w.num_blocks, w.block_size, w.free_order)
    from paged_kv_cache_266_gb300.runner import replay
    replay(a, w.alloc_ops)
    o.replay(w.alloc_ops)
    mb = w.max_blocks()
    assert np.array_equal(pkv.pkv_get_block_tables(a, w.seq_ids, mb), o.block_tables(w.seq_ids, mb))
    assert pkv.pkv_free_list(a).tolist() == o.free_list().tolist()
    seqs, pos = w.hist_positions(0, 5000)
    assert np.array_equal(pkv.pkv_slot_mapping(a, seqs, pos), o.slot_mapping(seqs, pos))
    pkv.pkv_allocator_destroy(a)


def test_allocator_errors(pkv):
    a = pkv.pkv_allocator_create(4, 16)
    with pytest.raises(pkv.PKVError) as e:
        pkv.pkv_seq_release(a, 3)
    assert e.value.status == pkv.PKV_ERR_NO_SEQ
    pkv.pkv_seq_reserve(a, 1, 40)  # 3 blocks
    with pytest.raises(pkv.PKVError) as e:
        pkv.pkv_seq_reserve(a, 2, 40)
    assert e.value.status == pkv.PKV_ERR_OOM
    with pytest.raises(pkv.PKVError) as e:
        pkv.pkv_seq_num_blocks(a, 2)  # the failed reserve created nothing
    assert e.value.status == pkv.PKV_ERR_NO_SEQ
    with pytest.raises(pkv.PKVError) as e:
        pkv.pkv_get_block_tables(a, [1], 2)
    assert e.value.status == pkv.PKV_ERR_BOUNDS
    with pytest.raises(pkv.PKVError) as e:
        pkv.pkv_slot_mapping(a, [1], [48])
    assert e.value.status == pkv.PKV_ERR_BOUNDS
    with pytest.raises(pkv.PKVError) as e:
        pkv.pkv_allocator_set_free_order(a, [0, 1, 2, 3])  # blocks are held
    assert e.value.status == pkv.PKV_ERR_INVALID_ARG
    pkv.pkv_seq_release(a, 1)
    with pytest.raises(pkv.PKVError):
        pkv.pkv_allocator_set_free_order(a, [0, 1, 1, 3])  # not a permutation
    pkv.pkv_allocator_destroy(a)


def test_reserve_many_equals_sequential_reserves(pkv):
    rng = np.random.default_rng(3)
    a = pkv.pkv_allocator_create(64, 16)
    o = oracle.Allocator(64, 16)
    seqs = np.arange(10, dtype=np.int64)
    toks = rng.integers(0, 60, 10)
    pkv.pkv_seq_reserve_many(a, seqs, toks)
    for s, n in zip(seqs, toks):
        assert o.reserve(int(s), int(n)) == 0
    _same_state(pkv, a, o, set(seqs.tolist()))
    # growth for every sequence, then one that cannot fit: earlier ones stay, the call reports OOM
    grow = toks + 16
    big = np.array(grow)
    big[5] = 10_000
    with pytest.raises(pkv.PKVError) as e:
        pkv.pkv_seq_reserve_many(a, seqs, big)
    assert e.value.status == pkv.PKV_ERR_OOM and "after 5 reservations" in str(e.value)
    for s in range(5):
        assert o.reserve(int(seqs[s]), int(grow[s])) == 0
    _same_state(pkv, a, o, set(seqs.tolist()))
    pkv.pkv_allocator_destroy(a)


def test_stage_calls_equal_their_composition(pkv):
    """pkv_stage_prefill / pkv_stage_decode against reserve + block tables + slot mapping run
    on a second allocator with the same state: identical outputs and identical free lists."""
    rng = np.random.default_rng(7)
    for bs in (16, 64):
        a, b = pkv.pkv_allocator_create(400, bs), pkv.pkv_allocator_create(400, bs)
        order = rng.permutation(400).astype(np.int32)
        pkv.pkv_allocator_set_free_order(a, order)
        pkv.pkv_allocator_set_free_order(b, order)
        held = {}
        for step in range(30):
            ids = rng.choice(60, size=int(rng.integers(1, 8)), replace=False).astype(np.int64)
            p0 = np.array([held.get(int(s), 0) for s in ids], dtype=np.int64)
            p1 = p0 + rng.integers(0, 40, len(ids))
            mb = 50
            slots, cu, ctx, tables = pkv.pkv_stage_prefill(a, ids, p0, p1, mb)
            for s, e in zip(ids, p1):
                pkv.pkv_seq_reserve(b, int(s), int(e))
            seqs = np.repeat(ids, p1 - p0)
            pos = np.concatenate([np.arange(x, y) for x, y in zip(p0, p1)]) if len(ids) else np.zeros(0)
            assert np.array_equal(slots, pkv.pkv_slot_mapping(b, seqs, pos))
            assert np.array_equal(tables, pkv.pkv_get_block_tables(b, ids, mb))
            assert cu.tolist() == [0] + np.cumsum(p1 - p0).tolist() and ctx.tolist() == p1.tolist()
            for s, e in zip(ids, p1):
                held[int(s)] = int(e)
            # one decode step over some held sequences, padded to a bucket
            dec = np.array(sorted(held)[: int(rng.integers(0, 6))], dtype=np.int64)
            dpos = np.array([held[int(s)] for s in dec], dtype=np.int64)
            n_pad = len(dec) + int(rng.integers(0, 3))
            t2, s2, l2 = pkv.pkv_stage_decode(a, dec, dpos, n_pad, mb)
            for s, q in zip(dec, dpos):
                pkv.pkv_seq_reserve(b, int(s), int(q) + 1)
            assert np.array_equal(t2[: len(dec)], pkv.pkv_get_block_tables(b, dec, mb))
            assert np.array_equal(s2[: len(dec)], pkv.pkv_slot_mapping(b, dec, dpos))
            assert l2[: len(dec)].tolist() == (dpos + 1).tolist()
            assert (t2[len(dec):] == -1).all() and (s2[len(dec):] == -1).all() and (l2[len(dec):] == 0).all()
            for s, q in zip(dec, dpos):
                held[int(s)] = int(q) + 1
            if rng.random() < 0.3 and held:  # a sequence finishes
                s = int(rng.choice(sorted(held)))
                pkv.pkv_seq_release(a, s)
                pkv.pkv_seq_release(b, s)
                del held[s]
            assert pkv.pkv_free_list(a).tolist() == pkv.pkv_free_list(b).tolist()
        L = pkv._L()
        one = np.zeros(4, np.int64)
        assert L.pkv_stage_prefill(a, one.ctypes.data, one.ctypes.data, one.ctypes.data, 1, 0, one.ctypes.data,
                                   one.ctypes.data, one.ctypes.data, one.ctypes.data) == pkv.PKV_ERR_INVALID_ARG
        bad = np.array([5], np.int64)
        assert L.pkv_stage_prefill(a, one.ctypes.data, bad.ctypes.data, one.ctypes.data, 1, 4, one.ctypes.data,
                                   one.ctypes.data, one.ctypes.data, one.ctypes.data) == pkv.PKV_ERR_INVALID_ARG  # p1 < p0
        assert L.pkv_stage_decode(a, one.ctypes.data, one.ctypes.data, 2, 1, 4, one.ctypes.data, one.ctypes.data,
                                  one.ctypes.data) == pkv.PKV_ERR_INVALID_ARG  # n_pad < n
        pkv.pkv_allocator_destroy(a)
        pkv.pkv_allocator_destroy(b)


def test_stage_calls_match_the_oracle_allocator(pkv):
    """The same random admission / decode script through pkv_stage_prefill / pkv_stage_decode
    and through the oracle's allocator replica: slots and block tables bit-identical."""
    rng = np.random.default_rng(31)
    a = pkv.pkv_allocator_create(300, 16)
    o = oracle.Allocator(300, 16)
    order = rng.permutation(300).astype(np.int32)
    pkv.pkv_allocator_set_free_order(a, order)
    assert o.set_free_order(order) == 0
    held, mb = {}, 40
    for step in range(25):
        new = [s for s in rng.choice(200, size=int(rng.integers(0, 4)), replace=False).tolist() if s not in held]
        if new:
            ids = np.array(new, dtype=np.int64)
            p1 = rng.integers(0, 120, len(ids)).astype(np.int64)
            slots, _, _, tables = pkv.pkv_stage_prefill(a, ids, np.zeros_like(p1), p1, mb)
            for s_, n_ in zip(new, p1.tolist()):
                assert o.reserve(s_, n_) == 0
            seqs = np.repeat(ids, p1)
            pos = np.concatenate([np.arange(n_) for n_ in p1.tolist()])
            assert np.array_equal(slots, o.slot_mapping(seqs, pos))
            assert np.array_equal(tables, o.block_tables(new, mb))
            held.update(zip(new, p1.tolist()))
        dec = np.array(sorted(held), dtype=np.int64)
        dpos = np.array([held[s_] for s_ in dec.tolist()], dtype=np.int64)
        t2, s2, _ = pkv.pkv_stage_decode(a, dec, dpos, len(dec) + 1, mb)
        for s_, q_ in zip(dec.tolist(), dpos.tolist()):
            assert o.reserve(s_, q_ + 1) == 0
            held[s_] = q_ + 1
        if len(dec):
            assert np.array_equal(s2[:-1], o.slot_mapping(dec, dpos))
            assert np.array_equal(t2[:-1], o.block_tables(dec.tolist(), mb))
        for s_ in [s_ for s_ in sorted(held) if rng.random() < 0.15]:
            assert pkv.pkv_seq_release(a, s_) is None and o.release(s_) == 0
            del held[s_]
        assert pkv.pkv_free_list(a).tolist() == o.free_list().tolist()
    pkv.pkv_allocator_destroy(a)


def _golden_splitmix():
    rows = []
    for line in open(os.path.join(os.path.dirname(__file__), "golden", "splitmix64.txt")):
        if line.strip() and not line.startswith("#"):
            seed, i, out = line.split()
            rows.append((int(seed), int(i), int(out, 16)))
    return rows


def test_input_generator_splitmix64_matches_its_published_outputs():
    """The seeded inputs of every workload come from splitmix64; its published reference outputs
    pin the generator (and, through the shuffle test below, the library's own restatement)."""
    import pkv_workloads as W
    for seed, i, out in _golden_splitmix():
        assert W.splitmix64_at(seed, i) == out


def test_shuffle_free_list_is_the_workloads_seeded_permutation(pkv):
    """pkv_allocator_shuffle_free_list on a fresh allocator gives the generator's seeded
    Fisher-Yates permutation, so a C caller reproduces the workloads' allocation state from the
    seed alone; on a list that is no longer 0..n-1 it applies the same permutation to the
    entries; held blocks are untouched."""
    import pkv_workloads as W
    for n in (1, 2, 3, 32, 1000, 8192):
        for seed in (0, 1, 266002, 2 ** 64 - 1, W.stream_seed(266 * 1000 + 2, W.TAG_PERM)):
            a = pkv.pkv_allocator_create(n, 16)
            pkv.pkv_allocator_shuffle_free_list(a, seed)
            assert np.array_equal(pkv.pkv_free_list(a), W.permutation(seed, n)), (n, seed)
            pkv.pkv_allocator_destroy(a)
    w = W.make_workload("c2")
    a = pkv.pkv_allocator_create(w.num_blocks, w.block_size)
    pkv.pkv_allocator_shuffle_free_list(a, W.stream_seed(w.seed, W.TAG_PERM))
    assert np.array_equal(pkv.pkv_free_list(a), w.free_order)
    pkv.pkv_allocator_destroy(a)
    # after some allocation: the remaining entries are permuted, the held blocks stay held
    a = pkv.pkv_allocator_create(64, 16)
    pkv.pkv_seq_reserve(a, 7, 16 * 5)
    pkv.pkv_seq_reserve(a, 8, 16 * 3)
    pkv.pkv_seq_release(a, 7)
    before = pkv.pkv_free_list(a)
    held = pkv.pkv_get_block_tables(a, [8], 3)[0]
    pkv.pkv_allocator_shuffle_free_list(a, 99)
    assert np.array_equal(pkv.pkv_free_list(a), before[W.permutation(99, len(before))])
    assert np.array_equal(pkv.pkv_get_block_tables(a, [8], 3)[0], held)
    pkv.pkv_allocator_destroy(a)
