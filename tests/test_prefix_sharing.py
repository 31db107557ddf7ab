"""Block reuse (prefix sharing with copy on write): oracle pins, the C allocator against the
oracle replica, and decode attention over sequences that share prefix blocks on the GPU."""
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_bits(x):
    import torch
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_prefix_share_golden_trace():
    a = oracle.Allocator(8, 4)
    ids = {}
    sid = lambda s: ids.setdefault(s, len(ids) + 100)
    for line in open(os.path.join(GOLDEN, "prefix_share_trace.txt")):
        if line.startswith("#") or not line.strip():
            continue
        lhs, rhs = [x.strip() for x in line.split("->")]
        op = lhs.split()
        fields = [f.strip() for f in rhs.split("|")]
        if op[0] == "reserve":
            assert a.reserve(sid(op[1]), int(op[2])) == 0
        elif op[0] == "release":
            assert a.release(sid(op[1])) == 0
        elif op[0] == "holders":
            assert a.holders(int(op[1])) == int(fields[0])
            continue
        elif op[0] == "share":
            rc, cs, cd = a.share_prefix(sid(op[1]), sid(op[2]), int(op[3]))
            if fields[0] == "noseq":
                assert rc == 3
                continue
            want = fields[0].split()
            assert rc == 0 and (cs, cd) == (int(want[2]), int(want[3])), line
        if len(fields) > 1 and fields[1]:
            name, pages = fields[1].split(":")
            s = sid(name.strip())
            assert a.block_tables([s], a.num_pages(s)).tolist() == [[int(x) for x in pages.split()]], line
        assert a.free_list().tolist() == [int(x) for x in fields[2].split(":")[1].split()], line


def _random_share_script(rng, nb, bs, n_ops):
    ops, live, nxt = [], [], 0
    for _ in range(n_ops):
        r = rng.random()
        if r < 0.35 or not live:
            ops.append(("reserve", nxt, int(rng.integers(0, 5 * bs))))
            live.append(nxt)
            nxt += 1
        elif r < 0.6:
            src = int(rng.choice(live))
            ops.append(("share", src, nxt, int(rng.integers(0, 5 * bs))))
            live.append(nxt)
            nxt += 1
        elif r < 0.8:
            s = int(rng.choice(live))
            ops.append(("reserve", s, int(rng.integers(0, 7 * bs))))
        else:
            s = int(rng.choice(live))
            ops.append(("release", s))
            live.remove(s)
    return ops


def test_holder_counts_are_conserved_under_sharing():
    rng = np.random.default_rng(5)
    a = oracle.Allocator(48, 8)
    tables = {}
    for op in _random_share_script(rng, 48, 8, 400):
        if op[0] == "reserve":
            if a.reserve(op[1], op[2]) == 0:
                tables[op[1]] = True
        elif op[0] == "share":
            rc, cs, cd = a.share_prefix(op[1], op[2], op[3])
            if rc == 0:
                tables[op[2]] = True
                assert (cs == -1) == (op[3] % 8 == 0)
        else:
            if a.release(op[1]) == 0:
                del tables[op[1]]
        held = {}
        for s in tables:
            for pg in a.block_tables([s], a.num_pages(s))[0]:
                held[pg] = held.get(pg, 0) + 1
        free = set(a.free_list().tolist())
        for pg in range(48):
            assert a.holders(pg) == held.get(pg, 0)
            assert (pg in free) == (held.get(pg, 0) == 0)


def test_shared_prefix_attends_exactly_like_its_source():
    """A sequence that shares (and copies the partial block of) another's first n tokens sees the
    same K/V: attention over its n tokens equals the source's over the same n tokens."""
    rng = np.random.default_rng(9)
    bs, Hkv, D, G = 16, 2, 64, 2
    for fp8 in (False, True):
        a = oracle.Allocator(20, bs)
        pool = oracle.Pool(20, bs, Hkv, D, fp8)
        L = 53
        assert a.reserve(1, L) == 0
        k, v = _bf16_bits(rng.standard_normal((L, Hkv, D))), _bf16_bits(rng.standard_normal((L, Hkv, D)))
        pool.append(k, v, a.slot_mapping([1] * L, np.arange(L)))
        for n in (16, 37, 53):
            rc, cs, cd = a.share_prefix(1, 100 + n, n)
            assert rc == 0
            if cs >= 0:
                pool.copy_block(cs, cd)
            q = _bf16_bits(rng.standard_normal((1, Hkv * G, D)))
            mb = a.num_pages(1)
            t_src = a.block_tables([1], mb)
            t_dst = a.block_tables([100 + n], mb) if a.num_pages(100 + n) == mb else np.pad(
                a.block_tables([100 + n], a.num_pages(100 + n)), ((0, 0), (0, mb - a.num_pages(100 + n))),
                constant_values=-1)
            o1 = pool.attention(q, t_src, np.array([n]), Hkv * G, 0.125)
            o2 = pool.attention(q, t_dst, np.array([n]), Hkv * G, 0.125)
            assert np.array_equal(o1, o2)


def test_c_allocator_matches_oracle_with_sharing():
    from paged_kv_cache_266_gb300 import build
    build.build()
    import paged_kv_cache_266_gb300 as pkv
    rng = np.random.default_rng(11)
    for trial in range(10):
        nb, bs = int(rng.integers(4, 80)), int(2 ** rng.integers(4, 7))
        a = pkv.pkv_allocator_create(nb, bs)
        o = oracle.Allocator(nb, bs)
        live = set()
        for op in _random_share_script(rng, nb, bs, 250):
            if op[0] == "reserve":
                rc_o = o.reserve(op[1], op[2])
                try:
                    pkv.pkv_seq_reserve(a, op[1], op[2])
                    rc = 0
                except pkv.PKVError as e:
                    rc = e.status
                assert rc == {0: 0, 2: pkv.PKV_ERR_OOM}[rc_o]
                if rc == 0:
                    live.add(op[1])
            elif op[0] == "share":
                rc_o, cs_o, cd_o = o.share_prefix(op[1], op[2], op[3])
                try:
                    cs, cd = pkv.pkv_seq_share_prefix(a, op[1], op[2], op[3])
                    rc = 0
                except pkv.PKVError as e:
                    rc = e.status
                assert rc == {0: 0, 2: pkv.PKV_ERR_OOM, 3: pkv.PKV_ERR_NO_SEQ, 4: pkv.PKV_ERR_BOUNDS,
                              1: pkv.PKV_ERR_INVALID_ARG}[rc_o]
                if rc == 0:
                    assert (cs, cd) == (cs_o, cd_o)
                    live.add(op[2])
            else:  # the script may name a sequence whose reserve or share failed
                rc_o = o.release(op[1])
                try:
                    pkv.pkv_seq_release(a, op[1])
                    rc = 0
                except pkv.PKVError as e:
                    rc = e.status
                assert rc == {0: 0, 3: pkv.PKV_ERR_NO_SEQ}[rc_o]
                live.discard(op[1])
            assert pkv.pkv_free_list(a).tolist() == o.free_list().tolist()
        for s in live:
            n = o.num_pages(s)
            assert pkv.pkv_get_block_tables(a, [s], n).tolist() == o.block_tables([s], n).tolist()
        for blk in range(nb):
            assert pkv.pkv_block_refcount(a, blk) == o.holders(blk)
        pkv.pkv_allocator_destroy(a)


@pytest.mark.gpu
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_decode_over_shared_prefixes_matches_oracle(kv_dtype):
    """A parent sequence and children forked at several prefix lengths (full-block and partial
    ends), each child then appending its own tokens: pool bytes bit-exact, attention within
    tolerance of the oracle, and the shared blocks are held, not duplicated."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_266_gb300 import build
    build.build()
    import paged_kv_cache_266_gb300 as pkv
    from paged_kv_cache_266_gb300.runner import _wrap_device
    rng = np.random.default_rng(21)
    fp8 = kv_dtype == "fp8_e4m3"
    bs, Hkv, D, G, nb = 16, 2, 128, 4, 64
    Hq = Hkv * G
    pool = pkv.KVPool(nb, bs, Hkv, D, pkv.PKV_KV_FP8_E4M3 if fp8 else pkv.PKV_KV_BF16)
    a = pool.allocator
    oa = oracle.Allocator(nb, bs)
    op = oracle.Pool(nb, bs, Hkv, D, fp8)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()

    def append(seq, pos, k, v):
        slots = pkv.pkv_slot_mapping(a, [seq] * len(pos), pos)
        assert np.array_equal(slots, oa.slot_mapping([seq] * len(pos), pos))
        pkv.pkv_append(pool.handle, dev(k), dev(v), torch.from_numpy(slots).cuda())
        op.append(k, v, slots)

    L = 150
    pkv.pkv_seq_reserve(a, 0, L)
    oa.reserve(0, L)
    append(0, np.arange(L), _bf16_bits(rng.standard_normal((L, Hkv, D))), _bf16_bits(rng.standard_normal((L, Hkv, D))))
    lens = {0: L}
    for child, n in ((1, 64), (2, 100), (3, 150), (4, 7)):
        cs, cd = pkv.pkv_seq_share_prefix(a, 0, child, n)
        rc, cs_o, cd_o = oa.share_prefix(0, child, n)
        assert rc == 0 and (cs, cd) == (cs_o, cd_o)
        if cs >= 0:
            pkv.pkv_pool_copy_block(pool.handle, cs, cd)
            op.copy_block(cs, cd)
        extra = int(rng.integers(1, 40))
        pkv.pkv_seq_reserve(a, child, n + extra)
        oa.reserve(child, n + extra)
        append(child, np.arange(n, n + extra), _bf16_bits(rng.standard_normal((extra, Hkv, D))),
               _bf16_bits(rng.standard_normal((extra, Hkv, D))))
        lens[child] = n + extra
    # block 0 is held by the parent and the three children forked at 64+ tokens; the child forked
    # at 7 tokens took a copy of it instead
    assert pkv.pkv_block_refcount(a, int(pkv.pkv_get_block_tables(a, [0], 10)[0, 0])) == 4
    for blk in range(nb):
        assert pkv.pkv_block_refcount(a, blk) == oa.holders(blk)
    seqs = list(lens)
    mb = max(-(-lens[s] // bs) for s in seqs)
    tables = pkv.pkv_get_block_tables(a, seqs, mb)
    assert np.array_equal(tables, oa.block_tables(seqs, mb))
    q = _bf16_bits(rng.standard_normal((len(seqs), Hq, D)))
    lens_arr = np.array([lens[s] for s in seqs], dtype=np.int32)
    out = torch.empty(len(seqs), Hq, D, dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(pkv.pkv_decode_workspace_bytes(pool.handle, len(seqs), Hq, mb), dtype=torch.uint8, device="cuda")
    pkv.pkv_decode_attention(pool.handle, dev(q), torch.from_numpy(tables).cuda(), torch.from_numpy(lens_arr).cuda(),
                             1 / math.sqrt(D), out, ws)
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_error(pool.handle) == pkv.PKV_OK
    kv_ptr, kv_bytes, sc_ptr, sc_bytes = pkv.pkv_pool_raw(pool.handle)
    assert np.array_equal(_wrap_device(kv_ptr, kv_bytes).cpu().numpy(), op.data)
    if fp8:
        assert np.array_equal(_wrap_device(sc_ptr, sc_bytes).cpu().numpy().view(np.float32), op.scales)
    ref = op.attention(q, tables, lens_arr, Hq, 1 / math.sqrt(D))
    got = oracle.bf16_bits_to_f64(out.view(torch.int16).cpu().numpy().view(np.uint16))
    err = np.abs(got - ref)
    assert err.max() <= (3e-2 if fp8 else 1e-2) and err.mean() <= 1e-3
    pool.close()


def _oracle_prefix(sc):
    """The oracle's replay of PrefixDecode(share=True): allocator, pool bytes, attention."""
    fp8 = sc.kv_dtype == "fp8_e4m3"
    a, pool = oracle.Allocator(sc.num_blocks, sc.block_size), oracle.Pool(sc.num_blocks, sc.block_size, sc.Hkv, sc.D, fp8)
    P = sc.P
    assert a.reserve(sc.parent, P) == 0
    pk, pv = sc.prefix_kv()
    pool.append(pk, pv, a.slot_mapping([sc.parent] * P, np.arange(P)))
    for b in range(sc.B):
        rc, cs, cd = a.share_prefix(sc.parent, b, P)
        assert rc == 0
        if cs >= 0:
            pool.copy_block(cs, cd)
        assert a.reserve(b, P + int(sc.suffix_lens[b]) + 1) == 0
        n = int(sc.suffix_lens[b])
        if n:
            sk, sv = sc.suffix_kv(b)
            pool.append(sk, sv, a.slot_mapping([b] * n, np.arange(P, P + n)))
    assert a.release(sc.parent) == 0
    k, v, q = sc.step_inputs()
    seqs = np.arange(sc.B)
    pool.append(k, v, a.slot_mapping(seqs, P + sc.suffix_lens))
    tables = a.block_tables(seqs, sc.max_blocks)
    return a, pool, tables, pool.attention(q, tables, sc.attend_lens, sc.Hq, 1 / math.sqrt(sc.D))


@pytest.mark.gpu
@pytest.mark.parametrize("kv_dtype,bs,P", [("bf16", 16, 37), ("bf16", 64, 128), ("fp8_e4m3", 16, 50),
                                           ("fp8_e4m3", 64, 64)])
def test_prefix_decode_step_matches_oracle(kv_dtype, bs, P):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_266_gb300 import build
    build.build()
    import paged_kv_cache_266_gb300 as pkv
    import pkv_workloads as W
    from paged_kv_cache_266_gb300.runner import PrefixDecode, _wrap_device
    sc = W.make_prefix_script(61, B=9, Hq=8, Hkv=2, D=128, block_size=bs, kv_dtype=kv_dtype, P=P, suffix_lo=0,
                              suffix_hi=150)
    oa, opool, otables, ref = _oracle_prefix(sc)
    st = PrefixDecode(sc, share=True)
    st.step()
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_error(st.pool.handle) == pkv.PKV_OK
    assert np.array_equal(st.tables_host, otables)
    assert st.blocks_held == sc.blocks_shared()
    kv_ptr, kv_bytes, sc_ptr, sc_bytes = pkv.pkv_pool_raw(st.pool.handle)
    assert np.array_equal(_wrap_device(kv_ptr, kv_bytes).cpu().numpy(), opool.data)
    if sc_bytes:
        assert np.array_equal(_wrap_device(sc_ptr, sc_bytes).cpu().numpy().view(np.float32), opool.scales)
    got = oracle.bf16_bits_to_f64(st.out_host())
    err = np.abs(got - ref)
    assert err.max() <= (3e-2 if kv_dtype == "fp8_e4m3" else 1e-2) and err.mean() <= 1e-3
    # the same logical contexts without sharing give the same bits (the kernel sees equal data)
    un = PrefixDecode(sc, share=False)
    un.step()
    torch.cuda.synchronize()
    assert un.blocks_held == sc.blocks_unshared()
    assert np.array_equal(un.out_host(), st.out_host())
    st.close()
    un.close()


@pytest.mark.gpu
def test_prefix_decode_full_size_sampled():
    """128 children of a 2048-token shared prompt (Llama-3-8B layer shapes, block 64): sampled
    children against dense attention over their logical history plus the step's token, and the
    unshared pool giving the same bits."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_266_gb300 import build
    build.build()
    import paged_kv_cache_266_gb300 as pkv
    import pkv_workloads as W
    from paged_kv_cache_266_gb300.runner import PrefixDecode
    sc = W.make_prefix_script()
    st = PrefixDecode(sc, share=True)
    st.step()
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_error(st.pool.handle) == pkv.PKV_OK
    got = oracle.bf16_bits_to_f64(st.out_host())
    k_new, v_new, q = sc.step_inputs()
    for b in (0, 17, 64, 127):
        K, V = sc.logical_kv(b)
        K = oracle.bf16_bits_to_f64(np.concatenate([K, k_new[b:b + 1]]))
        V = oracle.bf16_bits_to_f64(np.concatenate([V, v_new[b:b + 1]]))
        qb = oracle.bf16_bits_to_f64(q[b])
        for h in range(sc.Hkv):
            ref = oracle.dense_attention(qb[h * sc.G:(h + 1) * sc.G], K[:, h], V[:, h], 1 / math.sqrt(sc.D))
            err = np.abs(got[b, h * sc.G:(h + 1) * sc.G] - ref)
            assert err.max() <= 1e-2 and err.mean() <= 1e-3, (b, h)
    un = PrefixDecode(sc, share=False)
    un.step()
    torch.cuda.synchronize()
    assert np.array_equal(un.out_host(), st.out_host())
    st.close()
    un.close()
