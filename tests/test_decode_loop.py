"""The in-flight batching decode loop: sequences finish and join every step, blocks grow on
demand, each step runs append + attention (CUDA-graph replayed per batch bucket).  Every step's
output is compared with the oracle's replay of the same schedule, and the pool bytes at the end
must match the oracle's bit for bit."""
import numpy as np
import pytest

import oracle
import oracle.drive as odrive
import pkv_workloads as W

TOL_MEAN = 1e-3


def test_loop_schedule_fits_its_pool_and_conserves_blocks():
    sc = W.make_loop_script(n_steps=40)
    a = oracle.Allocator(sc.num_blocks, sc.block_size)
    lens, running = {}, []
    for t, (finished, joined) in enumerate(sc.steps):
        for s in finished:
            assert a.release(s) == 0
            running.remove(s)
            del lens[s]
        for s, n in joined:
            assert a.reserve(s, n) == 0
            lens[s] = n
            running.append(s)
        for s in running:
            assert a.reserve(s, lens[s] + 1) == 0
            lens[s] += 1
        held = sum(a.num_pages(s) for s in running)
        assert held + a.num_free() == sc.num_blocks
        assert held == sum(-(-L // sc.block_size) for L in lens.values())
        assert len(running) == sc.max_batch
    assert sum(len(f) for f, _ in sc.steps) > 0  # the schedule churns


@pytest.mark.gpu
@pytest.mark.parametrize("kv_dtype,bs,graphs,device_inputs", [("bf16", 16, True, False), ("bf16", 64, False, False),
                                                              ("fp8_e4m3", 16, True, False), ("bf16", 16, True, True),
                                                              ("int8", 64, False, True)])
def test_decode_loop_matches_oracle_every_step(kv_dtype, bs, graphs, device_inputs):
    """device_inputs: each step's q / new K / new V are written on the device into the loop's
    input region (as a QKV projection would) instead of being staged from the host."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_266_gb300 import build
    build.build()
    import paged_kv_cache_266_gb300 as pkv
    from paged_kv_cache_266_gb300.engine import DecodeLoop
    sc = W.make_loop_script(index=41 if kv_dtype == "bf16" else 42, n_steps=24, block_size=bs, kv_dtype=kv_dtype)
    ref, pool = odrive.run_loop(sc)
    loop = DecodeLoop(sc, graphs=graphs)
    tol = 3e-2 if kv_dtype != "bf16" else 1e-2
    for t in range(len(sc.steps)):
        if device_inputs:
            k, v, q = sc.step_inputs(t, ref[t][0])
            _, qd, kd, vd = loop.device_input_region(len(ref[t][0]))
            for dst, src in ((qd, q), (kd, k), (vd, v)):
                dst.copy_(torch.from_numpy(src.view(np.int16)).view(torch.bfloat16))
        run, out = loop.step(device_inputs=device_inputs)
        assert run == ref[t][0]
        err = np.abs(oracle.bf16_bits_to_f64(out) - ref[t][1])
        assert err.max() <= tol and err.mean() <= TOL_MEAN, (t, err.max(), err.mean())
    assert pkv.pkv_check_device_error(loop.pool.handle) == pkv.PKV_OK
    kv, kv_bytes, sc_ptr, sc_bytes = pkv.pkv_pool_raw(loop.pool.handle)
    from paged_kv_cache_266_gb300.runner import _wrap_device
    assert np.array_equal(_wrap_device(kv, kv_bytes).cpu().numpy(), pool.data)
    if sc_bytes:
        assert np.array_equal(_wrap_device(sc_ptr, sc_bytes).cpu().numpy().view(np.float32), pool.scales)
    loop.close()


def _golden_schedules():
    """Cases of tests/golden/chunked_schedule.txt: (name, chunk, system, reuse, steps), steps a
    list of (finished, joined, expected chunks, expected decoders)."""
    import os
    cases = []
    ids = lambda f: [] if f == "-" else [int(x) for x in f.split(",")]
    for line in open(os.path.join(os.path.dirname(__file__), "golden", "chunked_schedule.txt")):
        f = line.split()
        if not f or f[0].startswith("#"):
            continue
        if f[0] == "case":
            cases.append((f[1], int(f[3]), int(f[5]), bool(int(f[7])), []))
        else:  # step t fin F join J => pre P dec D
            join = [] if f[5] == "-" else [tuple(int(y) for y in x.split(":")) for x in f[5].split(",")]
            pre = [] if f[8] == "-" else [(int(x.split(":")[0]),) + tuple(int(y) for y in x.split(":")[1].split("-"))
                                          for x in f[8].split(",")]
            cases[-1][4].append((ids(f[3]), join, pre, ids(f[10])))
    return cases


def test_oracle_chunk_plan_matches_the_hand_traced_schedules():
    """The oracle's chunked-context planner against schedules traced by hand from the page's
    scheduler (joins, finishes, a prompt shorter than one chunk, a forked system prompt)."""
    for name, chunk, system, reuse, steps in _golden_schedules():
        plan = odrive.ChunkedContextPlan(chunk, system, reuse)
        for t, (fin, join, pre, dec) in enumerate(steps):
            assert plan.step(fin, join) == (pre, dec), (name, t)


def _oracle_plans(sc):
    plan = odrive.ChunkedContextPlan(sc.chunk, sc.system, sc.reuse)
    return [plan.step(f, j) for f, j in sc.steps]


@pytest.mark.parametrize("index,chunk,system,reuse", [(46, 48, 0, True), (47, 7, 0, True), (48, 48, 70, True),
                                                      (49, 16, 70, False), (50, 1, 5, True)])
def test_engine_scheduler_matches_the_oracle_plan(index, chunk, system, reuse):
    """The engine's scheduler and the oracle's planner, written separately, plan every step of
    the hand-traced cases and of seeded churn scripts identically."""
    from paged_kv_cache_266_gb300.engine import ChunkedContextScheduler
    scripts = [(steps, c, sy, r) for _, c, sy, r, steps in _golden_schedules()]
    sc = W.make_chunked_loop_script(index=index, n_steps=40, chunk=chunk, system=system, reuse=reuse)
    scripts.append(([(f, j, None, None) for f, j in sc.steps], chunk, system, reuse))
    for steps, c, sy, r in scripts:
        eng = ChunkedContextScheduler(c, sy, r)
        ora = odrive.ChunkedContextPlan(c, sy, r)
        for fin, join, _, _ in steps:
            for s in fin:
                eng.finish(s)
            for s, m in join:
                eng.admit(s, m)
            got = eng.plan()
            want = ora.step(fin, join)
            assert got == want
            for s in got[1]:
                assert eng.cached(s) == ora.cached(s)
            eng.mark_decoded(got[1])
            ora.decoded(set(want[1]))


def test_chunk_plans_cover_every_prompt_once():
    """Invariants of the oracle's plan on seeded scripts: every prompt is prefilled in order, in
    pieces of at most `chunk` tokens covering it exactly once; a sequence decodes only after its
    last piece (from the next step on); only sequences whose prompt is done finish."""
    for index, chunk, system, reuse in [(46, 48, 0, True), (48, 48, 70, True), (49, 16, 70, False)]:
        sc = W.make_chunked_loop_script(index=index, n_steps=40, chunk=chunk, system=system, reuse=reuse)
        covered, need, decoding, just_done = {}, {}, set(), set()
        for (fin, join), (pre, dec) in zip(sc.steps, _oracle_plans(sc)):
            for s in fin:
                assert covered[s] == need[s], "a sequence finished while prefilling"
                decoding.discard(s)
                just_done.discard(s)
            assert just_done <= set(dec), "a prefilled sequence did not decode in the next step"
            for s, m in join:
                need[s] = system + m
                covered[s] = system if (system and reuse) else 0
            for s, p0, p1 in pre:
                assert p0 == covered[s] and 0 < p1 - p0 <= chunk and p1 <= need[s]
                covered[s] = p1
            assert not set(dec) & {s for s, _, _ in pre}
            for s in dec:
                assert covered[s] == need[s]
            just_done = {s for s, _, p1 in pre if p1 == need[s]}
            decoding |= set(dec)
        assert decoding, "the script never decodes"


@pytest.mark.gpu
@pytest.mark.parametrize("bs,graphs,kv_dtype", [(16, True, "bf16"), (64, False, "bf16"), (16, True, "fp8_e4m3"),
                                                (64, False, "int8")])
def test_chunked_context_loop_matches_oracle_every_step(bs, graphs, kv_dtype):
    """Chunked context in the in-flight loop, on bf16 pools and on FP8 / INT8 pools (the chunks'
    K/V quantised by the append, the prefill widening the codes on chip): every step's
    prefill-chunk outputs and decode outputs against the oracle's replay, and the final pool bytes
    bit-exact."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_266_gb300 import build
    build.build()
    import paged_kv_cache_266_gb300 as pkv
    from paged_kv_cache_266_gb300.engine import DecodeLoop
    sc = W.make_chunked_loop_script(index=47, n_steps=20, block_size=bs, chunk=48, kv_dtype=kv_dtype)
    ref, pool = odrive.run_chunked_loop(sc)
    loop = DecodeLoop(sc, graphs=graphs)
    tol = 3e-2 if kv_dtype != "bf16" else 1e-2  # the decode bound of each pool type
    for t in range(len(sc.steps)):
        run, out = loop.step()
        assert run == ref[t][0]
        if run:
            err = np.abs(oracle.bf16_bits_to_f64(out) - ref[t][1])
            assert err.max() <= tol and err.mean() <= TOL_MEAN, ("decode", t, err.max(), err.mean())
        chunks, pre = loop.last_prefill
        assert chunks == ref[t][2]
        if chunks:
            got = oracle.bf16_bits_to_f64(pre.view(torch.int16).cpu().numpy().view(np.uint16))
            err = np.abs(got - ref[t][3])
            assert err.max() <= 1e-2 and err.mean() <= TOL_MEAN, ("prefill", t, err.max(), err.mean())
    assert pkv.pkv_check_device_error(loop.pool.handle) == pkv.PKV_OK
    kv, kv_bytes, sc_ptr, sc_bytes = pkv.pkv_pool_raw(loop.pool.handle)
    from paged_kv_cache_266_gb300.runner import _wrap_device
    assert np.array_equal(_wrap_device(kv, kv_bytes).cpu().numpy(), pool.data)
    if kv_dtype != "bf16":
        assert np.array_equal(_wrap_device(sc_ptr, sc_bytes).cpu().numpy().view(np.float32), pool.scales)
    loop.close()


@pytest.mark.gpu
@pytest.mark.parametrize("reuse", [True, False])
def test_chunked_loop_with_cached_system_prompt_matches_oracle(reuse):
    """Prefix caching in the loop: every prompt starts with a shared 70-token system prompt
    (a partial last block) cached once; joiners fork it and prefill only their own tokens. Every
    step's outputs against the oracle's replay (which forks the same way), final pool bit-exact,
    and the system prompt's whole blocks are held by every running request."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_266_gb300 import build
    build.build()
    import paged_kv_cache_266_gb300 as pkv
    from paged_kv_cache_266_gb300.engine import DecodeLoop
    sc = W.make_chunked_loop_script(index=48, n_steps=16, block_size=16, chunk=48, system=70, reuse=reuse)
    ref, pool = odrive.run_chunked_loop(sc)
    loop = DecodeLoop(sc, graphs=True, system_seq=W.SYSTEM_SEQ)
    for t in range(len(sc.steps)):
        run, out = loop.step()
        assert run == ref[t][0]
        if run:
            err = np.abs(oracle.bf16_bits_to_f64(out) - ref[t][1])
            assert err.max() <= 1e-2 and err.mean() <= TOL_MEAN, ("decode", t, err.max(), err.mean())
        chunks, pre = loop.last_prefill
        assert chunks == ref[t][2]
        if chunks:
            got = oracle.bf16_bits_to_f64(pre.view(torch.int16).cpu().numpy().view(np.uint16))
            err = np.abs(got - ref[t][3])
            assert err.max() <= 1e-2 and err.mean() <= TOL_MEAN, ("prefill", t, err.max(), err.mean())
    assert pkv.pkv_check_device_error(loop.pool.handle) == pkv.PKV_OK
    kv, kv_bytes, _, _ = pkv.pkv_pool_raw(loop.pool.handle)
    from paged_kv_cache_266_gb300.runner import _wrap_device
    assert np.array_equal(_wrap_device(kv, kv_bytes).cpu().numpy(), pool.data)
    first = int(pkv.pkv_get_block_tables(loop.alloc, [W.SYSTEM_SEQ], 5)[0, 0])
    assert pkv.pkv_block_refcount(loop.alloc, first) == (1 + len(loop.scheduler) if reuse else 1)
    loop.close()
