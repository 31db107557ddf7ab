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
@pytest.mark.parametrize("kv_dtype,bs,graphs", [("bf16", 16, True), ("bf16", 64, False), ("fp8_e4m3", 16, True)])
def test_decode_loop_matches_oracle_every_step(kv_dtype, bs, graphs):
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
    tol = 3e-2 if kv_dtype == "fp8_e4m3" else 1e-2
    for t in range(len(sc.steps)):
        run, out = loop.step()
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


def test_chunked_loop_schedule_matches_its_generator():
    """The per-step plan (prefill chunks, decoders) replays the generator's state: every prompt
    is prefilled in chunks of at most `chunk` tokens covering it exactly once, a sequence decodes
    only after its prompt, and only decoding sequences finish."""
    sc = W.make_chunked_loop_script(index=46, n_steps=40, chunk=48)
    state, covered = {}, {}
    for t in range(len(sc.steps)):
        finished, joined = sc.steps[t]
        for s in finished:
            assert state[s][1] == state[s][0], "a sequence finished while prefilling"
        prefill, decode = sc.plan_step(t, state)
        for s, p0, p1 in prefill:
            assert p0 == covered.get(s, 0) and 0 < p1 - p0 <= sc.chunk and p1 <= state[s][0]
            covered[s] = p1
            state[s][1] = p1
        for s in decode:
            assert state[s][1] == state[s][0] and s not in [c[0] for c in prefill]
            state[s][2] += 1
        assert len(state) <= sc.max_batch


@pytest.mark.gpu
@pytest.mark.parametrize("bs,graphs", [(16, True), (64, False)])
def test_chunked_context_loop_matches_oracle_every_step(bs, graphs):
    """Chunked context in the in-flight loop: every step's prefill-chunk outputs and decode
    outputs against the oracle's replay, and the final pool bytes bit-exact."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_266_gb300 import build
    build.build()
    import paged_kv_cache_266_gb300 as pkv
    from paged_kv_cache_266_gb300.engine import DecodeLoop
    sc = W.make_chunked_loop_script(index=47, n_steps=20, block_size=bs, chunk=48)
    ref, pool = odrive.run_chunked_loop(sc)
    loop = DecodeLoop(sc, graphs=graphs)
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
    loop = DecodeLoop(sc, graphs=True)
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
    assert pkv.pkv_block_refcount(loop.alloc, first) == (1 + len(loop.state) if reuse else 1)
    loop.close()
