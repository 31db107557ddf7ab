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
