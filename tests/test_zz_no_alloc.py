"""The allocation-free decode attention entry point.

Some callers cannot hand the library a workspace: an engine that has already given almost
all free device memory to its own KV pool, or a decode loop that must not call cudaMalloc
because it can stall the device.  pkv_decode_attention_static serves them from a fixed scratch
array inside the library.  These tests call it through the C ABI, twice in a row (the scratch
keeps the previous call's contents), and require the same output bits as the workspace-taking
entry point (the same plan and kernel run on both) and the oracle's result within tolerance.
A call right after one whose bounded waits ran out (merge tickets left mid-count in the shared
scratch) must give the same bits again, and a call needing more scratch than the fixed size is
refused."""
import ctypes

import numpy as np
import pytest

import oracle
import oracle.drive as odrive
import pkv_workloads as W

pytestmark = pytest.mark.gpu

TOL_MAX, TOL_MEAN, TOL_FP8_MAX = 1e-2, 1e-3, 3e-2


@pytest.fixture(scope="module")
def pkv():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_266_gb300 import build
    build.build()
    import paged_kv_cache_266_gb300 as m
    m._L()
    return m


def _static_call(pkv, step, out):
    import torch
    lib = pkv._L()
    return lib.pkv_decode_attention_static(
        step.pool.handle, step.q.data_ptr(), step.tables.data_ptr(), step.tables.shape[1], step.lens.data_ptr(),
        step.q.shape[0], step.q.shape[1], ctypes.c_float(step.scale), out.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


def _bits(out):
    import torch
    return out.view(torch.int16).cpu().numpy().view(np.uint16)


def _workload(name):
    if name == "long":  # one sequence split over every CTA: hundreds of partial states merged
        return W.custom_workload(310, 1, 8, 1, 128, 64, [40000])
    return W.make_workload(name)


@pytest.mark.parametrize("name", ["c2", "c4", "long"])
def test_static_scratch_matches_the_workspace_entry_point(pkv, name):
    import torch
    from paged_kv_cache_266_gb300.runner import DecodeStep
    w = _workload(name)
    step = DecodeStep(w)
    step.step()  # append, then attention with the caller-provided workspace
    torch.cuda.synchronize()
    want = step.out_host().copy()
    need = pkv.pkv_decode_workspace_bytes(step.pool.handle, w.B, w.Hq, step.tables.shape[1])
    assert need <= pkv.PKV_STATIC_WORKSPACE_BYTES
    pool, _, tables = odrive.build(w)
    ref = odrive.attention(w, pool, tables)
    tol = TOL_FP8_MAX if w.kv_dtype == "fp8_e4m3" else TOL_MAX
    for _ in range(2):
        out = torch.full_like(step.out, float("nan"))
        assert _static_call(pkv, step, out) == pkv.PKV_OK
        torch.cuda.synchronize()
        assert pkv.pkv_check_device_error(step.pool.handle) == pkv.PKV_OK
        got = _bits(out)
        assert np.array_equal(got, want), "static scratch output differs from the workspace call's"
        err = np.abs(oracle.bf16_bits_to_f64(got) - ref)
        assert err.max() <= tol and err.mean() <= TOL_MEAN, (err.max(), err.mean())
    step.close()


def test_static_scratch_after_a_timed_out_call(pkv, stall_hooks):
    """The bounded-wait hooks make one static call give up (PKV_ERR_TIMEOUT, no fault) and leave
    the shared scratch's merge tickets wherever they were; the next static call clears them itself
    and gives the workspace call's bits."""
    import torch
    from paged_kv_cache_266_gb300.runner import DecodeStep
    w = _workload("long")
    step = DecodeStep(w)
    step.step()
    torch.cuda.synchronize()
    want = step.out_host().copy()
    stall_hooks[0]()
    out = torch.zeros_like(step.out)
    assert _static_call(pkv, step, out) == pkv.PKV_OK  # launched; the device reports the timeout
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_error(step.pool.handle) == pkv.PKV_ERR_TIMEOUT
    stall_hooks[1]()
    for _ in range(2):
        out = torch.full_like(step.out, float("nan"))
        assert _static_call(pkv, step, out) == pkv.PKV_OK
        torch.cuda.synchronize()
        assert pkv.pkv_check_device_error(step.pool.handle) == pkv.PKV_OK
        assert np.array_equal(_bits(out), want)
    step.close()


def test_static_scratch_refuses_calls_beyond_its_size(pkv):
    import torch
    Hkv, D = 32, 128
    handle = pkv.pkv_pool_create(64, 64, Hkv, D, pkv.PKV_KV_BF16)
    B, Hq, max_blocks = 4096, Hkv * 8, 4
    assert pkv.pkv_decode_workspace_bytes(handle, B, Hq, max_blocks) > pkv.PKV_STATIC_WORKSPACE_BYTES
    q = torch.zeros(B, Hq, D, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(q)
    tables = torch.zeros(B, max_blocks, dtype=torch.int32, device="cuda")
    lens = torch.zeros(B, dtype=torch.int32, device="cuda")
    lib = pkv._L()
    rc = lib.pkv_decode_attention_static(handle, q.data_ptr(), tables.data_ptr(), max_blocks, lens.data_ptr(), B, Hq,
                                         ctypes.c_float(1.0), out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == pkv.PKV_ERR_INVALID_ARG
    with pytest.raises(pkv.PKVError, match="fixed limit"):
        pkv.pkv_decode_attention_static(handle, q, tables, lens, 1.0, out)
    torch.cuda.synchronize()
    pkv.pkv_pool_destroy(handle)
