"""The allocation-free decode attention entry point.

Some callers cannot hand the library a workspace: an engine that has already given almost
all free device memory to its own KV pool, or a decode loop that must not call cudaMalloc
because it can stall the device.  pkv_decode_attention_static serves them from a fixed scratch
array inside the library.  These tests call it through the C ABI and check it against the
workspace-taking entry point, twice in a row (the scratch keeps the previous call's contents),
and check that a call needing more scratch than the fixed size is refused."""
import ctypes

import numpy as np
import pytest

import oracle
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


@pytest.mark.parametrize("name", ["c2", "c4", "long"])
def test_static_scratch_matches_the_workspace_entry_point(pkv, name):
    import torch
    from paged_kv_cache_266_gb300.runner import DecodeStep
    w = W.custom_workload(310, 1, 8, 1, 128, 64, [40000]) if name == "long" else W.make_workload(name)
    step = DecodeStep(w)
    step.step()  # append, then attention with the caller-provided workspace
    torch.cuda.synchronize()
    ref = oracle.bf16_bits_to_f64(step.out_host())
    need = pkv.pkv_decode_workspace_bytes(step.pool.handle, w.B, w.Hq, step.tables.shape[1])
    assert need <= pkv.PKV_STATIC_WORKSPACE_BYTES
    tol = TOL_FP8_MAX if w.kv_dtype == "fp8_e4m3" else TOL_MAX
    for _ in range(2):
        out = torch.full_like(step.out, float("nan"))
        assert _static_call(pkv, step, out) == pkv.PKV_OK
        torch.cuda.synchronize()
        assert pkv.pkv_check_device_error(step.pool.handle) == pkv.PKV_OK
        got = oracle.bf16_bits_to_f64(out.view(torch.int16).cpu().numpy().view(np.uint16))
        err = np.abs(got - ref)
        assert np.isfinite(got).all()
        assert err.max() <= tol and err.mean() <= TOL_MEAN, (err.max(), err.mean())
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
