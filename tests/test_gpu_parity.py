"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle on the same seeded
inputs.  Block tables, slot mappings and appended pool bytes (and fp8 scales) must be
bit-exact; bf16 attention outputs within max |err| 1e-2 and mean |err| 1e-3 of the oracle,
fp8- and int8-KV outputs within 3e-2 (computed by the oracle from the same code bytes and
scales)."""
import math
import os

import numpy as np
import pytest

import oracle
import oracle.drive as odrive
import pkv_workloads as W
from boundary_rows import near_boundary_rows

pytestmark = pytest.mark.gpu

TOL_BF16_MAX, TOL_MEAN, TOL_FP8_MAX = 1e-2, 1e-3, 3e-2


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


def _run(pkv, w):
    import torch
    from paged_kv_cache_266_gb300.runner import DecodeStep
    step = DecodeStep(w)
    step.step()
    torch.cuda.synchronize()
    return step


def _errors(step, ref):
    got = oracle.bf16_bits_to_f64(step.out_host())
    err = np.abs(got - ref)
    return got, err


def _check_against_oracle(pkv, w, step, check_pool=True):
    assert pkv.pkv_check_device_error(step.pool.handle) == pkv.PKV_OK
    pool, alloc, tables = odrive.build(w)
    assert np.array_equal(step.tables_host, tables), "block tables differ from the oracle allocator"
    if w.append:
        assert np.array_equal(step.slots_new_host, alloc.slot_mapping(w.seq_ids, w.lens))
    if check_pool:
        kv, sc = step.pool_bytes_host()
        assert np.array_equal(kv, pool.data), "appended pool bytes differ from the oracle"
        if w.kv_dtype != "bf16":
            assert np.array_equal(sc, pool.scales), "block scales differ from the oracle"
    ref = odrive.attention(w, pool, tables)
    got, err = _errors(step, ref)
    tol = TOL_FP8_MAX if w.kv_dtype != "bf16" else TOL_BF16_MAX
    assert np.isfinite(got).all()
    assert err.max() <= tol, f"max |err| {err.max():.3e}"
    assert err.mean() <= TOL_MEAN, f"mean |err| {err.mean():.3e}"
    return got, ref


@pytest.mark.parametrize("name", W.WORKLOADS)
def test_workload_parity(pkv, name):
    """The five workloads at full size, every output compared."""
    w = W.make_workload(name)
    step = _run(pkv, w)
    _check_against_oracle(pkv, w, step)
    step.close()


def test_int8_churned_pool_parity(pkv):
    """The churned 200-request workload with an INT8 pool instead of fp8 (same shapes, blocks
    and inputs): pool codes and scales bit-exact, every output within the low-precision bound."""
    import dataclasses
    w = dataclasses.replace(W.make_workload("c4"), kv_dtype="int8")
    step = _run(pkv, w)
    _check_against_oracle(pkv, w, step)
    step.close()


@pytest.mark.parametrize("dtype", ["bf16", "fp8_e4m3", "int8"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bs", [16, 32, 64, 128])
def test_shapes(pkv, dtype, D, bs):
    """Head dims, block sizes, GQA ratios and ragged tails (lengths that end mid-tile)."""
    rng = np.random.default_rng(bs * 7 + D)
    for G, Hkv in ((1, 3), (3, 2), (8, 1)):
        lens = rng.integers(1, 700, size=5)
        lens[0] = 1
        w = W.custom_workload(200 + bs + D + G, 5, G * Hkv, Hkv, D, bs, lens, append=True, kv_dtype=dtype)
        step = _run(pkv, w)
        _check_against_oracle(pkv, w, step)
        step.close()


@pytest.mark.parametrize("name", ["c0", "c2", "c4", "c4-int8"])
def test_fused_step_equals_separate_calls(pkv, name):
    """pkv_decode_step gives the same pool bytes and outputs, bit for bit, as pkv_append followed
    by pkv_decode_attention: on bf16 pools the append kernel with the attention as a programmatic
    dependent launch, on one-byte pools (c4) the attention kernel quantising the tokens itself.
    Three steps in a row: the step's workspace words (tickets and the append's counters) are back
    at zero after each."""
    import dataclasses
    import torch
    from paged_kv_cache_266_gb300.runner import DecodeStep
    w = W.make_workload(name.split("-")[0])
    if name.endswith("int8"):
        w = dataclasses.replace(w, kv_dtype="int8")
    a, b = DecodeStep(w), DecodeStep(w)
    # merge tickets [B * Hkv], then from the next multiple of 32 ints the append's 32 counters
    # (32 ints apart) and its CTA count
    words = -(-w.B * w.Hkv // 32) * 32 + 32 * 32 + 1
    for _ in range(3):
        a.step(fused=True)
        torch.cuda.synchronize()
        assert not a.workspace[: words * 4].any(), "workspace words must return to zero"
    b.step(fused=False)
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_error(a.pool.handle) == pkv.PKV_OK
    assert np.array_equal(a.out_host(), b.out_host())
    ka, sa = a.pool_bytes_host()
    kb, sb = b.pool_bytes_host()
    assert np.array_equal(ka, kb) and np.array_equal(sa, sb)
    a.close()
    b.close()


@pytest.mark.parametrize("graph", [True, False])
@pytest.mark.parametrize("name", ["c0", "c3", "c4"])
def test_host_to_host_step_equals_device_step(pkv, name, graph):
    """The end-to-end step (allocator tables and slots into a pinned staging buffer, one copy to
    the device, fused step, output copied back) gives the device-resident step's output."""
    import torch
    from paged_kv_cache_266_gb300.runner import DecodeStep
    w = W.make_workload(name)
    step = DecodeStep(w)
    step.step()
    torch.cuda.synchronize()
    want = step.out_host().copy()
    if name == "c3":
        step.limit_batch(2)  # two of the long contexts keep the test short
        step.step()
        torch.cuda.synchronize()
        want = step.out_host().copy()
    for _ in range(3):
        step._host and step._host["out"].zero_()
        h2d, d2h = step.step_host(graph=graph)
        assert h2d > 0 and d2h == want.size * 2
        got = step._host["out"].numpy().view(np.uint16)
        assert np.array_equal(got, want)
    step.close()


def test_empty_and_single_token_contexts(pkv):
    w = W.custom_workload(300, 6, 8, 2, 128, 64, [0, 1, 0, 17, 64, 65], append=False)
    step = _run(pkv, w)
    got, ref = _check_against_oracle(pkv, w, step)
    out = step.out_host()
    assert not out[0].any() and not out[2].any(), "empty contexts must give zeros"
    # one cached token: the softmax weight is exactly 1, the output is that token's V row
    t = int(w.hist_offsets[1])  # sequence 1's only token in the concatenated history
    v = w.history_v(t, t + 1)[0]  # [Hkv][D]
    assert np.array_equal(out[1].reshape(2, 4, 128), np.repeat(v[:, None, :], 4, axis=1))
    step.close()


def test_stage_copy_moves_exact_bytes_and_refuses_pageable_memory(pkv):
    """Host-to-device, device-to-host and device-to-device copies of ragged sizes (multiples of
    16 bytes, from one vector to several grid-strides) return the bytes unchanged and touch
    nothing past the copied range; pageable host memory is refused without a launch."""
    import ctypes
    import torch
    rng = np.random.default_rng(11)
    for n in (16, 48, 4096, 4096 * 16 + 32, 3 * 2 ** 20 + 16 * 7):
        src = torch.from_numpy(rng.integers(0, 256, n + 64, dtype=np.uint8)).pin_memory()
        dev = torch.full((n + 64,), 0xA5, dtype=torch.uint8, device="cuda")
        back = torch.zeros(n + 64, dtype=torch.uint8).pin_memory()
        dev2 = torch.full((n + 64,), 0x5A, dtype=torch.uint8, device="cuda")
        pkv.pkv_stage_copy(dev, src, n)
        pkv.pkv_stage_copy(dev2, dev, n)
        pkv.pkv_stage_copy(back, dev2, n)
        torch.cuda.synchronize()
        assert torch.equal(back[:n], src[:n])
        assert not back[n:].any()
        assert (dev[n:].cpu() == 0xA5).all() and (dev2[n:].cpu() == 0x5A).all()
    pageable = np.zeros(1024, np.uint8)
    dev = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    L = pkv._L()
    stream = torch.cuda.current_stream().cuda_stream
    assert L.pkv_stage_copy(dev.data_ptr(), pageable.ctypes.data, 1024, stream) == pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_stage_copy(pageable.ctypes.data, dev.data_ptr(), 1024, stream) == pkv.PKV_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        pkv.pkv_stage_copy(dev, torch.zeros(1024, dtype=torch.uint8))  # not pinned


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_empty_batches_are_no_ops(pkv, kv):
    """Calls over zero tokens or zero sequences (an in-flight step where nothing joins, nothing
    decodes or nothing prefills) return OK and change neither the pool nor the outputs."""
    import torch
    from paged_kv_cache_266_gb300.runner import _wrap_device
    dev = torch.device("cuda")
    pool = pkv.KVPool(8, 16, 2, 128, pkv.KV_DTYPES[kv])
    g = torch.Generator().manual_seed(7)
    k = torch.randn(20, 2, 128, generator=g).to(torch.bfloat16).to(dev)
    v = torch.randn(20, 2, 128, generator=g).to(torch.bfloat16).to(dev)
    pkv.pkv_append(pool.handle, k, v, torch.arange(20, dtype=torch.int64, device=dev))

    def snapshot():
        torch.cuda.synchronize()
        kv_ptr, kv_bytes, sc_ptr, sc_bytes = pkv.pkv_pool_raw(pool.handle)
        return (_wrap_device(kv_ptr, kv_bytes).cpu().numpy().copy(),
                _wrap_device(sc_ptr, sc_bytes).cpu().numpy().copy() if sc_bytes else None)

    before = snapshot()
    e_kv = torch.empty(0, 2, 128, dtype=torch.bfloat16, device=dev)
    e_slot = torch.empty(0, dtype=torch.int64, device=dev)
    e_q = torch.empty(0, 8, 128, dtype=torch.bfloat16, device=dev)
    e_tab = torch.empty(0, 4, dtype=torch.int32, device=dev)
    e_len = torch.empty(0, dtype=torch.int32, device=dev)
    ws = torch.zeros(pkv.pkv_decode_workspace_bytes(pool.handle, 1, 8, 4), dtype=torch.uint8, device=dev)
    pkv.pkv_append(pool.handle, e_kv, e_kv, e_slot)
    pkv.pkv_append_rope(pool.handle, e_kv, e_kv, e_slot, e_slot, 10000.0, q=e_q)
    pkv.pkv_decode_attention(pool.handle, e_q, e_tab, e_len, 0.125, e_q, ws)
    pkv.pkv_decode_step(pool.handle, e_kv, e_kv, e_slot, e_q, e_tab, e_len, 0.125, e_q, ws)
    pkv.pkv_decode_step_rope(pool.handle, e_kv, e_kv, e_slot, e_slot, 10000.0, e_q, e_tab, e_len, 0.125, e_q, ws)
    pkv.pkv_decode_attention_static(pool.handle, e_q, e_tab, e_len, 0.125, e_q)
    if kv == "bf16":  # prefill: zero sequences, and sequences whose chunks are all empty
        cu = torch.zeros(1, dtype=torch.int32, device=dev)
        pkv.pkv_prefill_step(pool.handle, e_kv, e_kv, e_slot, e_q, cu, 0, e_tab, e_len, 0.125, e_q)
        tab = torch.tensor([[0, 1]], dtype=torch.int32, device=dev)
        ctx = torch.tensor([20], dtype=torch.int32, device=dev)
        pkv.pkv_prefill_attention(pool.handle, e_q, torch.zeros(2, dtype=torch.int32, device=dev), 0, tab, ctx,
                                  0.125, e_q)
    # a decode step over one sequence with no new token: attention only, the pool unchanged
    q = torch.randn(1, 8, 128, generator=g).to(torch.bfloat16).to(dev)
    out = torch.zeros(1, 8, 128, dtype=torch.bfloat16, device=dev)
    tab = torch.tensor([[0, 1, 0, 0]], dtype=torch.int32, device=dev)
    ctx = torch.tensor([20], dtype=torch.int32, device=dev)
    pkv.pkv_decode_step(pool.handle, e_kv, e_kv, e_slot, q, tab, ctx, 0.125, out, ws)
    after = snapshot()
    assert pkv.pkv_check_device_error(pool.handle) == pkv.PKV_OK
    assert np.array_equal(before[0], after[0])
    assert (before[1] is None) or np.array_equal(before[1], after[1])
    assert out.abs().sum().item() > 0
    pool.close()


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_maximum_batch_and_group(pkv, kv):
    """The largest batch one call takes (4096 sequences) with the largest query-head group (8
    per KV head): ragged short contexts, every output against the oracle.  One sequence more, or
    a larger group, is refused before any launch."""
    import torch
    rng = np.random.default_rng(4096)
    lens = rng.integers(0, 40, 4096)
    lens[::97] = 0
    w = W.custom_workload(310, 4096, 16, 2, 128, 16, lens, append=True, kv_dtype=kv)
    step = _run(pkv, w)
    _check_against_oracle(pkv, w, step)
    L = pkv._L()
    s = torch.cuda.current_stream().cuda_stream
    args = (step.q.data_ptr(), step.tables.data_ptr(), step.max_blocks, step.lens.data_ptr())
    tail = (1.0 / math.sqrt(w.D), step.out.data_ptr(), step.workspace.data_ptr(), step.ws_bytes, s)
    assert L.pkv_decode_attention(step.pool.handle, *args, 4097, 16, *tail) == pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_decode_attention(step.pool.handle, *args, 4096, 32, *tail) == pkv.PKV_ERR_INVALID_ARG
    step.close()


def test_long_context_split_over_every_cta(pkv):
    """One sequence of 40000 tokens: its 625 groups are spread over all CTAs, so the final
    output comes from the last-arriving CTA's merge of hundreds of partial states."""
    w = W.custom_workload(301, 1, 8, 1, 128, 64, [40000], append=True)
    step = _run(pkv, w)
    _check_against_oracle(pkv, w, step)
    step.close()


def test_results_are_deterministic_and_workspace_is_reusable(pkv):
    import torch
    w = W.make_workload("c2")
    step = _run(pkv, w)
    first = step.out_host().copy()
    for _ in range(3):
        step.attention()
    torch.cuda.synchronize()
    assert np.array_equal(step.out_host(), first)
    assert not step.workspace[: w.B * w.Hkv * 4].any(), "merge tickets must return to zero"
    step.close()



def test_out_of_range_block_id_is_flagged_not_faulted(pkv):
    import torch
    w = W.custom_workload(302, 3, 4, 2, 128, 16, [40, 40, 40], append=False)
    step = _run(pkv, w)
    good = step.out_host().copy()
    bad = step.tables_host.copy()
    bad[1, 1] = w.num_blocks + 7
    step.tables.copy_(torch.from_numpy(bad))
    step.attention()
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_error(step.pool.handle) == pkv.PKV_ERR_BOUNDS
    out = step.out_host()
    assert np.array_equal(out[0], good[0]) and np.array_equal(out[2], good[2])
    step.close()


def test_bounded_waits_report_timeout_and_leave_the_context_usable(pkv, stall_hooks):
    """Every mbarrier wait in the attention kernel is bounded.  With the test hooks the stages
    expect bytes no copy delivers and the waits give up after 20 ms: the call reports
    PKV_ERR_TIMEOUT, no fault, and the next normal call gives the same results as before."""
    import torch
    w = W.custom_workload(306, 3, 8, 2, 128, 64, [300, 70, 900], append=False)
    step = _run(pkv, w)
    good = step.out_host().copy()
    stall_hooks[0]()
    step.attention()
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_error(step.pool.handle) == pkv.PKV_ERR_TIMEOUT
    stall_hooks[1]()
    pkv.pkv_decode_workspace_init(step.workspace)  # merge tickets may have been left mid-count
    step.attention()
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_error(step.pool.handle) == pkv.PKV_OK
    assert np.array_equal(step.out_host(), good)
    step.close()


@pytest.mark.parametrize("kv_dtype", ["fp8_e4m3", "int8"])
def test_step_append_wait_is_bounded(pkv, monkeypatch, kv_dtype):
    """On a one-byte pool pkv_decode_step quantises its new tokens inside the attention kernel,
    whose producers wait until every row is in.  With the test hook that wait expects one row
    pair more than the kernel writes and gives up after 20 ms: the call reports PKV_ERR_TIMEOUT,
    no fault, and once the workspace is initialised again the next step stores the oracle's
    codes and scales and gives its outputs (the append is idempotent: same rows, same slots)."""
    import torch
    from paged_kv_cache_266_gb300.runner import DecodeStep
    w = W.custom_workload(307, 3, 8, 2, 128, 16, [300, 70, 900], append=True, kv_dtype=kv_dtype)
    step = DecodeStep(w)
    monkeypatch.setenv("PKV_TEST_STALL_APPENDS", "1")
    monkeypatch.setenv("PKV_TEST_WAIT_LIMIT_MS", "20")
    pkv.pkv_debug_reload_env()
    try:
        step.step()
        torch.cuda.synchronize()
        assert pkv.pkv_check_device_error(step.pool.handle) == pkv.PKV_ERR_TIMEOUT
    finally:
        monkeypatch.delenv("PKV_TEST_STALL_APPENDS", raising=False)
        monkeypatch.delenv("PKV_TEST_WAIT_LIMIT_MS", raising=False)
        pkv.pkv_debug_reload_env()
    pkv.pkv_decode_workspace_init(step.workspace)  # the wait's counters may have been left mid-count
    step.step()
    torch.cuda.synchronize()
    _check_against_oracle(pkv, w, step)
    step.close()


@pytest.mark.parametrize("kv_dtype", ["fp8_e4m3", "int8"])
def test_step_in_kernel_append_with_block_mates(pkv, kv_dtype):
    """pkv_decode_step on a one-byte pool appends inside the attention kernel, each row pair
    finding the call's other tokens in its block.  A call whose 40-odd tokens share six blocks in
    shuffled order (runs from offset 0, which open their block and derive its scale from all of
    the call's rows there, and runs from later offsets, which keep the stored scale), with a
    padding slot, into blocks the attention reads: the pool bytes, scales and outputs equal,
    bit for bit, those of pkv_append followed by pkv_decode_attention."""
    import torch
    from paged_kv_cache_266_gb300 import pkv_append, pkv_decode_attention, pkv_decode_step
    from paged_kv_cache_266_gb300.runner import DecodeStep
    w = W.custom_workload(308, 4, 8, 2, 128, 16, [200, 37, 500, 64], append=True, kv_dtype=kv_dtype)
    a, b = DecodeStep(w), DecodeStep(w)
    rng = np.random.default_rng(5 if kv_dtype == "int8" else 6)
    used = np.unique(a.tables_host[a.tables_host >= 0])
    blocks = rng.choice(used, size=6, replace=False)
    slots = []
    for j, blk in enumerate(blocks):
        start = 0 if j % 2 == 0 else int(rng.integers(1, 8))
        slots += [int(blk) * 16 + start + u for u in range(int(rng.integers(3, 9)))]
    slots.append(-1)
    slots = np.array(slots, dtype=np.int64)
    rng.shuffle(slots)
    N = len(slots)
    gen = torch.Generator().manual_seed(7)
    k = (torch.randn(N, w.Hkv, w.D, generator=gen) * 3).to(torch.bfloat16).cuda()
    v = (torch.randn(N, w.Hkv, w.D, generator=gen) * 3).to(torch.bfloat16).cuda()
    sd = torch.from_numpy(slots).cuda()
    pkv_decode_step(a.pool.handle, k, v, sd, a.q, a.tables, a.lens, a.scale, a.out, a.workspace)
    pkv_append(b.pool.handle, k, v, sd)
    pkv_decode_attention(b.pool.handle, b.q, b.tables, b.lens, b.scale, b.out, b.workspace)
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_error(a.pool.handle) == pkv.PKV_OK
    assert pkv.pkv_check_device_error(b.pool.handle) == pkv.PKV_OK
    ka, sa = a.pool_bytes_host()
    kb, sb = b.pool_bytes_host()
    assert np.array_equal(sa, sb), "block scales differ"
    assert np.array_equal(ka, kb), "pool bytes differ"
    assert np.array_equal(a.out_host(), b.out_host())
    a.close()
    b.close()


def test_context_longer_than_table_is_clamped_and_flagged(pkv):
    import torch
    w = W.custom_workload(303, 2, 4, 1, 64, 16, [30, 20], append=False)
    step = _run(pkv, w)
    good = step.out_host().copy()
    step.lens.copy_(torch.tensor([30, 10_000], dtype=torch.int32))
    step.attention()
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_error(step.pool.handle) == pkv.PKV_ERR_BOUNDS
    assert np.array_equal(step.out_host()[0], good[0])
    step.close()


def test_append_slot_out_of_range_is_skipped_and_flagged(pkv):
    import torch
    w = W.custom_workload(304, 2, 2, 2, 64, 16, [3, 3], append=True)
    step = _run(pkv, w)
    kv_before, _ = step.pool_bytes_host()
    step.slots_new.copy_(torch.tensor([w.num_blocks * 16 + 1, -1], dtype=torch.int64))
    step.append()
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_error(step.pool.handle) == pkv.PKV_ERR_BOUNDS
    kv_after, _ = step.pool_bytes_host()
    assert np.array_equal(kv_before, kv_after)
    step.close()


def test_fp8_decode_every_code(pkv):
    """Raw E4M3 codes written into V with unit scales: with one cached token the output is the
    decoded V row, which bf16 holds exactly — compared against the oracle's decode table."""
    import torch
    from paged_kv_cache_266_gb300.runner import _wrap_device
    w = W.custom_workload(305, 2, 1, 1, 128, 16, [1, 1], append=False, kv_dtype="fp8_e4m3")
    step = _run(pkv, w)
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    codes = np.concatenate([codes, codes[:2]])  # 256 bytes = two V rows of 128
    pool = oracle.Pool(w.num_blocks, 16, 1, 128, True)
    kv_ptr, kv_bytes, sc_ptr, sc_bytes = pkv.pkv_pool_raw(step.pool.handle)
    dev = _wrap_device(kv_ptr, kv_bytes)
    scd = _wrap_device(sc_ptr, sc_bytes)
    for b in range(2):
        blk = int(step.tables_host[b, 0])
        for d in range(128):
            dev[pool.elem_byte(blk, 1, 0, 0, d)] = int(codes[b * 128 + d])
        sc = torch.tensor([1.0, 1.0, 0.0, 0.0], dtype=torch.float32).view(torch.uint8)
        scd[blk * 16: blk * 16 + 16].copy_(sc)
    step.attention()
    torch.cuda.synchronize()
    got = oracle.bf16_bits_to_f64(step.out_host()).reshape(256)
    want = np.array([oracle.e4m3_decode(int(c)) for c in codes])
    assert np.array_equal(got, want)
    step.close()


def test_fp8_encode_matches_oracle_on_ties_and_subnormals(pkv):
    """Rows whose amax is 448 get scale 1, so stored codes are e4m3(x) directly: a sweep over
    grid midpoints (ties), subnormals, saturation and random values must match bit for bit."""
    import torch
    from paged_kv_cache_266_gb300 import pkv_append
    vals = np.array([oracle.e4m3_decode(c) for c in range(0x7F)])
    mids = (vals[:-1] + vals[1:]) / 2
    rng = np.random.default_rng(3)
    pool_vals = np.concatenate([mids, -mids, vals, rng.standard_normal(500) * 30, [447.9, -447.9, 1e-9, -0.0]])
    bf = torch.tensor(pool_vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    D = 128
    n_tok = -(-len(bf) // (D - 1))
    rows = np.zeros((n_tok, 1, D), dtype=np.uint16)
    flat = np.zeros(n_tok * (D - 1), dtype=np.uint16)
    flat[: len(bf)] = bf
    rows[:, 0, 1:] = flat.reshape(n_tok, D - 1)
    rows[:, 0, 0] = torch.tensor([448.0]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)[0]
    nb = n_tok
    handle = pkv.pkv_pool_create(nb, 16, 1, D, pkv.PKV_KV_FP8_E4M3)
    slots = np.arange(nb, dtype=np.int64) * 16  # each token opens its own block
    dk = torch.from_numpy(rows.view(np.int16)).view(torch.bfloat16).cuda()
    pkv_append(handle, dk, dk, torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_error(handle) == pkv.PKV_OK
    from paged_kv_cache_266_gb300.runner import _wrap_device
    kv_ptr, kv_bytes, sc_ptr, sc_bytes = pkv.pkv_pool_raw(handle)
    kv = _wrap_device(kv_ptr, kv_bytes).cpu().numpy()
    sc = _wrap_device(sc_ptr, sc_bytes).cpu().numpy().view(np.float32)
    ref = oracle.Pool(nb, 16, 1, D, True)
    assert ref.append(rows, rows, slots) == 0
    assert np.array_equal(sc, ref.scales)
    assert np.array_equal(kv, ref.data)
    pkv.pkv_pool_destroy(handle)


@pytest.mark.parametrize("dtype", ["fp8_e4m3", "int8"])
def test_one_byte_encode_at_rounding_boundaries(pkv, dtype):
    """Quantisation where x / s falls on or within a few fp32 steps of a code's rounding boundary,
    at power-of-two and other scales: the stored codes and scales match the oracle bit for bit,
    through the one-pass append (700 tokens) and the three-pass one (1100 tokens)."""
    import torch
    from paged_kv_cache_266_gb300 import pkv_append
    from paged_kv_cache_266_gb300.runner import _wrap_device
    D, n1, n2 = 128, 700, 1100
    rows = near_boundary_rows(dtype == "int8", n1 + n2, D, seed=11 if dtype == "int8" else 12)
    nb = n1 + n2
    handle = pkv.pkv_pool_create(nb, 16, 1, D, pkv.KV_DTYPES[dtype])
    ref = oracle.Pool(nb, 16, 1, D, odrive.KV_CODE[dtype])
    slots = np.arange(nb, dtype=np.int64) * 16  # each token opens its own block
    for a, b in ((0, n1), (n1, nb)):
        dk = torch.from_numpy(rows[a:b].view(np.int16)).view(torch.bfloat16).cuda()
        pkv_append(handle, dk, dk, torch.from_numpy(slots[a:b]).cuda())
        assert ref.append(rows[a:b], rows[a:b], slots[a:b]) == 0
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_error(handle) == pkv.PKV_OK
    kv_ptr, kv_bytes, sc_ptr, sc_bytes = pkv.pkv_pool_raw(handle)
    assert np.array_equal(_wrap_device(sc_ptr, sc_bytes).cpu().numpy().view(np.float32), ref.scales)
    assert np.array_equal(_wrap_device(kv_ptr, kv_bytes).cpu().numpy(), ref.data)
    pkv.pkv_pool_destroy(handle)


def _wide_range_queries(q_bits: np.ndarray, seed: int) -> np.ndarray:
    """bf16 query rows whose magnitudes span 2^-30 .. 2^40 (the f16 range is about 2^-24 ..
    65504): each row is the drawn N(0,1) row times 2^u for its own u, and a few rows mix
    magnitudes inside the row or hold values just above 65504 or bf16 subnormals.  Every result
    is a bf16 value (power-of-two multiples of bf16 values, or exactly written bits)."""
    B, Hq, D = q_bits.shape
    f = (q_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    rng = np.random.default_rng(seed)
    u = rng.choice([-30, -24, -16, -14, -8, 0, 4, 12, 16, 17, 24, 32, 40], size=(B, Hq))
    f = f * np.exp2(u)[:, :, None]
    f[0, 0, : D // 2] *= 2.0 ** 40  # one row spanning 2^-30 .. 2^40 inside itself
    f[0, 0, D // 2:] *= 2.0 ** -30
    f[0, 1, :] = np.where(np.arange(D) % 3 == 0, 98304.0, f[0, 1, :])  # beyond f16's largest finite value
    f[1, 0, :] = 69632.0 * np.where(f[1, 0, :] < 0, -1.0, 1.0)
    bits = (f.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64), f), "not bf16 values"
    bits[1, 1, :] = np.arange(1, D + 1, dtype=np.uint16) & 0x807F  # bf16 subnormals (and signs)
    return bits


@pytest.mark.parametrize("dtype", ["fp8_e4m3", "int8", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
def test_queries_across_the_bf16_range(pkv, dtype, D):
    """One-byte KV multiplies f16 operands: the query rows are scaled per head by a power of two
    into f16's range, so queries far outside it (2^-30 .. 2^40, values > 65504, bf16 subnormals)
    still give the oracle's result (the masked_mha decode of "TensorRT-LLM 推理加速实战" §7.2 with
    a bf16 query).  Outputs within the low-precision bound of the oracle run on the same codes."""
    import torch
    lens = [1, 37, 300, 64, 513, 129, 900, 2]
    w = W.custom_workload(320 + D, len(lens), 8, 2, D, 16, lens, append=True, kv_dtype=dtype)
    step = _run(pkv, w)
    q = _wide_range_queries(w.query(), 5 + D)
    step.q.copy_(torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).to(step.q.device))
    step.attention()
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_error(step.pool.handle) == pkv.PKV_OK
    pool, _, tables = odrive.build(w)
    ref = odrive.attention(w, pool, tables, q=q)
    got, err = _errors(step, ref)
    tol = TOL_FP8_MAX if dtype != "bf16" else TOL_BF16_MAX
    assert np.isfinite(got).all()
    assert err.max() <= tol, f"max |err| {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}"
    assert err.mean() <= TOL_MEAN, f"mean |err| {err.mean():.3e}"
    step.close()


@pytest.mark.parametrize("dtype", ["fp8_e4m3", "int8"])
@pytest.mark.parametrize("bs", [16, 64])
@pytest.mark.parametrize("D,Hkv", [(128, 2), (128, 12), (64, 20)])
def test_small_appends_with_several_tokens_per_block(pkv, dtype, bs, D, Hkv):
    """Appends of up to 1024 tokens (a decode step appends one per sequence) quantise in one
    pass, each token finding the call's other tokens in its block.  Calls whose tokens share
    blocks in shuffled order (blocks the call opens, blocks continued from earlier calls), with a
    padding slot, must store the oracle's codes and scales bit for bit after every call; so must
    a call of 1025 tokens (three passes).  Head counts: all of a token's 2 * Hkv rows loaded up
    front (Hkv 2), rows loaded after the slot scan (Hkv 12 at D 128), and rows past the 32nd,
    whose stored scale is read on its own (Hkv 20)."""
    import torch
    nb = 6400 // bs
    handle = pkv.pkv_pool_create(nb, bs, Hkv, D, pkv.KV_DTYPES[dtype])
    ref = oracle.Pool(nb, bs, Hkv, D, odrive.KV_CODE[dtype])
    rng = np.random.default_rng(bs + (7 if dtype == "int8" else 0) + Hkv)
    fill = np.zeros(nb, dtype=np.int64)
    from paged_kv_cache_266_gb300.runner import _wrap_device
    kv_ptr, kv_bytes, sc_ptr, sc_bytes = pkv.pkv_pool_raw(handle)
    for n in (1, 7, 33, 200, 1024, 1025, 3):
        slots = []
        while len(slots) < n - 1:
            b = int(rng.choice(np.flatnonzero(fill < bs)))
            run = int(min(n - 1 - len(slots), rng.integers(1, bs - fill[b] + 1)))
            slots += [b * bs + int(fill[b]) + u for u in range(run)]
            fill[b] += run
        slots.insert(int(rng.integers(0, len(slots) + 1)), -1)  # a padding token
        slots = np.array(slots, dtype=np.int64)
        rng.shuffle(slots)
        x = rng.standard_normal((2, n, Hkv, D)) * np.exp2(rng.integers(-3, 4, size=(2, n, 1, 1)))
        bits = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        dk = torch.from_numpy(bits[0].view(np.int16)).view(torch.bfloat16).cuda()
        dv = torch.from_numpy(bits[1].view(np.int16)).view(torch.bfloat16).cuda()
        pkv.pkv_append(handle, dk, dv, torch.from_numpy(slots).cuda())
        assert ref.append(bits[0], bits[1], slots) == 0
        torch.cuda.synchronize()
        assert pkv.pkv_check_device_error(handle) == pkv.PKV_OK
        assert np.array_equal(_wrap_device(sc_ptr, sc_bytes).cpu().numpy().view(np.float32), ref.scales), n
        assert np.array_equal(_wrap_device(kv_ptr, kv_bytes).cpu().numpy(), ref.data), n
    pkv.pkv_pool_destroy(handle)
