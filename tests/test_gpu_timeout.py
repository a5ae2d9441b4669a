"""The failure path of the kernels' bounded waits, exercised without any
fault: with KVP_LAUNCH_STALL_TEST one warp of every prefix-attention and
decode CTA waits on a barrier that nothing arrives on.  With a short
pipeline limit that wait gives up, the kernel reports KVP_DEVERR_TIMEOUT in
the pool's error word and returns; the host reads it as KVP_ERR_TIMEOUT.
The same context then runs the same step correctly (checked against the
oracle), so nothing was left stuck: no copy in flight, no tensor memory
held, no hung CTA."""
import time

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvp():
    from paged_prefix_reuse_gb300 import build

    build.build_library()
    import paged_prefix_reuse_gb300 as mod

    mod.load_library()
    return mod


def _small_mixed():
    # prefill over a cached prefix plus a decode batch split over its keys
    return wl.continuous_batching_step(n_decode=6, n_prefill=1, prefill_new=40, prefill_lo=60, prefill_hi=200,
                                       median=150, sigma=0.5, ctx_lo=20, ctx_hi=400, n_forks=2, num_blocks=256,
                                       Hq=10, Hkv=2, d=128)


@pytest.mark.parametrize("name,make", [("tiny", wl.tiny_correctness), ("mixed", _small_mixed)])
def test_stalled_wait_times_out_reports_and_leaves_context_usable(kvp, name, make):
    from paged_prefix_reuse_gb300.step import DeviceStep

    w = make()
    before = kvp.kvp_get_launch_options()
    st = DeviceStep(w)
    try:
        kvp.kvp_set_wait_limit_ns(2_000_000)  # 2 ms
        kvp.kvp_set_launch_options(before | kvp.LAUNCH_STALL_TEST)
        t0 = time.perf_counter()
        st.run()
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
    finally:
        kvp.kvp_set_launch_options(before)
        kvp.kvp_set_wait_limit_ns(0)
    assert kvp.kvp_get_wait_limit_ns() == 2_000_000_000
    bits = st.pool.errors()
    assert bits & kvp.DEVERR["timeout"], f"{name}: no timeout reported ({bits:#x})"
    assert not bits & ~kvp.DEVERR["timeout"], f"{name}: unexpected error bits {bits:#x}"
    with pytest.raises(kvp.KvpError) as e:
        kvp.kvp_pool_errors(st.pool)
    assert e.value.status == kvp.KVP_ERR_TIMEOUT
    assert elapsed < 30.0  # each stalled CTA gave up after ~2 ms (a few waves), not the 2 s default

    # the same context, the same buffers: a normal step matches the oracle
    st.pool.clear_errors()
    st.reset_pool()
    st.run()
    torch.cuda.synchronize()
    assert kvp.kvp_pool_errors(st.pool) == 0
    ref = oracle.run_step(w)
    tol = {"bf16": 2e-2, "f16": 5e-3}[w.dtype]
    if st.npf:
        o = st.out_pf.float().cpu().numpy().astype(np.float64).reshape(ref["prefill_out"].shape)
        assert np.abs(o - ref["prefill_out"]).max() <= tol
        l = st.lse_pf.cpu().numpy().astype(np.float64).T.reshape(-1)
        assert np.abs(l - ref["prefill_lse"]).max() <= 1e-3
    if st.ndec:
        o = st.out_dec.float().cpu().numpy().astype(np.float64).reshape(ref["decode_out"].shape)
        assert np.abs(o - ref["decode_out"]).max() <= tol
