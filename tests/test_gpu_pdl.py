"""Programmatic dependent launch changes only when a kernel may start, never
what it computes: the whole step (copy, slot mapping, append, prefix
attention with its merge, decode with its merge) gives bit-identical slots,
pool contents and outputs with the option on and off, launched directly and
replayed back to back from a CUDA graph (the overlap the benchmark times)."""
import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    from paged_prefix_reuse_gb300 import build

    build.build_library()
    import paged_prefix_reuse_gb300 as kvp

    kvp.load_library()
    yield
    kvp.kvp_set_launch_options(0)


def _snapshot(st):
    snap = [st.slots[: st.T].clone(), st.pool.k.clone(), st.pool.v.clone()]
    if st.npf:
        snap += [st.out_pf.clone(), st.lse_pf.clone()]
    if st.ndec:
        snap += [st.out_dec.clone(), st.lse_dec.clone()]
    return snap


def _same(a, b):
    for x, y in zip(a, b):
        assert x.shape == y.shape
        assert torch.equal(x.view(torch.uint8) if x.dtype != torch.int64 else x,
                           y.view(torch.uint8) if y.dtype != torch.int64 else y)


CASES = {
    "mixed_small": lambda: wl.continuous_batching_step(n_decode=10, n_prefill=2, prefill_new=70, prefill_lo=100,
                                                       prefill_hi=400, median=300, sigma=0.6, ctx_lo=20,
                                                       ctx_hi=900, n_forks=3, num_blocks=512, Hq=10, Hkv=2),
    "tiny": lambda: wl.make_config(1),
    "shared_prompt": lambda: wl.make_config(2),
    "mixed_full": lambda: wl.make_config(4),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("splits", [0, 3])
def test_step_is_bit_identical_with_and_without_pdl(name, splits):
    import paged_prefix_reuse_gb300 as kvp
    from paged_prefix_reuse_gb300.step import DeviceStep

    w = CASES[name]()
    kvp.kvp_set_launch_options(0)
    st = DeviceStep(w, prefix_splits=splits, decode_splits=splits)
    st.run()
    torch.cuda.synchronize()
    assert st.pool.errors() == 0
    want = _snapshot(st)

    kvp.kvp_set_launch_options(kvp.LAUNCH_PDL)
    assert kvp.kvp_get_launch_options() == kvp.LAUNCH_PDL
    st.reset_pool()
    for _ in range(4):  # each step may start under the previous one's tail
        st.run()
    torch.cuda.synchronize()
    assert st.pool.errors() == 0
    _same(_snapshot(st), want)

    st.reset_pool()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        st.run()
    for _ in range(4):
        g.replay()
    torch.cuda.synchronize()
    assert st.pool.errors() == 0
    _same(_snapshot(st), want)
