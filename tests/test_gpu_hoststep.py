"""The step from pinned host buffers (HostStep: groups of sequences on their
own streams, copies overlapping kernels) gives bit-identical slots, pool
bytes, outputs and LSE to the one-stream device step with the same split
counts, run after run, launched directly or replayed from one CUDA graph."""
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


CASES = {
    # prefill + decode + copy-on-write forks, GQA 5:1
    "mixed_small": lambda: wl.continuous_batching_step(n_decode=10, n_prefill=3, prefill_new=70, prefill_lo=100,
                                                       prefill_hi=400, median=300, sigma=0.6, ctx_lo=20,
                                                       ctx_hi=900, n_forks=3, num_blocks=512, Hq=10, Hkv=2),
    "ragged_f16": lambda: wl.make_random(48, [75, 130, 0, 260], [60, 33, 90, 1], Hq=8, Hkv=2, d=128, dtype="f16"),
    "shared_prompt": lambda: wl.make_config(2),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("groups", [1, 2, 3])
@pytest.mark.parametrize("graph", [False, True])
def test_host_step_matches_device_step(name, groups, graph):
    from paged_prefix_reuse_gb300.step import DeviceStep, HostStep

    w = CASES[name]()
    ref = DeviceStep(w)
    ref.run()
    torch.cuda.synchronize()
    assert ref.pool.errors() == 0

    st = DeviceStep(w)
    ref_pool0 = (st.pool.k.clone(), st.pool.v.clone())
    hs = HostStep(st, groups=groups)
    # device inputs start as garbage: everything must arrive from the host
    st.q.fill_(float("nan"))
    st.k_new.zero_()
    st.v_new.zero_()
    stream = torch.cuda.Stream()
    if graph:
        g = hs.capture(stream)
        st.q.fill_(float("nan"))  # the replays must bring everything again
        st.pool.k.copy_(ref_pool0[0])
        st.pool.v.copy_(ref_pool0[1])
        for _ in range(2):
            g.replay()
    else:
        for _ in range(2):
            hs.run(stream)
    torch.cuda.synchronize()
    assert st.pool.errors() == 0
    assert torch.equal(st.slots[: st.T], ref.slots[: ref.T])
    assert torch.equal(st.pool.k.view(torch.int16), ref.pool.k.view(torch.int16))
    assert torch.equal(st.pool.v.view(torch.int16), ref.pool.v.view(torch.int16))
    out = hs.out_host.view(torch.int16)
    if st.npf:
        assert torch.equal(out[: st.tq], ref.out_pf.cpu().view(torch.int16))
    if st.ndec:
        assert torch.equal(out[st.tq :], ref.out_dec.cpu().view(torch.int16))
    lse_ref = torch.cat([x for x in (ref.lse_pf.cpu() if st.npf else None, ref.lse_dec.cpu() if st.ndec else None)
                         if x is not None], dim=1)
    lse = torch.cat(hs.lse_host, dim=1)
    assert torch.equal(lse, lse_ref)
    assert hs.h2d_bytes > 0 and hs.d2h_bytes == out.numel() * 2 + lse.numel() * 4


@pytest.mark.parametrize("graph", [False, True])
def test_host_step_with_chunked_sequences_matches_device_step(graph):
    """More groups than sequences: each sequence's new tokens are cut into
    chunks whose queries see the keys up to the chunk's end, and a chunk
    follows the earlier chunks' appends.  With one key range per CTA the
    results are bit-identical to the one-stream step."""
    from paged_prefix_reuse_gb300.step import DeviceStep, HostStep

    w = wl.make_random(49, [900, 200], [600, 300], Hq=8, Hkv=2, d=128, dtype="bf16")
    ref = DeviceStep(w, prefix_splits=1)
    ref.run()
    torch.cuda.synchronize()
    st = DeviceStep(w, prefix_splits=1)
    hs = HostStep(st, groups=4)
    assert [g["t1"] - g["t0"] for g in hs.groups] == [512, 88, 256, 44]
    st.q.fill_(float("nan"))
    st.k_new.zero_()
    st.v_new.zero_()
    stream = torch.cuda.Stream()
    if graph:
        g = hs.capture(stream)
        st.q.fill_(float("nan"))
        g.replay()
    else:
        with torch.cuda.stream(stream):
            hs.run(stream)
    stream.synchronize()
    assert st.pool.errors() == 0
    assert torch.equal(st.slots[: st.T], ref.slots[: ref.T])
    assert torch.equal(st.pool.k, ref.pool.k) and torch.equal(st.pool.v, ref.pool.v)
    assert torch.equal(hs.out_host, ref.out_pf.cpu())
    assert torch.equal(torch.cat([l for l in hs.lse_host], dim=1), ref.lse_pf.cpu())
