"""The decode entry point that allocates nothing.

Some callers cannot hand the library device memory when they call it: a
runtime that owns a fixed memory budget through its own allocator, a plug-in
without access to the host application's allocator, or a serving loop that
bans cudaMalloc/cudaFree because they can synchronise the device.
kvp_decode_attn_noalloc serves them: its split partials live in a fixed
array inside the library instead of a caller workspace.  These tests check
it through the C ABI against kvp_decode_attn (which takes a workspace) on
two calls in a row, and that an oversized request is refused.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wl

TOL = {"bf16": 2e-2, "f16": 5e-3}
LSE_TOL = 1e-3


@pytest.fixture(scope="module")
def kvp():
    from paged_prefix_reuse_gb300 import build

    build.build_library()
    import paged_prefix_reuse_gb300 as mod

    mod.load_library()
    return mod


def _decode_batch(seed, contexts, dtype="bf16"):
    return wl.make_random(seed, [c - 1 for c in contexts], [1] * len(contexts), Hq=8, Hkv=2, d=128,
                          dtype=dtype, num_decode=len(contexts))


@pytest.mark.gpu
def test_noalloc_decode_matches_workspace_decode_on_two_calls(kvp):
    from paged_prefix_reuse_gb300.step import DeviceStep

    # Two different batches, so the second call runs over the first one's
    # leftover partials in the shared array.
    batches = [_decode_batch(71, [700, 31, 1500, 2]), _decode_batch(72, [1200, 90, 64, 999, 5])]
    splits = 5  # several key ranges per sequence: the partials need scratch
    for w in batches:
        st = DeviceStep(w, decode_splits=splits)
        st.run_slots()
        st.run_append()
        st.run_decode()  # kvp_decode_attn with a torch-allocated workspace
        torch.cuda.synchronize()
        want_o, want_l = st.out_dec.float().clone(), st.lse_dec.clone()
        assert kvp.kvp_workspace_size(1, w.B, w.num_q_heads, w.head_dim, splits) > 0

        q = st.q[st.tq :]
        out = torch.full_like(q, float("nan"))
        lse = torch.full((w.num_q_heads, w.B), float("nan"), dtype=torch.float32, device=q.device)
        lib = kvp.load_library()
        status = lib.kvp_decode_attn_noalloc(
            st.pool.c, ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(out.data_ptr()),
            ctypes.c_void_p(lse.data_ptr()), ctypes.c_void_p(st.ctx.data_ptr()), ctypes.c_void_p(st.bt.data_ptr()),
            int(st.bt.shape[1]), w.B, w.num_q_heads, st.max_ctx_dec, float(w.softmax_scale), splits,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert status == 0, kvp.kvp_status_string(status)
        torch.cuda.synchronize()
        assert st.pool.errors() == 0
        err = (out.float() - want_o).abs().max().item()
        lerr = (lse - want_l).abs().max().item()
        assert np.isfinite(err) and err <= TOL[w.dtype], err
        assert np.isfinite(lerr) and lerr <= LSE_TOL, lerr


def test_noalloc_decode_refuses_requests_beyond_its_scratch(kvp):
    """Refused on the host before any device work (no GPU needed)."""
    lib = kvp.load_library()
    pool = kvp._Pool(0x10000, 0x20000, 1 << 20, 16, 8, 128, 1, None)
    B, Hq, splits = 512, 64, 64
    assert kvp.kvp_workspace_size(1, B, Hq, 128, splits) > kvp.DECODE_NOALLOC_SCRATCH_BYTES
    status = lib.kvp_decode_attn_noalloc(ctypes.byref(pool), 0x30000, 0x40000, None, 0x50000, 0x60000, 2048, B,
                                         Hq, 32768, 0.088, splits, None)
    assert status == 3  # KVP_ERR_WORKSPACE
