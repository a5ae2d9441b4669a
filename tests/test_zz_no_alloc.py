"""The decode entry point that allocates nothing.

Some callers cannot hand the library device memory when they call it: a
runtime that owns a fixed memory budget through its own allocator, a plug-in
without access to the host application's allocator, or a serving loop that
bans cudaMalloc/cudaFree because they can synchronise the device.
kvp_decode_attn_noalloc serves them: its split partials live in a fixed
array inside the library instead of a caller workspace.

These tests call it through the C ABI.  Its kernels and split geometry are
those of kvp_decode_attn (which takes a workspace), so on the same inputs
and split count the two must agree bit for bit -- a partial left over from
an earlier call, or written to the wrong place in the shared array, would
show up as a difference.  Two different batches run back to back (the
second over the first one's leftovers), in bf16 and fp16, with an explicit
and with the library's own split count; one call is also checked against
the fp64 oracle.  A request whose nominal split count would overflow the
array but whose resolved count fits is accepted.

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


def _decode_batch(seed, contexts, dtype="bf16", Hq=8, Hkv=2):
    return wl.make_random(seed, [c - 1 for c in contexts], [1] * len(contexts), Hq=Hq, Hkv=Hkv, d=128,
                          dtype=dtype, num_decode=len(contexts))


def _noalloc(kvp, st, w, splits):
    """kvp_decode_attn_noalloc through ctypes into NaN-filled outputs."""
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
    return out, lse


def _workspace_decode(w, splits):
    """The same batch through kvp_decode_attn with a torch-allocated workspace."""
    from paged_prefix_reuse_gb300.step import DeviceStep

    st = DeviceStep(w, decode_splits=splits)
    st.run_slots()
    st.run_append()
    st.run_decode()
    torch.cuda.synchronize()
    assert st.pool.errors() == 0
    return st, st.out_dec.clone(), st.lse_dec.clone()


@pytest.mark.gpu
def test_noalloc_decode_is_bit_identical_to_workspace_decode_on_two_calls(kvp):
    import oracle

    # (dtype, requested splits, contexts): two different batches, so the
    # second call runs over the first one's leftover partials.
    cases = [("bf16", 5, [700, 31, 1500, 2]), ("f16", 0, [1200, 90, 64, 999, 5])]
    for i, (dtype, splits, contexts) in enumerate(cases):
        w = _decode_batch(71 + i, contexts, dtype)
        st, want_o, want_l = _workspace_decode(w, splits)
        assert st.decode_splits > 1  # the partials go through the scratch array
        out, lse = _noalloc(kvp, st, w, splits)
        assert st.pool.errors() == 0
        assert torch.equal(out, want_o), f"call {i}: out differs from kvp_decode_attn"
        assert torch.equal(lse, want_l), f"call {i}: lse differs from kvp_decode_attn"
        if i == 0:
            ref = oracle.run_step(w)
            o = out.float().cpu().numpy().astype(np.float64).reshape(ref["decode_out"].shape)
            l = lse.cpu().numpy().astype(np.float64).T.reshape(-1)
            assert np.abs(o - ref["decode_out"]).max() <= TOL[dtype]
            assert np.abs(l - ref["decode_lse"]).max() <= LSE_TOL


@pytest.mark.gpu
def test_noalloc_accepts_large_split_request_that_resolves_small(kvp):
    """64 splits requested over contexts of at most 100 keys: nominally 33 MB
    of partials, more than the array holds, but whole 32-key stages per split
    leave 4 splits (about 2 MB), so the call runs."""
    rng = np.random.default_rng(5)
    contexts = rng.integers(2, 101, size=64).tolist()
    w = _decode_batch(77, contexts, "bf16")
    assert kvp.kvp_workspace_size(1, w.B, w.num_q_heads, w.head_dim, 64) > kvp.DECODE_NOALLOC_SCRATCH_BYTES
    st, want_o, want_l = _workspace_decode(w, 64)
    out, lse = _noalloc(kvp, st, w, 64)
    assert torch.equal(out, want_o) and torch.equal(lse, want_l)


def test_noalloc_decode_refuses_requests_beyond_its_scratch(kvp):
    """Refused on the host before any device work (no GPU needed)."""
    lib = kvp.load_library()
    pool = kvp._Pool(0x10000, 0x20000, 1 << 20, 16, 8, 128, 1, None)
    B, Hq, splits = 512, 64, 64
    assert kvp.kvp_workspace_size(1, B, Hq, 128, splits) > kvp.DECODE_NOALLOC_SCRATCH_BYTES
    status = lib.kvp_decode_attn_noalloc(ctypes.byref(pool), 0x30000, 0x40000, None, 0x50000, 0x60000, 2048, B,
                                         Hq, 32768, 0.088, splits, None)
    assert status == 3  # KVP_ERR_WORKSPACE
