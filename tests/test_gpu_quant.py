"""GPU parity of the quantized KV pool (8/4 bits) through the C ABI against
the numpy oracle (oracle/quant.py) on the same seeded inputs.

Bars: quantization codes bit-exact and scale/min equal as fp16 values;
decode over a partly quantized context within max-abs 2e-2 (bf16) /
5e-3 (fp16) of the fp64 oracle over the dequantized values, LSE within 1e-3.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from oracle import quant

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f16": 5e-3}
LSE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _library():
    from paged_prefix_reuse_gb300 import build

    build.build_library()
    import paged_prefix_reuse_gb300 as kvp

    kvp.load_library()


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _qarrays(qp):
    return (qp.k_codes.cpu().numpy(), qp.v_codes.cpu().numpy(), qp.k_meta.cpu().numpy(), qp.v_meta.cpu().numpy())


@pytest.mark.parametrize("dtype,d,bits", [("bf16", 128, 8), ("bf16", 128, 4), ("f16", 96, 8), ("f16", 64, 4),
                                          ("bf16", 96, 4)])
def test_quantize_blocks_matches_oracle_bit_exact(dtype, d, bits):
    import paged_prefix_reuse_gb300 as kvp

    rng = np.random.default_rng(d * 10 + bits)
    nb, Hkv, bs = 40, 3, 16
    scale = np.geomspace(1e-2, 30, d).astype(np.float32)  # channels of very different ranges
    K = (rng.standard_normal((nb, Hkv, bs, d)) * scale).astype(np.float32)
    V = (rng.standard_normal((nb, Hkv, bs, d)) * rng.uniform(0.01, 10, (nb, Hkv, bs, 1))).astype(np.float32)
    K[3] = 0.625  # constant groups
    kb, vb = wl.round_to_bits(K, dtype), wl.round_to_bits(V, dtype)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    pool = kvp.PagedKVPool(torch.from_numpy(kb.view(np.int16)).view(tdt).cuda(),
                           torch.from_numpy(vb.view(np.int16)).view(tdt).cuda())
    qp = kvp.QuantKVPool.like(pool, 32, bits)
    src = rng.choice(nb, size=29, replace=False)
    src[0] = 3
    pairs = np.stack([src, rng.choice(32, size=29, replace=False)], 1).astype(np.int32)
    kvp.kvp_quantize_blocks(pool, qp, torch.from_numpy(pairs).cuda())
    torch.cuda.synchronize()
    assert pool.errors() == 0
    want, bad = quant.quantize_blocks(dtype, kb, vb, quant.empty_qpool(32, Hkv, bs, d, bits), bits, pairs)
    assert bad == 0
    got = _qarrays(qp)
    np.testing.assert_array_equal(got[0], want[0])
    np.testing.assert_array_equal(got[1], want[1])
    np.testing.assert_array_equal(got[2].astype(np.float32), want[2].astype(np.float32))
    np.testing.assert_array_equal(got[3].astype(np.float32), want[3].astype(np.float32))


def _decode_case(seed, contexts, dtype, d, Hq, Hkv, bits, qfrac, garbage_codes=False):
    """A decode batch whose first pages per sequence are moved to a quantized
    pool (a block index space of its own) and the rest stay 16-bit."""
    import paged_prefix_reuse_gb300 as kvp
    from paged_prefix_reuse_gb300.step import DeviceStep

    w = wl.make_random(seed, [c - 1 for c in contexts], [1] * len(contexts), Hq=Hq, Hkv=Hkv, d=d, dtype=dtype,
                       num_decode=len(contexts))
    st = DeviceStep(w)
    st.run_slots()
    st.run_append()
    torch.cuda.synchronize()
    kb, vb = _bits(st.pool.k), _bits(st.pool.v)
    rng = np.random.default_rng(seed)
    bs = w.block_size
    bt = st.bt.cpu().numpy().copy()
    ctx = st.ctx.cpu().numpy()
    qpages = []
    pairs = []
    for b, L in enumerate(ctx):
        n = (int(L) + bs - 1) // bs
        k = int(round(qfrac[b % len(qfrac)] * n))
        qpages.append(k)
        for p in range(k):
            pairs.append((int(bt[b, p]), len(pairs)))
            bt[b, p] = len(pairs) - 1
    nq = max(1, len(pairs))
    perm = rng.permutation(nq)  # scatter the quantized blocks
    for b, k in enumerate(qpages):
        bt[b, :k] = perm[bt[b, :k]]
    pairs = np.array([(s_, perm[d_]) for s_, d_ in pairs], dtype=np.int32).reshape(-1, 2)
    qp = kvp.QuantKVPool.like(st.pool, nq, bits)
    if garbage_codes:
        qp.k_codes.random_(0, 256)
        qp.v_codes.random_(0, 256)
    if len(pairs):
        kvp.kvp_quantize_blocks(st.pool, qp, torch.from_numpy(pairs).cuda())
    torch.cuda.synchronize()
    assert st.pool.errors() == 0
    oq, _ = quant.quantize_blocks(dtype, kb, vb, _qarrays(qp), bits, pairs)
    return w, st, qp, oq, bt, np.array(qpages, dtype=np.int32), kb, vb


@pytest.mark.parametrize("dtype,d,bits,splits", [("bf16", 128, 8, 1), ("bf16", 128, 4, 0), ("f16", 128, 8, 3),
                                                 ("f16", 96, 4, 1), ("bf16", 64, 8, 2), ("bf16", 96, 8, 0)])
def test_quantized_decode_matches_oracle(dtype, d, bits, splits):
    import paged_prefix_reuse_gb300 as kvp

    contexts = [700, 31, 1500, 2, 257, 16, 999]
    w, st, qp, oq, bt, qpages, kb, vb = _decode_case(100 + d + bits, contexts, dtype, d, 10, 2, bits,
                                                     qfrac=[1.0, 0.5, 0.9, 0.0, 1.0, 1.0, 0.3])
    tq = torch.from_numpy(qpages).cuda()
    tbt = torch.from_numpy(bt).cuda()
    q = st.q[st.tq:]
    out, lse = kvp.kvp_decode_attn_q(st.pool, qp, tq, q, st.ctx, tbt, st.max_ctx_dec, w.softmax_scale,
                                     num_splits=splits)
    torch.cuda.synchronize()
    assert st.pool.errors() == 0
    want, want_lse = quant.decode_attn_q(dtype, oq, bits, kb, vb, w.q[st.tq:], w.context_lens, bt, qpages,
                                         w.softmax_scale)
    o = out.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(o).all()
    err = np.abs(o - want).max()
    lerr = np.abs(lse.cpu().numpy().T.astype(np.float64) - want_lse).max()
    assert err <= TOL[dtype], err
    assert lerr <= LSE_TOL, lerr


def test_quantized_decode_without_quantized_pages_equals_16bit_decode():
    """qpages = 0 everywhere: every page takes the 16-bit path of the
    quantized-prefix kernel (fp16 products, a bf16 pool's values converted),
    which matches the oracle and the 16-bit decode at the dtype's tolerance."""
    import paged_prefix_reuse_gb300 as kvp

    w, st, qp, oq, bt, qpages, kb, vb = _decode_case(7, [300, 45, 1024], "f16", 128, 8, 2, 8, qfrac=[0.0])
    q = st.q[st.tq:]
    a, la = kvp.kvp_decode_attn(st.pool, q, st.ctx, st.bt, st.max_ctx_dec, w.softmax_scale, num_splits=2)
    b, lb = kvp.kvp_decode_attn_q(st.pool, qp, torch.zeros(3, dtype=torch.int32, device="cuda"), q, st.ctx, st.bt,
                                  st.max_ctx_dec, w.softmax_scale, num_splits=2)
    torch.cuda.synchronize()
    want, want_lse = quant.decode_attn_q("f16", oq, 8, kb, vb, w.q[st.tq:], w.context_lens, bt, qpages,
                                         w.softmax_scale)
    assert np.abs(b.float().cpu().numpy() - want).max() <= TOL["f16"]
    assert np.abs(lb.cpu().numpy().T - want_lse).max() <= LSE_TOL
    assert (b.float() - a.float()).abs().max().item() <= TOL["f16"]
    assert (lb - la).abs().max().item() <= LSE_TOL
    w, st, qp, oq, bt, qpages, kb, vb = _decode_case(8, [300, 45, 1024], "bf16", 128, 8, 2, 4, qfrac=[0.0])
    out, lse = kvp.kvp_decode_attn_q(st.pool, qp, torch.zeros(3, dtype=torch.int32, device="cuda"), st.q[st.tq:],
                                     st.ctx, st.bt, st.max_ctx_dec, w.softmax_scale, num_splits=2)
    torch.cuda.synchronize()
    want, want_lse = quant.decode_attn_q("bf16", oq, 4, kb, vb, w.q[st.tq:], w.context_lens, bt, qpages,
                                         w.softmax_scale)
    assert np.abs(out.float().cpu().numpy() - want).max() <= TOL["bf16"]
    assert np.abs(lse.cpu().numpy().T - want_lse).max() <= LSE_TOL


def test_quantized_decode_clamps_qpages_and_ignores_codes_past_the_context():
    """qpages larger than the page count is clamped; a fully quantized last
    page that is only partly inside the context (its codes past the context
    are garbage) still gives the oracle's result."""
    import paged_prefix_reuse_gb300 as kvp

    contexts = [37, 100, 16]
    w, st, qp, oq, bt, qpages, kb, vb = _decode_case(9, contexts, "f16", 64, 4, 2, 8, qfrac=[1.0],
                                                     garbage_codes=True)
    big = torch.tensor([100, 100, 100], dtype=torch.int32, device="cuda")
    out, lse = kvp.kvp_decode_attn_q(st.pool, qp, big, st.q[st.tq:], st.ctx, torch.from_numpy(bt).cuda(),
                                     st.max_ctx_dec, w.softmax_scale, num_splits=1)
    torch.cuda.synchronize()
    want, want_lse = quant.decode_attn_q("f16", oq, 8, kb, vb, w.q[st.tq:], w.context_lens, bt, qpages,
                                         w.softmax_scale)
    assert np.abs(out.float().cpu().numpy() - want).max() <= TOL["f16"]
    assert np.abs(lse.cpu().numpy().T - want_lse).max() <= LSE_TOL


def test_quantized_decode_bad_block_is_flagged_not_faulted():
    import paged_prefix_reuse_gb300 as kvp

    w, st, qp, oq, bt, qpages, kb, vb = _decode_case(11, [200, 90], "bf16", 128, 4, 2, 8, qfrac=[1.0])
    bt = bt.copy()
    bt[0, 1] = qp.num_blocks + 5  # outside the quantized pool
    out, _ = kvp.kvp_decode_attn_q(st.pool, qp, torch.from_numpy(qpages).cuda(), st.q[st.tq:], st.ctx,
                                   torch.from_numpy(bt).cuda(), st.max_ctx_dec, w.softmax_scale, num_splits=1)
    torch.cuda.synchronize()
    assert st.pool.errors() & kvp.DEVERR["bad_block"]
    assert torch.isfinite(out[1].float()).all()


def test_quantized_range_overflow_is_flagged():
    import paged_prefix_reuse_gb300 as kvp

    kb = wl.round_to_bits(np.full((2, 1, 16, 64), 1.0, np.float32), "bf16")
    kb[0, 0, 3, 5] = wl.round_to_bits(np.array([-1e6], np.float32), "bf16")[0]  # min beyond fp16
    pool = kvp.PagedKVPool(torch.from_numpy(kb.view(np.int16)).view(torch.bfloat16).cuda(),
                           torch.from_numpy(kb.view(np.int16)).view(torch.bfloat16).cuda())
    qp = kvp.QuantKVPool.like(pool, 2, 8)
    kvp.kvp_quantize_blocks(pool, qp, torch.tensor([[0, 1]], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert pool.errors() & 0x20


# --------------------------------------------------------------------------
# prefix attention over a quantized cached prefix (kvp_prefix_attn_q)
# --------------------------------------------------------------------------
def _prefill_q_case(w, bits, qfrac, into_new=False, seed=0):
    """Append the new tokens' K/V (16-bit pool), then move the first pages of
    every sequence to a quantized pool (scattered block ids; a block shared by
    several tables is quantized once).  qfrac[s] of the full cached pages
    (or, with into_new, of all pages: pages holding new tokens too)."""
    import paged_prefix_reuse_gb300 as kvp
    from paged_prefix_reuse_gb300.step import DeviceStep

    st = DeviceStep(w)
    st.run_slots()
    st.run_append()
    torch.cuda.synchronize()
    kb, vb = _bits(st.pool.k), _bits(st.pool.v)
    bs = w.block_size
    bt = st.bt.cpu().numpy().copy()
    ctx = st.ctx.cpu().numpy()
    new = np.diff(st.cu.cpu().numpy())
    qpages, qid = [], {}
    for s in range(w.B):
        full = (int(ctx[s]) + bs - 1) // bs if into_new else (int(ctx[s]) - int(new[s])) // bs
        k = int(round(qfrac[s % len(qfrac)] * full))
        qpages.append(k)
        for p in range(k):
            src = int(bt[s, p])
            if src not in qid:
                qid[src] = len(qid)
            bt[s, p] = qid[src]
    nq = max(1, len(qid))
    perm = np.random.default_rng(seed).permutation(nq)
    for s, k in enumerate(qpages):
        bt[s, :k] = perm[bt[s, :k]]
    pairs = np.array([(src, perm[i]) for src, i in qid.items()], dtype=np.int32).reshape(-1, 2)
    qp = kvp.QuantKVPool.like(st.pool, nq, bits)
    if len(pairs):
        kvp.kvp_quantize_blocks(st.pool, qp, torch.from_numpy(pairs).cuda())
    torch.cuda.synchronize()
    assert st.pool.errors() == 0
    oq, _ = quant.quantize_blocks(w.dtype, kb, vb, _qarrays(qp), bits, pairs)
    return st, qp, oq, bt, np.array(qpages, dtype=np.int32), kb, vb


def _run_prefill_q(st, qp, bt, qpages, w, splits=0):
    import paged_prefix_reuse_gb300 as kvp

    out, lse = kvp.kvp_prefix_attn_q(st.pool, qp, torch.from_numpy(qpages).cuda(), st.q[: st.tq],
                                     st.cu[: st.npf + 1], st.ctx[: st.npf], torch.from_numpy(bt[: st.npf]).cuda(),
                                     st.max_q_pf, st.max_ctx_pf, w.softmax_scale, num_splits=splits)
    torch.cuda.synchronize()
    assert st.pool.errors() == 0
    return out, lse


PREFILL_Q = [
    # dtype, d, bits, splits, Hq, Hkv, qfrac, into_new
    ("bf16", 128, 8, 1, 8, 2, [1.0, 0.5, 0.0], False),
    ("bf16", 128, 4, 2, 8, 2, [1.0, 0.7, 1.0], True),
    ("f16", 96, 8, 1, 4, 4, [1.0, 1.0, 0.3], False),
    ("f16", 64, 4, 0, 6, 3, [0.6, 1.0, 1.0], True),
    ("bf16", 96, 4, 3, 5, 1, [1.0, 0.0, 1.0], False),
    ("f16", 128, 8, 1, 16, 1, [1.0, 1.0, 1.0], False),
]


@pytest.mark.parametrize("dtype,d,bits,splits,Hq,Hkv,qfrac,into_new", PREFILL_Q)
def test_quantized_prefill_matches_oracle(dtype, d, bits, splits, Hq, Hkv, qfrac, into_new):
    """Ragged new-token counts (one chunk of 1 token, one crossing several
    query tiles), prefixes not a multiple of the block, a tile boundary inside
    the quantized range, splits over the key range."""
    w = wl.make_random(200 + d + bits + splits, [300, 77, 650], [131, 1, 40], Hq=Hq, Hkv=Hkv, d=d, dtype=dtype)
    st, qp, oq, bt, qpages, kb, vb = _prefill_q_case(w, bits, qfrac, into_new, seed=d)
    out, lse = _run_prefill_q(st, qp, bt, qpages, w, splits)
    want, want_lse = quant.prefix_attn_q(dtype, oq, bits, kb, vb, w.q, w.cu_seqlens_q, w.context_lens, bt, qpages,
                                         w.softmax_scale)
    o = out.float().cpu().numpy().astype(np.float64).reshape(want.shape)
    l = lse.cpu().numpy().astype(np.float64).T.reshape(-1)
    assert np.isfinite(o).all()
    assert np.abs(o - want).max() <= TOL[dtype], np.abs(o - want).max()
    assert np.abs(l - want_lse).max() <= LSE_TOL, np.abs(l - want_lse).max()


@pytest.mark.parametrize("bits", [8, 4])
def test_quantized_prefill_rag_chunks_at_full_size(bits):
    """The RAG chunk-reuse batch at full size (16 requests x 8 shared 256-token
    chunks, 32 kv heads, d = 96, fp16) with every cached chunk page stored
    quantized: sampled rows against the oracle, every output finite."""
    w = wl.make_config(3)
    st, qp, oq, bt, qpages, kb, vb = _prefill_q_case(w, bits, [1.0], seed=bits)
    assert (qpages == w.prefix_lens // 16).all()
    out, lse = _run_prefill_q(st, qp, bt, qpages, w)
    rng = np.random.default_rng(bits)
    T = int(w.cu_seqlens_q[-1])
    rows = np.unique(np.concatenate([rng.integers(0, T * w.num_q_heads, 40), [0, T * w.num_q_heads - 1]]))
    want, want_lse = quant.prefix_attn_q(w.dtype, oq, bits, kb, vb, w.q, w.cu_seqlens_q, w.context_lens, bt,
                                         qpages, w.softmax_scale, rows=rows)
    o = out.float().cpu().numpy().astype(np.float64).reshape(T * w.num_q_heads, -1)[rows]
    l = lse.cpu().numpy().astype(np.float64).T.reshape(-1)[rows]
    assert torch.isfinite(out.float()).all()
    assert np.abs(o - want).max() <= TOL[w.dtype]
    assert np.abs(l - want_lse).max() <= LSE_TOL


def test_quantized_prefill_bad_quantized_block_is_flagged():
    import paged_prefix_reuse_gb300 as kvp

    w = wl.make_random(250, [200], [30], Hq=4, Hkv=2, d=128, dtype="bf16")
    st, qp, oq, bt, qpages, kb, vb = _prefill_q_case(w, 8, [1.0])
    bt = bt.copy()
    bt[0, 1] = qp.num_blocks + 5  # outside the quantized pool (it is inside the 16-bit one)
    out, lse = kvp.kvp_prefix_attn_q(st.pool, qp, torch.from_numpy(qpages).cuda(), st.q, st.cu, st.ctx,
                                     torch.from_numpy(bt).cuda(), st.max_q_pf, st.max_ctx_pf, w.softmax_scale)
    torch.cuda.synchronize()
    assert st.pool.errors() & kvp.DEVERR["bad_block"]


@pytest.mark.parametrize("bits", [8, 4])
def test_quantize_codes_at_half_step_boundaries_match_oracle(bits):
    """Values placed half a quantization step apart, so that (x - z) / s lands
    within rounding distance of half-integers: the kernel's division-free
    code must still equal the correctly rounded division of the format."""
    import paged_prefix_reuse_gb300 as kvp

    rng = np.random.default_rng(300 + bits)
    nb, Hkv, bs, d = 24, 2, 16, 128
    levels = (1 << bits) - 1
    lo = rng.uniform(-3, 0, size=(nb, Hkv, 1, d)).astype(np.float32)
    step = rng.uniform(0.001, 0.05, size=(nb, Hkv, 1, d)).astype(np.float32)
    k = rng.integers(0, levels, size=(nb, Hkv, bs, d)).astype(np.float32)
    K = lo + (k + 0.5) * step
    K[:, :, 0] = lo[:, :, 0]                 # the group's minimum
    K[:, :, 1] = lo[:, :, 0] + levels * step[:, :, 0]  # and maximum
    Vlo = rng.uniform(-2, 0, size=(nb, Hkv, bs, 1)).astype(np.float32)
    Vst = rng.uniform(0.001, 0.05, size=(nb, Hkv, bs, 1)).astype(np.float32)
    V = Vlo + (rng.integers(0, levels, size=(nb, Hkv, bs, d)) + 0.5) * Vst
    V[..., 0:1] = Vlo
    V[..., 1:2] = Vlo + levels * Vst
    for dtype in ("f16", "bf16"):
        kb, vb = wl.round_to_bits(K, dtype), wl.round_to_bits(V.astype(np.float32), dtype)
        tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
        pool = kvp.PagedKVPool(torch.from_numpy(kb.view(np.int16)).view(tdt).cuda(),
                               torch.from_numpy(vb.view(np.int16)).view(tdt).cuda())
        qp = kvp.QuantKVPool.like(pool, nb, bits)
        pairs = np.stack([np.arange(nb), rng.permutation(nb)], 1).astype(np.int32)
        kvp.kvp_quantize_blocks(pool, qp, torch.from_numpy(pairs).cuda())
        torch.cuda.synchronize()
        assert pool.errors() == 0
        want, _ = quant.quantize_blocks(dtype, kb, vb, quant.empty_qpool(nb, Hkv, bs, d, bits), bits, pairs)
        got = _qarrays(qp)
        for a, b in zip(got, want):
            np.testing.assert_array_equal(a.astype(np.float32), b.astype(np.float32))


@pytest.mark.parametrize("dtype,d,bits,Hq,Hkv,splits", [("bf16", 128, 8, 32, 2, 0), ("f16", 96, 4, 12, 1, 2),
                                                        ("bf16", 64, 8, 9, 1, 1)])
def test_quantized_decode_groups_wider_than_eight_heads(dtype, d, bits, Hq, Hkv, splits):
    """Groups of more than 8 query heads per kv head run as blocks of 8 heads
    (one CTA each) over the same pages."""
    import paged_prefix_reuse_gb300 as kvp

    contexts = [300, 17, 1030, 64]
    w, st, qp, oq, bt, qpages, kb, vb = _decode_case(400 + Hq + bits, contexts, dtype, d, Hq, Hkv, bits,
                                                     qfrac=[1.0, 0.0, 0.6, 1.0])
    out, lse = kvp.kvp_decode_attn_q(st.pool, qp, torch.from_numpy(qpages).cuda(), st.q[st.tq:], st.ctx,
                                     torch.from_numpy(bt).cuda(), st.max_ctx_dec, w.softmax_scale, num_splits=splits)
    torch.cuda.synchronize()
    assert st.pool.errors() == 0
    want, want_lse = quant.decode_attn_q(dtype, oq, bits, kb, vb, w.q[st.tq:], w.context_lens, bt, qpages,
                                         w.softmax_scale)
    o = out.float().cpu().numpy().astype(np.float64)
    assert np.abs(o - want).max() <= TOL[dtype]
    assert np.abs(lse.cpu().numpy().T.astype(np.float64) - want_lse).max() <= LSE_TOL


@pytest.mark.parametrize("op", ["decode", "prefill"])
def test_quantized_kernels_stalled_wait_times_out_and_context_stays_usable(op):
    """KVP_LAUNCH_STALL_TEST on the quantized-prefix kernels: one warp of every
    CTA waits on a barrier nothing arrives on, gives up after the 2 ms limit
    and reports KVP_DEVERR_TIMEOUT; the same call then runs normally and
    matches the oracle."""
    import paged_prefix_reuse_gb300 as kvp

    if op == "decode":
        w, st, qp, oq, bt, qpages, kb, vb = _decode_case(61, [300, 45, 700], "bf16", 128, 10, 2, 8,
                                                         qfrac=[1.0, 0.5, 0.9])

        def call(splits):
            return kvp.kvp_decode_attn_q(st.pool, qp, torch.from_numpy(qpages).cuda(), st.q[st.tq:], st.ctx,
                                         torch.from_numpy(bt).cuda(), st.max_ctx_dec, w.softmax_scale,
                                         num_splits=splits)

        def want():
            return quant.decode_attn_q("bf16", oq, 8, kb, vb, w.q[st.tq:], w.context_lens, bt, qpages,
                                       w.softmax_scale)
    else:
        w = wl.make_random(62, [300, 77], [131, 40], Hq=8, Hkv=2, d=128, dtype="bf16")
        st, qp, oq, bt, qpages, kb, vb = _prefill_q_case(w, 8, [1.0, 0.5])

        def call(splits):
            return kvp.kvp_prefix_attn_q(st.pool, qp, torch.from_numpy(qpages).cuda(), st.q[: st.tq],
                                         st.cu[: st.npf + 1], st.ctx[: st.npf], torch.from_numpy(bt[: st.npf]).cuda(),
                                         st.max_q_pf, st.max_ctx_pf, w.softmax_scale, num_splits=splits)

        def want():
            return quant.prefix_attn_q("bf16", oq, 8, kb, vb, w.q, w.cu_seqlens_q, w.context_lens, bt, qpages,
                                       w.softmax_scale)
    before = kvp.kvp_get_launch_options()
    try:
        kvp.kvp_set_wait_limit_ns(2_000_000)  # 2 ms
        kvp.kvp_set_launch_options(before | kvp.LAUNCH_STALL_TEST)
        for splits in (1, 2):
            call(splits)
        torch.cuda.synchronize()
    finally:
        kvp.kvp_set_launch_options(before)
        kvp.kvp_set_wait_limit_ns(0)
    bits = st.pool.errors()
    assert bits & kvp.DEVERR["timeout"], f"no timeout reported ({bits:#x})"
    assert not bits & ~kvp.DEVERR["timeout"], f"unexpected error bits {bits:#x}"
    st.pool.clear_errors()
    out, lse = call(2)
    torch.cuda.synchronize()
    assert st.pool.errors() == 0
    o_want, l_want = want()
    o = out.float().cpu().numpy().astype(np.float64).reshape(o_want.shape)
    assert np.abs(o - o_want).max() <= TOL["bf16"]
    l = lse.cpu().numpy().astype(np.float64).T.reshape(l_want.shape)
    assert np.abs(l - l_want).max() <= LSE_TOL


@pytest.mark.parametrize("bits", [8, 4])
def test_quantized_decode_mixed_batch_at_full_size(bits):
    """The decode batch of the continuous-batching step at full size, every
    complete page quantized, in the benchmark's launch configuration
    (automatic split count).  Eight sequences (the longest, the shortest and
    six at random) are checked against the oracle, which quantizes their
    pages itself from the 16-bit pool."""
    import paged_prefix_reuse_gb300 as kvp
    from paged_prefix_reuse_gb300.step import DeviceStep

    w = wl.make_config(4)
    st = DeviceStep(w)
    st.run_slots()
    st.run_append()
    torch.cuda.synchronize()
    pool, bs = st.pool, w.block_size
    ctx = st.ctx[st.npf:].cpu().numpy()
    bt = st.bt[st.npf:].cpu().numpy().copy()
    qpages = (ctx // bs).astype(np.int32)
    pairs, bt_q = [], bt.copy()
    for b in range(len(ctx)):
        for pg in range(int(qpages[b])):
            pairs.append((int(bt[b, pg]), len(pairs)))
            bt_q[b, pg] = len(pairs) - 1
    qp = kvp.QuantKVPool.like(pool, len(pairs), bits)
    kvp.kvp_quantize_blocks(pool, qp, torch.tensor(pairs, dtype=torch.int32, device="cuda"))
    q = st.q[st.tq:]
    out, lse = kvp.kvp_decode_attn_q(pool, qp, torch.from_numpy(qpages).cuda(), q, st.ctx[st.npf:],
                                     torch.from_numpy(bt_q).cuda(), int(ctx.max()), w.softmax_scale)
    torch.cuda.synchronize()
    assert pool.errors() == 0

    rng = np.random.default_rng(500 + bits)
    pick = np.unique(np.concatenate([[int(ctx.argmax()), int(ctx.argmin())], rng.choice(len(ctx), 6, replace=False)]))
    # The oracle's own pools: the picked sequences' blocks, gathered and renumbered.
    blocks = sorted({int(bt[b, p]) for b in pick for p in range((int(ctx[b]) + bs - 1) // bs)})
    where = {blk: i for i, blk in enumerate(blocks)}
    idx = torch.tensor(blocks, dtype=torch.int64, device="cuda")
    kb, vb = _bits(pool.k.index_select(0, idx)), _bits(pool.v.index_select(0, idx))
    npg = (ctx[pick] + bs - 1) // bs
    bt_o = np.zeros((len(pick), int(npg.max())), dtype=np.int64)
    opairs = []
    for r, b in enumerate(pick):
        for p in range(int(npg[r])):
            blk = where[int(bt[b, p])]
            if p < int(qpages[b]):
                opairs.append((blk, len(opairs)))
                bt_o[r, p] = len(opairs) - 1
            else:
                bt_o[r, p] = blk
    Hkv, d = pool.num_kv_heads, pool.head_dim
    oq, _ = quant.quantize_blocks(w.dtype, kb, vb, quant.empty_qpool(max(1, len(opairs)), Hkv, bs, d, bits), bits,
                                  np.array(opairs, dtype=np.int64))
    want, want_lse = quant.decode_attn_q(w.dtype, oq, bits, kb, vb, w.q[st.tq:][pick], ctx[pick], bt_o,
                                         qpages[pick], w.softmax_scale)
    o = out.float().cpu().numpy().astype(np.float64)[pick]
    assert np.isfinite(o).all()
    assert np.abs(o - want).max() <= TOL[w.dtype]
    assert np.abs(lse.cpu().numpy().T.astype(np.float64)[pick] - want_lse).max() <= LSE_TOL
