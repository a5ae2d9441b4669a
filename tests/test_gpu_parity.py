"""GPU parity: libkvp (through its C ABI) against the fp64 CPU oracle on the
same seeded inputs.

Bars: slot indexing, append and copy bit-exact; attention outputs within a
max-abs error of 2e-2 (bf16) / 5e-3 (fp16) and the log-sum-exp within 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f16": 5e-3}
LSE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _library():
    from paged_prefix_reuse_gb300 import build

    build.build_library()
    import paged_prefix_reuse_gb300 as kvp

    kvp.load_library()


def _step(w, **kw):
    from paged_prefix_reuse_gb300.step import DeviceStep

    return DeviceStep(w, **kw)


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def _compare_attn(dtype, out_gpu, lse_gpu, out_ref, lse_ref, rows=None, what=""):
    """out_gpu [T, Hq, d], lse_gpu [Hq, T]; out_ref [nrows, d] and lse_ref
    [nrows] in flat row order t * Hq + h (all rows, or the given ones)."""
    T, Hq, d = out_gpu.shape
    o = _f64(out_gpu).reshape(T * Hq, d)
    l = _f64(lse_gpu).T.reshape(T * Hq)
    if rows is not None:
        o, l = o[rows], l[rows]
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    err = np.abs(o - out_ref).max()
    lerr = np.abs(l - lse_ref).max()
    assert err <= TOL[dtype], f"{what}: max |out - oracle| = {err:.3e} > {TOL[dtype]}"
    assert lerr <= LSE_TOL, f"{what}: max |lse - oracle| = {lerr:.3e} > {LSE_TOL}"
    return err, lerr


def _check_step(w, rows=None, decode_rows=None, **kw):
    st = _step(w, **kw)
    st.run()
    torch.cuda.synchronize()
    assert st.pool.errors() == 0
    ref = oracle.run_step(w, rows=rows, decode_rows=decode_rows)
    assert ref["bad"] == 0
    if rows is None:
        np.testing.assert_array_equal(st.slots[: st.T].cpu().numpy(), ref["slots"])
        np.testing.assert_array_equal(_bits(st.pool.k), ref["k_pool"])
        np.testing.assert_array_equal(_bits(st.pool.v), ref["v_pool"])
    if st.npf:
        _compare_attn(w.dtype, st.out_pf, st.lse_pf, ref["prefill_out"], ref["prefill_lse"], rows, "prefill")
    if st.ndec:
        _compare_attn(w.dtype, st.out_dec, st.lse_dec, ref["decode_out"], ref["decode_lse"], decode_rows, "decode")
    return st, ref


# --------------------------------------------------------------------------
# small cases the oracle computes completely (several tiles + ragged tails)
# --------------------------------------------------------------------------
SMALL = {
    "tiny_correctness": lambda: wl.tiny_correctness(),
    # GQA 8:1, d=128, bf16, one shared 2-block-aligned prefix, 3 query tiles per kv head
    "shared_prompt_small": lambda: wl.shared_system_prompt(B=3, prefix=304, new=48, num_blocks=256),
    # d=96 fp16, no GQA, chunks reused with replacement, ragged N
    "rag_small": lambda: wl.rag_chunk_reuse(B=3, library=6, chunk=64, chunks_per_request=4, new_lo=20,
                                           new_hi=150, num_blocks=256),
    # GQA 5:1 (rows straddle tokens), mixed prefill + decode, CoW forks
    "mixed_step_small": lambda: wl.continuous_batching_step(n_decode=10, n_prefill=2, prefill_new=70,
                                                            prefill_lo=100, prefill_hi=400, median=300, sigma=0.6,
                                                            ctx_lo=20, ctx_hi=900, n_forks=3, num_blocks=512,
                                                            Hq=10, Hkv=2),
    "p0_causal_d64_bf16": lambda: wl.make_random(41, [0, 0], [200, 131], Hq=4, Hkv=2, d=64, dtype="bf16"),
    "block8_gqa4_f16": lambda: wl.make_random(42, [75, 130], [60, 33], Hq=8, Hkv=2, d=128, dtype="f16", bs=8),
    "block32_d96_bf16": lambda: wl.make_random(43, [300, 5], [40, 100], Hq=6, Hkv=3, d=96, dtype="bf16", bs=32),
    "zero_new_tokens": lambda: wl.make_random(44, [50, 20, 70], [30, 0, 17], Hq=2, Hkv=1, d=64, dtype="f16"),
    "gqa16_d128": lambda: wl.make_random(45, [260], [20], Hq=16, Hkv=1, d=128, dtype="bf16"),
    # logits with std ~6: row maxima jump by more than 2^8 between tiles and
    # between the two 64-key halves of a tile (the rescaling paths)
    "large_logits_bf16": lambda: wl.make_random(46, [300, 0], [200, 150], Hq=4, Hkv=2, d=128, dtype="bf16",
                                                q_std=6.0),
    "large_logits_f16_d64": lambda: wl.make_random(47, [520, 33], [90, 260], Hq=6, Hkv=3, d=64, dtype="f16",
                                                   q_std=6.0),
}


# CTAs with one live query tile over long key ranges (odd and even tile
# counts), a one-token chunk over a long prefix, a chunk of exactly one tile
# with no prefix, one just over a tile, and logits large enough that row
# maxima jump by far more than 2^8 between distant tiles.
SMALL.update({
    "key_split_g1_bf16": lambda: wl.make_random(81, [500, 1000, 0, 37], [100, 3, 128, 129], Hq=4, Hkv=4, d=128,
                                                dtype="bf16"),
    "key_split_g2_f16_d64": lambda: wl.make_random(82, [700, 260, 5], [60, 17, 64], Hq=4, Hkv=2, d=64,
                                                   dtype="f16"),
    "key_split_d96_large_logits": lambda: wl.make_random(83, [900, 1], [70, 120], Hq=3, Hkv=3, d=96, dtype="f16",
                                                         q_std=6.0),
    "key_split_bs8_gqa5": lambda: wl.make_random(84, [333, 2000], [25, 1], Hq=10, Hkv=2, d=128, dtype="bf16",
                                                 bs=8),
})


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_workloads_match_oracle(name):
    _check_step(SMALL[name]())


@pytest.mark.parametrize("splits", [2, 3])
def test_single_tile_ctas_with_split_kv(splits):
    """Single-tile CTAs whose key range is cut across CTAs, the partials
    merged by log-sum-exp."""
    w = wl.make_random(85, [1500, 777], [90, 40], Hq=6, Hkv=6, d=128, dtype="bf16")
    _check_step(w, prefix_splits=splits)


@pytest.mark.parametrize("splits", [1, 2, 3, 7])
def test_prefix_split_kv_counts(splits):
    w = wl.make_random(51, [900, 260], [150, 64], Hq=8, Hkv=2, d=128, dtype="bf16")
    _check_step(w, prefix_splits=splits)


@pytest.mark.parametrize("splits", [1, 2, 5, 40])
def test_decode_split_counts(splits):
    w = wl.make_random(52, [700, 31, 1500, 0], [1, 1, 1, 1], Hq=8, Hkv=2, d=128, dtype="bf16", num_decode=4)
    _check_step(w, decode_splits=splits)


def test_decode_merge_of_more_than_128_partials():
    """100 key ranges of two partials each for the longest context: the merge
    takes the weights of partials past the first 128 from broadcast loads."""
    w = wl.make_random(54, [3300, 31, 1500, 0], [1, 1, 1, 1], Hq=8, Hkv=2, d=128, dtype="bf16", num_decode=4)
    _check_step(w, decode_splits=100)


@pytest.mark.parametrize("d,dtype,bs", [(64, "f16", 16), (96, "bf16", 8), (128, "f16", 32), (96, "f16", 16)])
def test_decode_head_dims_and_blocks(d, dtype, bs):
    w = wl.make_random(53, [3, 77, 400, 1023], [1, 1, 1, 1], Hq=4, Hkv=1, d=d, dtype=dtype, bs=bs, num_decode=4)
    _check_step(w)


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------
def test_physical_placement_permutation_is_bit_identical():
    w = wl.make_random(61, [333, 64], [77, 50], Hq=8, Hkv=2, d=128, dtype="bf16", num_blocks=128)
    w2 = wl.permute_placement(w, 7)
    a, b = _step(w), _step(w2)
    a.run()
    b.run()
    torch.cuda.synchronize()
    assert torch.equal(a.out_pf, b.out_pf)
    assert torch.equal(a.lse_pf, b.lse_pf)


def test_cow_fork_keeps_shared_blocks_byte_identical():
    w = wl.continuous_batching_step(n_decode=8, n_prefill=1, prefill_new=40, prefill_lo=50, prefill_hi=90,
                                    median=200, sigma=0.3, ctx_lo=40, ctx_hi=400, n_forks=4, num_blocks=256,
                                    Hq=8, Hkv=2, d=64)
    shared = set()
    for i in range(4):
        a, b = w.block_tables[w.num_prefill + 2 * i], w.block_tables[w.num_prefill + 2 * i + 1]
        shared |= set(np.intersect1d(a[a >= 0], b[b >= 0]).tolist())
    shared = np.array(sorted(shared))
    st, ref = _check_step(w)
    np.testing.assert_array_equal(_bits(st.pool.k)[shared], w.k_pool[shared])
    np.testing.assert_array_equal(_bits(st.pool.v)[shared], w.v_pool[shared])


def test_garbage_in_unwritten_slots_never_reaches_the_output():
    """Rows of a partial last block past the context (and unused blocks) may
    hold anything, NaN included; they must not influence the result."""
    w = wl.make_random(62, [100, 37], [29, 1], Hq=4, Hkv=2, d=128, dtype="bf16", num_blocks=64)
    ref = oracle.run_step(w)
    k = w.k_pool.copy()
    v = w.v_pool.copy()
    for s in range(w.B):
        L = int(w.context_lens[s])
        last = w.block_tables[s, (L - 1) // 16]
        k[last, :, L % 16 or 16 :] = 0x7FC0  # bf16 NaN
        v[last, :, L % 16 or 16 :] = 0x7FC0
    unused = np.setdiff1d(np.arange(64), w.used_blocks())
    k[unused] = 0x7FC0
    v[unused] = 0x7FC0
    w.k_pool, w.v_pool = k, v
    st = _step(w)
    st.run()
    torch.cuda.synchronize()
    _compare_attn(w.dtype, st.out_pf, st.lse_pf, ref["prefill_out"], ref["prefill_lse"], what="nan-pool")


def test_bad_block_id_is_flagged_not_faulted():
    w = wl.make_random(63, [40], [10], Hq=2, Hkv=2, d=64, dtype="f16", num_blocks=16)
    w.block_tables = w.block_tables.copy()
    w.block_tables[0, 1] = 1000  # outside the 16-block pool
    st = _step(w)
    st.run()
    torch.cuda.synchronize()
    from paged_prefix_reuse_gb300 import DEVERR

    assert st.pool.errors() & DEVERR["bad_block"]
    # the context is still usable afterwards
    good = _step(wl.make_random(64, [40], [10], Hq=2, Hkv=2, d=64, dtype="f16", num_blocks=16))
    good.run()
    torch.cuda.synchronize()
    assert good.pool.errors() == 0


def test_bad_slot_and_pair_are_flagged():
    import paged_prefix_reuse_gb300 as kvp

    w = wl.make_random(65, [16], [4], Hq=2, Hkv=2, d=64, dtype="f16", num_blocks=8)
    st = _step(w)
    before = st.pool.k.clone()
    slots = torch.tensor([-1, 8 * 16, -5, 3], dtype=torch.int64, device="cuda")
    kvp.kvp_cache_append(st.pool, st.k_new, st.v_new, slots)
    pairs = torch.tensor([[0, 99]], dtype=torch.int32, device="cuda")
    kvp.kvp_block_copy(st.pool, pairs)
    torch.cuda.synchronize()
    e = st.pool.errors()
    assert e & kvp.DEVERR["bad_slot"] and e & kvp.DEVERR["bad_pair"]
    changed = (st.pool.k != before).reshape(-1, 64).any(dim=1).nonzero().flatten().tolist()
    # only slot 3 (block 0, row 3) was written, for both kv heads
    assert changed and all(r in (3, 16 + 3) for r in changed)


def test_empty_calls_are_no_ops():
    import paged_prefix_reuse_gb300 as kvp

    w = wl.make_random(66, [16], [4], Hq=2, Hkv=2, d=64, dtype="f16", num_blocks=8)
    st = _step(w)
    before = st.pool.k.clone()
    kvp.kvp_cache_append(st.pool, st.k_new[:0], st.v_new[:0], st.slots[:0])
    kvp.kvp_block_copy(st.pool, torch.empty((0, 2), dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(before, st.pool.k)


# --------------------------------------------------------------------------
# full sizes, in the launch configuration the benchmark times: sampled rows
# --------------------------------------------------------------------------
def _sample_rows(w, sub, n, rng):
    """Flat rows t * Hq + h within a sub-batch: first, last and random tokens."""
    cu = w.cu_seqlens_q
    if sub == "prefill":
        seqs = range(w.num_prefill)
        base = 0
    else:
        seqs = range(w.num_prefill, w.B)
        base = int(cu[w.num_prefill])
    toks = []
    for s in seqs:
        a, b = int(cu[s]) - base, int(cu[s + 1]) - base
        if b > a:
            toks += [a, b - 1]
    toks = np.array(toks + list(rng.choice(np.concatenate([np.arange(int(cu[s]) - base, int(cu[s + 1]) - base)
                                                           for s in seqs]), size=n, replace=True)))
    heads = rng.integers(0, w.num_q_heads, size=toks.shape[0])
    return np.unique(toks * w.num_q_heads + heads)


_CONFIGS = {}


def _config(cfg):
    """Full-size workloads are generated once per module (seconds each)."""
    if cfg not in _CONFIGS:
        _CONFIGS[cfg] = wl.make_config(cfg)
    return _CONFIGS[cfg]


@pytest.mark.parametrize("cfg", [2, 3, 4, 5])
def test_full_size_configs_sampled_rows(cfg):
    w = _config(cfg)
    rng = np.random.default_rng(cfg)
    rows = _sample_rows(w, "prefill", 48, rng) if w.num_prefill else None
    drows = _sample_rows(w, "decode", 48, rng) if w.num_decode else None
    st = _step(w)
    st.run()
    torch.cuda.synchronize()
    assert st.pool.errors() == 0
    ref = oracle.run_step(w, rows=rows, decode_rows=drows)
    # indexing and data movement: bit-exact at full size
    np.testing.assert_array_equal(st.slots[: st.T].cpu().numpy(), ref["slots"])
    touched = np.unique(np.concatenate([ref["slots"] // w.block_size, w.cow_pairs.reshape(-1)]))
    idx = torch.from_numpy(touched).to(st.pool.k.device)
    np.testing.assert_array_equal(_bits(st.pool.k[idx]), ref["k_pool"][touched])
    np.testing.assert_array_equal(_bits(st.pool.v[idx]), ref["v_pool"][touched])
    if rows is not None:
        _compare_attn(w.dtype, st.out_pf, st.lse_pf, ref["prefill_out"], ref["prefill_lse"], rows, f"cfg{cfg}")
        assert torch.isfinite(st.out_pf.float()).all()
    if drows is not None:
        _compare_attn(w.dtype, st.out_dec, st.lse_dec, ref["decode_out"], ref["decode_lse"], drows, f"cfg{cfg}-dec")
        assert torch.isfinite(st.out_dec.float()).all()


@pytest.mark.parametrize("splits", [2, 4])
def test_long_context_split_kv_at_full_size(splits):
    """The long-context batch (4 x 32768 cached + 2048 new tokens) with its
    key range split: each query tile's keys are cut into `splits` ranges of up
    to 8 K keys, written as fp32 partials and merged by log-sum-exp.  (The
    library itself picks one split here: 4 x 8 x 32 = 1024 CTAs already fill
    the GPU.)  Sampled rows against the oracle, every row finite."""
    w = _config(5)
    rng = np.random.default_rng(100 + splits)
    rows = _sample_rows(w, "prefill", 48, rng)
    st = _step(w, prefix_splits=splits)
    assert st.prefix_splits == splits
    st.run()
    torch.cuda.synchronize()
    assert st.pool.errors() == 0
    ref = oracle.run_step(w, rows=rows)
    _compare_attn(w.dtype, st.out_pf, st.lse_pf, ref["prefill_out"], ref["prefill_lse"], rows, f"split{splits}")
    assert torch.isfinite(st.out_pf.float()).all() and torch.isfinite(st.lse_pf).all()


# --------------------------------------------------------------------------
# host <-> device block swap (the CPU page pool of preempted sequences)
# --------------------------------------------------------------------------
def _bits_host(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("dtype,d,bs", [("bf16", 128, 16), ("f16", 96, 32), ("bf16", 64, 8)])
def test_block_swap_out_and_in_is_bit_exact(dtype, d, bs):
    import paged_prefix_reuse_gb300 as kvp

    nb = 128
    w = wl.make_random(60 + d, [500, 300], [20, 7], Hq=8, Hkv=4, d=d, dtype=dtype, bs=bs, num_blocks=nb,
                       fill_all_blocks=True)
    st = _step(w)
    host = kvp.HostKVPool.like(st.pool, 40)
    rng = np.random.default_rng(d)
    host.k.view(torch.int16).copy_(torch.from_numpy(rng.integers(-32768, 32767, size=host.k.shape, dtype=np.int16)))
    host.v.view(torch.int16).copy_(torch.from_numpy(rng.integers(-32768, 32767, size=host.v.shape, dtype=np.int16)))
    hk0, hv0 = _bits_host(host.k).copy(), _bits_host(host.v).copy()
    dev_k0, dev_v0 = _bits(st.pool.k), _bits(st.pool.v)

    # swap out 23 scattered device blocks to scattered host blocks, on a side stream
    src = rng.choice(nb, size=23, replace=False)
    dst = rng.choice(40, size=23, replace=False)
    out_pairs = np.stack([src, dst], 1).astype(np.int32)
    side = torch.cuda.Stream()
    pairs_d = torch.from_numpy(out_pairs).cuda()
    side.wait_stream(torch.cuda.current_stream())
    kvp.kvp_block_swap(st.pool, host, pairs_d, kvp.HostKVPool.SWAP_OUT, stream=side)
    side.synchronize()
    assert st.pool.errors() == 0
    want_k, want_v, bad = oracle.block_swap(dev_k0, dev_v0, hk0, hv0, out_pairs)
    assert bad == 0
    np.testing.assert_array_equal(_bits_host(host.k), want_k)
    np.testing.assert_array_equal(_bits_host(host.v), want_v)

    # swap those host blocks back in to other (free) device blocks
    free = np.setdiff1d(np.arange(nb), src)
    back = np.stack([dst, rng.choice(free, size=23, replace=False)], 1).astype(np.int32)
    kvp.kvp_block_swap(st.pool, host, torch.from_numpy(back).cuda(), kvp.HostKVPool.SWAP_IN)
    torch.cuda.synchronize()
    assert st.pool.errors() == 0
    want_dk, want_dv, bad = oracle.block_swap(want_k, want_v, dev_k0, dev_v0, back)
    assert bad == 0
    np.testing.assert_array_equal(_bits(st.pool.k), want_dk)
    np.testing.assert_array_equal(_bits(st.pool.v), want_dv)
    np.testing.assert_array_equal(want_dk[back[:, 1]], dev_k0[src])  # the round trip


def test_block_swap_bad_pairs_are_flagged_not_faulted():
    import paged_prefix_reuse_gb300 as kvp

    w = wl.make_random(70, [100], [4], Hq=4, Hkv=2, d=64, dtype="f16", num_blocks=16, fill_all_blocks=True)
    st = _step(w)
    host = kvp.HostKVPool.like(st.pool, 8)
    host.k.zero_()
    host.v.zero_()
    dev_k0 = _bits(st.pool.k)
    pairs = torch.tensor([[3, 8], [16, 0], [2, 1], [-1, 2]], dtype=torch.int32, device="cuda")
    kvp.kvp_block_swap(st.pool, host, pairs, kvp.HostKVPool.SWAP_OUT)
    torch.cuda.synchronize()
    assert st.pool.errors() & kvp.DEVERR["bad_pair"]
    np.testing.assert_array_equal(_bits_host(host.k)[1], dev_k0[2])  # the valid pair still moved
    assert not _bits_host(host.k)[[0, 2, 3]].any()
    st.pool.clear_errors()
    kvp.kvp_block_swap(st.pool, host, pairs[:0], kvp.HostKVPool.SWAP_IN)  # n == 0
    torch.cuda.synchronize()
    assert st.pool.errors() == 0
    np.testing.assert_array_equal(_bits(st.pool.k), dev_k0)
