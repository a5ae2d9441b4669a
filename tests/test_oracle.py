"""Pins for the fp64 CPU oracle: each check ties it to something other than
itself -- a library routine, a closed form, an invariant of the mathematics,
brute force on small inputs, or a value printed on the pages.

Each test names the mistake it is there to catch.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# independent helpers (test side): logical gather + dense textbook attention
# --------------------------------------------------------------------------
def logical_kv(w, pool_bits, s, kvh):
    """Logical key/value rows of sequence s for kv head kvh, read through the
    table with numpy indexing: token j -> block bt[s, j // bs], row j % bs."""
    L = int(w.context_lens[s])
    j = np.arange(L)
    blocks = w.block_tables[s, j // w.block_size]
    return wl.bits_to_float32(pool_bits[blocks, kvh, j % w.block_size], w.dtype).astype(np.float64)


def dense_reference(w, k_pool=None, v_pool=None):
    """softmax(scale * Q K^T + bottom-right causal mask) V per sequence and head,
    by numpy matrix products and scipy's logsumexp; returns (out, lse) with
    rows ordered t * Hq + h like the oracle."""
    from scipy.special import logsumexp

    kp = w.k_pool if k_pool is None else k_pool
    vp = w.v_pool if v_pool is None else v_pool
    g = w.num_q_heads // w.num_kv_heads
    cu = w.cu_seqlens_q
    out = np.zeros((w.T * w.num_q_heads, w.head_dim))
    lse = np.zeros(w.T * w.num_q_heads)
    qf = wl.bits_to_float32(w.q, w.dtype).astype(np.float64)
    for s in range(w.B):
        n = int(w.new_lens[s])
        L = int(w.context_lens[s])
        if n == 0:
            continue
        for h in range(w.num_q_heads):
            K = logical_kv(w, kp, s, h // g)
            V = logical_kv(w, vp, s, h // g)
            Q = qf[cu[s] : cu[s + 1], h]
            X = w.softmax_scale * Q @ K.T  # [n, L]
            pos = L - n + np.arange(n)
            mask = np.arange(L)[None, :] > pos[:, None]
            X = np.where(mask, -np.inf, X)
            l = logsumexp(X, axis=1)
            Pm = np.exp(X - l[:, None])
            rows = (cu[s] + np.arange(n)) * w.num_q_heads + h
            out[rows] = Pm @ V
            lse[rows] = l
    return out, lse


def run_oracle(w, k_pool=None, v_pool=None, rows=None):
    kp = w.k_pool if k_pool is None else k_pool
    vp = w.v_pool if v_pool is None else v_pool
    return oracle.prefix_attn(
        w.dtype, kp, vp, w.q, w.cu_seqlens_q, w.context_lens, w.block_tables, w.softmax_scale, rows
    )


# --------------------------------------------------------------------------
# storage formats
# --------------------------------------------------------------------------
def test_f16_decoding_matches_numpy_for_every_bit_pattern():
    """Catches a wrong exponent bias, subnormal scale or sign handling."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode_bits(bits, "f16")
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_bf16_decoding_matches_torch_for_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode_bits(bits, "bf16")
    want = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


# --------------------------------------------------------------------------
# attention = textbook dense attention over the logical sequence
# --------------------------------------------------------------------------
CASES = [
    # (prefix_lens, new_lens, Hq, Hkv, d, dtype, bs)
    ([0], [7], 2, 2, 64, "f16", 16),  # P = 0: plain causal attention
    ([32], [16], 2, 2, 64, "f16", 16),  # the tiny correctness shape
    ([21, 0, 40], [5, 9, 1], 4, 2, 64, "bf16", 8),  # GQA 2:1, ragged, block 8
    ([33], [19], 8, 2, 96, "f16", 32),  # GQA 4:1, d = 96, block 32
    ([50, 17], [3, 30], 6, 3, 128, "bf16", 16),  # d = 128, partial blocks
]


@pytest.mark.parametrize("P,N,Hq,Hkv,d,dtype,bs", CASES)
def test_oracle_matches_dense_numpy(P, N, Hq, Hkv, d, dtype, bs):
    """Catches a wrong causal offset, GQA head map, scale or lse formula."""
    w = wl.make_random(7, P, N, Hq=Hq, Hkv=Hkv, d=d, dtype=dtype, bs=bs)
    out, lse, bad = run_oracle(w)
    assert bad == 0
    ref_out, ref_lse = dense_reference(w)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_oracle_matches_torch_sdpa_float64():
    """A second library routine: torch SDPA in float64 with an explicit mask."""
    w = wl.make_random(11, [24, 40], [10, 6], Hq=4, Hkv=2, d=64, dtype="bf16", bs=16)
    out, lse, _ = run_oracle(w)
    g = w.num_q_heads // w.num_kv_heads
    qf = torch.from_numpy(wl.bits_to_float32(w.q, w.dtype).astype(np.float64))
    for s in range(w.B):
        n, L = int(w.new_lens[s]), int(w.context_lens[s])
        cu = w.cu_seqlens_q
        K = torch.stack([torch.from_numpy(logical_kv(w, w.k_pool, s, h // g)) for h in range(w.num_q_heads)])
        V = torch.stack([torch.from_numpy(logical_kv(w, w.v_pool, s, h // g)) for h in range(w.num_q_heads)])
        Q = qf[cu[s] : cu[s + 1]].transpose(0, 1)  # [Hq, n, d]
        pos = torch.arange(L - n, L)
        allowed = torch.arange(L)[None, :] <= pos[:, None]
        o = torch.nn.functional.scaled_dot_product_attention(
            Q[None], K[None], V[None], attn_mask=allowed, scale=w.softmax_scale
        )[0]
        rows = (cu[s] + np.arange(n))[:, None] * w.num_q_heads + np.arange(w.num_q_heads)[None, :]
        np.testing.assert_allclose(out[rows.ravel()], o.transpose(0, 1).reshape(-1, w.head_dim).numpy(), atol=1e-12)


def test_brute_force_tiny_config_elementwise():
    """Brute force on the tiny correctness shape: every logit by an explicit
    Python loop over keys (no matrix routine), softmax by its definition."""
    w = wl.tiny_correctness()
    out, lse, _ = run_oracle(w)
    qf = wl.bits_to_float32(w.q, w.dtype).astype(np.float64)
    kf = wl.bits_to_float32(w.k_pool, w.dtype).astype(np.float64)
    vf = wl.bits_to_float32(w.v_pool, w.dtype).astype(np.float64)
    bs = w.block_size
    for t in range(0, w.T, 5):
        for h in range(w.num_q_heads):
            p = 32 + t
            logits = []
            for j in range(p + 1):
                blk = w.block_tables[0, j // bs]
                logits.append(w.softmax_scale * sum(qf[t, h, c] * kf[blk, h, j % bs, c] for c in range(w.head_dim)))
            m = max(logits)
            e = [math.exp(x - m) for x in logits]
            z = sum(e)
            want = np.zeros(w.head_dim)
            for j in range(p + 1):
                blk = w.block_tables[0, j // bs]
                want += e[j] / z * vf[blk, h, j % bs]
            r = t * w.num_q_heads + h
            np.testing.assert_allclose(out[r], want, atol=1e-12)
            assert abs(lse[r] - (m + math.log(z))) < 1e-12


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------
def _set_all_keys(w, kvec_bits):
    kp = w.k_pool.copy()
    kp[w.used_blocks()] = kvec_bits
    return kp


def test_equal_keys_give_mean_of_visible_values():
    """All keys equal: weights are uniform over the p+1 visible keys, so
    o = mean(v_0..v_p) and lse = x + ln(p+1).  Catches a wrong visible count."""
    w = wl.make_random(3, [20], [12], Hq=2, Hkv=1, d=64, dtype="f16", bs=8)
    kvec = wl.round_to_bits(np.linspace(-1, 1, 64, dtype=np.float32), "f16")
    kp = _set_all_keys(w, kvec)
    out, lse, _ = run_oracle(w, k_pool=kp)
    qf = wl.bits_to_float32(w.q, "f16").astype(np.float64)
    kf = wl.bits_to_float32(kvec, "f16").astype(np.float64)
    for t in range(w.T):
        p = 20 + t
        V = logical_kv(w, w.v_pool, 0, 0)[: p + 1]
        for h in range(2):
            r = t * 2 + h
            np.testing.assert_allclose(out[r], V.mean(axis=0), atol=1e-12)
            x = w.softmax_scale * float(qf[t, h] @ kf)
            assert abs(lse[r] - (x + math.log(p + 1))) < 1e-12


def test_single_visible_key_and_decode_of_length_one():
    """P = 0: the first new token sees only itself (o = v_0, lse = x_00).
    Decode with context 1 likewise returns its own value."""
    w = wl.make_random(5, [0, 0], [4, 1], Hq=2, Hkv=2, d=64, dtype="bf16", bs=16)
    out, lse, _ = run_oracle(w)
    qf = wl.bits_to_float32(w.q, "bf16").astype(np.float64)
    for s, t in ((0, 0), (1, 4)):
        for h in range(2):
            K = logical_kv(w, w.k_pool, s, h)
            V = logical_kv(w, w.v_pool, s, h)
            r = t * 2 + h
            np.testing.assert_array_equal(out[r], V[0])
            assert abs(lse[r] - w.softmax_scale * float(qf[t, h] @ K[0])) < 1e-12
    # decode entry: one query per sequence
    o2, l2, _ = oracle.decode_attn("bf16", w.k_pool, w.v_pool, w.q[[0, 4]], [1, 1], w.block_tables, w.softmax_scale)
    np.testing.assert_array_equal(o2, out[[0, 1, 8, 9]])
    np.testing.assert_array_equal(l2, lse[[0, 1, 8, 9]])


def test_constant_values_give_that_constant():
    w = wl.make_random(9, [37], [9], Hq=4, Hkv=2, d=96, dtype="f16", bs=16)
    vp = w.v_pool.copy()
    c = wl.round_to_bits(np.full(96, 0.375, dtype=np.float32), "f16")
    vp[w.used_blocks()] = c
    out, _, _ = run_oracle(w, v_pool=vp)
    np.testing.assert_allclose(out, 0.375, atol=1e-15)


def test_two_keys_worked_by_hand():
    """q = e_0, k_0 = e_0, k_1 = 0, scale 1: logits (1, 0) for the second
    query, so o = (e v_0 + v_1)/(e + 1) and lse = ln(e + 1)."""
    w = wl.make_random(13, [0], [2], Hq=1, Hkv=1, d=64, dtype="f16", bs=16, scale=1.0)
    e0 = np.zeros(64, dtype=np.float32)
    e0[0] = 1.0
    q = w.q.copy()
    q[:, 0] = wl.round_to_bits(e0, "f16")
    kp = w.k_pool.copy()
    blk = w.block_tables[0, 0]
    kp[blk, 0, 0] = wl.round_to_bits(e0, "f16")
    kp[blk, 0, 1] = wl.round_to_bits(np.zeros(64, dtype=np.float32), "f16")
    w.q = q
    out, lse, _ = run_oracle(w, k_pool=kp)
    v0 = wl.bits_to_float32(w.v_pool[blk, 0, 0], "f16").astype(np.float64)
    v1 = wl.bits_to_float32(w.v_pool[blk, 0, 1], "f16").astype(np.float64)
    e = math.e
    np.testing.assert_allclose(out[1], (e * v0 + v1) / (e + 1), atol=1e-13)
    assert abs(lse[1] - math.log(e + 1)) < 1e-13
    np.testing.assert_array_equal(out[0], v0)  # first query sees only k_0
    assert abs(lse[0] - 1.0) < 1e-13


# --------------------------------------------------------------------------
# paging invariants
# --------------------------------------------------------------------------
def test_prefix_from_cache_plus_chunk_equals_full_sequence():
    """(P cached, N new) rows equal the last N rows of (0 cached, P+N new)
    over the same blocks.  Catches a causal window anchored at the chunk
    start instead of its absolute position."""
    w = wl.make_random(17, [45, 64], [19, 8], Hq=4, Hkv=4, d=64, dtype="bf16", bs=16)
    out, lse, _ = run_oracle(w)
    full = wl.Workload(**{**w.__dict__})
    full.prefix_lens = np.zeros(2, dtype=np.int32)
    full.new_lens = w.context_lens.copy()
    qf = []
    # give the full-sequence run queries whose last N rows are the chunk's
    rng = np.random.default_rng(0)
    for s in range(w.B):
        lead = wl.round_to_bits(rng.standard_normal((int(w.prefix_lens[s]), 4, 64), dtype=np.float32), "bf16")
        qf.append(np.concatenate([lead, w.q[w.cu_seqlens_q[s] : w.cu_seqlens_q[s + 1]]]))
    full.q = np.concatenate(qf)
    o2, l2, _ = run_oracle(full)
    for s in range(w.B):
        n = int(w.new_lens[s])
        a = np.arange(w.cu_seqlens_q[s], w.cu_seqlens_q[s + 1])
        b = np.arange(full.cu_seqlens_q[s + 1] - n, full.cu_seqlens_q[s + 1])
        ra = (a[:, None] * 4 + np.arange(4)).ravel()
        rb = (b[:, None] * 4 + np.arange(4)).ravel()
        np.testing.assert_array_equal(out[ra], o2[rb])
        np.testing.assert_array_equal(lse[ra], l2[rb])


def test_physical_placement_permutation_is_invisible():
    w = wl.make_random(19, [70, 33, 0], [5, 20, 11], Hq=4, Hkv=2, d=64, dtype="f16", bs=16, num_blocks=64)
    w2 = wl.permute_placement(w, 99)
    assert not np.array_equal(w.block_tables, w2.block_tables)
    o1, l1, _ = run_oracle(w)
    o2, l2, _ = run_oracle(w2)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_duplicate_physical_blocks_in_one_table():
    """A table naming the same block twice reads it twice (chunk reuse with
    replacement); the dense reference sees the same logical sequence."""
    w = wl.rag_chunk_reuse(B=2, library=3, chunk=32, chunks_per_request=4, new_lo=5, new_hi=20, num_blocks=64)
    dup = any(len(set(r[r >= 0])) < (r >= 0).sum() for r in w.block_tables)
    assert dup
    out, lse, _ = run_oracle(w)
    ref, rlse = dense_reference(w)
    np.testing.assert_allclose(out, ref, atol=1e-12)
    np.testing.assert_allclose(lse, rlse, atol=1e-12)


# --------------------------------------------------------------------------
# split-KV merge identity
# --------------------------------------------------------------------------
def test_merge_of_dense_partials_equals_full_softmax():
    """Partials over disjoint key ranges (numpy), merged by the oracle, equal
    the unsplit result; an empty range (lse = -inf) contributes nothing."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal(300) * 3
    V = rng.standard_normal((300, 32))
    cuts = [0, 17, 17, 150, 299, 300]
    parts_o, parts_l = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        if a == b:
            parts_o.append(np.zeros(32))
            parts_l.append(-np.inf)
            continue
        m = x[a:b].max()
        e = np.exp(x[a:b] - m)
        parts_o.append(e @ V[a:b] / e.sum())
        parts_l.append(m + np.log(e.sum()))
    o, l = oracle.lse_merge(np.array(parts_o), np.array(parts_l))
    m = x.max()
    e = np.exp(x - m)
    np.testing.assert_allclose(o, e @ V / e.sum(), atol=1e-13)
    assert abs(l - (m + np.log(e.sum()))) < 1e-13


# --------------------------------------------------------------------------
# slot mapping, append, copy-on-write
# --------------------------------------------------------------------------
def _read_chunking_golden():
    vals = {}
    with open(os.path.join(GOLDEN, "chunking_example.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                vals[k] = int(v)
    return vals


def test_slot_mapping_reproduces_pages_chunking_example():
    """kvboost 'How it works' > Chunking: 1000 tokens at 128 per chunk are
    7 full chunks plus a 104-token tail."""
    g = _read_chunking_golden()
    bs, n = g["block_size"], g["tokens"]
    table = np.arange(16, dtype=np.int32)[None, :]
    slots, bad = oracle.slot_mapping([0, n], [n], table, bs, 16)
    assert bad == 0
    counts = np.bincount(slots // bs)
    assert (counts == bs).sum() == g["full_blocks"]
    assert counts[-1] == g["tail_tokens"] and len(counts) == g["full_blocks"] + 1


def test_slot_mapping_round_trips_through_the_block_table():
    """Append by the oracle's slots, then gather the logical sequence by
    numpy indexing: positions P..L-1 must hold the new tokens in order."""
    w = wl.make_random(23, [13, 0, 48], [21, 3, 16], Hq=2, Hkv=2, d=64, dtype="f16", bs=8)
    slots, bad = oracle.slot_mapping(w.cu_seqlens_q, w.context_lens, w.block_tables, w.block_size, w.num_blocks)
    assert bad == 0
    assert len(np.unique(slots)) == len(slots)
    kp, vp, bad = oracle.cache_append(w.k_pool, w.v_pool, w.k_new, w.v_new, slots)
    assert bad == 0
    for s in range(w.B):
        for h in range(2):
            K = logical_kv(w, kp, s, h)
            V = logical_kv(w, vp, s, h)
            a, b = w.cu_seqlens_q[s], w.cu_seqlens_q[s + 1]
            np.testing.assert_array_equal(K[w.prefix_lens[s] :], wl.bits_to_float32(w.k_new[a:b, h], "f16"))
            np.testing.assert_array_equal(V[w.prefix_lens[s] :], wl.bits_to_float32(w.v_new[a:b, h], "f16"))
            # the cached prefix is untouched
            np.testing.assert_array_equal(K[: w.prefix_lens[s]], logical_kv(w, w.k_pool, s, h)[: w.prefix_lens[s]])


def test_slot_mapping_flags_invalid_table_entries():
    bt = np.array([[0, -1, 3], [2, 99, 1]], dtype=np.int32)
    slots, bad = oracle.slot_mapping([0, 4, 8], [20, 24], bt, 8, 16)
    # seq 0: positions 16..19 -> logical block 2 -> block 3
    assert list(slots[:4]) == [24, 25, 26, 27]
    # seq 1: positions 20..23 -> logical block 2 -> block 1 (valid)
    assert list(slots[4:]) == [12, 13, 14, 15]
    slots, bad = oracle.slot_mapping([0, 2], [10], bt[:1], 8, 16)  # positions 8,9 -> entry -1
    assert bad == 2 and list(slots) == [-1, -1]


def test_append_skips_minus_one_and_changes_nothing_else():
    w = wl.make_random(29, [10], [6], Hq=2, Hkv=2, d=64, dtype="bf16", bs=16)
    slots, _ = oracle.slot_mapping(w.cu_seqlens_q, w.context_lens, w.block_tables, 16, w.num_blocks)
    slots[2] = -1
    kp, vp, bad = oracle.cache_append(w.k_pool, w.v_pool, w.k_new, w.v_new, slots)
    assert bad == 0
    changed = np.argwhere(np.any(kp != w.k_pool, axis=-1))
    written = {(int(s // 16), h, int(s % 16)) for s in slots if s >= 0 for h in range(2)}
    assert {tuple(int(x) for x in c) for c in changed} <= written
    blk, row = divmod(int(slots[3]), 16)
    np.testing.assert_array_equal(kp[blk, 1, row], w.k_new[3, 1])
    # an out-of-range slot is skipped and counted, never written
    _, _, bad = oracle.cache_append(w.k_pool, w.v_pool, w.k_new[:1], w.v_new[:1], np.array([w.num_blocks * 16]))
    assert bad == 1


def test_copy_on_write_fork_leaves_shared_blocks_and_parent_unchanged():
    """kvstream 'Request lifecycle' 3: a forked table shares pages; the one
    partial page about to be written is copied first.  After copy + append
    into both children, every shared block is byte-identical and the
    parent's attention equals its attention computed without the child."""
    w = wl.continuous_batching_step(n_decode=4, n_prefill=0, n_forks=2, median=60, sigma=0.3, ctx_lo=20,
                                    ctx_hi=100, num_blocks=64, Hq=4, Hkv=2, d=64)
    assert w.cow_pairs.shape == (2, 2)
    shared = np.intersect1d(w.block_tables[0][w.block_tables[0] >= 0], w.block_tables[1][w.block_tables[1] >= 0])
    before_k, before_v = w.k_pool[shared].copy(), w.v_pool[shared].copy()
    res = oracle.run_step(w)
    assert res["bad"] == 0
    np.testing.assert_array_equal(res["k_pool"][shared], before_k)
    np.testing.assert_array_equal(res["v_pool"][shared], before_v)
    src, dst = w.cow_pairs[0]
    # the copy equals the source on every row written before the fork
    c = int(w.prefix_lens[0]) % w.block_size
    assert c > 0
    np.testing.assert_array_equal(res["k_pool"][dst, :, :c], w.k_pool[src, :, :c])
    np.testing.assert_array_equal(res["k_pool"][src, :, :c], w.k_pool[src, :, :c])
    # each child's new token went to its own block
    np.testing.assert_array_equal(res["k_pool"][src, :, c], w.k_new[0])
    np.testing.assert_array_equal(res["k_pool"][dst, :, c], w.k_new[1])
    # the parent's output equals a world in which the child never forked
    slots, _ = oracle.slot_mapping([0, 1], w.context_lens[:1], w.block_tables[:1], w.block_size, w.num_blocks)
    kp, vp, _ = oracle.cache_append(w.k_pool, w.v_pool, w.k_new[:1], w.v_new[:1], slots)
    solo, solo_lse, _ = oracle.decode_attn(w.dtype, kp, vp, w.q[:1], w.context_lens[:1], w.block_tables[:1],
                                           w.softmax_scale)
    np.testing.assert_array_equal(solo, res["decode_out"][:4])
    np.testing.assert_array_equal(solo_lse, res["decode_lse"][:4])


def test_block_copy_copies_exactly_the_pairs():
    w = wl.make_random(31, [40], [8], Hq=2, Hkv=2, d=64, dtype="f16", bs=16, num_blocks=16, fill_all_blocks=True)
    pairs = np.array([[1, 5], [7, 2]], dtype=np.int32)
    kp, vp, bad = oracle.block_copy(w.k_pool, w.v_pool, pairs)
    assert bad == 0
    np.testing.assert_array_equal(kp[5], w.k_pool[1])
    np.testing.assert_array_equal(vp[2], w.v_pool[7])
    others = [b for b in range(16) if b not in (5, 2)]
    np.testing.assert_array_equal(kp[others], w.k_pool[others])
    _, _, bad = oracle.block_copy(w.k_pool, w.v_pool, np.array([[0, 16]], dtype=np.int32))
    assert bad == 1


def test_block_swap_moves_blocks_between_pools_and_round_trips():
    """Swap out then back in to other blocks: the device blocks come back
    byte-identical, untouched blocks of both pools are unchanged, and a pair
    outside either pool is skipped and counted."""
    w = wl.make_random(32, [70], [9], Hq=4, Hkv=2, d=64, dtype="bf16", bs=16, num_blocks=12, fill_all_blocks=True)
    rng = np.random.default_rng(5)
    host_k = rng.integers(0, 1 << 16, size=(6,) + w.k_pool.shape[1:], dtype=np.uint16)
    host_v = rng.integers(0, 1 << 16, size=host_k.shape, dtype=np.uint16)
    out = np.array([[3, 0], [7, 4], [11, 5]], dtype=np.int32)
    hk, hv, bad = oracle.block_swap(w.k_pool, w.v_pool, host_k, host_v, out)
    assert bad == 0
    for src, dst in out:
        np.testing.assert_array_equal(hk[dst], w.k_pool[src])
        np.testing.assert_array_equal(hv[dst], w.v_pool[src])
    np.testing.assert_array_equal(hk[[1, 2, 3]], host_k[[1, 2, 3]])
    back = np.array([[0, 1], [4, 2], [5, 9]], dtype=np.int32)
    dk, dv, bad = oracle.block_swap(hk, hv, w.k_pool, w.v_pool, back)
    assert bad == 0
    np.testing.assert_array_equal(dk[[1, 2, 9]], w.k_pool[[3, 7, 11]])
    np.testing.assert_array_equal(dv[[1, 2, 9]], w.v_pool[[3, 7, 11]])
    keep = [b for b in range(12) if b not in (1, 2, 9)]
    np.testing.assert_array_equal(dk[keep], w.k_pool[keep])
    _, _, bad = oracle.block_swap(w.k_pool, w.v_pool, host_k, host_v, np.array([[12, 0], [0, 6], [-1, 1]]))
    assert bad == 3


def test_pool_page_size_matches_the_pages_formula():
    """kvstream.yaml: one page = block_size x heads x head_dim x 2 x dtype_bytes."""
    vals = {}
    with open(os.path.join(GOLDEN, "page_geometry.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, *v = line.split()
                vals[k] = [int(x) for x in v]
    w = wl.shared_system_prompt(B=1, prefix=32, new=16, num_blocks=vals["pool_blocks_example"][0])
    assert w.block_size == vals["block_size"][0] and w.block_size in vals["allowed_block_sizes"]
    page = (w.k_pool[0].nbytes + w.v_pool[0].nbytes)
    assert page == w.block_size * w.num_kv_heads * w.head_dim * 2 * vals["dtype_bytes"][0]
    assert w.k_pool.shape[0] == vals["pool_blocks_example"][0]
