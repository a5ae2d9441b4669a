"""The benchmark's algorithmic work counts, which every reported rate
divides by: the FLOP convention 4 * d * Hq * sum_s (N_s * P_s + N_s (N_s + 1) / 2)
of the prefill, checked against a count of the visible (query, key) pairs
and against the shared-prompt batch's value worked by hand; the decode's
unique K/V bytes against a per-sequence sum."""
import numpy as np
import pytest

import bench
import workloads as wl


def _visible_pairs(w):
    """Brute force: for every prefill query row, the keys it attends to."""
    total = 0
    for s in range(w.num_prefill):
        P = int(w.prefix_lens[s])
        for i in range(int(w.new_lens[s])):
            total += P + i + 1  # keys 0 .. P + i
    return total * w.num_q_heads


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_prefill_flops_is_four_d_per_visible_pair(seed):
    rng = np.random.default_rng(seed)
    n = rng.integers(0, 40, size=5)
    p = rng.integers(0, 200, size=5)
    w = wl.make_random(seed, p, n, Hq=6, Hkv=2, d=64, dtype="f16")
    # q.k and p.v each take d multiply-adds (2 d FLOP) per visible pair
    assert bench.prefill_flops(w) == 4 * w.head_dim * _visible_pairs(w)
    # the per-row form used for the CPU baseline's samples sums to the same
    rows = np.arange(int(w.cu_seqlens_q[w.num_prefill]) * w.num_q_heads)
    assert bench.row_flops(w, rows) == pytest.approx(bench.prefill_flops(w), rel=0, abs=0.5)


def test_shared_prompt_batch_flops_by_hand():
    # 8 requests x 16 query heads x d 128, prefix 1024, 256 new tokens each
    w = wl.make_config(2)
    by_hand = 4 * 128 * 16 * 8 * (256 * 1024 + 256 * 257 // 2)
    assert by_hand == 65_536 * 295_040 == 19_335_741_440
    assert bench.prefill_flops(w) == by_hand


def test_decode_bytes_are_each_contexts_k_and_v_once():
    w = wl.make_config(4)
    ctx = w.context_lens[w.num_prefill :]
    per_seq = [int(L) * w.num_kv_heads * w.head_dim * 2 * 2 for L in ctx]
    assert bench.decode_kv_bytes(w) == sum(per_seq)
    assert 600e6 < bench.decode_kv_bytes(w) < 700e6  # the mixed batch's ~643 MB


def test_long_context_batch_flops_by_hand():
    # 4 requests x 64 query heads x d 128, prefix 32768, 2048 new tokens each
    w = wl.make_config(5)
    by_hand = 4 * 128 * 64 * 4 * (2048 * 32768 + 2048 * 2049 // 2)
    assert by_hand == 9_071_105_146_880
    assert bench.prefill_flops(w) == by_hand
