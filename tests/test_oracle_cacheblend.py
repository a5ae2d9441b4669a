"""Pins of the CacheBlend oracle (oracle/cacheblend.py): closed-form
deviations and a selection worked by hand."""
import numpy as np

import workloads as wl
from oracle import cacheblend as cb


def _pool_with(vectors_k, vectors_v, dtype="f16"):
    """A pool whose slot t (block t // 16, row t % 16) holds the given K and V."""
    T = len(vectors_k)
    hkv, d = vectors_k[0].shape
    kp = np.zeros(((T + 15) // 16, hkv, 16, d), np.float32)
    vp = np.zeros_like(kp)
    for t in range(T):
        kp[t // 16, :, t % 16] = vectors_k[t]
        vp[t // 16, :, t % 16] = vectors_v[t]
    return wl.round_to_bits(kp, dtype), wl.round_to_bits(vp, dtype)


def test_closed_form_deviations():
    rng = np.random.default_rng(0)
    k = [rng.integers(-4, 5, size=(2, 8)).astype(np.float32) for _ in range(6)]
    v = [rng.integers(-4, 5, size=(2, 8)).astype(np.float32) for _ in range(6)]
    kf = np.stack([k[0], -k[1], 2 * k[2], k[3], np.zeros((2, 8)), np.zeros((2, 8))]).astype(np.float32)
    vf = np.stack([v[0], -v[1], 2 * v[2], v[3], np.zeros((2, 8)), np.zeros((2, 8))]).astype(np.float32)
    # token 3: fresh V made orthogonal to [K;V] cached by construction below
    k[3] = np.zeros((2, 8), np.float32)
    v[3] = np.zeros((2, 8), np.float32)
    v[3][0, 0] = 1.0
    kf[3] = 0
    vf[3] = 0
    vf[3][0, 1] = 3.0
    k[5] = np.zeros((2, 8), np.float32)
    v[5] = np.zeros((2, 8), np.float32)
    kp, vp = _pool_with(k, v)
    dev = cb.kv_deviation("f16", kp, vp, wl.round_to_bits(kf, "f16"), wl.round_to_bits(vf, "f16"), np.arange(6))
    np.testing.assert_allclose(dev, [0.0, 2.0, 0.0, 1.0, 1.0, 0.0], atol=1e-12)


def test_selection_worked_example_and_ties():
    # n = 5, 400 per mille: k = ceil(2.0) = 2; the two 0.5s, by position
    mask, cnt = cb.select_recompute([0.1, 0.5, 0.3, 0.5, 0.0], [0, 5], permille=400)
    assert cnt.tolist() == [2] and np.flatnonzero(mask).tolist() == [1, 3]
    # ties beyond k: the lower positions win
    mask, cnt = cb.select_recompute([0.2] * 7, [0, 7], permille=300)
    assert cnt.tolist() == [3] and np.flatnonzero(mask).tolist() == [0, 1, 2]
    # the pages' ~15%: 20 tokens -> 3 (0.15 * 20 is 3.0000000000000004 in floating point),
    # 21 -> 4, 1 -> 1, 0 -> 0; sequences are independent
    dev = np.arange(42, dtype=float)[::-1].copy()
    mask, cnt = cb.select_recompute(dev, [0, 20, 41, 42, 42])
    assert cnt.tolist() == [3, 4, 1, 0]
    assert np.flatnonzero(mask).tolist() == [0, 1, 2, 20, 21, 22, 23, 41]


def test_deviation_identities_on_random_vectors():
    """1 - cos(a, b) = |a/|a| - b/|b||^2 / 2, symmetric in (cached, fresh) and
    unchanged by positive scaling of either side (checked on values that the
    16-bit format holds exactly)."""
    rng = np.random.default_rng(3)
    T, hkv, d = 40, 2, 16
    k = [rng.integers(-6, 7, size=(hkv, d)).astype(np.float32) for _ in range(T)]
    v = [rng.integers(-6, 7, size=(hkv, d)).astype(np.float32) for _ in range(T)]
    kf = rng.integers(-6, 7, size=(T, hkv, d)).astype(np.float32)
    vf = rng.integers(-6, 7, size=(T, hkv, d)).astype(np.float32)
    kp, vp = _pool_with(k, v)
    dev = cb.kv_deviation("f16", kp, vp, wl.round_to_bits(kf, "f16"), wl.round_to_bits(vf, "f16"), np.arange(T))
    for t in range(T):
        a = np.concatenate([k[t].ravel(), v[t].ravel()]).astype(np.float64)
        b = np.concatenate([kf[t].ravel(), vf[t].ravel()]).astype(np.float64)
        half_sq = 0.5 * np.sum((a / np.linalg.norm(a) - b / np.linalg.norm(b)) ** 2)
        assert abs(dev[t] - half_sq) < 1e-12
    # swap the roles of cached and fresh: same deviations
    kp2, vp2 = _pool_with(list(kf), list(vf))
    dev2 = cb.kv_deviation("f16", kp2, vp2, wl.round_to_bits(np.stack(k), "f16"),
                           wl.round_to_bits(np.stack(v), "f16"), np.arange(T))
    np.testing.assert_allclose(dev2, dev, atol=1e-12)
    # scale the fresh side by 4 (exact in fp16 for these integers): same deviations
    dev4 = cb.kv_deviation("f16", kp, vp, wl.round_to_bits(4 * kf, "f16"), wl.round_to_bits(4 * vf, "f16"),
                           np.arange(T))
    np.testing.assert_allclose(dev4, dev, atol=1e-12)


def test_selection_properties_on_random_inputs_with_ties():
    """Per sequence: exactly ceil(n * permille / 1000) tokens; every selected
    deviation >= every unselected one; among tokens at the threshold value
    the selected ones are the lowest positions."""
    rng = np.random.default_rng(4)
    lens = rng.integers(0, 60, size=12)
    cu = np.concatenate([[0], np.cumsum(lens)])
    dev = rng.integers(0, 6, size=int(cu[-1])) / 4.0  # few distinct values: many ties
    for permille in (0, 1, 150, 333, 999, 1000):
        mask, cnt = cb.select_recompute(dev, cu, permille=permille)
        for s in range(len(lens)):
            a, b = int(cu[s]), int(cu[s + 1])
            n = b - a
            k = -(-n * permille // 1000)
            sel = np.flatnonzero(mask[a:b])
            assert cnt[s] == k == len(sel)
            if 0 < k < n:
                unsel = np.setdiff1d(np.arange(n), sel)
                d = dev[a:b]
                assert d[sel].min() >= d[unsel].max()
                thr = d[sel].min()
                at_thr = np.flatnonzero(d == thr)
                chosen = np.intersect1d(sel, at_thr)
                assert chosen.tolist() == at_thr[: len(chosen)].tolist()
