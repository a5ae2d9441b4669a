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
