"""GPU parity of CacheBlend recompute selection against the oracle
(oracle/cacheblend.py): deviations within 1e-5 of fp64; the selection, an
integer decision, bit-exact against the oracle's selection applied to the
same fp32 deviations (ties to the lower position); the overwrite bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from oracle import cacheblend as cb

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    from paged_prefix_reuse_gb300 import build

    build.build_library()
    import paged_prefix_reuse_gb300 as kvp

    kvp.load_library()


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _dev(a, dtype):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    return torch.from_numpy(a.view(np.int16)).view(tdt).cuda()


@pytest.mark.parametrize("dtype,d,hkv", [("bf16", 128, 8), ("f16", 96, 4), ("bf16", 64, 2)])
def test_deviation_select_overwrite_match_oracle(dtype, d, hkv):
    import paged_prefix_reuse_gb300 as kvp

    rng = np.random.default_rng(d + hkv)
    lens = [0, 1, 7, 20, 21, 300, 1500]
    T = sum(lens)
    nb, bs = (T + 15) // 16 + 8, 16
    kp = wl.round_to_bits(rng.standard_normal((nb, hkv, bs, d)).astype(np.float32), dtype)
    vp = wl.round_to_bits(rng.standard_normal((nb, hkv, bs, d)).astype(np.float32), dtype)
    slots = rng.permutation(nb * bs)[:T].astype(np.int64)
    Kc = oracle.decode_bits(kp, dtype)[slots // bs, :, slots % bs]  # cached K [T, hkv, d]
    Vc = oracle.decode_bits(vp, dtype)[slots // bs, :, slots % bs]
    noise = rng.uniform(0, 1.5, size=(T, 1, 1))  # per-token perturbation strength
    Kf = (Kc + noise * rng.standard_normal(Kc.shape)).astype(np.float32)
    Vf = (Vc + noise * rng.standard_normal(Vc.shape)).astype(np.float32)
    Kf[0], Vf[0] = Kc[0], Vc[0]          # identical -> 0
    Kf[1], Vf[1] = -Kc[1], -Vc[1]        # negated -> 2
    Kf[2], Vf[2] = 0, 0                  # fresh zero -> 1
    Kf[40:60], Vf[40:60] = Kc[40:60], Vc[40:60]  # a run of exact ties at 0
    kf, vf = wl.round_to_bits(Kf, dtype), wl.round_to_bits(Vf, dtype)
    pool = kvp.PagedKVPool(_dev(kp, dtype), _dev(vp, dtype))
    ts = torch.from_numpy(slots).cuda()
    dev = kvp.kvp_kv_deviation(pool, _dev(kf, dtype), _dev(vf, dtype), ts)
    torch.cuda.synchronize()
    assert pool.errors() == 0
    g = dev.cpu().numpy()
    want = cb.kv_deviation(dtype, kp, vp, kf, vf, slots)
    assert np.abs(g - want).max() <= 1e-5
    assert g[0] == 0.0 and abs(g[1] - 2.0) < 1e-6 and g[2] == 1.0

    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    for permille in (0, 150, 400, 1000):
        rs, counts = kvp.kvp_select_recompute(dev, ts, torch.from_numpy(cu).cuda(), permille)
        torch.cuda.synchronize()
        mask, want_counts = cb.select_recompute(g.astype(np.float64), cu, permille)
        np.testing.assert_array_equal(counts.cpu().numpy(), want_counts)
        np.testing.assert_array_equal(rs.cpu().numpy(), np.where(mask, slots, -1))

    # overwrite the ~15% selected tokens' entries with their fresh K/V
    rs, counts = kvp.kvp_select_recompute(dev, ts, torch.from_numpy(cu).cuda(), 150)
    kvp.kvp_cache_append(pool, _dev(kf, dtype), _dev(vf, dtype), rs)
    torch.cuda.synchronize()
    assert pool.errors() == 0
    want_k, want_v, bad = oracle.cache_append(kp, vp, kf, vf, rs.cpu().numpy())
    assert bad == 0
    np.testing.assert_array_equal(_bits(pool.k), want_k)
    np.testing.assert_array_equal(_bits(pool.v), want_v)


def test_selection_on_a_long_sequence_with_ties():
    """One 200 000-token sequence (many 1024-wide scan tiles) whose deviations
    take only 50 distinct values: the threshold falls inside a huge tie."""
    import paged_prefix_reuse_gb300 as kvp

    rng = np.random.default_rng(1)
    n = 200_000
    g = rng.integers(0, 50, size=n).astype(np.float32) / 25.0
    slots = np.arange(n, dtype=np.int64) * 3
    cu = np.array([0, n], dtype=np.int32)
    for permille in (1, 150, 999):
        rs, counts = kvp.kvp_select_recompute(torch.from_numpy(g).cuda(), torch.from_numpy(slots).cuda(),
                                              torch.from_numpy(cu).cuda(), permille)
        torch.cuda.synchronize()
        mask, want = cb.select_recompute(g.astype(np.float64), cu, permille)
        assert counts.item() == want[0]
        np.testing.assert_array_equal(rs.cpu().numpy(), np.where(mask, slots, -1))


def test_bad_slot_is_flagged():
    import paged_prefix_reuse_gb300 as kvp

    pool = kvp.PagedKVPool.allocate(4, 2, 16, 64, dtype=torch.float16)
    pool.k.zero_()
    pool.v.zero_()
    f = torch.zeros((2, 2, 64), dtype=torch.float16, device="cuda")
    dev = kvp.kvp_kv_deviation(pool, f, f, torch.tensor([3, 64], dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert pool.errors() & kvp.DEVERR["bad_slot"]
    assert dev.cpu().tolist() == [0.0, -1.0]
