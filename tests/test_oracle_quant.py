"""Pins of the quantized-pool oracle (oracle/quant.py) against things other
than itself: a worked example derived by hand, closed-form error bounds, the
orientation of the groups, the nibble order, and exactness on inputs that lie
on the quantization grid (where quantized decode must equal 16-bit decode)."""
import os

import numpy as np
import pytest

import oracle
import workloads as wl
from oracle import quant

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden():
    vals = {}
    with open(os.path.join(GOLDEN, "quant_example.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = [float(t) for t in v.split()]
    return vals


@pytest.mark.parametrize("bits", [8, 4])
def test_worked_example(bits):
    g = _golden()
    x = np.array(g["values"], dtype=np.float32)
    codes, s, z = quant.quantize_groups(x[None, :], bits, axis=1)
    assert float(s[0]) == g[f"int{bits}_scale"][0]
    assert float(z[0]) == g[f"int{bits}_min"][0]
    np.testing.assert_array_equal(codes[0], np.array(g[f"int{bits}_codes"], dtype=np.uint8))
    deq = codes[0].astype(np.float64) * float(s[0]) + float(z[0])
    np.testing.assert_array_equal(deq, np.array(g[f"int{bits}_dequant"]))
    if bits == 4:
        np.testing.assert_array_equal(quant.pack_codes(codes, 4)[0], np.array(g["int4_packed"], dtype=np.uint8))


def test_directed_fp16_rounding():
    x = np.array([4 / 255, -1 / 3, 1e-8, 70000.0, -70000.0, 0.0], dtype=np.float32)
    up = quant.f16_directed(x, True).astype(np.float64)
    dn = quant.f16_directed(x, False).astype(np.float64)
    assert np.all(up[:3] >= x[:3]) and np.all(dn[:3] <= x[:3])
    assert up[3] == np.inf and dn[4] == -np.inf and up[5] == 0 and dn[5] == 0
    assert np.all(np.nextafter(dn[:3].astype(np.float16), np.float16(np.inf)).astype(np.float64) >= x[:3])


@pytest.mark.parametrize("bits", [8, 4])
def test_error_bound_and_group_orientation(bits):
    """K is grouped per channel over tokens and V per token over channels:
    every element reconstructs within s/2 + (min - z) of its own group.  The
    page mixes channels (and tokens) of wildly different ranges, so grouping
    along the wrong axis breaks the bound by orders of magnitude."""
    rng = np.random.default_rng(bits)
    Hkv, bs, d = 2, 16, 64
    chan_scale = np.geomspace(1e-3, 1e2, d).astype(np.float32)
    tok_scale = np.geomspace(1e-3, 1e2, bs).astype(np.float32)
    Kf = (rng.standard_normal((Hkv, bs, d)) * chan_scale).astype(np.float32)
    Vf = (rng.standard_normal((Hkv, bs, d)) * tok_scale[:, None]).astype(np.float32)
    kbits = wl.round_to_bits(Kf, "f16")
    vbits = wl.round_to_bits(Vf, "f16")
    qp = quant.empty_qpool(3, Hkv, bs, d, bits)
    qp, bad = quant.quantize_blocks("f16", kbits[None], vbits[None], qp, bits, [[0, 2]])
    assert bad == 0
    K = oracle.decode_bits(kbits, "f16")
    V = oracle.decode_bits(vbits, "f16")
    Kd, Vd = quant.dequantize_block(qp, bits, 2, d)
    ks = qp[2][2, :, 0, :].astype(np.float64)[:, None, :]
    kz = qp[2][2, :, 1, :].astype(np.float64)[:, None, :]
    kmin = K.min(axis=1, keepdims=True)
    assert np.all(np.abs(Kd - K) <= ks / 2 + (kmin - kz) + 1e-12 * np.abs(K))
    vs = qp[3][2, :, :, 0].astype(np.float64)[:, :, None]
    vz = qp[3][2, :, :, 1].astype(np.float64)[:, :, None]
    vmin = V.min(axis=2, keepdims=True)
    assert np.all(np.abs(Vd - V) <= vs / 2 + (vmin - vz) + 1e-12 * np.abs(V))
    # the smallest-range channel of K stays within a step of its own range
    # (grouped per token instead, its error would be ~1e5 times larger)
    rng0 = (K[:, :, 0].max(axis=1) - K[:, :, 0].min(axis=1)).max()
    assert np.abs(Kd - K)[:, :, 0].max() <= rng0 / quant.LEVELS[bits]
    # untouched blocks stay zero
    assert not qp[0][[0, 1]].any() and not qp[2][[0, 1]].any()


def test_constant_group_and_codes_range():
    x = np.full((1, 16), 0.375, dtype=np.float32)
    codes, s, z = quant.quantize_groups(x, 8, axis=1)
    assert float(s[0]) == 0.0 and float(z[0]) == 0.375 and not codes.any()
    rng = np.random.default_rng(3)
    y = rng.standard_normal((5, 33)).astype(np.float32) * 7
    for bits in (8, 4):
        codes, s, z = quant.quantize_groups(y, bits, axis=1)
        assert codes.max() <= quant.LEVELS[bits] and codes.min() == 0
        assert np.all(codes.max(axis=1) >= quant.LEVELS[bits] - 1)


def test_int4_nibble_order_round_trip():
    rng = np.random.default_rng(4)
    c = rng.integers(0, 16, size=(3, 5, 64), dtype=np.uint8)
    p = quant.pack_codes(c, 4)
    assert p.shape == (3, 5, 32)
    np.testing.assert_array_equal(p[..., 0], c[..., 0] | (c[..., 1] << 4))
    np.testing.assert_array_equal(quant.unpack_codes(p, 4, 64), c)


def _grid_pool(rng, nb, Hkv, bs, d, bits):
    """A bf16 pool whose every K channel (per page, head) and every V token
    lies exactly on a quantization grid with power-of-two step and fp16/bf16
    exact min, with both ends of the code range present: quantize-dequantize
    is then exact."""
    levels = quant.LEVELS[bits]
    step = 2.0 ** -4 if bits == 8 else 0.5
    lo = -8.0 if bits == 8 else -4.0
    kc = rng.integers(0, levels + 1, size=(nb, Hkv, bs, d))
    kc[:, :, 0, :] = 0
    kc[:, :, 1, :] = levels
    vc = rng.integers(0, levels + 1, size=(nb, Hkv, bs, d))
    vc[:, :, :, 0] = 0
    vc[:, :, :, 1] = levels
    K = (lo + kc * step).astype(np.float32)
    V = (lo + vc * step).astype(np.float32)
    return wl.round_to_bits(K, "bf16"), wl.round_to_bits(V, "bf16"), K, V


@pytest.mark.parametrize("bits", [8, 4])
def test_quantized_decode_is_exact_on_grid_inputs(bits):
    """On grid inputs dequant(quant(x)) == x, so decode over the quantized
    pool must equal the 16-bit decode oracle (a different implementation,
    C fp64) on the original pool, whichever pages are read quantized."""
    rng = np.random.default_rng(10 + bits)
    nb, Hkv, bs, d, Hq, B = 24, 2, 16, 64, 6, 3
    kb, vb, K, V = _grid_pool(rng, nb, Hkv, bs, d, bits)
    np.testing.assert_array_equal(oracle.decode_bits(kb, "bf16"), K)
    qp = quant.empty_qpool(nb, Hkv, bs, d, bits)
    qp, bad = quant.quantize_blocks("bf16", kb, vb, qp, bits, np.stack([np.arange(nb)] * 2, 1))
    assert bad == 0
    for blk in (0, 7, 23):
        Kd, Vd = quant.dequantize_block(qp, bits, blk, d)
        np.testing.assert_array_equal(Kd, K[blk])
        np.testing.assert_array_equal(Vd, V[blk])
    ctx = np.array([70, 16, 113], dtype=np.int32)
    bt = np.full((B, 8), -1, dtype=np.int32)
    perm = rng.permutation(nb)
    k = 0
    for b in range(B):
        n = (ctx[b] + bs - 1) // bs
        bt[b, :n] = perm[k:k + n]
        k += n
    q = wl.round_to_bits(rng.standard_normal((B, Hq, d)).astype(np.float32) * 0.2, "bf16")
    want, want_lse, _ = oracle.decode_attn("bf16", kb, vb, q, ctx, bt, 0.125)
    for qpages in ([0, 0, 0], [2, 1, 5], [5, 1, 8]):
        out, lse = quant.decode_attn_q("bf16", qp, bits, kb, vb, q, ctx, bt, np.array(qpages), 0.125)
        np.testing.assert_allclose(out.reshape(B * Hq, d), want, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse.reshape(B * Hq), want_lse, rtol=0, atol=1e-12)


def test_quantize_skips_out_of_range_pairs():
    rng = np.random.default_rng(6)
    kb = wl.round_to_bits(rng.standard_normal((4, 1, 16, 64)).astype(np.float32), "f16")
    qp = quant.empty_qpool(2, 1, 16, 64, 8)
    qp2, bad = quant.quantize_blocks("f16", kb, kb, qp, 8, [[4, 0], [0, 2], [-1, 1], [1, 1]])
    assert bad == 3
    assert not qp2[0][0].any() and qp2[0][1].any()


def _prefill_tables(rng, nb, bs, ctx, width):
    bt = np.full((len(ctx), width), -1, dtype=np.int32)
    perm = rng.permutation(nb)
    k = 0
    for b, L in enumerate(ctx):
        n = (int(L) + bs - 1) // bs
        bt[b, :n] = perm[k:k + n]
        k += n
    return bt


@pytest.mark.parametrize("bits", [8, 4])
def test_quantized_prefill_is_exact_on_grid_inputs(bits):
    """Prefix attention over a quantized cached prefix: on grid inputs
    dequant(quant(x)) == x, so it must equal the 16-bit C prefix-attention
    oracle (a different implementation) on the original pool for any split
    of the pages between the two pools -- none, part of the prefix, the whole
    prefix, and pages holding new tokens too (quantized after their append)."""
    rng = np.random.default_rng(20 + bits)
    nb, Hkv, bs, d, Hq = 40, 2, 16, 64, 6
    kb, vb, K, V = _grid_pool(rng, nb, Hkv, bs, d, bits)
    qp = quant.empty_qpool(nb, Hkv, bs, d, bits)
    qp, bad = quant.quantize_blocks("bf16", kb, vb, qp, bits, np.stack([np.arange(nb)] * 2, 1))
    assert bad == 0
    new = np.array([37, 1, 20], dtype=np.int64)
    ctx = np.array([150, 16, 260], dtype=np.int32)  # prefixes 113, 15, 240 tokens
    cu = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    bt = _prefill_tables(rng, nb, bs, ctx, 20)
    T = int(cu[-1])
    q = wl.round_to_bits(rng.standard_normal((T, Hq, d)).astype(np.float32) * 0.2, "bf16")
    want, want_lse, badr = oracle.prefix_attn("bf16", kb, vb, q, cu, ctx, bt, 0.125)
    assert badr == 0
    for qpages in ([0, 0, 0], [3, 0, 7], [7, 0, 15], [10, 1, 17]):
        out, lse = quant.prefix_attn_q("bf16", qp, bits, kb, vb, q, cu, ctx, bt, np.array(qpages), 0.125)
        np.testing.assert_allclose(out, want, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, want_lse, rtol=0, atol=1e-12)


def test_quantized_prefill_without_quantized_pages_is_16bit_attention():
    """qpages = 0 everywhere: the quantized pool is never read (it holds only
    zeros here), and random, off-grid inputs give the 16-bit C oracle's
    answer; sampled rows equal the corresponding rows of the full answer."""
    rng = np.random.default_rng(31)
    nb, Hkv, bs, d, Hq = 30, 2, 16, 128, 8
    kb = wl.round_to_bits(rng.standard_normal((nb, Hkv, bs, d)).astype(np.float32), "f16")
    vb = wl.round_to_bits(rng.standard_normal((nb, Hkv, bs, d)).astype(np.float32), "f16")
    new = np.array([5, 40], dtype=np.int64)
    ctx = np.array([100, 200], dtype=np.int32)
    cu = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    bt = _prefill_tables(rng, nb, bs, ctx, 16)
    q = wl.round_to_bits(rng.standard_normal((45, Hq, d)).astype(np.float32), "f16")
    qp = quant.empty_qpool(4, Hkv, bs, d, 8)
    want, want_lse, _ = oracle.prefix_attn("f16", kb, vb, q, cu, ctx, bt, 0.088)
    out, lse = quant.prefix_attn_q("f16", qp, 8, kb, vb, q, cu, ctx, bt, np.zeros(2, np.int32), 0.088)
    np.testing.assert_allclose(out, want, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, want_lse, rtol=0, atol=1e-12)
    rows = np.array([0, 7, 44 * Hq + 3, 20 * Hq + 5])
    o2, l2 = quant.prefix_attn_q("f16", qp, 8, kb, vb, q, cu, ctx, bt, np.zeros(2, np.int32), 0.088, rows=rows)
    np.testing.assert_array_equal(o2, out[rows])
    np.testing.assert_array_equal(l2, lse[rows])


@pytest.mark.parametrize("bits", [8, 4])
def test_quantized_prefill_of_one_token_is_quantized_decode(bits):
    """With one new token per sequence, prefix attention over a partly
    quantized context is decode attention over it (decode_attn_q, written
    separately), on off-grid inputs where quantization changes the values."""
    rng = np.random.default_rng(40 + bits)
    nb, Hkv, bs, d, Hq = 30, 2, 16, 96, 4
    kb = wl.round_to_bits(rng.standard_normal((nb, Hkv, bs, d)).astype(np.float32), "bf16")
    vb = wl.round_to_bits(rng.standard_normal((nb, Hkv, bs, d)).astype(np.float32), "bf16")
    qp = quant.empty_qpool(nb, Hkv, bs, d, bits)
    qp, _ = quant.quantize_blocks("bf16", kb, vb, qp, bits, np.stack([np.arange(nb)] * 2, 1))
    ctx = np.array([77, 16, 130], dtype=np.int32)
    cu = np.arange(4, dtype=np.int32)
    bt = _prefill_tables(rng, nb, bs, ctx, 10)
    q = wl.round_to_bits(rng.standard_normal((3, Hq, d)).astype(np.float32) * 0.3, "bf16")
    qpages = np.array([4, 1, 6], dtype=np.int32)
    out, lse = quant.prefix_attn_q("bf16", qp, bits, kb, vb, q, cu, ctx, bt, qpages, 0.1)
    want, want_lse = quant.decode_attn_q("bf16", qp, bits, kb, vb, q, ctx, bt, qpages, 0.1)
    np.testing.assert_allclose(out, want.reshape(3 * Hq, d), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, want_lse.reshape(3 * Hq), rtol=0, atol=1e-12)
    # and quantization did change the answer (the pages are off the grid)
    plain, _, _ = oracle.prefix_attn("bf16", kb, vb, q, cu, ctx, bt, 0.1)
    assert np.abs(out - plain).max() > 1e-4
