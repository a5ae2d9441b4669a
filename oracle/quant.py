"""Oracle for the quantized KV pool -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this module.  Plain numpy; it shares no code with the CUDA
library.

What it follows (kvboost 0.6.0, "Optional: KV quantization"): cached K/V
tensors are stored with 8 or 4 bits, K quantized per channel and V per token
(the asymmetry of the KIVI paper), for about 2x / 4x less memory.  The pages
give nothing more, so these readings are taken:

* The quantization group is one page of one kv head: K per (page, head,
  channel) over the page's block_size tokens, V per (page, head, token) over
  the head_dim channels.
* Asymmetric min/max quantization (KIVI's): levels = 2^bits - 1,
  s = (max - min) / levels, code = clamp(round((x - min) / s), 0, levels),
  x' = code * s + min, exactly: the quantized cache stands for these values,
  and an implementation's own rounding of them (the CUDA kernel computes
  them in fp16, unit roundoff 2^-11) is part of its error, not of the
  method.
* s and min are stored as fp16: s rounded up and min rounded down, so that
  the grid still spans the group; the codes are computed against the stored
  (rounded) values, in fp32: d = x - z, q = d / s, code = round-half-even(q),
  each step one IEEE fp32 operation.  A group with max == min has s = 0 and
  all codes 0.
* Layout per block: codes uint8 [Hkv][bs][d * bits / 8], channels in order,
  two 4-bit codes per byte with the even channel in the low nibble; K meta
  fp16 [Hkv][2][d] (scale row, then min row); V meta fp16 [Hkv][bs][2]
  (scale, min) per token.
* The cached prefix is what is quantized: for sequence s the first
  qpages[s] entries of its block table index the quantized pool, the rest
  (the live suffix) the 16-bit pool.
"""
from __future__ import annotations

import numpy as np

from . import decode_bits

LEVELS = {8: 255, 4: 15}


def f16_directed(x, up: bool) -> np.ndarray:
    """fp32 -> fp16 rounded toward +inf (up) or -inf (down)."""
    x = np.asarray(x, dtype=np.float32)
    with np.errstate(over="ignore"):
        h = x.astype(np.float16)
    back = h.astype(np.float32)
    with np.errstate(invalid="ignore"):
        fix = back < x if up else back > x
    if np.any(fix):
        h = np.where(fix, np.nextafter(h, np.float16(np.inf if up else -np.inf)), h)
    return h.astype(np.float16)


def quantize_groups(x: np.ndarray, bits: int, axis: int):
    """Quantize fp32 ``x`` in groups along ``axis`` (the reduced axis).

    Returns (codes uint8 same shape as x, scale fp16, min fp16) with the
    reduced axis removed from scale and min."""
    levels = LEVELS[bits]
    x = np.asarray(x, dtype=np.float32)
    mn = x.min(axis=axis)
    mx = x.max(axis=axis)
    s32 = ((mx - mn).astype(np.float32) / np.float32(levels)).astype(np.float32)
    s_h = f16_directed(s32, up=True)
    z_h = f16_directed(mn, up=False)
    sf = np.expand_dims(s_h.astype(np.float32), axis)
    zf = np.expand_dims(z_h.astype(np.float32), axis)
    d = (x - zf).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(sf > 0, d / np.where(sf > 0, sf, np.float32(1)), np.float32(0)).astype(np.float32)
    codes = np.clip(np.rint(q), 0, levels).astype(np.uint8)
    return codes, s_h, z_h


def pack_codes(codes: np.ndarray, bits: int) -> np.ndarray:
    """[..., d] codes -> [..., d * bits / 8] bytes (even channel in the low nibble at 4 bits)."""
    if bits == 8:
        return codes.astype(np.uint8)
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)


def unpack_codes(packed: np.ndarray, bits: int, d: int) -> np.ndarray:
    if bits == 8:
        return packed.astype(np.uint8)
    out = np.empty(packed.shape[:-1] + (d,), dtype=np.uint8)
    out[..., 0::2] = packed & 0x0F
    out[..., 1::2] = packed >> 4
    return out


def empty_qpool(num_blocks: int, num_kv_heads: int, block_size: int, head_dim: int, bits: int):
    """Zeroed (k_codes, v_codes, k_meta, v_meta) arrays of a quantized pool."""
    cb = head_dim * bits // 8
    return (np.zeros((num_blocks, num_kv_heads, block_size, cb), np.uint8),
            np.zeros((num_blocks, num_kv_heads, block_size, cb), np.uint8),
            np.zeros((num_blocks, num_kv_heads, 2, head_dim), np.float16),
            np.zeros((num_blocks, num_kv_heads, block_size, 2), np.float16))


def quantize_blocks(dtype: str, k_pool, v_pool, qpool, bits: int, pairs):
    """For each (src, dst) pair: block src of the 16-bit pool, quantized, into
    block dst of the quantized pool (K per channel, V per token).  Returns the
    updated qpool arrays and the number of pairs skipped as out of range."""
    kc, vc, km, vm = (np.array(a, copy=True) for a in qpool)
    nb16 = k_pool.shape[0]
    bad = 0
    for src, dst in np.asarray(pairs, dtype=np.int64).reshape(-1, 2):
        if not (0 <= src < nb16 and 0 <= dst < kc.shape[0]):
            bad += 1
            continue
        K = decode_bits(k_pool[src], dtype).astype(np.float32)  # [Hkv, bs, d]
        V = decode_bits(v_pool[src], dtype).astype(np.float32)
        codes, s, z = quantize_groups(K, bits, axis=1)           # per channel over tokens
        kc[dst] = pack_codes(codes, bits)
        km[dst, :, 0, :] = s
        km[dst, :, 1, :] = z
        codes, s, z = quantize_groups(V, bits, axis=2)           # per token over channels
        vc[dst] = pack_codes(codes, bits)
        vm[dst, :, :, 0] = s
        vm[dst, :, :, 1] = z
    return (kc, vc, km, vm), bad


def dequantize_block(qpool, bits: int, blk: int, head_dim: int):
    """K, V of one quantized block as float64 [Hkv, bs, d]: code * s + min."""
    kc, vc, km, vm = qpool
    K = unpack_codes(kc[blk], bits, head_dim).astype(np.float64)
    V = unpack_codes(vc[blk], bits, head_dim).astype(np.float64)
    K = K * km[blk, :, 0, :].astype(np.float64)[:, None, :] + km[blk, :, 1, :].astype(np.float64)[:, None, :]
    V = V * vm[blk, :, :, 0].astype(np.float64)[:, :, None] + vm[blk, :, :, 1].astype(np.float64)[:, :, None]
    return K, V


def decode_attn_q(dtype: str, qpool, bits: int, k_pool, v_pool, q, context_lens, block_tables, qpages, scale):
    """Decode attention (one query token per sequence, all L keys) where the
    first qpages[s] pages of sequence s come from the quantized pool and the
    rest from the 16-bit pool.  fp64 softmax.  Returns (out [B, Hq, d],
    lse [B, Hq], natural log)."""
    B, Hq, d = q.shape
    nb16, Hkv, bs, _ = k_pool.shape
    g = Hq // Hkv
    qf = decode_bits(q, dtype).astype(np.float64)
    out = np.zeros((B, Hq, d))
    lse = np.zeros((B, Hq))
    for b in range(B):
        L = int(context_lens[b])
        npg = (L + bs - 1) // bs
        Ks, Vs = [], []
        for p in range(npg):
            blk = int(block_tables[b][p])
            if p < int(qpages[b]):
                K, V = dequantize_block(qpool, bits, blk, d)
            else:
                K = decode_bits(k_pool[blk], dtype).astype(np.float64)
                V = decode_bits(v_pool[blk], dtype).astype(np.float64)
            Ks.append(K)
            Vs.append(V)
        K = np.concatenate(Ks, axis=1)[:, :L]  # [Hkv, L, d]
        V = np.concatenate(Vs, axis=1)[:, :L]
        for h in range(Hq):
            x = K[h // g] @ qf[b, h] * scale
            m = x.max()
            e = np.exp(x - m)
            l = e.sum()
            out[b, h] = e @ V[h // g] / l
            lse[b, h] = m + np.log(l)
    return out, lse


def prefix_attn_q(dtype: str, qpool, bits: int, k_pool, v_pool, q, cu_seqlens_q, context_lens, block_tables,
                  qpages, scale, rows=None):
    """Causal attention of each sequence's new tokens over its cached prefix
    plus its own K/V (kvboost "How it works" step 5), where the cached prefix
    is held in the quantized pool ("Optional: KV quantization"): the first
    qpages[s] pages of sequence s are dequantized from ``qpool`` (code * s +
    min, exactly), the rest read from the 16-bit pool.  New token i of
    sequence s sits at position context_lens[s] - N_s + i and sees keys 0 ..
    that position.  fp64 softmax.

    q: bit patterns [T, Hq, d].  Returns (out, lse) for the flat rows
    t * Hq + h given in ``rows`` (all rows when None): out [n, d], lse [n]
    (natural log)."""
    T, Hq, d = q.shape
    nb16, Hkv, bs, _ = k_pool.shape
    g = Hq // Hkv
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    qf = decode_bits(q, dtype).astype(np.float64)
    if rows is None:
        rows = np.arange(T * Hq)
    rows = np.asarray(rows, dtype=np.int64)
    out = np.zeros((len(rows), d))
    lse = np.zeros(len(rows))
    seq_of = np.searchsorted(cu, rows // Hq, side="right") - 1
    cache = {}
    for n, r in enumerate(rows):
        t, h = int(r // Hq), int(r % Hq)
        s = int(seq_of[n])
        if s not in cache:
            L = int(context_lens[s])
            npg = (L + bs - 1) // bs
            qp = min(max(int(qpages[s]), 0), npg)
            Ks, Vs = [], []
            for p in range(npg):
                blk = int(block_tables[s][p])
                if p < qp:
                    K, V = dequantize_block(qpool, bits, blk, d)
                else:
                    K = decode_bits(k_pool[blk], dtype).astype(np.float64)
                    V = decode_bits(v_pool[blk], dtype).astype(np.float64)
                Ks.append(K)
                Vs.append(V)
            cache = {s: (np.concatenate(Ks, axis=1)[:, :L], np.concatenate(Vs, axis=1)[:, :L], L)}
        K, V, L = cache[s]
        N = int(cu[s + 1] - cu[s])
        pos = L - N + (t - int(cu[s]))
        x = K[h // g, : pos + 1] @ qf[t, h] * scale
        m = x.max()
        e = np.exp(x - m)
        l = e.sum()
        out[n] = e @ V[h // g, : pos + 1] / l
        lse[n] = m + np.log(l)
    return out, lse
