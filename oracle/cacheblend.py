"""Oracle for CacheBlend recompute selection -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this module.  Plain numpy, fp64; no code shared with the CUDA
library.

What it follows (kvboost 0.6.0, "How it works" > "4. Seam repair"): the
cacheblend strategy runs one forward pass, measures per-token cosine
deviation between the cached K/V and what the K/V would be with full
context, and recomputes only the ~15% most-deviated tokens; content-hash
(approximate) matches always take this path.

Readings taken where the pages are silent:
* a token's vector is its K and V for all kv heads, concatenated;
  deviation = 1 - cos(cached, fresh), clamped to [0, 2] (the range of
  1 - cos, which rounding can leave by an ulp); a zero vector on either
  side gives deviation 1 (no direction to agree with) unless both are zero
  (deviation 0);
* per sequence, k = ceil(n * permille / 1000) tokens are selected (150 per
  mille, the pages' ~15%, by default; integer arithmetic, so every
  implementation gets the same k), the largest deviations first, ties to the
  lower position;
* "recompute" overwrites the selected tokens' pool entries with their fresh
  K/V (this build has no model; the fresh K/V are an input).
"""
from __future__ import annotations

import math

import numpy as np

from . import decode_bits


def kv_deviation(dtype: str, k_pool, v_pool, k_fresh, v_fresh, slots):
    """deviation[t] = 1 - cos([K;V] at pool slot slots[t], [K;V] fresh[t]), fp64."""
    nb, hkv, bs, d = k_pool.shape
    T = len(slots)
    dev = np.zeros(T)
    kf = decode_bits(k_fresh, dtype).reshape(T, -1)
    vf = decode_bits(v_fresh, dtype).reshape(T, -1)
    for t in range(T):
        s = int(slots[t])
        if not 0 <= s < nb * bs:
            dev[t] = -1.0  # no cached entry to compare
            continue
        blk, off = s // bs, s % bs
        a = np.concatenate([decode_bits(k_pool[blk, :, off], dtype).ravel(),
                            decode_bits(v_pool[blk, :, off], dtype).ravel()])
        b = np.concatenate([kf[t], vf[t]])
        na, nb_ = math.sqrt(a @ a), math.sqrt(b @ b)
        if na == 0.0 and nb_ == 0.0:
            dev[t] = 0.0
        elif na == 0.0 or nb_ == 0.0:
            dev[t] = 1.0
        else:
            dev[t] = min(max(1.0 - (a @ b) / (na * nb_), 0.0), 2.0)  # cos is in [-1, 1]
    return dev


def select_recompute(deviation, cu_seqlens, permille: int = 150):
    """Per sequence the ceil(n * permille / 1000) largest deviations (ties to
    the lower position).  Returns (mask bool [T], counts int [B])."""
    dev = np.asarray(deviation)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    mask = np.zeros(len(dev), dtype=bool)
    counts = np.zeros(len(cu) - 1, dtype=np.int64)
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        n = b - a
        k = (n * permille + 999) // 1000
        order = sorted(range(a, b), key=lambda t: (-dev[t], t))
        mask[order[:k]] = True
        counts[s] = k
    return mask, counts
