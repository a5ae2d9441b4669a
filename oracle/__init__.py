"""fp64 CPU oracle for paged prefix-reuse attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  It shares no code with the CUDA library
(``paged_prefix_reuse_gb300``) and never imports it; the only module both
sides use is the seeded input generator ``workloads``.

The arithmetic lives in ``kvp_oracle.c`` (plain C, fp64, OpenMP over query
rows); this module builds it with gcc on first use and marshals numpy arrays.
Every function states the passage it follows in the C source.  Pins that tie
the oracle to something other than itself are in ``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvp_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/liboracle.so`` (gcc, -O2, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            lib.oracle_decode_bits.argtypes = [ctypes.c_int, P, P, i64]
            lib.oracle_decode_bits.restype = None
            lib.oracle_slot_mapping.argtypes = [i32, P, P, P, i32, i32, i64, P]
            lib.oracle_slot_mapping.restype = i64
            lib.oracle_cache_append.argtypes = [P, P, i64, i32, i32, i32, P, P, P, i32]
            lib.oracle_cache_append.restype = i64
            lib.oracle_block_copy.argtypes = [P, P, i64, i64, P, i32]
            lib.oracle_block_copy.restype = i64
            lib.oracle_prefix_attn.argtypes = [
                i32, P, P, i64, i32, i32, i32, P, i32, P, P, P, i32, i32, f64, P, i64, P, P,
            ]
            lib.oracle_prefix_attn.restype = i64
            lib.oracle_lse_merge.argtypes = [i32, i32, P, P, P, P]
            lib.oracle_lse_merge.restype = None
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


_DT = {"f16": 0, "bf16": 1}


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def decode_bits(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Stored fp16/bf16 bit patterns -> float64 values (format definitions)."""
    lib = _load()
    b = _c(bits, np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    lib.oracle_decode_bits(_DT[dtype], _ptr(b), _ptr(out), b.size)
    return out


def slot_mapping(cu_seqlens_q, context_lens, block_tables, block_size: int, num_blocks: int):
    """Pool slot of every new token; -1 where the table has no valid block.

    Returns ``(slots int64 [T], n_invalid)``.
    """
    lib = _load()
    cu = _c(cu_seqlens_q, np.int32)
    cl = _c(context_lens, np.int32)
    bt = _c(block_tables, np.int32)
    B = cl.shape[0]
    T = int(cu[-1])
    slots = np.empty(T, dtype=np.int64)
    bad = lib.oracle_slot_mapping(B, _ptr(cu), _ptr(cl), _ptr(bt), bt.shape[1], block_size, num_blocks, _ptr(slots))
    return slots, int(bad)


def cache_append(k_pool, v_pool, k_new, v_new, slots):
    """Return (k_pool', v_pool', n_out_of_range) after writing every slot != -1."""
    lib = _load()
    kp = np.array(k_pool, dtype=np.uint16, copy=True, order="C")
    vp = np.array(v_pool, dtype=np.uint16, copy=True, order="C")
    nb, hkv, bs, d = kp.shape
    kn = _c(k_new, np.uint16)
    vn = _c(v_new, np.uint16)
    sl = _c(slots, np.int64)
    bad = lib.oracle_cache_append(_ptr(kp), _ptr(vp), nb, hkv, bs, d, _ptr(kn), _ptr(vn), _ptr(sl), sl.shape[0])
    return kp, vp, int(bad)


def block_copy(k_pool, v_pool, pairs):
    """Return (k_pool', v_pool', n_invalid) after pool[dst] = pool[src] per pair."""
    lib = _load()
    kp = np.array(k_pool, dtype=np.uint16, copy=True, order="C")
    vp = np.array(v_pool, dtype=np.uint16, copy=True, order="C")
    pr = _c(pairs, np.int32).reshape(-1, 2)
    nb = kp.shape[0]
    block_elems = int(np.prod(kp.shape[1:]))
    bad = lib.oracle_block_copy(_ptr(kp), _ptr(vp), nb, block_elems, _ptr(pr), pr.shape[0])
    return kp, vp, int(bad)


def block_swap(src_k, src_v, dst_k, dst_v, pairs):
    """Swap between a device pool and a host page pool (kvstream "Features":
    low-priority sequences spill to a CPU page pool; kvboost's CPU paging:
    blocks that do not fit on the GPU move to system RAM).  For each
    (src, dst) pair in order, dst_pool[dst] = src_pool[src], whole block, K
    and V; a pair naming a block outside its pool is skipped and counted.
    Returns (dst_k', dst_v', n_invalid)."""
    dk = np.array(dst_k, copy=True)
    dv = np.array(dst_v, copy=True)
    pr = np.asarray(pairs, dtype=np.int64).reshape(-1, 2)
    bad = 0
    for src, dst in pr:
        if not (0 <= src < src_k.shape[0] and 0 <= dst < dk.shape[0]):
            bad += 1
            continue
        dk[dst] = src_k[src]
        dv[dst] = src_v[src]
    return dk, dv, bad


def prefix_attn(dtype, k_pool, v_pool, q, cu_seqlens_q, context_lens, block_tables, scale, rows=None):
    """Causal attention of every new token over its sequence's logical K/V.

    ``rows`` (optional) selects flat rows ``t * Hq + h``.  Returns
    ``(out float64 [nrows, d], lse float64 [nrows], n_invalid)``.
    """
    lib = _load()
    kp = _c(k_pool, np.uint16)
    vp = _c(v_pool, np.uint16)
    qq = _c(q, np.uint16)
    nb, hkv, bs, d = kp.shape
    T, hq, _ = qq.shape
    cu = _c(cu_seqlens_q, np.int32)
    cl = _c(context_lens, np.int32)
    bt = _c(block_tables, np.int32)
    if rows is None:
        nrows = T * hq
        rp = None
    else:
        r = _c(rows, np.int64)
        nrows = r.shape[0]
        rp = _ptr(r)
    out = np.empty((nrows, d), dtype=np.float64)
    lse = np.empty(nrows, dtype=np.float64)
    bad = lib.oracle_prefix_attn(
        _DT[dtype], _ptr(kp), _ptr(vp), nb, hkv, bs, d, _ptr(qq), hq, _ptr(cu), _ptr(cl), _ptr(bt),
        bt.shape[1], cl.shape[0], float(scale), rp, nrows, _ptr(out), _ptr(lse),
    )
    return out, lse, int(bad)


def decode_attn(dtype, k_pool, v_pool, q, context_lens, block_tables, scale, rows=None):
    """One query per sequence (the decode batch): prefix attention with N_s = 1."""
    B = np.asarray(context_lens).shape[0]
    cu = np.arange(B + 1, dtype=np.int32)
    return prefix_attn(dtype, k_pool, v_pool, q, cu, context_lens, block_tables, scale, rows)


def lse_merge(o_parts: np.ndarray, lse_parts: np.ndarray):
    """Merge partials of one row over disjoint key sets -> (o [d], lse)."""
    lib = _load()
    op = _c(o_parts, np.float64)
    lp = _c(lse_parts, np.float64)
    n, d = op.shape
    o = np.empty(d, dtype=np.float64)
    lse = np.empty(1, dtype=np.float64)
    lib.oracle_lse_merge(n, d, _ptr(op), _ptr(lp), _ptr(o), _ptr(lse))
    return o, float(lse[0])


# ---- whole-step convenience over a workloads.Workload -------------------
def run_step(w, rows=None, decode_rows=None):
    """The whole path on one workload: fork copies, slot mapping, append,
    then attention for the prefill sequences and for the decode batch.

    Returns a dict with the updated pools, the slots and the outputs.
    ``rows``/``decode_rows`` optionally restrict which attention rows are
    computed (flat ``t * Hq + h`` within each sub-batch).
    """
    kp, vp, bad_copy = block_copy(w.k_pool, w.v_pool, w.cow_pairs)
    slots, bad_slots = slot_mapping(w.cu_seqlens_q, w.context_lens, w.block_tables, w.block_size, w.num_blocks)
    kp, vp, bad_app = cache_append(kp, vp, w.k_new, w.v_new, slots)
    res = {"k_pool": kp, "v_pool": vp, "slots": slots, "bad": bad_copy + bad_slots + bad_app}
    npf = w.num_prefill
    cu = w.cu_seqlens_q
    if npf > 0:
        tq = int(cu[npf])
        out, lse, bad = prefix_attn(
            w.dtype, kp, vp, w.q[:tq], cu[: npf + 1], w.context_lens[:npf], w.block_tables[:npf],
            w.softmax_scale, rows,
        )
        res.update(prefill_out=out, prefill_lse=lse)
        res["bad"] += bad
    if w.num_decode > 0:
        tq = int(cu[npf])
        out, lse, bad = decode_attn(
            w.dtype, kp, vp, w.q[tq:], w.context_lens[npf:], w.block_tables[npf:], w.softmax_scale, decode_rows,
        )
        res.update(decode_out=out, decode_lse=lse)
        res["bad"] += bad
    return res
