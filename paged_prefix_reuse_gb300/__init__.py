"""paged_prefix_reuse_gb300 -- Python binding of libkvp, the sm_103a library
for attention over a paged, prefix-sharing KV cache.

This module only marshals arguments: torch tensors become device pointers
and the current CUDA stream is passed along.  Every step of the path runs
in libkvp's CUDA kernels; there is no CPU or PyTorch fallback.  If the
shared library has not been built, importing works but the first call
raises ``KvpLibraryMissing``.

Functions carry the names of the C entry points declared in
``include/kvp.h``: ``kvp_slot_mapping``, ``kvp_cache_append``,
``kvp_block_copy``, ``kvp_block_swap``, ``kvp_quantize_blocks``,
``kvp_kv_deviation``, ``kvp_select_recompute``, ``kvp_prefix_attn``,
``kvp_decode_attn``, ``kvp_decode_attn_noalloc``, ``kvp_decode_attn_q``,
``kvp_prefix_attn_q``, ``kvp_pool_errors``, ``kvp_set_wait_limit_ns``,
``kvp_workspace_size``, the split-count helpers and
``kvp_set_launch_options``.  ``BlockManager`` and ``kvp_hash_chunks`` wrap
the host block manager of ``include/kvp_blockmgr.h``.  ``step`` runs a
whole step from device buffers (``DeviceStep``) or from pinned host buffers
(``HostStep``).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "KvpError",
    "KvpLibraryMissing",
    "PagedKVPool",
    "HostKVPool",
    "QuantKVPool",
    "BlockManager",
    "NoBlocks",
    "kvp_hash_chunks",
    "EXPORTED_SYMBOLS",
    "lib_path",
    "load_library",
    "kvp_slot_mapping",
    "kvp_cache_append",
    "kvp_block_copy",
    "kvp_block_swap",
    "kvp_quantize_blocks",
    "kvp_kv_deviation",
    "kvp_select_recompute",
    "kvp_prefix_attn",
    "kvp_decode_attn",
    "kvp_decode_attn_q",
    "kvp_prefix_attn_q",
    "kvp_decode_attn_noalloc",
    "kvp_workspace_size",
    "kvp_prefix_num_splits",
    "kvp_decode_num_splits",
    "kvp_status_string",
    "kvp_set_launch_options",
    "kvp_get_launch_options",
    "kvp_set_wait_limit_ns",
    "kvp_get_wait_limit_ns",
    "kvp_pool_errors",
    "LAUNCH_PDL",
    "LAUNCH_STALL_TEST",
    "DEVERR",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libkvp.so")

KVP_F16, KVP_BF16 = 0, 1
_DTYPES = {torch.float16: KVP_F16, torch.bfloat16: KVP_BF16}

LAUNCH_PDL = 0x1  # KVP_LAUNCH_PDL in kvp.h
LAUNCH_STALL_TEST = 0x2  # KVP_LAUNCH_STALL_TEST: exercises the timed-out-wait path (tests only)
KVP_ERR_TIMEOUT = 5

# Device error-word bits (KVP_DEVERR_* in kvp.h).
DEVERR = {"bad_block": 0x1, "bad_slot": 0x2, "bad_pair": 0x4, "bad_len": 0x8, "timeout": 0x10, "qrange": 0x20}

# Every extern "C" symbol declared in include/kvp.h.
EXPORTED_SYMBOLS = (
    "kvp_slot_mapping",
    "kvp_cache_append",
    "kvp_block_copy",
    "kvp_block_swap",
    "kvp_quantize_blocks",
    "kvp_kv_deviation",
    "kvp_select_recompute",
    "kvp_prefix_attn",
    "kvp_decode_attn",
    "kvp_decode_attn_q",
    "kvp_prefix_attn_q",
    "kvp_decode_attn_noalloc",
    "kvp_prefix_num_splits",
    "kvp_decode_num_splits",
    "kvp_workspace_size",
    "kvp_status_string",
    "kvp_set_launch_options",
    "kvp_get_launch_options",
    "kvp_set_wait_limit_ns",
    "kvp_get_wait_limit_ns",
    "kvp_pool_errors",
    "kvp_version",
)

# Host block manager entry points (include/kvp_blockmgr.h).
BLOCKMGR_SYMBOLS = (
    "kvp_bm_create",
    "kvp_bm_destroy",
    "kvp_hash_chunks",
    "kvp_bm_admit",
    "kvp_bm_append",
    "kvp_bm_append_batch",
    "kvp_bm_fork",
    "kvp_bm_finish",
    "kvp_bm_table",
    "kvp_bm_evict_one",
    "kvp_bm_stats",
    "kvp_bm_audit",
)


class KvpError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_status_text(status)} (kvp_status {status})")


class KvpLibraryMissing(RuntimeError):
    pass


class _QPool(ctypes.Structure):
    _fields_ = [
        ("k_codes", ctypes.c_void_p),
        ("v_codes", ctypes.c_void_p),
        ("k_meta", ctypes.c_void_p),
        ("v_meta", ctypes.c_void_p),
        ("num_blocks", ctypes.c_int64),
        ("block_size", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("bits", ctypes.c_int32),
    ]


class _HostPool(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p), ("num_blocks", ctypes.c_int64)]


class _Pool(ctypes.Structure):
    _fields_ = [
        ("k_pool", ctypes.c_void_p),
        ("v_pool", ctypes.c_void_p),
        ("num_blocks", ctypes.c_int64),
        ("block_size", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("err_word", ctypes.c_void_p),
    ]


_lib = None
_lock = threading.Lock()


def lib_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libkvp.so (built by ``paged_prefix_reuse_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise KvpLibraryMissing(
                f"{_LIB_PATH} is not built; run `python -m paged_prefix_reuse_gb300.build` first"
            )
        lib = ctypes.CDLL(_LIB_PATH)
        P, i32, i64, sz, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
        PP = ctypes.POINTER(_Pool)
        lib.kvp_slot_mapping.argtypes = [PP, P, P, P, i32, i32, i32, P, P]
        lib.kvp_cache_append.argtypes = [PP, P, P, P, i32, P]
        lib.kvp_block_copy.argtypes = [PP, P, i32, P]
        lib.kvp_block_swap.argtypes = [PP, ctypes.POINTER(_HostPool), P, i32, i32, P]
        lib.kvp_kv_deviation.argtypes = [PP, P, P, P, i32, P, P]
        lib.kvp_select_recompute.argtypes = [P, P, P, i32, i32, P, P, P]
        QP = ctypes.POINTER(_QPool)
        lib.kvp_quantize_blocks.argtypes = [PP, QP, P, i32, P]
        lib.kvp_decode_attn_q.argtypes = [PP, QP, P, P, P, P, P, P, i32, i32, i32, i32, f32, i32, P, sz, P]
        lib.kvp_prefix_attn_q.argtypes = [PP, QP, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, f32, i32, P, sz,
                                          P]
        lib.kvp_prefix_attn.argtypes = [PP, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, f32, i32, P, sz, P]
        lib.kvp_decode_attn.argtypes = [PP, P, P, P, P, P, i32, i32, i32, i32, f32, i32, P, sz, P]
        lib.kvp_decode_attn_noalloc.argtypes = [PP, P, P, P, P, P, i32, i32, i32, i32, f32, i32, P]
        i64p, i32p, i8p = ctypes.POINTER(i64), ctypes.POINTER(i32), ctypes.POINTER(ctypes.c_int8)
        lib.kvp_bm_create.argtypes = [i64, i32, i32]
        lib.kvp_bm_create.restype = P
        lib.kvp_bm_destroy.argtypes = [P]
        lib.kvp_bm_destroy.restype = None
        lib.kvp_hash_chunks.argtypes = [i32p, i64, i32, P, P]
        lib.kvp_hash_chunks.restype = i64
        lib.kvp_bm_admit.argtypes = [P, i64, i32p, i64, i32p, i32, i64p, i8p, i64]
        lib.kvp_bm_append.argtypes = [P, i64, i64, i32p, i32, i32p, i32, i32p]
        lib.kvp_bm_append_batch.argtypes = [P, P, P, i32, P, i32, P, i32p, i32p]
        lib.kvp_bm_append_batch.restype = ctypes.c_int
        lib.kvp_bm_fork.argtypes = [P, i64, i64]
        lib.kvp_bm_finish.argtypes = [P, i64, i32p, i64]
        lib.kvp_bm_table.argtypes = [P, i64, i32p, i32, i64p]
        lib.kvp_bm_evict_one.argtypes = [P]
        lib.kvp_bm_evict_one.restype = i32
        lib.kvp_bm_stats.argtypes = [P, i64p]
        lib.kvp_bm_stats.restype = None
        lib.kvp_bm_audit.argtypes = [P]
        for name in ("kvp_bm_admit", "kvp_bm_append", "kvp_bm_fork", "kvp_bm_finish", "kvp_bm_table", "kvp_bm_audit"):
            getattr(lib, name).restype = ctypes.c_int
        for name in ("kvp_slot_mapping", "kvp_cache_append", "kvp_block_copy", "kvp_block_swap",
                     "kvp_quantize_blocks", "kvp_kv_deviation", "kvp_select_recompute", "kvp_prefix_attn",
                     "kvp_decode_attn", "kvp_decode_attn_q", "kvp_prefix_attn_q",
                     "kvp_decode_attn_noalloc"):
            getattr(lib, name).restype = ctypes.c_int
        lib.kvp_prefix_num_splits.argtypes = [i32, i32, i32, i32, i32, i32]
        lib.kvp_prefix_num_splits.restype = i32
        lib.kvp_decode_num_splits.argtypes = [i32, i32, i32, i32]
        lib.kvp_decode_num_splits.restype = i32
        lib.kvp_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        lib.kvp_workspace_size.restype = sz
        lib.kvp_status_string.argtypes = [ctypes.c_int]
        lib.kvp_status_string.restype = ctypes.c_char_p
        lib.kvp_set_launch_options.argtypes = [ctypes.c_uint32]
        lib.kvp_set_launch_options.restype = None
        lib.kvp_get_launch_options.argtypes = []
        lib.kvp_get_launch_options.restype = ctypes.c_uint32
        lib.kvp_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        lib.kvp_set_wait_limit_ns.restype = None
        lib.kvp_get_wait_limit_ns.argtypes = []
        lib.kvp_get_wait_limit_ns.restype = ctypes.c_uint64
        lib.kvp_pool_errors.argtypes = [PP, ctypes.POINTER(ctypes.c_uint32), P]
        lib.kvp_pool_errors.restype = ctypes.c_int
        lib.kvp_version.argtypes = []
        lib.kvp_version.restype = i32
        _lib = lib
        return lib


def _status_text(status: int) -> str:
    try:
        return load_library().kvp_status_string(status).decode()
    except Exception:  # pragma: no cover
        return "unknown"


def kvp_status_string(status: int) -> str:
    return load_library().kvp_status_string(status).decode()


def kvp_set_launch_options(flags: int) -> None:
    """Process-wide launch options (``LAUNCH_PDL``: each kernel may start
    while the one before it on the stream finishes; see kvp.h for the
    caller's side of that contract)."""
    load_library().kvp_set_launch_options(int(flags))


def kvp_get_launch_options() -> int:
    return int(load_library().kvp_get_launch_options())


def kvp_set_wait_limit_ns(ns: int) -> None:
    """Limit of the kernels' pipeline waits before they give up and report
    ``DEVERR["timeout"]`` (0: the default, 2 s)."""
    load_library().kvp_set_wait_limit_ns(int(ns))


def kvp_get_wait_limit_ns() -> int:
    return int(load_library().kvp_get_wait_limit_ns())


def kvp_pool_errors(pool: "PagedKVPool", stream=None) -> int:
    """The pool's error bits after the work queued on ``stream``; raises
    ``KvpError`` (status KVP_ERR_TIMEOUT) when a kernel's wait gave up."""
    bits = ctypes.c_uint32(0)
    st = load_library().kvp_pool_errors(pool.c, ctypes.byref(bits), _stream(stream))
    if st not in (0, KVP_ERR_TIMEOUT):
        _check(st, "kvp_pool_errors")
    if st == KVP_ERR_TIMEOUT:
        raise KvpError(st, f"kvp_pool_errors (error bits {bits.value:#x})")
    return int(bits.value)


def _check(status: int, where: str) -> None:
    if status != 0:
        raise KvpError(status, where)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dev_i32(x, device) -> torch.Tensor:
    t = torch.as_tensor(x, dtype=torch.int32)
    return t.to(device, non_blocking=True).contiguous()


def _arg(t, name: str, dtype, ndim: int | None = None, tail: tuple | None = None, optional: bool = False):
    """The C ABI sees only a pointer, so check here what it cannot: the
    element type, the layout (dense, row-major), the device and the trailing
    shape.  An fp16 q against a bf16 pool, or a transposed view, would
    otherwise be read as garbage without an error."""
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor, not {type(t).__name__}")
    if t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}; expected {dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, not {t.dim()}")
    if tail is not None and tuple(t.shape[-len(tail):]) != tuple(tail):
        raise ValueError(f"{name} has shape {tuple(t.shape)}; its trailing dimensions must be {tuple(tail)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (row-major, no strides or transposes)")


def _on_device(**tensors):
    """After the structural checks of a call: every tensor is device memory."""
    for name, t in tensors.items():
        if t is not None and not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")


def _decode_index_args(q, context_lens, block_tables, out, lse):
    _arg(context_lens, "context_lens", torch.int32, 1)
    _arg(block_tables, "block_tables", torch.int32, 2)
    _arg(out, "out", q.dtype, 3, tuple(q.shape), optional=True)
    _arg(lse, "lse", torch.float32, 2, (q.shape[1], q.shape[0]), optional=True)
    if context_lens.shape[0] != q.shape[0] or block_tables.shape[0] < q.shape[0]:
        raise ValueError("context_lens and block_tables need one row per sequence of q")


class PagedKVPool:
    """A pool of physical KV blocks: k/v tensors [num_blocks, Hkv, block_size, d].

    The tensors are caller-owned device memory; the library keeps no state.
    ``err_word`` is a device uint32 (int32 tensor of one element) that the
    kernels OR ``DEVERR`` bits into.
    """

    def __init__(self, k_pool: torch.Tensor, v_pool: torch.Tensor, err_word: torch.Tensor | None = None):
        if k_pool.shape != v_pool.shape or k_pool.dtype != v_pool.dtype or k_pool.dim() != 4:
            raise ValueError("k_pool and v_pool must be [num_blocks, Hkv, block_size, head_dim] of one dtype")
        if not (k_pool.is_cuda and v_pool.is_cuda and k_pool.is_contiguous() and v_pool.is_contiguous()):
            raise ValueError("pools must be contiguous CUDA tensors")
        if k_pool.dtype not in _DTYPES:
            raise ValueError(f"unsupported dtype {k_pool.dtype}")
        self.k = k_pool
        self.v = v_pool
        if err_word is None:
            err_word = torch.zeros(1, dtype=torch.int32, device=k_pool.device)
        self.err_word = err_word
        nb, hkv, bs, d = k_pool.shape
        self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim = int(nb), int(hkv), int(bs), int(d)
        self.dtype = k_pool.dtype
        self._c = _Pool(
            k_pool.data_ptr(), v_pool.data_ptr(), nb, bs, hkv, d, _DTYPES[k_pool.dtype], err_word.data_ptr()
        )

    @classmethod
    def allocate(cls, num_blocks, num_kv_heads, block_size, head_dim, dtype=torch.bfloat16, device="cuda"):
        k = torch.empty((num_blocks, num_kv_heads, block_size, head_dim), dtype=dtype, device=device)
        v = torch.empty_like(k)
        return cls(k, v)

    @property
    def c(self):
        return ctypes.byref(self._c)

    def errors(self) -> int:
        return int(self.err_word.item()) & 0xFFFFFFFF

    def clear_errors(self) -> None:
        self.err_word.zero_()


def kvp_kv_deviation(pool: PagedKVPool, k_fresh: torch.Tensor, v_fresh: torch.Tensor, slots: torch.Tensor,
                     out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Per-token 1 - cos([K;V] in the pool at slots[t], [K;V] fresh[t]) (float32 [T])."""
    T = int(slots.shape[0])
    tail = (pool.num_kv_heads, pool.head_dim)
    _arg(k_fresh, "k_fresh", pool.dtype, 3, tail)
    _arg(v_fresh, "v_fresh", pool.dtype, 3, tail)
    _arg(slots, "slots", torch.int64, 1)
    _arg(out, "out", torch.float32, 1, optional=True)
    if k_fresh.shape[0] != T or v_fresh.shape[0] != T:
        raise ValueError("k_fresh, v_fresh and slots must have one row per token")
    _on_device(k_fresh=k_fresh, v_fresh=v_fresh, slots=slots, out=out)
    if out is None:
        out = torch.empty(T, dtype=torch.float32, device=slots.device)
    _check(load_library().kvp_kv_deviation(pool.c, _ptr(k_fresh), _ptr(v_fresh), _ptr(slots), T, _ptr(out),
                                           _stream(stream)), "kvp_kv_deviation")
    return out


def kvp_select_recompute(deviation: torch.Tensor, slots: torch.Tensor, cu_seqlens: torch.Tensor,
                         permille: int = 150, stream=None):
    """CacheBlend selection: -> (recompute_slots int64 [T] (-1 = keep), counts int32 [B]).
    Follow with kvp_cache_append(pool, k_fresh, v_fresh, recompute_slots)."""
    _arg(deviation, "deviation", torch.float32, 1)
    _arg(slots, "slots", torch.int64, 1)
    _arg(cu_seqlens, "cu_seqlens", torch.int32, 1)
    _on_device(deviation=deviation, slots=slots, cu_seqlens=cu_seqlens)
    B = int(cu_seqlens.shape[0]) - 1
    rs = torch.empty_like(slots)
    counts = torch.empty(max(B, 0), dtype=torch.int32, device=slots.device)
    _check(load_library().kvp_select_recompute(_ptr(deviation), _ptr(slots), _ptr(cu_seqlens), B, int(permille),
                                               _ptr(rs), _ptr(counts), _stream(stream)), "kvp_select_recompute")
    return rs, counts


class QuantKVPool:
    """A quantized block pool (8 or 4 bits; K per channel, V per token; see
    ``kvp_qpool`` in kvp.h): device tensors k_codes/v_codes uint8
    [num_blocks, Hkv, bs, d*bits/8], k_meta float16 [num_blocks, Hkv, 2, d]
    (scale row, min row), v_meta float16 [num_blocks, Hkv, bs, 2]."""

    def __init__(self, k_codes, v_codes, k_meta, v_meta, bits: int):
        nb, hkv, bs, cb = (int(x) for x in k_codes.shape)
        d = cb * 8 // bits
        if bits not in (8, 4) or tuple(v_codes.shape) != (nb, hkv, bs, cb):
            raise ValueError("bad code tensors")
        if tuple(k_meta.shape) != (nb, hkv, 2, d) or tuple(v_meta.shape) != (nb, hkv, bs, 2):
            raise ValueError("bad meta tensors")
        for t in (k_codes, v_codes, k_meta, v_meta):
            if not (t.is_cuda and t.is_contiguous()):
                raise ValueError("quantized pool tensors must be contiguous CUDA tensors")
        self.k_codes, self.v_codes, self.k_meta, self.v_meta = k_codes, v_codes, k_meta, v_meta
        self.bits, self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim = bits, nb, hkv, bs, d
        self._c = _QPool(k_codes.data_ptr(), v_codes.data_ptr(), k_meta.data_ptr(), v_meta.data_ptr(), nb, bs, hkv,
                         d, bits)

    @classmethod
    def like(cls, pool: "PagedKVPool", num_blocks: int, bits: int):
        dev = pool.k.device
        cb = pool.head_dim * bits // 8
        shape = (num_blocks, pool.num_kv_heads, pool.block_size, cb)
        return cls(torch.zeros(shape, dtype=torch.uint8, device=dev), torch.zeros(shape, dtype=torch.uint8, device=dev),
                   torch.zeros((num_blocks, pool.num_kv_heads, 2, pool.head_dim), dtype=torch.float16, device=dev),
                   torch.zeros((num_blocks, pool.num_kv_heads, pool.block_size, 2), dtype=torch.float16, device=dev),
                   bits)

    @property
    def c(self):
        return ctypes.byref(self._c)


def kvp_quantize_blocks(pool: PagedKVPool, qpool: QuantKVPool, pairs: torch.Tensor, stream=None) -> None:
    """qpool[dst] = quantize(pool[src]) per (src, dst) row of ``pairs`` (device int32 [n, 2])."""
    _arg(pairs, "pairs", torch.int32, 2, (2,))
    _on_device(pairs=pairs)
    lib = load_library()
    n = int(pairs.shape[0]) if pairs.numel() else 0
    _check(lib.kvp_quantize_blocks(pool.c, qpool.c, _ptr(pairs) if n else None, n, _stream(stream)),
           "kvp_quantize_blocks")


def kvp_decode_attn_q(pool: PagedKVPool, qpool: QuantKVPool, qpages: torch.Tensor, q: torch.Tensor,
                      context_lens: torch.Tensor, block_tables: torch.Tensor, max_context_len: int,
                      softmax_scale: float, num_splits: int = 0, out: torch.Tensor | None = None,
                      lse: torch.Tensor | None = None, workspace: torch.Tensor | None = None, want_lse: bool = True,
                      stream=None):
    """Decode attention where the first ``qpages[s]`` table entries of each
    sequence name blocks of the quantized pool and the rest blocks of the
    16-bit pool.  Returns (out [B, Hq, d], lse [Hq, B] float32 or None)."""
    _arg(q, "q", pool.dtype, 3, (pool.head_dim,))
    _arg(qpages, "qpages", torch.int32, 1)
    _decode_index_args(q, context_lens, block_tables, out, lse)
    _on_device(q=q, qpages=qpages, context_lens=context_lens, block_tables=block_tables, out=out, lse=lse)
    lib = load_library()
    B, Hq, d = (int(x) for x in q.shape)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((Hq, B), dtype=torch.float32, device=q.device)
    splits = num_splits or kvp_decode_num_splits(B, pool.num_kv_heads, pool.block_size, max_context_len)
    need = kvp_workspace_size(1, B, Hq, d, splits)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.kvp_decode_attn_q(pool.c, qpool.c, _ptr(qpages), _ptr(q), _ptr(out), _ptr(lse), _ptr(context_lens),
                                 _ptr(block_tables), int(block_tables.shape[1]), B, Hq, int(max_context_len),
                                 float(softmax_scale), int(splits), _ptr(workspace), ws_bytes, _stream(stream)),
           "kvp_decode_attn_q")
    return out, lse


def kvp_prefix_attn_q(pool: PagedKVPool, qpool: QuantKVPool, qpages: torch.Tensor, q: torch.Tensor,
                      cu_seqlens_q: torch.Tensor, context_lens: torch.Tensor, block_tables: torch.Tensor,
                      max_q_len: int, max_context_len: int, softmax_scale: float, num_splits: int = 0,
                      out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None, want_lse: bool = True, stream=None):
    """Prefix attention where the first ``qpages[s]`` table entries of each
    sequence name blocks of the quantized pool (the cached prefix) and the
    rest blocks of the 16-bit pool.  Returns (out [T, Hq, d], lse [Hq, T]
    float32 or None)."""
    _arg(q, "q", pool.dtype, 3, (pool.head_dim,))
    _arg(qpages, "qpages", torch.int32, 1)
    _arg(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _arg(context_lens, "context_lens", torch.int32, 1)
    _arg(block_tables, "block_tables", torch.int32, 2)
    _arg(out, "out", pool.dtype, 3, tuple(q.shape), optional=True)
    _arg(lse, "lse", torch.float32, 2, (q.shape[1], q.shape[0]), optional=True)
    _on_device(q=q, qpages=qpages, cu_seqlens_q=cu_seqlens_q, context_lens=context_lens, block_tables=block_tables,
               out=out, lse=lse)
    lib = load_library()
    T, Hq, d = (int(x) for x in q.shape)
    B = int(context_lens.shape[0])
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((Hq, T), dtype=torch.float32, device=q.device)
    splits = num_splits or kvp_prefix_num_splits(B, Hq, pool.num_kv_heads, d, max_q_len, max_context_len)
    need = kvp_workspace_size(0, T, Hq, d, splits)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.kvp_prefix_attn_q(pool.c, qpool.c, _ptr(qpages), _ptr(q), _ptr(out), _ptr(lse), _ptr(cu_seqlens_q),
                                 _ptr(context_lens), _ptr(block_tables), int(block_tables.shape[1]), B, T, Hq,
                                 int(max_q_len), int(max_context_len), float(softmax_scale), int(splits),
                                 _ptr(workspace), ws_bytes, _stream(stream)),
           "kvp_prefix_attn_q")
    return out, lse


KVP_ERR_NO_BLOCKS = 6


class NoBlocks(KvpError):
    """The block manager could not supply enough blocks, even after eviction
    (its state is unchanged)."""


def kvp_hash_chunks(tokens, chunk_size: int):
    """The two-level hashes of the full chunks: (prefix_hashes, content_hashes),
    lists of 32-byte digests (see kvp_blockmgr.h)."""
    import numpy as np

    t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    nc = len(t) // chunk_size
    pre = ctypes.create_string_buffer(32 * max(nc, 1))
    con = ctypes.create_string_buffer(32 * max(nc, 1))
    got = load_library().kvp_hash_chunks(t.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), len(t), chunk_size,
                                          pre, con)
    if got < 0:
        raise ValueError("bad arguments")
    pr, cr = pre.raw, con.raw
    return [pr[32 * c:32 * c + 32] for c in range(got)], [cr[32 * c:32 * c + 32] for c in range(got)]


class BlockManager:
    """Host block manager (include/kvp_blockmgr.h): chunk hashing and prefix
    reuse, page allocation, copy-on-write forks, registration and eviction.
    Sequence ids are integers chosen by the caller."""

    def __init__(self, num_blocks: int, block_size: int, chunk_size: int, max_blocks_per_seq: int = 4096):
        self._lib = load_library()
        self._h = self._lib.kvp_bm_create(num_blocks, block_size, chunk_size)
        if not self._h:
            raise ValueError("bad block manager sizes")
        self.num_blocks, self.block_size, self.chunk_size = num_blocks, block_size, chunk_size
        self.max_blocks = max_blocks_per_seq
        import numpy as np

        self._tbuf = np.full(max_blocks_per_seq, -1, dtype=np.int32)  # reused table buffer
        self._tptr = self._tbuf.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        self._pbuf = np.zeros(2, dtype=np.int32)
        self._pptr = self._pbuf.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h:
            self._lib.kvp_bm_destroy(h)

    @staticmethod
    def _i32(a):
        import numpy as np

        if not (isinstance(a, np.ndarray) and a.dtype == np.int32 and a.flags.c_contiguous):
            a = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
        return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))

    def _table_list(self):
        import numpy as np

        neg = np.flatnonzero(self._tbuf < 0)
        return self._tbuf[: neg[0] if len(neg) else len(self._tbuf)].tolist()

    def _status(self, st, where):
        if st == KVP_ERR_NO_BLOCKS:
            raise NoBlocks(st, where)
        _check(st, where)

    def admit(self, seq: int, tokens):
        """-> (table list, cached_tokens, match kinds per full chunk)."""
        import numpy as np

        t, tp = self._i32(tokens)
        cached = ctypes.c_int64(0)
        nc = max(1, len(t) // self.chunk_size)
        kinds = (ctypes.c_int8 * nc)()
        self._status(self._lib.kvp_bm_admit(self._h, seq, tp, len(t), self._tptr, self.max_blocks,
                                            ctypes.byref(cached), kinds, nc), "kvp_bm_admit")
        return self._table_list(), int(cached.value), list(kinds)[: len(t) // self.chunk_size]

    def append(self, seq: int, n: int):
        """-> (table list, copy-on-write pairs [(src, dst)])."""
        import numpy as np

        npairs = ctypes.c_int32(0)
        self._status(self._lib.kvp_bm_append(self._h, seq, n, self._tptr, self.max_blocks, self._pptr, 1,
                                             ctypes.byref(npairs)), "kvp_bm_append")
        return self._table_list(), [tuple(self._pbuf.tolist())] if npairs.value else []

    def append_batch(self, seqs, n_tokens, max_blocks: int | None = None):
        """One decode step for many sequences: -> (tables int32 [count,
        max_blocks] (-1 padded), cow_pairs int32 [k, 2]).  On running out of
        blocks raises NoBlocks with ``.done`` = sequences appended."""
        import numpy as np

        mb = max_blocks or self.max_blocks
        s = np.ascontiguousarray(np.asarray(seqs, dtype=np.int64))
        n, np_ = self._i32(n_tokens)
        tables = np.full((len(s), mb), -1, dtype=np.int32)
        pairs = np.zeros((max(len(s), 1), 2), dtype=np.int32)
        npairs, done = ctypes.c_int32(0), ctypes.c_int32(0)
        st = self._lib.kvp_bm_append_batch(self._h, s.ctypes.data, n.ctypes.data, len(s), tables.ctypes.data, mb,
                                           pairs.ctypes.data, ctypes.byref(npairs), ctypes.byref(done))
        if st == KVP_ERR_NO_BLOCKS:
            e = NoBlocks(st, "kvp_bm_append_batch")
            e.done = int(done.value)
            raise e
        _check(st, "kvp_bm_append_batch")
        return tables, pairs[: npairs.value]

    def fork(self, parent: int, child: int):
        self._status(self._lib.kvp_bm_fork(self._h, parent, child), "kvp_bm_fork")

    def finish(self, seq: int, tokens):
        t, tp = self._i32(tokens)
        self._status(self._lib.kvp_bm_finish(self._h, seq, tp, len(t)), "kvp_bm_finish")

    def table(self, seq: int):
        import numpy as np

        n = ctypes.c_int64(0)
        self._status(self._lib.kvp_bm_table(self._h, seq, self._tptr, self.max_blocks, ctypes.byref(n)),
                     "kvp_bm_table")
        return self._table_list(), int(n.value)

    def evict_one(self) -> bool:
        return bool(self._lib.kvp_bm_evict_one(self._h))

    def stats(self) -> dict:
        out = (ctypes.c_int64 * 5)()
        self._lib.kvp_bm_stats(self._h, out)
        return dict(zip(("free", "cached", "used", "hits", "misses"), list(out)))

    def audit(self) -> bool:
        return self._lib.kvp_bm_audit(self._h) == 0


class HostKVPool:
    """The swap buffer: k/v tensors [num_blocks, Hkv, block_size, d] in pinned
    host memory, with the block geometry and dtype of a device pool.

    Pinned (page-locked) host memory is mapped into the device's address
    space on a unified-address system, which is what ``kvp_block_swap``
    reads and writes.
    """

    SWAP_OUT, SWAP_IN = 0, 1

    def __init__(self, k_pool: torch.Tensor, v_pool: torch.Tensor):
        if k_pool.shape != v_pool.shape or k_pool.dtype != v_pool.dtype or k_pool.dim() != 4:
            raise ValueError("k_pool and v_pool must be [num_blocks, Hkv, block_size, head_dim] of one dtype")
        if k_pool.is_cuda or v_pool.is_cuda or not (k_pool.is_pinned() and v_pool.is_pinned()):
            raise ValueError("a host pool must be pinned host memory")
        if not (k_pool.is_contiguous() and v_pool.is_contiguous()):
            raise ValueError("host pool tensors must be contiguous")
        self.k, self.v = k_pool, v_pool
        self.num_blocks = int(k_pool.shape[0])
        self._c = _HostPool(k_pool.data_ptr(), v_pool.data_ptr(), self.num_blocks)

    @classmethod
    def like(cls, pool: "PagedKVPool", num_blocks: int):
        shape = (num_blocks, pool.num_kv_heads, pool.block_size, pool.head_dim)
        k = torch.empty(shape, dtype=pool.dtype, pin_memory=True)
        v = torch.empty(shape, dtype=pool.dtype, pin_memory=True)
        return cls(k, v)

    @property
    def c(self):
        return ctypes.byref(self._c)


def kvp_block_swap(pool: PagedKVPool, host: HostKVPool, pairs: torch.Tensor, direction: int, stream=None) -> None:
    """Move whole blocks between the device pool and the host pool:
    ``direction`` HostKVPool.SWAP_OUT copies pool[src] -> host[dst],
    HostKVPool.SWAP_IN copies host[src] -> pool[dst], per (src, dst) row of
    ``pairs`` (device int32 [n, 2])."""
    if tuple(host.k.shape[1:]) != (pool.num_kv_heads, pool.block_size, pool.head_dim) or host.k.dtype != pool.dtype:
        raise ValueError("host pool geometry or dtype differs from the device pool")
    _arg(pairs, "pairs", torch.int32, 2, (2,))
    _on_device(pairs=pairs)
    lib = load_library()
    n = int(pairs.shape[0]) if pairs.numel() else 0
    _check(lib.kvp_block_swap(pool.c, host.c, _ptr(pairs) if n else None, n, int(direction), _stream(stream)),
           "kvp_block_swap")


def kvp_workspace_size(op: int, rows: int, num_q_heads: int, head_dim: int, num_splits: int) -> int:
    return int(load_library().kvp_workspace_size(op, rows, num_q_heads, head_dim, num_splits))


def kvp_prefix_num_splits(B, num_q_heads, num_kv_heads, head_dim, max_q_len, max_context_len) -> int:
    return int(load_library().kvp_prefix_num_splits(B, num_q_heads, num_kv_heads, head_dim, max_q_len,
                                                    max_context_len))


def kvp_decode_num_splits(B, num_kv_heads, block_size, max_context_len) -> int:
    return int(load_library().kvp_decode_num_splits(B, num_kv_heads, block_size, max_context_len))


def kvp_slot_mapping(pool: PagedKVPool, cu_seqlens_q: torch.Tensor, context_lens: torch.Tensor,
                     block_tables: torch.Tensor, total_q: int, out: torch.Tensor | None = None,
                     stream=None) -> torch.Tensor:
    """Pool slot of every new token (int64 [total_q]); see kvp.h."""
    _arg(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _arg(context_lens, "context_lens", torch.int32, 1)
    _arg(block_tables, "block_tables", torch.int32, 2)
    _arg(out, "out", torch.int64, 1, optional=True)
    _on_device(cu_seqlens_q=cu_seqlens_q, context_lens=context_lens, block_tables=block_tables, out=out)
    lib = load_library()
    if out is None:
        out = torch.empty(total_q, dtype=torch.int64, device=pool.k.device)
    B = int(context_lens.shape[0])
    _check(lib.kvp_slot_mapping(pool.c, _ptr(cu_seqlens_q), _ptr(context_lens), _ptr(block_tables),
                                int(block_tables.shape[1]), B, int(total_q), _ptr(out), _stream(stream)),
           "kvp_slot_mapping")
    return out


def kvp_cache_append(pool: PagedKVPool, k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
                     stream=None) -> None:
    """Scatter new K/V [T, Hkv, d] into the pool slots (-1 = skip)."""
    tail = (pool.num_kv_heads, pool.head_dim)
    _arg(k_new, "k_new", pool.dtype, 3, tail)
    _arg(v_new, "v_new", pool.dtype, 3, tail)
    _arg(slot_mapping, "slot_mapping", torch.int64, 1)
    T = int(k_new.shape[0])
    if v_new.shape[0] != T or slot_mapping.shape[0] < T:
        raise ValueError("k_new, v_new and slot_mapping must have one row per token")
    _on_device(k_new=k_new, v_new=v_new, slot_mapping=slot_mapping)
    lib = load_library()
    _check(lib.kvp_cache_append(pool.c, _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), T, _stream(stream)),
           "kvp_cache_append")


def kvp_block_copy(pool: PagedKVPool, pairs: torch.Tensor, stream=None) -> None:
    """Copy-on-write fork: pool[dst] = pool[src] for each (src, dst) row of ``pairs``."""
    _arg(pairs, "pairs", torch.int32, 2, (2,))
    _on_device(pairs=pairs)
    lib = load_library()
    n = int(pairs.shape[0]) if pairs.numel() else 0
    _check(lib.kvp_block_copy(pool.c, _ptr(pairs) if n else None, n, _stream(stream)), "kvp_block_copy")


def kvp_prefix_attn(pool: PagedKVPool, q: torch.Tensor, cu_seqlens_q: torch.Tensor, context_lens: torch.Tensor,
                    block_tables: torch.Tensor, max_q_len: int, max_context_len: int, softmax_scale: float,
                    num_splits: int = 0, out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                    workspace: torch.Tensor | None = None, want_lse: bool = True, stream=None):
    """Causal attention of the packed new tokens q [T, Hq, d] over their
    sequences' paged K/V.  Returns (out [T, Hq, d], lse [Hq, T] float32 or None)."""
    _arg(q, "q", pool.dtype, 3, (pool.head_dim,))
    _arg(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _arg(context_lens, "context_lens", torch.int32, 1)
    _arg(block_tables, "block_tables", torch.int32, 2)
    _arg(out, "out", pool.dtype, 3, tuple(q.shape), optional=True)
    _arg(lse, "lse", torch.float32, 2, (q.shape[1], q.shape[0]), optional=True)
    _on_device(q=q, cu_seqlens_q=cu_seqlens_q, context_lens=context_lens, block_tables=block_tables, out=out, lse=lse)
    lib = load_library()
    T, Hq, d = (int(x) for x in q.shape)
    B = int(context_lens.shape[0])
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((Hq, T), dtype=torch.float32, device=q.device)
    splits = num_splits or kvp_prefix_num_splits(B, Hq, pool.num_kv_heads, d, max_q_len, max_context_len)
    need = kvp_workspace_size(0, T, Hq, d, splits)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.kvp_prefix_attn(pool.c, _ptr(q), _ptr(out), _ptr(lse), _ptr(cu_seqlens_q), _ptr(context_lens),
                               _ptr(block_tables), int(block_tables.shape[1]), B, T, Hq, int(max_q_len),
                               int(max_context_len), float(softmax_scale), int(splits), _ptr(workspace),
                               ws_bytes, _stream(stream)),
           "kvp_prefix_attn")
    return out, lse


def kvp_decode_attn(pool: PagedKVPool, q: torch.Tensor, context_lens: torch.Tensor, block_tables: torch.Tensor,
                    max_context_len: int, softmax_scale: float, num_splits: int = 0,
                    out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                    workspace: torch.Tensor | None = None, want_lse: bool = True, stream=None):
    """One query per sequence q [B, Hq, d] over its paged context.
    Returns (out [B, Hq, d], lse [Hq, B] float32 or None)."""
    _arg(q, "q", pool.dtype, 3, (pool.head_dim,))
    _decode_index_args(q, context_lens, block_tables, out, lse)
    _on_device(q=q, context_lens=context_lens, block_tables=block_tables, out=out, lse=lse)
    lib = load_library()
    B, Hq, d = (int(x) for x in q.shape)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((Hq, B), dtype=torch.float32, device=q.device)
    splits = num_splits or kvp_decode_num_splits(B, pool.num_kv_heads, pool.block_size, max_context_len)
    need = kvp_workspace_size(1, B, Hq, d, splits)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.kvp_decode_attn(pool.c, _ptr(q), _ptr(out), _ptr(lse), _ptr(context_lens), _ptr(block_tables),
                               int(block_tables.shape[1]), B, Hq, int(max_context_len), float(softmax_scale),
                               int(splits), _ptr(workspace), ws_bytes, _stream(stream)),
           "kvp_decode_attn")
    return out, lse


# Bytes of split partials the no-allocation decode entry point can hold.
DECODE_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def kvp_decode_attn_noalloc(pool: PagedKVPool, q: torch.Tensor, context_lens: torch.Tensor,
                            block_tables: torch.Tensor, max_context_len: int, softmax_scale: float,
                            num_splits: int = 0, out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                            want_lse: bool = True, stream=None):
    """Decode attention without a workspace: the split partials use the
    library's fixed device array (see kvp.h).  The caller still provides
    ``out`` and ``lse`` (allocated here only when omitted)."""
    _arg(q, "q", pool.dtype, 3, (pool.head_dim,))
    _decode_index_args(q, context_lens, block_tables, out, lse)
    _on_device(q=q, context_lens=context_lens, block_tables=block_tables, out=out, lse=lse)
    lib = load_library()
    B, Hq, d = (int(x) for x in q.shape)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((Hq, B), dtype=torch.float32, device=q.device)
    _check(lib.kvp_decode_attn_noalloc(pool.c, _ptr(q), _ptr(out), _ptr(lse), _ptr(context_lens),
                                       _ptr(block_tables), int(block_tables.shape[1]), B, Hq,
                                       int(max_context_len), float(softmax_scale), int(num_splits),
                                       _stream(stream)),
           "kvp_decode_attn_noalloc")
    return out, lse
