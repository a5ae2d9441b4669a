"""Seeded synthetic workloads for paged prefix-reuse attention.

This module only *draws inputs*: shapes, random values rounded to the storage
dtype, and the physical placement of KV blocks in the pool (the part a host
block allocator plays in the kvstream "Request lifecycle", steps 2-3, and in
the kvboost "CPU paged attention" pool).  It performs none of the method's own
arithmetic -- no slot indexing, no attention, no merge -- so that the CPU
oracle and the CUDA library both consume exactly the same bytes and share no
code beyond this generator.

Everything is a numpy array.  Floating-point tensors are held as ``uint16``
bit patterns of IEEE binary16 (``"f16"``) or bfloat16 (``"bf16"``).

Layouts (the pages fix only the page size, kvstream.yaml ``memory`` comment:
one page is block_size x heads x head_dim x 2 x dtype_bytes):

* ``k_pool``, ``v_pool``: ``[num_blocks, Hkv, block_size, head_dim]``
* ``q``: ``[T, Hq, head_dim]``; ``k_new``, ``v_new``: ``[T, Hkv, head_dim]``,
  where the new tokens of all sequences are packed back to back (sequence s
  owns rows ``cu_seqlens_q[s] .. cu_seqlens_q[s+1]-1``).
* ``block_tables``: ``int32 [B, max_blocks]``, logical block -> physical
  block, padded with -1.
* ``cow_pairs``: ``int32 [n, 2]`` of (src, dst) physical blocks that must be
  copied before the step's append (copy-on-write fork of a shared partial
  block).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

DTYPE_CODES = {"f16": 0, "bf16": 1}


def round_to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to the storage dtype; return the uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        import torch  # bfloat16 rounding (round-to-nearest-even) from torch

        t = torch.from_numpy(x).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    raise ValueError(dtype)


def bits_to_float32(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Widen stored bit patterns to float32 (exact for both formats)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float32)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32)
    raise ValueError(dtype)


@dataclass
class Workload:
    name: str
    dtype: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    prefix_lens: np.ndarray  # int32 [B]: cached tokens P_s already in the pool
    new_lens: np.ndarray  # int32 [B]: new tokens N_s of this step
    block_tables: np.ndarray  # int32 [B, max_blocks], -1 padded
    k_pool: np.ndarray  # uint16 [num_blocks, Hkv, bs, d]
    v_pool: np.ndarray
    q: np.ndarray  # uint16 [T, Hq, d]
    k_new: np.ndarray  # uint16 [T, Hkv, d]
    v_new: np.ndarray
    cow_pairs: np.ndarray  # int32 [n, 2] (src, dst)
    softmax_scale: float
    num_decode: int = 0  # the last num_decode sequences have N_s == 1 (decode batch)
    notes: dict = field(default_factory=dict)

    # ---- plain input bookkeeping (no method arithmetic) ----
    @property
    def B(self) -> int:
        return int(self.prefix_lens.shape[0])

    @property
    def T(self) -> int:
        return int(self.new_lens.sum())

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def context_lens(self) -> np.ndarray:
        return (self.prefix_lens + self.new_lens).astype(np.int32)

    @property
    def cu_seqlens_q(self) -> np.ndarray:
        out = np.zeros(self.B + 1, dtype=np.int32)
        out[1:] = np.cumsum(self.new_lens)
        return out

    @property
    def num_prefill(self) -> int:
        return self.B - self.num_decode

    def used_blocks(self) -> np.ndarray:
        bt = self.block_tables
        return np.unique(bt[bt >= 0])


class _BlockAllocator:
    """Hands out physical blocks in a seeded random order (the placement)."""

    def __init__(self, num_blocks: int, rng: np.random.Generator):
        self.free = list(rng.permutation(num_blocks).astype(np.int64))
        self.num_blocks = num_blocks

    def take(self, n: int) -> list[int]:
        if n > len(self.free):
            raise ValueError(f"pool of {self.num_blocks} blocks exhausted")
        out, self.free = self.free[:n], self.free[n:]
        return [int(b) for b in out]


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def _finish(
    name,
    rng,
    *,
    dtype,
    Hq,
    Hkv,
    d,
    bs,
    num_blocks,
    prefix_lens,
    new_lens,
    tables,
    q_std,
    scale,
    cow_pairs=(),
    num_decode=0,
    fill_all_blocks=False,
    notes=None,
):
    """Fill pool blocks and new-token tensors with seeded N(0,1) values."""
    B = len(tables)
    max_blocks = max(1, max(len(t) for t in tables))
    bt = np.full((B, max_blocks), -1, dtype=np.int32)
    for s, t in enumerate(tables):
        bt[s, : len(t)] = t
    k_pool = np.zeros((num_blocks, Hkv, bs, d), dtype=np.uint16)
    v_pool = np.zeros((num_blocks, Hkv, bs, d), dtype=np.uint16)
    used = set(int(b) for b in bt[bt >= 0].ravel())
    used.update(int(b) for pr in cow_pairs for b in pr)
    blocks = np.arange(num_blocks) if fill_all_blocks else np.array(sorted(used), dtype=np.int64)
    per_block = Hkv * bs * d
    # Draw in a fixed order, a few thousand blocks at a time to bound memory.
    for lo in range(0, len(blocks), 2048):
        ids = blocks[lo : lo + 2048]
        k_pool[ids] = round_to_bits(
            rng.standard_normal(len(ids) * per_block, dtype=np.float32), dtype
        ).reshape(len(ids), Hkv, bs, d)
        v_pool[ids] = round_to_bits(
            rng.standard_normal(len(ids) * per_block, dtype=np.float32), dtype
        ).reshape(len(ids), Hkv, bs, d)
    T = int(np.sum(new_lens))
    q = round_to_bits(rng.standard_normal((T, Hq, d), dtype=np.float32) * np.float32(q_std), dtype)
    k_new = round_to_bits(rng.standard_normal((T, Hkv, d), dtype=np.float32), dtype)
    v_new = round_to_bits(rng.standard_normal((T, Hkv, d), dtype=np.float32), dtype)
    pairs = np.array(list(cow_pairs), dtype=np.int32).reshape(-1, 2)
    return Workload(
        name=name,
        dtype=dtype,
        num_q_heads=Hq,
        num_kv_heads=Hkv,
        head_dim=d,
        block_size=bs,
        num_blocks=num_blocks,
        prefix_lens=np.asarray(prefix_lens, dtype=np.int32),
        new_lens=np.asarray(new_lens, dtype=np.int32),
        block_tables=bt,
        k_pool=k_pool,
        v_pool=v_pool,
        q=q.reshape(T, Hq, d),
        k_new=k_new.reshape(T, Hkv, d),
        v_new=v_new.reshape(T, Hkv, d),
        cow_pairs=pairs,
        softmax_scale=float(scale),
        num_decode=num_decode,
        notes=notes or {},
    )


# --------------------------------------------------------------------------
# Generic shapes (tests: edge cases, ragged lengths, shrunken configs)
# --------------------------------------------------------------------------
def make_random(
    seed: int,
    prefix_lens,
    new_lens,
    *,
    Hq: int = 2,
    Hkv: int = 2,
    d: int = 64,
    dtype: str = "f16",
    bs: int = 16,
    num_blocks: int | None = None,
    shared_prefix: bool = False,
    q_std: float = 1.0,
    scale: float | None = None,
    num_decode: int = 0,
    fill_all_blocks: bool = False,
    name: str = "random",
) -> Workload:
    """Independent sequences with the given cached/new lengths.

    With ``shared_prefix=True`` every sequence reuses the *same* physical
    blocks for its first ``min(prefix_lens)`` tokens, rounded down to whole
    blocks (shared system prompt); the rest of each table is private.
    """
    rng = np.random.default_rng(seed)
    prefix_lens = [int(p) for p in prefix_lens]
    new_lens = [int(n) for n in new_lens]
    need = sum(_ceil_div(p + n, bs) for p, n in zip(prefix_lens, new_lens))
    if num_blocks is None:
        num_blocks = max(8, need + need // 2 + 4)
    alloc = _BlockAllocator(num_blocks, rng)
    shared = []
    if shared_prefix and prefix_lens:
        shared = alloc.take(min(prefix_lens) // bs)
    tables = []
    for p, n in zip(prefix_lens, new_lens):
        nb = _ceil_div(p + n, bs)
        own = alloc.take(nb - len(shared[:nb]))
        tables.append(shared[:nb] + own)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    return _finish(
        name,
        rng,
        dtype=dtype,
        Hq=Hq,
        Hkv=Hkv,
        d=d,
        bs=bs,
        num_blocks=num_blocks,
        prefix_lens=prefix_lens,
        new_lens=new_lens,
        tables=tables,
        q_std=q_std,
        scale=scale,
        num_decode=num_decode,
        fill_all_blocks=fill_all_blocks,
    )


# --------------------------------------------------------------------------
# The five workload shapes (sizes as stated for each use case)
# --------------------------------------------------------------------------
def tiny_correctness(seed: int = 1001) -> Workload:
    """1 sequence, 2 q / 2 kv heads, d=64, fp16, 8-block pool of 16-token blocks.

    A 32-token cached prefix (2 blocks) placed by a seeded permutation, plus
    16 new tokens appended into one fresh block.  Q, K, V ~ N(0,1); the
    softmax scale is 1/sqrt(64).
    """
    return make_random(
        seed, [32], [16], Hq=2, Hkv=2, d=64, dtype="f16", bs=16, num_blocks=8, name="tiny_correctness"
    )


def shared_system_prompt(seed: int = 1002, B: int = 8, prefix: int = 1024, new: int = 256,
                         num_blocks: int = 8192) -> Workload:
    """Qwen2.5-3B-shaped layer: Hq=16, Hkv=2 (GQA 8:1), d=128, bf16.

    B requests share one cached prefix (the same physical blocks in every
    table: copy-on-write sharing of full blocks), each with its own new
    tokens, causal.  K, V ~ N(0,1), Q ~ N(0,1)/sqrt(128); since Q is
    pre-scaled the softmax scale is 1.
    """
    rng = np.random.default_rng(seed)
    bs = 16
    alloc = _BlockAllocator(num_blocks, rng)
    shared = alloc.take(prefix // bs)
    tail = prefix % bs
    tables = []
    for _ in range(B):
        # A partial last prefix block is never shared: each request owns it.
        own = alloc.take(_ceil_div(prefix + new, bs) - len(shared))
        tables.append(shared + own)
    w = _finish(
        "shared_system_prompt",
        rng,
        dtype="bf16",
        Hq=16,
        Hkv=2,
        d=128,
        bs=bs,
        num_blocks=num_blocks,
        prefix_lens=[prefix] * B,
        new_lens=[new] * B,
        tables=tables,
        q_std=1.0 / np.sqrt(128.0),
        scale=1.0,
    )
    if tail:
        # The private copies of a partial prefix block hold the same prefix tokens.
        src = tables[0][len(shared)]
        for t in tables[1:]:
            w.k_pool[t[len(shared)], :, :tail] = w.k_pool[src, :, :tail]
            w.v_pool[t[len(shared)], :, :tail] = w.v_pool[src, :, :tail]
    w.notes["shared_blocks"] = np.array(shared, dtype=np.int32)
    return w


def rag_chunk_reuse(seed: int = 1003, B: int = 16, library: int = 64, chunk: int = 256,
                    chunks_per_request: int = 8, new_lo: int = 100, new_hi: int = 300,
                    num_blocks: int = 2048) -> Workload:
    """Phi-3-mini-shaped layer: Hq=Hkv=32, d=96, fp16.

    A library of ``library`` distinct pre-encoded document chunks of
    ``chunk`` tokens sits in the pool.  Each request's cached prefix is the
    concatenation of ``chunks_per_request`` chunks drawn uniformly with
    replacement (so one table may name the same physical block twice),
    followed by a new query of N tokens, N uniform in [new_lo, new_hi] and
    not a multiple of 16.  Q, K, V ~ N(0,1), scale 1/sqrt(96).
    """
    rng = np.random.default_rng(seed)
    bs = 16
    alloc = _BlockAllocator(num_blocks, rng)
    lib = [alloc.take(chunk // bs) for _ in range(library)]
    picks = rng.integers(0, library, size=(B, chunks_per_request))
    new_lens = []
    for _ in range(B):
        n = int(rng.integers(new_lo, new_hi + 1))
        while n % 16 == 0:
            n = int(rng.integers(new_lo, new_hi + 1))
        new_lens.append(n)
    tables = []
    for s in range(B):
        t = [b for c in picks[s] for b in lib[int(c)]]
        t += alloc.take(_ceil_div(new_lens[s], bs))
        tables.append(t)
    prefix = chunk * chunks_per_request
    w = _finish(
        "rag_chunk_reuse",
        rng,
        dtype="f16",
        Hq=32,
        Hkv=32,
        d=96,
        bs=bs,
        num_blocks=num_blocks,
        prefix_lens=[prefix] * B,
        new_lens=new_lens,
        tables=tables,
        q_std=1.0,
        scale=1.0 / np.sqrt(96.0),
    )
    w.notes["chunk_picks"] = picks
    return w


def continuous_batching_step(seed: int = 1004, n_decode: int = 64, n_prefill: int = 4,
                             prefill_new: int = 512, prefill_lo: int = 1024, prefill_hi: int = 4096,
                             median: float = 2048.0, sigma: float = 0.6, ctx_lo: int = 512,
                             ctx_hi: int = 8192, n_forks: int = 8, num_blocks: int = 32768,
                             Hq: int = 40, Hkv: int = 8, d: int = 128, dtype: str = "bf16") -> Workload:
    """Qwen2.5-32B-shaped layer: Hq=40, Hkv=8, d=128, bf16; one mixed step.

    ``n_prefill`` chunks of ``prefill_new`` new tokens over cached prefixes
    P ~ U[prefill_lo, prefill_hi], then ``n_decode`` decode sequences (one new
    token each) whose cached context is lognormal (median, sigma) clipped to
    [ctx_lo, ctx_hi].  The first 2*n_forks decode sequences form n_forks
    forked pairs: both children share every block of a cached prefix whose
    last block is partial; the second child's table names a fresh block
    that receives a copy of that partial block (one ``cow_pairs`` row) before
    the step's append.  Q, K, V ~ N(0,1), scale 1/sqrt(128).
    """
    rng = np.random.default_rng(seed)
    bs = 16
    alloc = _BlockAllocator(num_blocks, rng)
    prefix_lens, new_lens, tables, pairs = [], [], [], []
    for _ in range(n_prefill):
        p = int(rng.integers(prefill_lo, prefill_hi + 1))
        prefix_lens.append(p)
        new_lens.append(prefill_new)
        tables.append(alloc.take(_ceil_div(p + prefill_new, bs)))
    ctx = np.exp(np.log(median) + sigma * rng.standard_normal(n_decode))
    ctx = np.clip(np.rint(ctx), ctx_lo, ctx_hi).astype(np.int64)
    s = 0
    while s < n_decode:
        c = int(ctx[s])
        if s < 2 * n_forks and s + 1 < n_decode:
            if c % bs == 0:
                c += 1  # a forked prefix ends in a partial block
            parent = alloc.take(_ceil_div(c + 1, bs))
            dst = alloc.take(1)[0]
            child = parent[:-1] + [dst]
            pairs.append((parent[-1], dst))
            for t in (parent, child):
                prefix_lens.append(c)
                new_lens.append(1)
                tables.append(t)
            s += 2
        else:
            prefix_lens.append(c)
            new_lens.append(1)
            tables.append(alloc.take(_ceil_div(c + 1, bs)))
            s += 1
    w = _finish(
        "continuous_batching_step",
        rng,
        dtype=dtype,
        Hq=Hq,
        Hkv=Hkv,
        d=d,
        bs=bs,
        num_blocks=num_blocks,
        prefix_lens=prefix_lens,
        new_lens=new_lens,
        tables=tables,
        q_std=1.0,
        scale=1.0 / np.sqrt(d),
        cow_pairs=pairs,
        num_decode=n_decode,
    )
    return w


def long_context_prefix(seed: int = 1005, B: int = 4, prefix: int = 32768, new: int = 2048,
                        num_blocks: int = 16384) -> Workload:
    """Hq=64, Hkv=8, d=128, bf16: B requests with a long cached prefix each.

    Every prefix block sits at a seeded random physical place in the pool.
    K, V ~ N(0,1), Q ~ N(0,1)/sqrt(128), scale 1.
    """
    rng = np.random.default_rng(seed)
    bs = 16
    alloc = _BlockAllocator(num_blocks, rng)
    tables = [alloc.take(_ceil_div(prefix + new, bs)) for _ in range(B)]
    return _finish(
        "long_context_prefix",
        rng,
        dtype="bf16",
        Hq=64,
        Hkv=8,
        d=128,
        bs=bs,
        num_blocks=num_blocks,
        prefix_lens=[prefix] * B,
        new_lens=[new] * B,
        tables=tables,
        q_std=1.0 / np.sqrt(128.0),
        scale=1.0,
    )


CONFIGS = {
    1: tiny_correctness,
    2: shared_system_prompt,
    3: rag_chunk_reuse,
    4: continuous_batching_step,
    5: long_context_prefix,
}


def make_config(cfg: int, **kw) -> Workload:
    return CONFIGS[cfg](**kw)


def permute_placement(w: Workload, seed: int) -> Workload:
    """Same logical content, every used block moved to a new physical place.

    Returns a new Workload whose pool and tables are relabelled by a seeded
    permutation of the pool (the cow pairs are relabelled too).
    """
    rng = np.random.default_rng(seed)
    perm = rng.permutation(w.num_blocks).astype(np.int64)  # old -> new
    k_pool = np.empty_like(w.k_pool)
    v_pool = np.empty_like(w.v_pool)
    k_pool[perm] = w.k_pool
    v_pool[perm] = w.v_pool
    bt = w.block_tables.copy()
    m = bt >= 0
    bt[m] = perm[bt[m]]
    pairs = w.cow_pairs.copy()
    if pairs.size:
        pairs = perm[pairs].astype(np.int32)
    out = Workload(**{**w.__dict__})
    out.k_pool, out.v_pool, out.block_tables, out.cow_pairs = k_pool, v_pool, bt.astype(np.int32), pairs
    out.notes = dict(w.notes)
    if "shared_blocks" in out.notes:
        out.notes["shared_blocks"] = perm[out.notes["shared_blocks"]].astype(np.int32)
    return out
