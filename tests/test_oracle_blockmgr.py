"""Pins of the reference block manager and hash chain (oracle/blockmgr.py)
against the pages' worked example, published SHA-256 answers, the kvstream
request lifecycle, and reference-count invariants checked from scratch."""
import hashlib
import os

import numpy as np
import pytest

from oracle import blockmgr as bm

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_sha256_known_answers():
    with open(os.path.join(GOLDEN, "sha256_vectors.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                msg, want = line.rsplit(":", 1)
                assert hashlib.sha256(msg.encode()).hexdigest() == want.strip()


def test_chunking_example_and_chain_properties():
    """kvboost "1. Chunking": 1000 tokens at 128 -> 7 full chunks (hashed) + a 104-token tail."""
    rng = np.random.default_rng(0)
    t = rng.integers(0, 50000, size=1000)
    pre, con = bm.hash_chunks(t, 128)
    assert len(pre) == len(con) == 7
    assert pre[0] == con[0]  # no history before the first chunk
    assert con[1] == hashlib.sha256(t[128:256].astype("<i4").tobytes()).digest()
    assert pre[1] == hashlib.sha256(pre[0] + t[128:256].astype("<i4").tobytes()).digest()
    u = t.copy()
    u[300] += 1  # a change inside chunk 2
    pu, cu = bm.hash_chunks(u, 128)
    assert pu[:2] == pre[:2] and all(a != b for a, b in zip(pu[2:], pre[2:]))
    assert cu[3:] == con[3:] and cu[2] != con[2]  # later chunks keep their content hash
    sw = np.concatenate([t[128:256], t[:128], t[256:]])  # two chunks swapped
    ps, cs = bm.hash_chunks(sw, 128)
    assert cs[0] == con[1] and cs[1] == con[0] and ps[0] != pre[0] and ps[2:] != pre[2:]


def test_lifecycle_admit_finish_reuse_fork_cow():
    m = bm.BlockManager(64, 16, 32)
    rng = np.random.default_rng(1)
    system = list(rng.integers(0, 1000, size=96))  # 3 chunks
    a = system + list(rng.integers(0, 1000, size=20))
    table, cached, kinds = m.admit("a", a)
    assert cached == 0 and kinds == [0, 0, 0] and len(table) == 8 and len(set(table)) == 8
    m.audit()
    # decode grows one slot per token (kvstream lifecycle 2)
    table, pairs = m.append("a", 13)
    assert len(table) == 9 and pairs == []
    m.finish("a", a + [7] * 13)  # registers its 4 full chunks, pages return
    m.audit()
    assert m.stats()["cached"] == 8 and m.stats()["free"] == 56
    # a second request with the same system prompt reuses those pages (lifecycle 3)
    b = system + list(rng.integers(0, 1000, size=5))
    tb, cached, kinds = m.admit("b", b)
    assert cached == 96 and kinds == [1, 1, 1] and tb[:6] == table[:6]
    m.audit()
    # fork: the child shares every page; appending into the shared partial
    # last page copies it first (copy-on-write), and the parent is untouched
    m.fork("b", "c")
    tc, pairs = m.append("c", 3)
    assert len(pairs) == 1 and pairs[0][0] == tb[-1] and tc[-1] == pairs[0][1] and tc[:-1] == tb[:-1]
    assert m.seqs["b"]["table"] == tb
    m.audit()
    # the whole prompt cached: its last chunk stays live
    td, cached, kinds = m.admit("d", system)
    assert cached == 64 and kinds == [1, 1, 2]
    m.audit()
    for s in ("b", "c", "d"):
        m.finish(s, (b + [1] * 3) if s == "c" else (b if s == "b" else system))
    m.audit()


def test_frequency_eviction_order_and_no_blocks():
    m = bm.BlockManager(8, 16, 16)  # one block per chunk
    rng = np.random.default_rng(2)
    prompts = [list(rng.integers(0, 1000, size=17)) for _ in range(4)]  # 1 full chunk + 1-token tail
    for i, p in enumerate(prompts):
        m.admit(i, p)
        m.finish(i, p)
    # 4 cached chunk blocks, 4 free.  Hit chunk 0 three times and chunk 2 once.
    for k in range(3):
        m.admit(("h", k), prompts[0])
        m.finish(("h", k), prompts[0])
    m.admit("h2", prompts[2])
    m.finish("h2", prompts[2])
    m.audit()
    # a long prompt needs 7 blocks: the 4 free ones plus 3 evictions, fewest hits first
    m.admit("big", list(rng.integers(0, 1000, size=100)))
    left = [h for h, e in m.chunks.items()]
    assert len(left) == 1 and m.chunks[left[0]]["hits"] == 3  # the most-reused chunk survives
    m.audit()
    with pytest.raises(bm.NoBlocks):
        m.admit("x", list(range(40)))
    m.audit()


def test_random_operation_streams_keep_invariants():
    rng = np.random.default_rng(3)
    m = bm.BlockManager(96, 16, 32)
    prompts = [list(rng.integers(0, 50, size=int(rng.integers(1, 150)))) for _ in range(6)]
    live = {}
    for step in range(400):
        op = rng.integers(0, 4)
        try:
            if op == 0 or not live:
                sid = step
                p = prompts[rng.integers(0, 6)] + list(rng.integers(0, 50, size=int(rng.integers(0, 20))))
                m.admit(sid, p)
                live[sid] = list(p)
            elif op == 1:
                sid = list(live)[rng.integers(0, len(live))]
                n = int(rng.integers(1, 20))
                m.append(sid, n)
                live[sid] += list(rng.integers(0, 50, size=n))
            elif op == 2:
                sid = list(live)[rng.integers(0, len(live))]
                m.fork(sid, ("f", step))
                live[("f", step)] = list(live[sid])
            else:
                sid = list(live)[rng.integers(0, len(live))]
                m.finish(sid, live.pop(sid))
        except bm.NoBlocks:
            pass
        m.audit()
    for sid in list(live):
        m.finish(sid, live.pop(sid))
    m.audit()
    while m._evict_one():
        pass
    assert m.stats()["free"] == 96


def test_block_shared_by_two_cached_chunks_is_freed_after_both_evictions():
    """Fork inside a chunk, then diverge: both children register the chunk
    (different prefix hashes) over one shared block; eviction must still free it."""
    m = bm.BlockManager(16, 16, 32)
    p = list(range(16))  # fills the chunk's first block exactly
    m.admit("p", p)
    m.fork("p", "c")
    m.append("p", 16)
    m.append("c", 16)
    m.finish("p", p + [1] * 16)
    m.finish("c", p + [2] * 16)
    m.audit()
    assert len(m.chunks) == 2 and m.stats()["free"] == 13
    while m._evict_one():
        m.audit()
    assert m.stats()["free"] == 16 and not m.chunks
