"""The native host block manager (include/kvp_blockmgr.h) against the
reference (oracle/blockmgr.py): the same tables, cached-prefix lengths,
match kinds, copy-on-write pairs, counters and out-of-blocks refusals over
random operation streams, and its own reference-count audit after each one.
No GPU needed."""
import os
import re

import numpy as np
import pytest

import paged_prefix_reuse_gb300 as kvp
from oracle import blockmgr as ref

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_prefix_reuse_gb300 import build

    build.build_library()
    kvp.load_library()


def test_header_symbols_are_exported():
    src = open(os.path.join(ROOT, "include", "kvp_blockmgr.h")).read()
    names = sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]*?\b(kvp_\w+)\s*\(", src, flags=re.M)))
    assert names == sorted(kvp.BLOCKMGR_SYMBOLS)
    lib = kvp.load_library()
    for n in names:
        assert hasattr(lib, n), n


def test_hash_chain_matches_reference():
    rng = np.random.default_rng(0)
    for n, cs in ((1000, 128), (0, 16), (15, 16), (257, 32), (64, 1)):
        t = rng.integers(-2**31, 2**31 - 1, size=n, dtype=np.int64).astype(np.int32)
        assert kvp.kvp_hash_chunks(t, cs) == ref.hash_chunks(t, cs)


def test_argument_errors():
    with pytest.raises(ValueError):
        kvp.BlockManager(16, 16, 24)
    m = kvp.BlockManager(16, 16, 32, max_blocks_per_seq=2)
    with pytest.raises(kvp.KvpError):
        m.append(5, 1)  # unknown sequence
    m.admit(1, list(range(20)))
    with pytest.raises(kvp.KvpError):
        m.admit(1, [1])  # sequence already known
    with pytest.raises(kvp.KvpError):
        m.append(1, 40)  # table would exceed its capacity
    with pytest.raises(kvp.KvpError):
        m.finish(1, list(range(5)))  # fewer tokens than the sequence holds
    assert m.audit()


def _state(native, model, live_ids):
    for sid in live_ids:
        t, L = native.table(sid)
        assert t == model.seqs[sid]["table"] and L == model.seqs[sid]["len"]
    s = native.stats()
    r = model.stats()
    assert s == r, (s, r)


@pytest.mark.parametrize("seed,nb,bs,cs", [(1, 96, 16, 32), (2, 40, 8, 32), (3, 200, 16, 128), (4, 24, 16, 16)])
def test_random_streams_match_reference(seed, nb, bs, cs):
    rng = np.random.default_rng(seed)
    native = kvp.BlockManager(nb, bs, cs)
    model = ref.BlockManager(nb, bs, cs)
    prompts = [list(rng.integers(0, 40, size=int(rng.integers(1, 6 * cs)))) for _ in range(6)]
    live = {}
    next_id = 0
    seen = {"cow": 0, "noblocks": 0}
    for step in range(500):
        op = int(rng.integers(0, 5))
        if op in (0, 4) or not live:
            sid, next_id = next_id, next_id + 1
            p = prompts[int(rng.integers(0, 6))] + list(rng.integers(0, 40, size=int(rng.integers(0, cs))))
            try:
                want = model.admit(sid, p)
            except ref.NoBlocks:
                seen["noblocks"] += 1
                with pytest.raises(kvp.NoBlocks):
                    native.admit(sid, p)
            else:
                assert native.admit(sid, p) == want
                live[sid] = list(p)
        elif op == 1:
            sid = list(live)[int(rng.integers(0, len(live)))]
            n = int(rng.integers(0, 2 * bs))
            try:
                want = model.append(sid, n)
            except ref.NoBlocks:
                seen["noblocks"] += 1
                with pytest.raises(kvp.NoBlocks):
                    native.append(sid, n)
            else:
                assert native.append(sid, n) == want
                seen["cow"] += len(want[1])
                live[sid] += list(rng.integers(0, 40, size=n))
        elif op == 2:
            sid = list(live)[int(rng.integers(0, len(live)))]
            cid, next_id = next_id, next_id + 1
            model.fork(sid, cid)
            native.fork(sid, cid)
            live[cid] = list(live[sid])
        else:
            sid = list(live)[int(rng.integers(0, len(live)))]
            toks = live.pop(sid)
            model.finish(sid, toks)
            native.finish(sid, toks)
        model.audit()
        assert native.audit()
        _state(native, model, live)
    # the streams reach every path: reuse, copy-on-write, refusal, eviction
    assert model.hits > 0 and seen["cow"] > 0 and seen["noblocks"] > 0, (model.hits, seen)
    for sid in list(live):
        toks = live.pop(sid)
        model.finish(sid, toks)
        native.finish(sid, toks)
    while True:
        a, b = model._evict_one(), native.evict_one()
        assert a == b
        if not a:
            break
    assert native.stats()["free"] == nb and native.audit()


def test_append_batch_equals_sequential_appends():
    rng = np.random.default_rng(9)
    a, b = kvp.BlockManager(64, 16, 32, 64), kvp.BlockManager(64, 16, 32, 64)
    seqs = list(range(6))
    prompts = [list(rng.integers(0, 9, size=int(rng.integers(5, 60)))) for _ in seqs]
    for m in (a, b):
        for s, p in zip(seqs, prompts):
            m.admit(s, p)
        m.fork(0, 100)
        m.fork(3, 103)
    order = [0, 100, 3, 103, 5, 1]
    for step in range(6):
        n = [int(x) for x in rng.integers(0, 9, size=len(order))]
        tables, pairs = a.append_batch(order, n)
        want_pairs = []
        for i, (s, k) in enumerate(zip(order, n)):
            t, p = b.append(s, k)
            assert tables[i][: len(t)].tolist() == t and (tables[i][len(t):] == -1).all()
            want_pairs += p
        assert [tuple(r) for r in pairs.tolist()] == want_pairs
        assert a.audit() and b.audit() and a.stats() == b.stats()
    # running out of blocks part-way: the first `done` sequences appended, the rest unchanged
    with pytest.raises(kvp.NoBlocks) as ei:
        a.append_batch(order, [16 * 40] * len(order))
    assert ei.value.done < len(order)
    assert a.audit()
