"""The host block manager driving the device path end to end, against the
oracle: request A is prefilled and finished (its chunks registered); request
B shares A's first chunks, is admitted with that cached prefix, and only its
live suffix is prefilled over the reused pages; B is then forked and both
branches decode, the fork's copy-on-write pair going through kvp_block_copy.

Synthetic K/V of a token depend only on (position, token id), so pages
reused by prefix hash hold exactly what recomputing them would give."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

HKV, HQ, D, BS, CS = 2, 8, 64, 16, 128
DT = "bf16"


@pytest.fixture(scope="module", autouse=True)
def _library():
    from paged_prefix_reuse_gb300 import build

    build.build_library()
    import paged_prefix_reuse_gb300 as kvp

    kvp.load_library()


def _kv(pos, tok):
    r = np.random.default_rng(int(pos) * 1000003 + int(tok))
    return r.standard_normal((2, HKV, D)).astype(np.float32)


def _tensor(a):
    return torch.from_numpy(wl.round_to_bits(a, DT).view(np.int16)).view(torch.bfloat16).cuda()


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _prefill(kvp, pool, table, tokens, cached, rng):
    """Append the live suffix's K/V and run prefix attention for it; returns
    (out, lse, q bits, table bits)."""
    n = len(tokens)
    live = list(range(cached, n))
    kv = np.stack([_kv(p, tokens[p]) for p in live])  # [N, 2, Hkv, d]
    q = rng.standard_normal((len(live), HQ, D)).astype(np.float32) * 0.3
    bt = torch.tensor([table + [-1] * (64 - len(table))], dtype=torch.int32, device="cuda")
    cu = torch.tensor([0, len(live)], dtype=torch.int32, device="cuda")
    ctx = torch.tensor([n], dtype=torch.int32, device="cuda")
    slots = kvp.kvp_slot_mapping(pool, cu, ctx, bt, len(live))
    kvp.kvp_cache_append(pool, _tensor(kv[:, 0]), _tensor(kv[:, 1]), slots)
    qt = _tensor(q)
    out, lse = kvp.kvp_prefix_attn(pool, qt, cu, ctx, bt, max_q_len=len(live), max_context_len=n,
                                   softmax_scale=0.125)
    torch.cuda.synchronize()
    assert pool.errors() == 0
    return out, lse, wl.round_to_bits(q, DT), bt.cpu().numpy()


def test_block_manager_tables_drive_prefix_reuse_and_forked_decode():
    import paged_prefix_reuse_gb300 as kvp

    rng = np.random.default_rng(5)
    pool = kvp.PagedKVPool.allocate(128, HKV, BS, D, dtype=torch.bfloat16)
    pool.k.zero_()
    pool.v.zero_()
    bm = kvp.BlockManager(128, BS, CS)
    system = list(rng.integers(0, 500, size=300))
    a = system + list(rng.integers(0, 500, size=100))
    ta, cached, kinds = bm.admit(1, a)
    assert cached == 0
    _prefill(kvp, pool, ta, a, 0, rng)
    bm.finish(1, a)

    b = system + list(rng.integers(500, 900, size=150))
    tb, cached, kinds = bm.admit(2, b)
    assert cached == 256 and kinds == [1, 1, 0] and tb[:16] == ta[:16]
    out, lse, qb, bt = _prefill(kvp, pool, tb, b, cached, rng)
    kp, vp = _bits(pool.k), _bits(pool.v)
    cu = np.array([0, len(b) - cached], dtype=np.int32)
    want, want_lse, bad = oracle.prefix_attn(DT, kp, vp, qb, cu, np.array([len(b)], np.int32), bt, 0.125)
    assert bad == 0
    o = out.float().cpu().numpy().reshape(-1, D).astype(np.float64)
    assert np.abs(o - want).max() <= 2e-2
    assert np.abs(lse.cpu().numpy().T.reshape(-1) - want_lse).max() <= 1e-3
    # the cached pages hold exactly the K/V a full recomputation would give
    for p in range(cached):
        blk, off = tb[p // BS], p % BS
        np.testing.assert_array_equal(kp[blk, :, off], wl.round_to_bits(_kv(p, b[p])[0], DT))

    # fork B; both branches decode one token each: the fork's shared partial
    # last page is copied before the child writes into it
    bm.fork(2, 3)
    seqs = {2: list(b), 3: list(b)}
    qdec, tables = [], []
    for sid in (2, 3):
        tok = int(rng.integers(0, 500))
        table, pairs = bm.append(sid, 1)
        # the first branch to write into the shared partial page gets a copy of it
        assert len(pairs) == (1 if sid == 2 else 0)
        if pairs:
            kvp.kvp_block_copy(pool, torch.tensor(pairs, dtype=torch.int32, device="cuda"))
        seqs[sid].append(tok)
        pos = len(seqs[sid]) - 1
        kv = _kv(pos, tok)
        bt1 = torch.tensor([table + [-1] * (64 - len(table))], dtype=torch.int32, device="cuda")
        cu1 = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
        ctx1 = torch.tensor([len(seqs[sid])], dtype=torch.int32, device="cuda")
        slots = kvp.kvp_slot_mapping(pool, cu1, ctx1, bt1, 1)
        kvp.kvp_cache_append(pool, _tensor(kv[None, 0]), _tensor(kv[None, 1]), slots)
        tables.append(table)
        qdec.append(rng.standard_normal((HQ, D)).astype(np.float32) * 0.3)
    assert tables[0][-1] != tables[1][-1]  # the two branches write different pages
    bt2 = torch.tensor([t + [-1] * (64 - len(t)) for t in tables], dtype=torch.int32, device="cuda")
    ctx2 = torch.tensor([len(seqs[2]), len(seqs[3])], dtype=torch.int32, device="cuda")
    q2 = _tensor(np.stack(qdec))
    out, lse = kvp.kvp_decode_attn(pool, q2, ctx2, bt2, int(ctx2.max()), 0.125, num_splits=2)
    torch.cuda.synchronize()
    assert pool.errors() == 0
    kp, vp = _bits(pool.k), _bits(pool.v)
    want, want_lse, bad = oracle.decode_attn(DT, kp, vp, wl.round_to_bits(np.stack(qdec), DT), ctx2.cpu().numpy(),
                                             bt2.cpu().numpy(), 0.125)
    assert bad == 0
    assert np.abs(out.float().cpu().numpy().reshape(-1, D) - want).max() <= 2e-2
    assert np.abs(lse.cpu().numpy().T.reshape(-1) - want_lse).max() <= 1e-3
    # each branch sees its own last token: the shared prefix page was copied, not overwritten
    for sid, t in zip((2, 3), tables):
        p = len(seqs[sid]) - 1
        np.testing.assert_array_equal(kp[t[p // BS], :, p % BS], wl.round_to_bits(_kv(p, seqs[sid][p])[0], DT))
    for sid in (2, 3):
        bm.finish(sid, seqs[sid])
    assert bm.audit()
