"""Reference block manager and hash chain -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this module.  Plain Python (dicts and lists, hashlib for
SHA-256); it shares no code with the library's native block manager.

What it follows:

* kvboost 0.6.0, "How it works" > "1. Chunking": the token stream is split
  into fixed-size chunks (default 128); a 1000-token prompt is 7 full chunks
  and a 104-token tail.  > "2. Two-level hashing": per chunk,
      prefix_hash  = SHA256(previous_chunk.prefix_hash || this_chunk.tokens)
      content_hash = SHA256(this_chunk.tokens).
  > "3. Lookup and assembly": lookup by prefix hash, content hash as a
  flagged (approximate) fallback; the prompt splits into a cached prefix and
  a live suffix; the cache keeps frequently reused chunks and evicts
  one-off chunks first (frequency-based eviction).
* kvstream 0.1.0, "Request lifecycle": pages are allocated for the prompt
  on admission, the page table then grows one slot per generated token, a
  cached prefix's block table is forked copy-on-write (shared pages never
  duplicated), and a finished request's prefix is registered for reuse while
  its pages return to the pool.

Readings taken where the pages are silent:
* tokens are hashed as little-endian int32, 4 bytes each; the first chunk's
  previous prefix hash is empty, so its prefix hash equals its content hash;
* only full chunks are hashed and cached; the tail is always live;
* chunk_size is a multiple of block_size, so a chunk is whole blocks;
* a prompt fully covered by cached chunks still keeps its last chunk live
  (the model needs at least one token to run);
* content-hash-only matches are reported, not reused (their K/V would need
  correction first);
* free blocks are handed out lowest id first; eviction drops the cached,
  unreferenced chunk with the fewest hits, then the least recently used;
* a block shared by several sequences that receives a token is first copied
  to a fresh block (copy-on-write), and the (src, dst) pair is returned.
"""
from __future__ import annotations

import hashlib
import heapq

import numpy as np


def hash_chunks(tokens, chunk_size: int):
    """(prefix_hashes, content_hashes): lists of 32-byte digests of the full chunks."""
    toks = np.asarray(tokens, dtype="<i4")
    pre, con = [], []
    prev = b""
    for c in range(len(toks) // chunk_size):
        data = toks[c * chunk_size:(c + 1) * chunk_size].tobytes()
        con.append(hashlib.sha256(data).digest())
        prev = hashlib.sha256(prev + data).digest()
        pre.append(prev)
    return pre, con


class NoBlocks(Exception):
    pass


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int, chunk_size: int):
        assert chunk_size % block_size == 0
        self.nb, self.bs, self.cs = num_blocks, block_size, chunk_size
        self.bpc = chunk_size // block_size
        self.ref = [0] * num_blocks
        self.creg = [0] * num_blocks  # references held by cached chunks (a block may be in several)
        self.free = list(range(num_blocks))  # min-heap of free ids
        heapq.heapify(self.free)
        self.seqs = {}       # seq -> {"table": [...], "len": int}
        self.chunks = {}     # prefix_hash -> {"blocks": [...], "hits": int, "last": int, "content": bytes}
        self.by_content = {}  # content_hash -> prefix_hash
        self.clock = 0
        self.hits = self.misses = 0

    # ---- allocation -------------------------------------------------------
    def _evictable(self):
        """Cached chunks none of whose blocks a live sequence holds."""
        return [h for h, e in self.chunks.items() if all(self.ref[b] == self.creg[b] for b in e["blocks"])]

    def _evict_one(self) -> bool:
        cands = self._evictable()
        if not cands:
            return False
        h = min(cands, key=lambda k: (self.chunks[k]["hits"], self.chunks[k]["last"], k))
        e = self.chunks.pop(h)
        if self.by_content.get(e["content"]) == h:
            del self.by_content[e["content"]]
        for b in e["blocks"]:
            self.creg[b] -= 1
            self.ref[b] -= 1
            if self.ref[b] == 0:
                heapq.heappush(self.free, b)
        return True

    def _can_alloc(self, n: int) -> bool:
        avail = len(self.free)
        if avail >= n:
            return True
        # blocks that eviction could free
        seen = set()
        for h in self._evictable():
            seen.update(self.chunks[h]["blocks"])
        return avail + len(seen) >= n

    def _alloc(self) -> int:
        while not self.free:
            if not self._evict_one():
                raise NoBlocks
        b = heapq.heappop(self.free)
        self.ref[b] = 1
        return b

    def _release(self, b: int):
        self.ref[b] -= 1
        if self.ref[b] == 0:
            heapq.heappush(self.free, b)

    # ---- operations -------------------------------------------------------
    def admit(self, seq, tokens):
        """Returns (table, cached_tokens, match_kinds) -- kinds per full
        chunk: 0 miss, 1 exact (reused), 2 content-only (reported)."""
        assert seq not in self.seqs
        n = len(tokens)
        pre, con = hash_chunks(tokens, self.cs)
        kinds = [0] * len(pre)
        exact = 0
        for c in range(len(pre)):
            if pre[c] in self.chunks:
                exact += 1
            else:
                break
        if exact > 0 and exact * self.cs >= n:
            exact -= 1  # keep at least the last chunk live
        for c in range(len(pre)):
            if c < exact:
                kinds[c] = 1
            elif con[c] in self.by_content:
                kinds[c] = 2
        cached = exact * self.cs
        need = -(-(n - cached) // self.bs)
        if not self._can_alloc_after_refs(pre[:exact], need):
            raise NoBlocks
        table = []
        for c in range(exact):
            e = self.chunks[pre[c]]
            self.clock += 1
            e["hits"] += 1
            e["last"] = self.clock
            for b in e["blocks"]:
                self.ref[b] += 1
                table.append(b)
        self.hits += exact
        self.misses += len(pre) - exact
        for _ in range(need):
            table.append(self._alloc())
        self.seqs[seq] = {"table": table, "len": n}
        return list(table), cached, kinds

    def _can_alloc_after_refs(self, hashes, need):
        # the chunks about to be referenced can no longer be evicted
        keep = set()
        for h in hashes:
            keep.update(self.chunks[h]["blocks"])
        avail = len(self.free)
        seen = set()
        for h in self._evictable():
            bl = self.chunks[h]["blocks"]
            if not keep.intersection(bl):
                seen.update(bl)
        return avail + len(seen) >= need

    def append(self, seq, n: int):
        """Grow by n tokens; returns (table, cow_pairs)."""
        s = self.seqs[seq]
        table, L = s["table"], s["len"]
        pairs = []
        # count blocks needed first, so that a failure changes nothing
        need = 0
        last = (L - 1) // self.bs if L > 0 else -1
        if L % self.bs != 0 and last < len(table) and self.ref[table[last]] > 1:
            need += 1
        need += max(0, -(-(L + n) // self.bs) - len(table))
        if not self._can_alloc(need):
            raise NoBlocks
        if L % self.bs != 0 and self.ref[table[last]] > 1 and n > 0:
            old = table[last]
            new = self._alloc()
            self.ref[old] -= 1
            table[last] = new
            pairs.append((old, new))
        while len(table) * self.bs < L + n:
            table.append(self._alloc())
        s["len"] = L + n
        return list(table), pairs

    def fork(self, parent, child):
        assert child not in self.seqs
        p = self.seqs[parent]
        for b in p["table"]:
            self.ref[b] += 1
        self.seqs[child] = {"table": list(p["table"]), "len": p["len"]}

    def finish(self, seq, tokens):
        """Register the sequence's full chunks (tokens = its first len tokens)
        for reuse, then drop its references."""
        s = self.seqs.pop(seq)
        table = s["table"]
        pre, con = hash_chunks(tokens[:s["len"]], self.cs)
        for c in range(len(pre)):
            blocks = table[c * self.bpc:(c + 1) * self.bpc]
            if pre[c] in self.chunks:
                continue
            self.clock += 1
            self.chunks[pre[c]] = {"blocks": list(blocks), "hits": 0, "last": self.clock, "content": con[c]}
            self.by_content.setdefault(con[c], pre[c])
            for b in blocks:
                self.ref[b] += 1
                self.creg[b] += 1
        for b in table:
            self._release(b)

    def audit(self):
        """Reference counts recomputed from the holders (sequence tables and
        cached chunks); raises if they or the free list disagree."""
        ref = [0] * self.nb
        for s_ in self.seqs.values():
            for b in s_["table"]:
                ref[b] += 1
        for e in self.chunks.values():
            for b in e["blocks"]:
                ref[b] += 1
        assert ref == self.ref, "reference counts"
        creg = [0] * self.nb
        for e in self.chunks.values():
            for b in e["blocks"]:
                creg[b] += 1
        assert creg == self.creg, "cached-chunk references"
        assert sorted(self.free) == [b for b in range(self.nb) if ref[b] == 0], "free list"

    def stats(self):
        cached = set()
        for e in self.chunks.values():
            cached.update(e["blocks"])
        used = sum(1 for r in self.ref if r > 0)
        return {"free": len(self.free), "cached": len(cached), "used": used, "hits": self.hits,
                "misses": self.misses}
