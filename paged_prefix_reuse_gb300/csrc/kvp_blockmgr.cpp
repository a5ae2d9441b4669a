// kvp_blockmgr.cpp -- host block manager of the paged KV cache (see
// include/kvp_blockmgr.h for what it follows and the readings it takes):
// two-level chunk hashing, prefix reuse on admission, one slot per appended
// token, copy-on-write forks, registration on finish and frequency-based
// eviction.  Plain C++17, no CUDA.
#include <cstring>
#include <map>
#include <set>
#include <unordered_map>
#include <vector>

#include "kvp_blockmgr.h"

namespace {

// ---- SHA-256, written from the Secure Hash Standard (FIPS 180-4) ----------
constexpr uint32_t kK[64] = {
    0x428a2f98, 0x71374491, 0xb5c0fbcf, 0xe9b5dba5, 0x3956c25b, 0x59f111f1, 0x923f82a4, 0xab1c5ed5,
    0xd807aa98, 0x12835b01, 0x243185be, 0x550c7dc3, 0x72be5d74, 0x80deb1fe, 0x9bdc06a7, 0xc19bf174,
    0xe49b69c1, 0xefbe4786, 0x0fc19dc6, 0x240ca1cc, 0x2de92c6f, 0x4a7484aa, 0x5cb0a9dc, 0x76f988da,
    0x983e5152, 0xa831c66d, 0xb00327c8, 0xbf597fc7, 0xc6e00bf3, 0xd5a79147, 0x06ca6351, 0x14292967,
    0x27b70a85, 0x2e1b2138, 0x4d2c6dfc, 0x53380d13, 0x650a7354, 0x766a0abb, 0x81c2c92e, 0x92722c85,
    0xa2bfe8a1, 0xa81a664b, 0xc24b8b70, 0xc76c51a3, 0xd192e819, 0xd6990624, 0xf40e3585, 0x106aa070,
    0x19a4c116, 0x1e376c08, 0x2748774c, 0x34b0bcb5, 0x391c0cb3, 0x4ed8aa4a, 0x5b9cca4f, 0x682e6ff3,
    0x748f82ee, 0x78a5636f, 0x84c87814, 0x8cc70208, 0x90befffa, 0xa4506ceb, 0xbef9a3f7, 0xc67178f2};

inline uint32_t rotr(uint32_t x, int n) { return (x >> n) | (x << (32 - n)); }

void sha256_block(uint32_t (&h)[8], const uint8_t* p) {
    uint32_t w[64];
    for (int t = 0; t < 16; ++t)
        w[t] = (uint32_t(p[4 * t]) << 24) | (uint32_t(p[4 * t + 1]) << 16) | (uint32_t(p[4 * t + 2]) << 8) |
               uint32_t(p[4 * t + 3]);
    for (int t = 16; t < 64; ++t) {
        const uint32_t s0 = rotr(w[t - 15], 7) ^ rotr(w[t - 15], 18) ^ (w[t - 15] >> 3);
        const uint32_t s1 = rotr(w[t - 2], 17) ^ rotr(w[t - 2], 19) ^ (w[t - 2] >> 10);
        w[t] = s1 + w[t - 7] + s0 + w[t - 16];
    }
    uint32_t a = h[0], b = h[1], c = h[2], d = h[3], e = h[4], f = h[5], g = h[6], hh = h[7];
    for (int t = 0; t < 64; ++t) {
        const uint32_t S1 = rotr(e, 6) ^ rotr(e, 11) ^ rotr(e, 25);
        const uint32_t ch = (e & f) ^ (~e & g);
        const uint32_t t1 = hh + S1 + ch + kK[t] + w[t];
        const uint32_t S0 = rotr(a, 2) ^ rotr(a, 13) ^ rotr(a, 22);
        const uint32_t maj = (a & b) ^ (a & c) ^ (b & c);
        const uint32_t t2 = S0 + maj;
        hh = g;
        g = f;
        f = e;
        e = d + t1;
        d = c;
        c = b;
        b = a;
        a = t1 + t2;
    }
    h[0] += a; h[1] += b; h[2] += c; h[3] += d; h[4] += e; h[5] += f; h[6] += g; h[7] += hh;
}

struct Digest {
    uint8_t b[32];
    bool operator==(const Digest& o) const { return std::memcmp(b, o.b, 32) == 0; }
};
struct DigestHash {
    size_t operator()(const Digest& d) const {
        size_t v;
        std::memcpy(&v, d.b, sizeof v);
        return v;
    }
};

// Streaming SHA-256: 64-byte blocks are compressed straight from the input;
// only the last partial block and the padding go through the buffer.
struct Sha256 {
    uint32_t h[8] = {0x6a09e667, 0xbb67ae85, 0x3c6ef372, 0xa54ff53a, 0x510e527f, 0x9b05688c, 0x1f83d9ab, 0x5be0cd19};
    uint8_t buf[64];
    size_t nbuf = 0;
    uint64_t total = 0;
    void update(const uint8_t* p, size_t n) {
        total += n;
        if (nbuf) {
            const size_t k = n < 64 - nbuf ? n : 64 - nbuf;
            std::memcpy(buf + nbuf, p, k);
            nbuf += k;
            p += k;
            n -= k;
            if (nbuf < 64) return;
            sha256_block(h, buf);
            nbuf = 0;
        }
        for (; n >= 64; p += 64, n -= 64) sha256_block(h, p);
        std::memcpy(buf, p, n);
        nbuf = n;
    }
    Digest final() {
        const uint64_t bits = total * 8;
        buf[nbuf++] = 0x80;
        if (nbuf > 56) {
            std::memset(buf + nbuf, 0, 64 - nbuf);
            sha256_block(h, buf);
            nbuf = 0;
        }
        std::memset(buf + nbuf, 0, 56 - nbuf);
        for (int i = 0; i < 8; ++i) buf[56 + i] = uint8_t(bits >> (8 * (7 - i)));
        sha256_block(h, buf);
        Digest d;
        for (int i = 0; i < 8; ++i)
            for (int j = 0; j < 4; ++j) d.b[4 * i + j] = uint8_t(h[i] >> (24 - 8 * j));
        return d;
    }
};

// The full chunks' (prefix, content) hashes; tokens serialised little-endian.
void hash_chunks(const int32_t* tokens, int64_t n, int32_t cs, std::vector<Digest>* pre, std::vector<Digest>* con) {
    const int64_t nc = n / cs;
    pre->resize(nc);
    con->resize(nc);
    std::vector<uint8_t> data(size_t(cs) * 4);
    for (int64_t c = 0; c < nc; ++c) {
        for (int32_t i = 0; i < cs; ++i) {
            const uint32_t t = uint32_t(tokens[c * cs + i]);
            data[4 * i] = uint8_t(t);
            data[4 * i + 1] = uint8_t(t >> 8);
            data[4 * i + 2] = uint8_t(t >> 16);
            data[4 * i + 3] = uint8_t(t >> 24);
        }
        Sha256 hc;
        hc.update(data.data(), data.size());
        (*con)[c] = hc.final();
        Sha256 hp;
        if (c > 0) hp.update((*pre)[c - 1].b, 32);
        hp.update(data.data(), data.size());
        (*pre)[c] = hp.final();
    }
}

struct Chunk {
    std::vector<int32_t> blocks;
    int64_t hits = 0, last = 0;
    Digest content;
};
struct Seq {
    std::vector<int32_t> table;
    int64_t len = 0;
};

}  // namespace

struct kvp_block_manager {
    int64_t nb;
    int32_t bs, cs, bpc;
    std::vector<int32_t> ref, creg;  // references; references held by cached chunks
    std::set<int32_t> free;          // lowest id first
    std::unordered_map<int64_t, Seq> seqs;
    std::unordered_map<Digest, Chunk, DigestHash> chunks;
    std::unordered_map<Digest, Digest, DigestHash> by_content;
    int64_t clock = 0, hits = 0, misses = 0;

    bool evictable(const Chunk& c) const {
        for (int32_t b : c.blocks)
            if (ref[b] != creg[b]) return false;
        return true;
    }
    // Blocks that evicting every evictable chunk not touching `keep` frees.
    int64_t evictable_blocks(const std::set<int32_t>& keep) const {
        std::set<int32_t> seen;
        for (const auto& kv : chunks) {
            if (!evictable(kv.second)) continue;
            bool touches = false;
            for (int32_t b : kv.second.blocks) touches |= keep.count(b) != 0;
            if (!touches) seen.insert(kv.second.blocks.begin(), kv.second.blocks.end());
        }
        return int64_t(seen.size());
    }
    bool can_alloc(int64_t n, const std::set<int32_t>& keep = {}) const {
        return int64_t(free.size()) >= n || int64_t(free.size()) + evictable_blocks(keep) >= n;
    }
    bool evict_one() {
        const Digest* best = nullptr;
        const Chunk* bc = nullptr;
        for (const auto& kv : chunks) {
            if (!evictable(kv.second)) continue;
            const Chunk& c = kv.second;
            if (!bc || c.hits < bc->hits || (c.hits == bc->hits && c.last < bc->last)) {
                best = &kv.first;
                bc = &c;
            }
        }
        if (!best) return false;
        const Digest h = *best;
        Chunk c = chunks[h];
        chunks.erase(h);
        auto it = by_content.find(c.content);
        if (it != by_content.end() && it->second == h) by_content.erase(it);
        for (int32_t b : c.blocks) {
            --creg[b];
            if (--ref[b] == 0) free.insert(b);
        }
        return true;
    }
    int32_t alloc() {
        while (free.empty())
            if (!evict_one()) return -1;
        const int32_t b = *free.begin();
        free.erase(free.begin());
        ref[b] = 1;
        return b;
    }
    void release(int32_t b) {
        if (--ref[b] == 0) free.insert(b);
    }
};

namespace {
void write_table(const std::vector<int32_t>& t, int32_t* out, int32_t max_blocks) {
    for (int32_t i = 0; i < max_blocks; ++i) out[i] = i < int32_t(t.size()) ? t[i] : -1;
}
}  // namespace

extern "C" {

kvp_block_manager* kvp_bm_create(int64_t num_blocks, int32_t block_size, int32_t chunk_size) {
    if (num_blocks < 1 || num_blocks > (int64_t(1) << 31) - 1 || block_size < 1 || chunk_size < 1 ||
        chunk_size % block_size != 0)
        return nullptr;
    kvp_block_manager* bm = new kvp_block_manager;
    bm->nb = num_blocks;
    bm->bs = block_size;
    bm->cs = chunk_size;
    bm->bpc = chunk_size / block_size;
    bm->ref.assign(size_t(num_blocks), 0);
    bm->creg.assign(size_t(num_blocks), 0);
    for (int64_t b = 0; b < num_blocks; ++b) bm->free.insert(int32_t(b));
    return bm;
}

void kvp_bm_destroy(kvp_block_manager* bm) { delete bm; }

int64_t kvp_hash_chunks(const int32_t* tokens, int64_t n, int32_t chunk_size, uint8_t* prefix_hashes,
                        uint8_t* content_hashes) {
    if (n < 0 || chunk_size < 1 || (n > 0 && !tokens)) return -1;
    std::vector<Digest> pre, con;
    hash_chunks(tokens, n, chunk_size, &pre, &con);
    for (size_t c = 0; c < pre.size(); ++c) {
        if (prefix_hashes) std::memcpy(prefix_hashes + 32 * c, pre[c].b, 32);
        if (content_hashes) std::memcpy(content_hashes + 32 * c, con[c].b, 32);
    }
    return int64_t(pre.size());
}

kvp_status kvp_bm_admit(kvp_block_manager* bm, int64_t seq, const int32_t* tokens, int64_t n, int32_t* table,
                        int32_t max_blocks, int64_t* cached_tokens, int8_t* match_kinds, int64_t max_chunks) {
    if (!bm || n < 0 || (n > 0 && !tokens) || !table || max_blocks < 0 || !cached_tokens || bm->seqs.count(seq))
        return KVP_ERR_INVALID_ARG;
    std::vector<Digest> pre, con;
    hash_chunks(tokens, n, bm->cs, &pre, &con);
    int64_t exact = 0;
    while (exact < int64_t(pre.size()) && bm->chunks.count(pre[exact])) ++exact;
    if (exact > 0 && exact * bm->cs >= n) --exact;  // keep the last chunk live
    const int64_t cached = exact * bm->cs;
    const int64_t need = (n - cached + bm->bs - 1) / bm->bs;
    if (exact * bm->bpc + need > max_blocks) return KVP_ERR_INVALID_ARG;
    std::set<int32_t> keep;
    for (int64_t c = 0; c < exact; ++c) {
        const Chunk& ch = bm->chunks.at(pre[c]);
        keep.insert(ch.blocks.begin(), ch.blocks.end());
    }
    if (!bm->can_alloc(need, keep)) return KVP_ERR_NO_BLOCKS;
    if (match_kinds)
        for (int64_t c = 0; c < int64_t(pre.size()) && c < max_chunks; ++c)
            match_kinds[c] = c < exact ? 1 : (bm->by_content.count(con[c]) ? 2 : 0);
    Seq s;
    for (int64_t c = 0; c < exact; ++c) {
        Chunk& ch = bm->chunks.at(pre[c]);
        ch.hits += 1;
        ch.last = ++bm->clock;
        for (int32_t b : ch.blocks) {
            ++bm->ref[b];
            s.table.push_back(b);
        }
    }
    bm->hits += exact;
    bm->misses += int64_t(pre.size()) - exact;
    for (int64_t i = 0; i < need; ++i) s.table.push_back(bm->alloc());
    s.len = n;
    write_table(s.table, table, max_blocks);
    *cached_tokens = cached;
    bm->seqs.emplace(seq, std::move(s));
    return KVP_OK;
}

kvp_status kvp_bm_append(kvp_block_manager* bm, int64_t seq, int64_t n, int32_t* table, int32_t max_blocks,
                         int32_t* cow_pairs, int32_t max_pairs, int32_t* n_pairs) {
    if (!bm || n < 0 || !table || !n_pairs) return KVP_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return KVP_ERR_INVALID_ARG;
    Seq& s = it->second;
    const int64_t L = s.len;
    const int64_t last = L > 0 ? (L - 1) / bm->bs : -1;
    const bool shared_tail =
        L % bm->bs != 0 && last < int64_t(s.table.size()) && bm->ref[s.table[last]] > 1;
    const int64_t blocks_after = (L + n + bm->bs - 1) / bm->bs;
    const int64_t grow = blocks_after > int64_t(s.table.size()) ? blocks_after - int64_t(s.table.size()) : 0;
    const int64_t need = (shared_tail ? 1 : 0) + grow;
    if (int64_t(s.table.size()) + grow > max_blocks) return KVP_ERR_INVALID_ARG;
    const bool cow = shared_tail && n > 0;
    if (cow && (!cow_pairs || max_pairs < 1)) return KVP_ERR_INVALID_ARG;
    if (!bm->can_alloc(need)) return KVP_ERR_NO_BLOCKS;
    *n_pairs = 0;
    if (cow) {
        const int32_t old = s.table[last];
        const int32_t fresh = bm->alloc();
        --bm->ref[old];
        s.table[last] = fresh;
        cow_pairs[0] = old;
        cow_pairs[1] = fresh;
        *n_pairs = 1;
    }
    while (int64_t(s.table.size()) * bm->bs < L + n) s.table.push_back(bm->alloc());
    s.len = L + n;
    write_table(s.table, table, max_blocks);
    return KVP_OK;
}

kvp_status kvp_bm_append_batch(kvp_block_manager* bm, const int64_t* seqs, const int32_t* n_tokens, int32_t count,
                               int32_t* tables, int32_t max_blocks, int32_t* cow_pairs, int32_t* n_pairs,
                               int32_t* done) {
    if (!bm || count < 0 || (count > 0 && (!seqs || !n_tokens || !tables || !cow_pairs)) || !n_pairs || !done)
        return KVP_ERR_INVALID_ARG;
    *n_pairs = 0;
    *done = 0;
    for (int32_t i = 0; i < count; ++i) {
        int32_t np_i = 0;
        const kvp_status st = kvp_bm_append(bm, seqs[i], n_tokens[i], tables + int64_t(i) * max_blocks, max_blocks,
                                            cow_pairs + 2 * int64_t(*n_pairs), 1, &np_i);
        if (st != KVP_OK) return st;
        *n_pairs += np_i;
        *done = i + 1;
    }
    return KVP_OK;
}

kvp_status kvp_bm_fork(kvp_block_manager* bm, int64_t parent, int64_t child) {
    if (!bm || bm->seqs.count(child)) return KVP_ERR_INVALID_ARG;
    auto it = bm->seqs.find(parent);
    if (it == bm->seqs.end()) return KVP_ERR_INVALID_ARG;
    Seq c = it->second;
    for (int32_t b : c.table) ++bm->ref[b];
    bm->seqs.emplace(child, std::move(c));
    return KVP_OK;
}

kvp_status kvp_bm_finish(kvp_block_manager* bm, int64_t seq, const int32_t* tokens, int64_t n) {
    if (!bm) return KVP_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return KVP_ERR_INVALID_ARG;
    if (n < it->second.len || (it->second.len > 0 && !tokens)) return KVP_ERR_INVALID_ARG;
    Seq s = std::move(it->second);
    bm->seqs.erase(it);
    std::vector<Digest> pre, con;
    hash_chunks(tokens, s.len, bm->cs, &pre, &con);
    for (size_t c = 0; c < pre.size(); ++c) {
        if (bm->chunks.count(pre[c])) continue;
        Chunk ch;
        ch.blocks.assign(s.table.begin() + c * bm->bpc, s.table.begin() + (c + 1) * bm->bpc);
        ch.last = ++bm->clock;
        ch.content = con[c];
        for (int32_t b : ch.blocks) {
            ++bm->ref[b];
            ++bm->creg[b];
        }
        bm->chunks.emplace(pre[c], std::move(ch));
        bm->by_content.emplace(con[c], pre[c]);  // keeps an existing entry
    }
    for (int32_t b : s.table) bm->release(b);
    return KVP_OK;
}

kvp_status kvp_bm_table(const kvp_block_manager* bm, int64_t seq, int32_t* table, int32_t max_blocks, int64_t* len) {
    if (!bm || !table || !len) return KVP_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end() || int64_t(it->second.table.size()) > max_blocks) return KVP_ERR_INVALID_ARG;
    write_table(it->second.table, table, max_blocks);
    *len = it->second.len;
    return KVP_OK;
}

int32_t kvp_bm_evict_one(kvp_block_manager* bm) { return bm && bm->evict_one() ? 1 : 0; }

void kvp_bm_stats(const kvp_block_manager* bm, int64_t* out) {
    if (!bm || !out) return;
    int64_t cached = 0, used = 0;
    for (int64_t b = 0; b < bm->nb; ++b) {
        cached += bm->creg[b] > 0;
        used += bm->ref[b] > 0;
    }
    out[0] = int64_t(bm->free.size());
    out[1] = cached;
    out[2] = used;
    out[3] = bm->hits;
    out[4] = bm->misses;
}

kvp_status kvp_bm_audit(const kvp_block_manager* bm) {
    if (!bm) return KVP_ERR_INVALID_ARG;
    std::vector<int32_t> ref(size_t(bm->nb), 0), creg(size_t(bm->nb), 0);
    for (const auto& kv : bm->seqs)
        for (int32_t b : kv.second.table) {
            if (b < 0 || b >= bm->nb) return KVP_ERR_INVALID_ARG;
            ++ref[b];
        }
    for (const auto& kv : bm->chunks)
        for (int32_t b : kv.second.blocks) {
            ++ref[b];
            ++creg[b];
        }
    if (ref != bm->ref || creg != bm->creg) return KVP_ERR_INVALID_ARG;
    int64_t nfree = 0;
    for (int64_t b = 0; b < bm->nb; ++b) {
        const bool listed = bm->free.count(int32_t(b)) != 0;
        if (listed != (ref[b] == 0)) return KVP_ERR_INVALID_ARG;
        nfree += listed;
    }
    return nfree == int64_t(bm->free.size()) ? KVP_OK : KVP_ERR_INVALID_ARG;
}

}  // extern "C"
