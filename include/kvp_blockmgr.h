/* kvp_blockmgr.h -- the host block manager of the paged KV cache: chunk
 * hashing, prefix reuse, page allocation, copy-on-write forks and
 * frequency-based eviction.  It produces the block tables, cached-prefix
 * lengths and copy-on-write pairs that the device entry points of kvp.h take.
 * Host code only (no CUDA calls); one manager is not thread-safe.
 *
 * What it follows:
 *  - kvboost 0.6.0, "How it works" > "1. Chunking": the token stream is cut
 *    into fixed-size chunks (default 128); > "2. Two-level hashing":
 *        prefix_hash  = SHA256(previous_chunk.prefix_hash || this_chunk.tokens)
 *        content_hash = SHA256(this_chunk.tokens);
 *    > "3. Lookup and assembly": prefix-hash lookup with a content-hash
 *    fallback that is flagged approximate; the prompt splits into a cached
 *    prefix and a live suffix; frequently reused chunks stay, one-off chunks
 *    are evicted first.
 *  - kvstream 0.1.0, "Request lifecycle": pages are allocated on admission,
 *    the page table then grows one slot per token, a cached prefix's block
 *    table is forked copy-on-write, and a finished request's prefix is
 *    registered for reuse while its pages return to the pool.
 * Readings where the pages are silent: tokens are hashed as little-endian
 * int32; the first chunk's previous prefix hash is empty; only full chunks
 * are hashed and cached (the tail is always live); chunk_size is a multiple
 * of block_size; a prompt wholly covered by cached chunks keeps its last
 * chunk live; content-only matches are reported, not reused; free blocks are
 * handed out lowest id first; eviction drops the cached chunk that no live
 * sequence holds with the fewest hits, then the least recently used. */
#ifndef KVP_BLOCKMGR_H
#define KVP_BLOCKMGR_H

#include <stdint.h>

#include "kvp.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct kvp_block_manager kvp_block_manager;

/* A manager of blocks 0 .. num_blocks-1 of block_size tokens, hashing
 * chunks of chunk_size tokens (a multiple of block_size).  NULL if the
 * sizes are not positive or chunk_size is not a multiple of block_size. */
kvp_block_manager *kvp_bm_create(int64_t num_blocks, int32_t block_size, int32_t chunk_size);
void kvp_bm_destroy(kvp_block_manager *bm);

/* The two-level hashes of the full chunks of tokens[0..n): writes 32 bytes
 * per chunk to prefix_hashes and content_hashes (either may be NULL).
 * Returns the number of full chunks, n / chunk_size, or -1 on bad args. */
int64_t kvp_hash_chunks(const int32_t *tokens, int64_t n, int32_t chunk_size, uint8_t *prefix_hashes,
                        uint8_t *content_hashes);

/* Admit sequence `seq` (a new id) with its prompt tokens[0..n): its leading
 * full chunks found by prefix hash are shared (their hit counts grow), the
 * rest of the prompt gets fresh blocks.  Writes table[0..max_blocks) (the
 * sequence's blocks, -1 padded), *cached_tokens (tokens whose K/V are
 * already in the pool: the cached prefix P) and, if match_kinds is not
 * NULL, one byte per full chunk (up to max_chunks): 0 miss, 1 exact (reused),
 * 2 content-hash-only (approximate, not reused).  KVP_ERR_NO_BLOCKS if the
 * pool cannot supply the blocks even after eviction; KVP_ERR_INVALID_ARG for
 * a known seq id or a table too short. */
kvp_status kvp_bm_admit(kvp_block_manager *bm, int64_t seq, const int32_t *tokens, int64_t n, int32_t *table,
                        int32_t max_blocks, int64_t *cached_tokens, int8_t *match_kinds, int64_t max_chunks);

/* Grow sequence `seq` by n tokens (one slot per token): fresh blocks as
 * pages fill; if the partly filled last block is shared with another
 * sequence it is first replaced by a fresh copy and the (src, dst) pair is
 * written to cow_pairs (at most one pair per call) for kvp_block_copy.
 * Writes the updated table and *n_pairs. */
kvp_status kvp_bm_append(kvp_block_manager *bm, int64_t seq, int64_t n, int32_t *table, int32_t max_blocks,
                         int32_t *cow_pairs, int32_t max_pairs, int32_t *n_pairs);

/* One decode step for a batch: kvp_bm_append(seqs[i], n_tokens[i]) for i in
 * order, writing sequence i's table to tables[i][0..max_blocks) (the
 * [count][max_blocks] block-table array the device calls take) and its
 * copy-on-write pair, if any, to the next free row of cow_pairs[count][2];
 * *n_pairs counts them.  Stops at the first failure: *done is the number of
 * sequences appended (all of them on KVP_OK), the rest unchanged. */
kvp_status kvp_bm_append_batch(kvp_block_manager *bm, const int64_t *seqs, const int32_t *n_tokens, int32_t count,
                               int32_t *tables, int32_t max_blocks, int32_t *cow_pairs, int32_t *n_pairs,
                               int32_t *done);

/* `child` (a new id) shares every block of `parent` (copy-on-write). */
kvp_status kvp_bm_fork(kvp_block_manager *bm, int64_t parent, int64_t child);

/* Finish `seq`: its full chunks (tokens[0..n) are its tokens, n >= its
 * length) are registered for reuse unless their prefix hash already is,
 * then its references are dropped; blocks nobody holds return to the pool. */
kvp_status kvp_bm_finish(kvp_block_manager *bm, int64_t seq, const int32_t *tokens, int64_t n);

/* The current table and length of `seq`. */
kvp_status kvp_bm_table(const kvp_block_manager *bm, int64_t seq, int32_t *table, int32_t max_blocks, int64_t *len);

/* Evict one cached chunk that no live sequence holds; 1 if one was evicted. */
int32_t kvp_bm_evict_one(kvp_block_manager *bm);

/* out[0..4] = free blocks, blocks held by cached chunks, blocks in use,
 * chunk hits, chunk misses (over all admissions). */
void kvp_bm_stats(const kvp_block_manager *bm, int64_t *out);

/* Recompute every block's reference count from its holders (sequence
 * tables and cached chunks) and compare with the maintained counts and the
 * free list: KVP_OK, or KVP_ERR_INVALID_ARG if anything disagrees. */
kvp_status kvp_bm_audit(const kvp_block_manager *bm);

#ifdef __cplusplus
}
#endif

#endif /* KVP_BLOCKMGR_H */
