/*
 * kvp.h -- C ABI of libkvp: paged prefix-reuse attention on one GB300 GPU.
 *
 * The operation (kvboost 0.6.0, "How it works" step 5 and "CPU paged
 * attention"; kvstream 0.1.0, "Request lifecycle" and "Configuration"):
 * a request's new tokens attend causally to the K/V of a cached prefix plus
 * their own K/V.  K/V live in a pool of fixed-size physical blocks addressed
 * through a per-request block table; a block may be named by several tables
 * (shared copy-on-write); new tokens' K/V are written into the pool one slot
 * per token.  Paging changes where bytes live, not the mathematics: the
 * result is ordinary causal softmax attention over the logical sequence.
 *
 * Conventions shared by every call
 * --------------------------------
 * Pool:   k_pool and v_pool are separate device arrays laid out
 *         [num_blocks][num_kv_heads][block_size][head_dim], elements fp16 or
 *         bf16.  One block of K plus V is block_size x heads x head_dim x 2
 *         x dtype_bytes, the page size of the kvstream.yaml "memory" comment.
 * Tokens: the new tokens of B sequences are packed back to back: sequence s
 *         owns rows cu_seqlens_q[s] .. cu_seqlens_q[s+1]-1 of q/out/k_new.
 *         context_lens[s] = cached prefix tokens + new tokens of sequence s.
 *         New token i of sequence s sits at absolute position
 *         context_lens[s] - N_s + i (bottom-right causal alignment) and sees
 *         keys 0 .. that position.
 * Tables: block_tables is int32 [B][max_blocks]; logical token j of sequence
 *         s lives in physical block block_tables[s][j / block_size], row
 *         j % block_size.  Entries past ceil(context_lens[s]/block_size) are
 *         never read.
 * GQA:    query head h reads kv head h / (num_q_heads / num_kv_heads).
 * Memory: every pointer argument is caller-owned; device pointers must stay
 *         valid until the enqueued work completes.  The library allocates
 *         nothing and keeps no per-call state.
 * Async:  every call enqueues kernels on `stream` (a cudaStream_t, NULL =
 *         legacy default stream) and returns after launch.  It does not
 *         synchronise.
 * Errors: arguments checkable on the host are validated before any launch
 *         and reported by the return value (nothing is enqueued then).
 *         Device-resident indices (block ids, slots, lengths) are checked in
 *         the kernels: a bad entry is skipped and a KVP_DEVERR_* bit is
 *         OR-ed into *pool->err_word when err_word is non-NULL.  No kernel
 *         traps.  Every wait inside a kernel is bounded; a wait that gives
 *         up sets KVP_DEVERR_TIMEOUT and the kernel returns.
 */
#ifndef KVP_H_
#define KVP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KVP_OK = 0,
    KVP_ERR_INVALID_ARG = 1, /* null/misaligned pointer, negative size, Hq % Hkv != 0 ... */
    KVP_ERR_UNSUPPORTED = 2, /* head_dim not 64/96/128, dtype, block_size not 8/16/32 */
    KVP_ERR_WORKSPACE = 3,   /* workspace missing or smaller than kvp_workspace_size() */
    KVP_ERR_CUDA = 4,        /* a CUDA runtime/driver call or launch failed */
    KVP_ERR_TIMEOUT = 5,     /* kvp_pool_errors: a kernel's bounded wait gave up (KVP_DEVERR_TIMEOUT) */
    KVP_ERR_NO_BLOCKS = 6    /* block manager: too few free or evictable blocks (state unchanged) */
} kvp_status;

typedef enum { KVP_F16 = 0, KVP_BF16 = 1 } kvp_dtype;

/* Bits OR-ed into *err_word by the kernels. */
#define KVP_DEVERR_BAD_BLOCK 0x1u /* a block-table entry outside [0, num_blocks) */
#define KVP_DEVERR_BAD_SLOT 0x2u  /* a slot outside [0, num_blocks*block_size), not -1 */
#define KVP_DEVERR_BAD_PAIR 0x4u  /* a copy pair naming a block outside the pool */
#define KVP_DEVERR_BAD_LEN 0x8u   /* context_len < new tokens, or a table too short */
#define KVP_DEVERR_TIMEOUT 0x10u  /* a bounded in-kernel wait gave up */
#define KVP_DEVERR_QRANGE 0x20u   /* a quantization group's scale or min is not a finite fp16 */

typedef struct {
    void *k_pool;          /* device, [num_blocks][num_kv_heads][block_size][head_dim], 16-B aligned */
    void *v_pool;          /* device, same shape and dtype as k_pool */
    int64_t num_blocks;    /* physical blocks in the pool, >= 1 */
    int32_t block_size;    /* tokens per block: 8, 16 or 32 (kvstream.yaml: power of two 8/16/32) */
    int32_t num_kv_heads;  /* >= 1 */
    int32_t head_dim;      /* 64, 96 or 128 (kvboost "Flash Attention (CUDA)" table) */
    int32_t dtype;         /* kvp_dtype: fp16 or bf16 (same table) */
    uint32_t *err_word;    /* device uint32 that kernels OR KVP_DEVERR_* bits into; may be NULL */
} kvp_pool;

/* Slot of every new token (kvstream "Request lifecycle" step 2: the page
 * table grows one slot per token).  For token i of sequence s at position
 * p = context_lens[s] - N_s + i:
 *     slot_mapping[cu_seqlens_q[s] + i] = block_tables[s][p / bs] * bs + p % bs.
 * cu_seqlens_q: device int32 [B+1], non-decreasing, cu_seqlens_q[B] == total_q.
 * context_lens: device int32 [B].  block_tables: device int32 [B][max_blocks].
 * slot_mapping: device int64 [total_q], written.  A token whose table entry
 * is missing or outside the pool gets slot -1 and sets KVP_DEVERR_BAD_BLOCK
 * (or KVP_DEVERR_BAD_LEN when p / bs >= max_blocks or p < 0). */
kvp_status kvp_slot_mapping(const kvp_pool *pool, const int32_t *cu_seqlens_q, const int32_t *context_lens,
                            const int32_t *block_tables, int32_t max_blocks, int32_t B, int32_t total_q,
                            int64_t *slot_mapping, void *stream);

/* Append (kvstream "Request lifecycle" step 2; kvboost "How it works" step
 * 5, write-back of newly seen chunks): for every token t with
 * slot = slot_mapping[t] != -1 and every kv head h,
 *     k_pool[slot / bs][h][slot % bs][:] = k_new[t][h][:]   (same for V).
 * k_new, v_new: device [T][num_kv_heads][head_dim] in the pool dtype, 16-B
 * aligned.  slot_mapping: device int64 [T].  Slots must be distinct (two
 * tokens writing one slot race).  A slot outside the pool is skipped and
 * sets KVP_DEVERR_BAD_SLOT.  T == 0 is a no-op. */
kvp_status kvp_cache_append(const kvp_pool *pool, const void *k_new, const void *v_new,
                            const int64_t *slot_mapping, int32_t T, void *stream);

/* Copy-on-write fork (kvboost "CPU paged attention": shared prefixes share
 * physical blocks copy-on-write; kvstream "Request lifecycle" step 3: a
 * forked table shares pages, which are never duplicated): before a sequence
 * writes into a block it shares, the block is copied to a private one:
 *     k_pool[pairs[i][1]] = k_pool[pairs[i][0]]  (whole block, all heads; same for V).
 * pairs: device int32 [n][2] = (src, dst).  Destinations must be distinct
 * and no destination may also be a source in the same call; otherwise the
 * result is undefined.  A pair naming a block outside the pool is skipped
 * and sets KVP_DEVERR_BAD_PAIR.  n == 0 is a no-op; n <= 65535 per call. */
kvp_status kvp_block_copy(const kvp_pool *pool, const int32_t *pairs, int32_t n, void *stream);

/* A quantized block pool (kvboost "Optional: KV quantization": cached K/V
 * stored in 8 or 4 bits, K quantized per channel and V per token, the
 * asymmetry of the KIVI paper).  The pages give nothing more; the format
 * taken here: the quantization group is one page of one kv head, K per
 * (block, head, channel) over the block's tokens and V per (block, head,
 * token) over the channels; asymmetric min/max codes, levels = 2^bits - 1,
 *     s = fp16_round_up((max - min) / levels),  z = fp16_round_down(min),
 *     code = clamp(round_half_even((x - z) / s), 0, levels)   (fp32 steps),
 *     x' = code * s + z;
 * a group with max == min has s = 0 and codes 0.
 *   k_codes, v_codes: device uint8 [num_blocks][Hkv][bs][head_dim*bits/8],
 *       channels in order; at 4 bits two codes per byte, the even channel in
 *       the low nibble.
 *   k_meta: device fp16 [num_blocks][Hkv][2][head_dim] (scale row, min row).
 *   v_meta: device fp16 [num_blocks][Hkv][bs][2] (scale, min) per token.
 * All four 16-byte aligned, caller-owned.  num_kv_heads, block_size and
 * head_dim must equal those of the 16-bit pool it is used with. */
typedef struct kvp_qpool {
    void *k_codes;
    void *v_codes;
    void *k_meta;
    void *v_meta;
    int64_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t bits; /* 8 or 4 */
} kvp_qpool;

/* Quantize whole blocks of the 16-bit pool into the quantized pool (the
 * write-back of cached chunks in quantized form): for each pair,
 *     qpool[pairs[i][1]] = quantize(pool[pairs[i][0]])   (K and V, all heads).
 * pairs: device int32 [n][2] = (src block of pool, dst block of qpool);
 * destinations must be distinct.  A pair outside either pool is skipped and
 * sets KVP_DEVERR_BAD_PAIR; a group whose scale or min overflows fp16 sets
 * KVP_DEVERR_QRANGE (in pool.err_word).  n == 0 is a no-op; n <= 65535.
 * Errors: KVP_ERR_INVALID_ARG (null/misaligned pointer, n < 0, geometry of
 * the two pools differs), KVP_ERR_UNSUPPORTED (bits not 8 or 4). */
kvp_status kvp_quantize_blocks(const kvp_pool *pool, const kvp_qpool *qpool, const int32_t *pairs, int32_t n,
                               void *stream);

/* Decode attention over a context whose cached prefix is quantized: as
 * kvp_decode_attn, except that for sequence s the first qpages[s] entries of
 * its block table name blocks of qpool and the remaining entries name blocks
 * of the 16-bit pool (the live suffix).  The codes are dequantized inside the
 * products: q.k = sum_c (q_c s_c) code_c + q.z with q_c s_c carried as an
 * fp16 pair hi + lo, and sum_t P_t v_t = sum_t (P_t sv_t) code_t + sum_t P_t
 * zv_t with P_t sv_t rounded to fp16; the products q_c s_c must lie in fp16
 * range.  The tensor-core products of this call run in fp16 whatever the pool
 * dtype (q and a bf16 pool's suffix pages are converted to fp16;
 * accumulation, softmax, O and LSE in fp32, O written in the pool dtype).
 * qpages: device int32 [B], 0 <= qpages[s] <= pages of s (a larger value is
 * clamped).  block_size must be 16 (else KVP_ERR_UNSUPPORTED), and
 * qpool.num_blocks * num_kv_heads * 16 < 2^31 (else KVP_ERR_INVALID_ARG).
 * Workspace, splits, outputs and errors as kvp_decode_attn
 * (kvp_workspace_size op 1 covers it). */
kvp_status kvp_decode_attn_q(const kvp_pool *pool, const kvp_qpool *qpool, const int32_t *qpages, const void *q,
                             void *out, float *lse, const int32_t *context_lens, const int32_t *block_tables,
                             int32_t max_blocks, int32_t B, int32_t num_q_heads, int32_t max_context_len,
                             float softmax_scale, int32_t num_splits, void *workspace, size_t workspace_bytes,
                             void *stream);

/* Prefix attention over a context whose cached prefix is quantized
 * (kvboost "Optional: KV quantization" with "How it works" step 5: the
 * cached chunks are stored in 8 or 4 bits and the live suffix attends to
 * them): as kvp_prefix_attn, except that for sequence s the first qpages[s]
 * entries of its block table name blocks of qpool (dequantized inside the
 * kernel, code * s + z, into the tiles the tensor cores read) and the
 * remaining entries name blocks of the 16-bit pool (the live suffix, whose
 * K/V kvp_cache_append wrote).  The tensor-core products of this call run in
 * fp16 whatever the pool dtype (q and a bf16 pool's suffix pages are
 * converted to fp16; accumulation, softmax, O and LSE in fp32, O written in
 * the pool dtype), so K/V values must lie within fp16 range.
 * qpages: device int32 [B], 0 <= qpages[s] <= pages of s (a larger value is
 * clamped).  block_size must be 16 (else KVP_ERR_UNSUPPORTED).  Workspace,
 * splits, outputs and errors as kvp_prefix_attn (kvp_workspace_size op 0);
 * a table entry outside the pool it names sets KVP_DEVERR_BAD_BLOCK. */
kvp_status kvp_prefix_attn_q(const kvp_pool *pool, const kvp_qpool *qpool, const int32_t *qpages, const void *q,
                             void *out, float *lse, const int32_t *cu_seqlens_q, const int32_t *context_lens,
                             const int32_t *block_tables, int32_t max_blocks, int32_t B, int32_t total_q,
                             int32_t num_q_heads, int32_t max_q_len, int32_t max_context_len, float softmax_scale,
                             int32_t num_splits, void *workspace, size_t workspace_bytes, void *stream);

/* CacheBlend recompute selection (kvboost "How it works" > "4. Seam
 * repair": the cacheblend strategy measures per-token cosine deviation
 * between the cached K/V and the K/V with full context in one forward pass
 * and recomputes only the ~15% most-deviated tokens; content-hash matches
 * always take it).  Three calls: kvp_kv_deviation, kvp_select_recompute,
 * then kvp_cache_append(pool, k_fresh, v_fresh, recompute_slots, T), which
 * overwrites the selected tokens' pool entries with their fresh K/V.
 *
 * Deviation: for token t with pool slot slots[t], the vector of its K and V
 * for all kv heads, cached (in the pool) and fresh (k_fresh/v_fresh, device
 * [T][num_kv_heads][head_dim] in the pool dtype, 16-byte aligned):
 *     deviation[t] = 1 - cos(cached, fresh), clamped to [0, 2] (fp32; 0 if both vectors are
 *     zero, 1 if only one is).
 * A slot outside the pool gives -1 and sets KVP_DEVERR_BAD_SLOT.
 * deviation: device float [T], written.  T == 0 is a no-op. */
kvp_status kvp_kv_deviation(const kvp_pool *pool, const void *k_fresh, const void *v_fresh, const int64_t *slots,
                            int32_t T, float *deviation, void *stream);

/* Selection: tokens of sequence s are t in [cu_seqlens[s], cu_seqlens[s+1]);
 * k_s = ceil(n_s * permille / 1000) of them (integer arithmetic; 150 per
 * mille = the pages' ~15%) are selected, the largest deviations first, ties
 * to the lower position.  recompute_slots[t] = slots[t] if selected, else -1
 * (device int64 [T]); counts[s] = k_s (device int32 [B]).  permille in
 * [0, 1000].  B == 0 is a no-op. */
kvp_status kvp_select_recompute(const float *deviation, const int64_t *slots, const int32_t *cu_seqlens, int32_t B,
                                int32_t permille, int64_t *recompute_slots, int32_t *counts, void *stream);

/* Launch options, process-wide (all devices, all streams); default 0.
 * KVP_LAUNCH_PDL: every kernel the library launches may begin before the
 * kernel queued before it on the same stream has finished (programmatic
 * dependent launch), overlapping its start-up (barrier setup, tensor memory,
 * reads of metadata, block tables and q) with that kernel's tail.  Before
 * its first global write and before reading any pool, slot, workspace or
 * deviation buffer, every kernel waits for the preceding kernel to complete
 * (griddepcontrol.wait), so completions stay ordered down the stream.
 * Contract with the caller when enabled: the kernel queued immediately
 * before a kvp_* call must not write that call's q, cu_seqlens_q,
 * context_lens, block_tables or qpages.  (Within the library's own step --
 * copy, slot mapping, append, prefix attention, decode -- this holds.) */
#define KVP_LAUNCH_PDL 0x1u
/* KVP_LAUNCH_STALL_TEST exercises the failure path of the bounded waits
 * without faulting anything: in every prefix-attention and decode CTA one
 * warp first waits on a shared-memory barrier that nothing ever arrives on.
 * That wait gives up when the pipeline wait limit (kvp_set_wait_limit_ns)
 * runs out, sets KVP_DEVERR_TIMEOUT and an abort flag, and the CTA winds down
 * the way it does after any wait that gave up: the other warps leave their
 * waits, copies already in flight are waited for (with the default limit),
 * tensor memory is freed, and the kernel returns.  Outputs are then
 * unspecified; the context stays usable.  For tests only -- with the default
 * 2 s limit each CTA would stall for 2 s. */
#define KVP_LAUNCH_STALL_TEST 0x2u
void kvp_set_launch_options(uint32_t flags);
uint32_t kvp_get_launch_options(void);

/* How long a kernel's pipeline waits (a warp waiting for a copy, a
 * tensor-core result or another warp's data) last before they give up and
 * report KVP_DEVERR_TIMEOUT; process-wide, read at each call; 0 restores the
 * default of 2 s.  A healthy wait lasts microseconds, so the limit only
 * decides how soon a stuck kernel is reported.  The waits of a CTA that is
 * winding down (for its own copies in flight and its last tensor-core
 * commit) always keep the default, so nothing lands in its memory after it
 * exits. */
void kvp_set_wait_limit_ns(uint64_t ns);
uint64_t kvp_get_wait_limit_ns(void);

/* Reads pool->err_word on the host after everything queued on `stream`
 * before it: synchronises `stream`, stores the KVP_DEVERR_* bits in *bits
 * and returns KVP_ERR_TIMEOUT when KVP_DEVERR_TIMEOUT is among them, else
 * KVP_OK (data errors -- bad blocks, slots, pairs, lengths -- are reported in
 * *bits only).  With err_word NULL, *bits = 0.  The word is not cleared.
 * Errors: KVP_ERR_INVALID_ARG (pool or bits NULL), KVP_ERR_CUDA. */
kvp_status kvp_pool_errors(const kvp_pool *pool, uint32_t *bits, void *stream);

/* A pool of blocks in host memory with the same block geometry (num_kv_heads,
 * block_size, head_dim, dtype) as a device pool: the swap buffer of
 * preempted sequences.  k_pool, v_pool: host [num_blocks][Hkv][bs][d],
 * 16-byte aligned, page-locked and mapped into the device's address space
 * (cudaHostAlloc / cudaMallocHost memory on a unified-address system, or
 * cudaHostRegister'ed memory).  Caller-owned; the library keeps no state. */
typedef struct kvp_host_pool {
    void *k_pool;
    void *v_pool;
    int64_t num_blocks;
} kvp_host_pool;

enum { KVP_SWAP_OUT = 0, KVP_SWAP_IN = 1 };

/* Swap whole blocks between the device pool and the host pool (kvstream
 * "Features": low-priority sequences are spilled to a CPU page pool rather
 * than dropped, and its configuration sizes that pool in num_cpu_blocks with
 * preemption_policy "swap"; the kvboost post on CPU paging: KV blocks that
 * do not fit on the GPU move to system RAM by asynchronous DMA).
 *     direction KVP_SWAP_OUT: host.k_pool[pairs[i][1]] = pool.k_pool[pairs[i][0]]
 *     direction KVP_SWAP_IN:  pool.k_pool[pairs[i][1]] = host.k_pool[pairs[i][0]]
 * (whole block, all heads; same for V).  One kernel moves every pair, reading
 * or writing the host pool directly over the host link, so a list of
 * scattered blocks costs one launch, asynchronous on `stream` (a copy stream
 * lets it overlap compute on another).  pairs: device int32 [n][2] =
 * (src, dst), block ids of the source and destination pool.  Destinations
 * must be distinct; otherwise the result is undefined.  A pair naming a block
 * outside its pool is skipped and sets KVP_DEVERR_BAD_PAIR in the device
 * pool's err_word.  n == 0 is a no-op; n <= 65535 per call.  Errors:
 * KVP_ERR_INVALID_ARG for a null or misaligned pointer, a negative block
 * count or an unknown direction; no device work is queued then. */
kvp_status kvp_block_swap(const kvp_pool *pool, const kvp_host_pool *host, const int32_t *pairs, int32_t n,
                          int32_t direction, void *stream);

/* Causal attention of a chunk of new tokens over the cached prefix plus the
 * chunk itself (kvboost "How it works" step 5 and "Flash Attention (CUDA)":
 * tiled online softmax, fp16/bf16, head_dim 64/96/128, any length, causal
 * with future tiles skipped):
 *     out[t][h] = sum_j softmax_j(scale * q[t][h] . K_s[j]) V_s[j],  j <= position(t)
 *     lse[h][t] = ln(sum_j exp(scale * q[t][h] . K_s[j]))            (natural log)
 * where K_s, V_s is sequence s's logical K/V read through block_tables and
 * kv head h / (num_q_heads / num_kv_heads).  ALL keys are read from the
 * pool, so the chunk's own K/V must have been appended first.
 * q, out: device [total_q][num_q_heads][head_dim], pool dtype, 16-B aligned.
 * lse: device float [num_q_heads][total_q], or NULL.
 * max_q_len >= every N_s; max_context_len >= every context_lens[s] (they size
 * the grid; larger values only waste empty blocks).
 * num_splits: 0 = the library chooses (kvp_prefix_num_splits); >= 1 splits
 * every query tile's key range into that many parts merged by log-sum-exp.
 * When the resolved count is > 1 the call needs workspace_bytes >=
 * kvp_workspace_size(0, total_q, num_q_heads, head_dim, splits) of device
 * memory (its contents need no initialisation). */
kvp_status kvp_prefix_attn(const kvp_pool *pool, const void *q, void *out, float *lse, const int32_t *cu_seqlens_q,
                           const int32_t *context_lens, const int32_t *block_tables, int32_t max_blocks, int32_t B,
                           int32_t total_q, int32_t num_q_heads, int32_t max_q_len, int32_t max_context_len,
                           float softmax_scale, int32_t num_splits, void *workspace, size_t workspace_bytes,
                           void *stream);

/* Decode attention for a continuous batch (kvstream "Why KVStream?" and
 * "Request lifecycle": one new token per sequence per step): prefix
 * attention with N_s = 1 for every sequence, keys 0 .. context_lens[s]-1.
 * q, out: device [B][num_q_heads][head_dim]; lse: device float
 * [num_q_heads][B] or NULL.  num_q_heads / num_kv_heads must be <= 16.
 * num_splits: 0 = the library chooses (kvp_decode_num_splits); otherwise the
 * longest context is cut into at most that many key ranges, each processed
 * by its own CTA and merged by log-sum-exp; the call then needs
 * workspace_bytes >= kvp_workspace_size(1, B, num_q_heads, head_dim, splits). */
kvp_status kvp_decode_attn(const kvp_pool *pool, const void *q, void *out, float *lse, const int32_t *context_lens,
                           const int32_t *block_tables, int32_t max_blocks, int32_t B, int32_t num_q_heads,
                           int32_t max_context_len, float softmax_scale, int32_t num_splits, void *workspace,
                           size_t workspace_bytes, void *stream);

/* Bytes of split partials that kvp_decode_attn_noalloc can hold (32 MiB). */
#define KVP_DECODE_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/* Decode attention that allocates nothing and takes no workspace.  The pages
 * have no counterpart of this call: it exists for callers that cannot hand
 * the library device memory at the point of the call -- a runtime that owns
 * a fixed memory budget through its own allocator, a plug-in that has no
 * access to the host application's allocator, or a serving loop that bans
 * cudaMalloc/cudaFree because they can synchronise the device.
 * Arguments, results and errors are those of kvp_decode_attn without
 * `workspace` and `workspace_bytes`.  The split partials go to one fixed
 * array of KVP_DECODE_NOALLOC_SCRATCH_BYTES in the library's device image,
 * which every GPU that loads the library holds until the process exits.
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it; make that
 * first call before any stream capture.  Every call uses the same array and
 * it keeps the last call's contents; nothing in it needs to start at zero,
 * because each call writes every partial it reads.  Calls whose kernels
 * overlap on the GPU (e.g. on two streams without ordering) race on the
 * array: order them on one stream or with events.
 * Arguments are validated first, with kvp_decode_attn's error codes.  Then
 * the call returns KVP_ERR_WORKSPACE, launching nothing, when the split count
 * kvp_decode_attn would resolve (num_splits, or the library's choice for 0,
 * after rounding each split up to whole 32-key stages -- so a large
 * num_splits over short contexts may resolve to far fewer) needs more than
 * the array holds, i.e. when kvp_workspace_size(1, B, num_q_heads, head_dim,
 * resolved splits) exceeds KVP_DECODE_NOALLOC_SCRATCH_BYTES; pass a smaller
 * num_splits or batch.
 * It calls no cudaMalloc, cudaFree or other allocating routine. */
kvp_status kvp_decode_attn_noalloc(const kvp_pool *pool, const void *q, void *out, float *lse,
                                   const int32_t *context_lens, const int32_t *block_tables, int32_t max_blocks,
                                   int32_t B, int32_t num_q_heads, int32_t max_context_len, float softmax_scale,
                                   int32_t num_splits, void *stream);

/* Split counts the library picks for num_splits == 0. */
int32_t kvp_prefix_num_splits(int32_t B, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                              int32_t max_q_len, int32_t max_context_len);
int32_t kvp_decode_num_splits(int32_t B, int32_t num_kv_heads, int32_t block_size, int32_t max_context_len);

/* Device workspace bytes for op 0 (prefix: rows = total_q) or op 1 (decode:
 * rows = B) at a given split count; 0 when num_splits <= 1. */
size_t kvp_workspace_size(int32_t op, int32_t rows, int32_t num_q_heads, int32_t head_dim, int32_t num_splits);

/* Static, NUL-terminated description of a status code. */
const char *kvp_status_string(kvp_status status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int32_t kvp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVP_H_ */
