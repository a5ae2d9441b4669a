// kvp_cache.cu -- slot indexing, slot-mapped append and copy-on-write block
// copy.  All three are pure data movement: HBM-bound, 16-byte vector loads
// and stores, grid-stride loops sized to the SM count.
//
// Pages: kvstream 0.1.0, "Request lifecycle" steps 2-3 (one slot per new
// token; a forked block table shares pages copy-on-write); kvboost 0.6.0,
// "CPU paged attention" (fixed block pool, shared prefixes share physical
// blocks copy-on-write) and "How it works" step 5 (newly seen K/V written
// back to the cache).
#include "kvp_internal.cuh"

namespace kvp {
namespace {

constexpr int kThreads = 256;

int grid_for(int64_t work, int per_cta) {
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 148;
    }
    int64_t need = (work + per_cta - 1) / per_cta;
    int64_t cap = static_cast<int64_t>(sms) * 8;
    if (need < 1) need = 1;
    return static_cast<int>(need < cap ? need : cap);
}

// One thread per new token.  The owning sequence is found by binary search
// over cu_seqlens_q (the largest s with cu_seqlens_q[s] <= t, which skips
// sequences without new tokens).
__global__ void slot_mapping_kernel(PoolView pool, const int32_t* __restrict__ cu,
                                    const int32_t* __restrict__ ctx, const int32_t* __restrict__ bt,
                                    int32_t max_blocks, int32_t B, int32_t total_q,
                                    int64_t* __restrict__ slots) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < total_q; t += stride) {
        int lo = 0, hi = B;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(cu + mid) <= t) lo = mid; else hi = mid;
        }
        const int s = lo;
        const int64_t n = __ldg(cu + s + 1) - __ldg(cu + s);
        const int64_t pos = static_cast<int64_t>(__ldg(ctx + s)) - n + (t - __ldg(cu + s));
        const int64_t logical = pos >= 0 ? pos / pool.block_size : -1;
        int64_t slot = -1;
        if (pos < 0 || logical >= max_blocks) {
            report(pool.err_word, KVP_DEVERR_BAD_LEN);
        } else {
            const int64_t blk = __ldg(bt + static_cast<int64_t>(s) * max_blocks + logical);
            if (blk >= 0 && blk < pool.num_blocks)
                slot = blk * pool.block_size + pos % pool.block_size;
            else
                report(pool.err_word, KVP_DEVERR_BAD_BLOCK);
        }
        slots[t] = slot;
    }
}

// One thread per 16-byte vector of a (token, kv head) row, K and V together.
__global__ void append_kernel(PoolView pool, uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                              const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                              const int64_t* __restrict__ slots, int32_t T) {
    const int vec_per_head = pool.head_dim / 8;  // 16-byte vectors of 8 x 16-bit
    const int64_t vec_per_tok = static_cast<int64_t>(pool.num_kv_heads) * vec_per_head;
    const int64_t total = vec_per_tok * T;
    const int64_t num_slots = pool.num_blocks * pool.block_size;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; v < total; v += stride) {
        const int64_t t = v / vec_per_tok;
        const int64_t rem = v - t * vec_per_tok;
        const int64_t slot = __ldg(slots + t);
        if (slot == -1) continue;
        if (slot < 0 || slot >= num_slots) {
            if (rem == 0) report(pool.err_word, KVP_DEVERR_BAD_SLOT);
            continue;
        }
        const int64_t h = rem / vec_per_head;
        const int64_t c = rem - h * vec_per_head;
        const int64_t blk = slot / pool.block_size;
        const int64_t row = slot - blk * pool.block_size;
        const int64_t dst = ((blk * pool.num_kv_heads + h) * pool.block_size + row) * vec_per_head + c;
        const uint4 kv = __ldcs(k_new + v);
        const uint4 vv = __ldcs(v_new + v);
        k_pool[dst] = kv;
        v_pool[dst] = vv;
    }
}

// One thread per 16-byte vector of a whole block (all heads), K and V together.
__global__ void block_copy_kernel(PoolView pool, uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                                  const int32_t* __restrict__ pairs, int32_t n) {
    const int64_t vec_per_block =
        static_cast<int64_t>(pool.num_kv_heads) * pool.block_size * (pool.head_dim / 8);
    const int64_t total = vec_per_block * n;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; v < total; v += stride) {
        const int64_t i = v / vec_per_block;
        const int64_t e = v - i * vec_per_block;
        const int64_t src = __ldg(pairs + 2 * i);
        const int64_t dst = __ldg(pairs + 2 * i + 1);
        if (src < 0 || src >= pool.num_blocks || dst < 0 || dst >= pool.num_blocks) {
            if (e == 0) report(pool.err_word, KVP_DEVERR_BAD_PAIR);
            continue;
        }
        const uint4 kv = k_pool[src * vec_per_block + e];
        const uint4 vv = v_pool[src * vec_per_block + e];
        k_pool[dst * vec_per_block + e] = kv;
        v_pool[dst * vec_per_block + e] = vv;
    }
}

}  // namespace

cudaError_t launch_slot_mapping(const PoolView& pool, const int32_t* cu_seqlens_q, const int32_t* context_lens,
                                const int32_t* block_tables, int32_t max_blocks, int32_t B, int32_t total_q,
                                int64_t* slot_mapping, cudaStream_t stream) {
    if (total_q <= 0) return cudaSuccess;
    slot_mapping_kernel<<<grid_for(total_q, kThreads), kThreads, 0, stream>>>(
        pool, cu_seqlens_q, context_lens, block_tables, max_blocks, B, total_q, slot_mapping);
    return cudaGetLastError();
}

cudaError_t launch_cache_append(const PoolView& pool, void* k_pool, void* v_pool, const void* k_new,
                                const void* v_new, const int64_t* slot_mapping, int32_t T, cudaStream_t stream) {
    if (T <= 0) return cudaSuccess;
    const int64_t total = static_cast<int64_t>(T) * pool.num_kv_heads * (pool.head_dim / 8);
    append_kernel<<<grid_for(total, kThreads), kThreads, 0, stream>>>(
        pool, static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), static_cast<const uint4*>(k_new),
        static_cast<const uint4*>(v_new), slot_mapping, T);
    return cudaGetLastError();
}

cudaError_t launch_block_copy(const PoolView& pool, void* k_pool, void* v_pool, const int32_t* pairs, int32_t n,
                              cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    const int64_t total =
        static_cast<int64_t>(n) * pool.num_kv_heads * pool.block_size * (pool.head_dim / 8);
    block_copy_kernel<<<grid_for(total, kThreads), kThreads, 0, stream>>>(
        pool, static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), pairs, n);
    return cudaGetLastError();
}

}  // namespace kvp
