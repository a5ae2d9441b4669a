// kvp_cache.cu -- slot indexing, slot-mapped append and copy-on-write block
// copy.  All three are pure data movement: HBM-bound, 16-byte vector loads
// and stores, grid-stride loops sized to the SM count.
//
// Pages: kvstream 0.1.0, "Request lifecycle" steps 2-3 (one slot per new
// token; a forked block table shares pages copy-on-write) and "Features"
// (swap and preemption to a CPU page pool); kvboost 0.6.0,
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
    pdl_trigger();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    bool waited = false;
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
        if (!waited) {
            pdl_wait();  // before the first write: the slots may still be read upstream
            waited = true;
        }
        slots[t] = slot;
    }
    if (!waited) pdl_wait();
}

// Append.  A token's K (and V) rows for all kv heads are vpt = Hkv * d / 8
// 16-byte vectors.  A 256-thread block covers tpb = max(1, 256 / vpt) tokens
// per step; thread i owns vector i % vpt of token i / vpt (computed once, in
// 32-bit arithmetic) and walks tokens with a grid stride, kUnroll tokens per
// pass.  The new K/V rows do not depend on the slot, so each pass issues the
// data loads together with the slot loads -- one memory round trip, not two
// -- and stores once both have arrived.  (A token whose slot is -1 has its
// rows read for nothing; padding tokens are rare.)
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kThreads) append_kernel(PoolView pool, uint4* __restrict__ k_pool,
                                                          uint4* __restrict__ v_pool, const uint4* __restrict__ k_new,
                                                          const uint4* __restrict__ v_new,
                                                          const int64_t* __restrict__ slots, int32_t T, int32_t vpt,
                                                          int32_t tpb) {
    pdl_trigger();
    pdl_wait();  // the slots come from the kernel before
    const int vph = pool.head_dim / 8;  // vectors per (token, head)
    const int64_t num_slots = pool.num_blocks * pool.block_size;
    const bool wide = vpt >= kThreads;          // one token per step, several vectors per thread
    const int span = wide ? vpt : tpb * vpt;    // vector positions a block covers per step (<= 256 if !wide)
    for (int j0 = threadIdx.x; j0 < span; j0 += kThreads) {
        const int tok_local = wide ? 0 : j0 / vpt;
        const int j = j0 - tok_local * vpt;
        const int h = j / vph, c = j - h * vph;
        const int64_t step = static_cast<int64_t>(gridDim.x) * tpb;
        for (int64_t t0 = static_cast<int64_t>(blockIdx.x) * tpb + tok_local; t0 < T; t0 += step * kUnroll) {
            uint4 kv[kUnroll], vv[kUnroll];
            int64_t sl[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t t = t0 + u * step;
                sl[u] = -1;
                if (t < T) {
                    sl[u] = __ldg(slots + t);
                    kv[u] = __ldcs(k_new + t * vpt + j);
                    vv[u] = __ldcs(v_new + t * vpt + j);
                }
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t slot = sl[u];
                if (slot >= 0 && slot < num_slots) {
                    const int64_t blk = slot / pool.block_size;
                    const int64_t row = slot - blk * pool.block_size;
                    const int64_t dst = ((blk * pool.num_kv_heads + h) * pool.block_size + row) * vph + c;
                    k_pool[dst] = kv[u];
                    v_pool[dst] = vv[u];
                } else if (slot != -1 && j == 0) {
                    report(pool.err_word, KVP_DEVERR_BAD_SLOT);
                }
            }
        }
    }
}

// Block moves: copy-on-write within the device pool, and swap between the
// device pool and a host pool (read or written over the host link through
// the host memory's device mapping).  A block of either pool is vpb =
// Hkv * bs * d / 8 16-byte vectors; blockIdx.y picks the pair and blockIdx.x
// a 512-vector chunk of it, each thread moving two vectors of K and two of V
// with all four loads issued before the stores.
__global__ void __launch_bounds__(kThreads) block_move_kernel(const uint4* __restrict__ ks,
                                                              const uint4* __restrict__ vs, int64_t src_blocks,
                                                              uint4* __restrict__ kd, uint4* __restrict__ vd,
                                                              int64_t dst_blocks, const int32_t* __restrict__ pairs,
                                                              int32_t vpb, uint32_t* err_word) {
    pdl_trigger();
    pdl_wait();
    const int i = blockIdx.y;
    const int64_t src = __ldg(pairs + 2 * i);
    const int64_t dst = __ldg(pairs + 2 * i + 1);
    if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks) {
        if (threadIdx.x == 0 && blockIdx.x == 0) report(err_word, KVP_DEVERR_BAD_PAIR);
        return;
    }
    const int e0 = blockIdx.x * 2 * kThreads + threadIdx.x, e1 = e0 + kThreads;
    const uint4* kss = ks + src * vpb;
    const uint4* vss = vs + src * vpb;
    uint4* kdd = kd + dst * vpb;
    uint4* vdd = vd + dst * vpb;
    uint4 k0, v0, k1, v1;
    if (e0 < vpb) {
        k0 = kss[e0];
        v0 = vss[e0];
    }
    if (e1 < vpb) {
        k1 = kss[e1];
        v1 = vss[e1];
    }
    if (e0 < vpb) {
        kdd[e0] = k0;
        vdd[e0] = v0;
    }
    if (e1 < vpb) {
        kdd[e1] = k1;
        vdd[e1] = v1;
    }
}

}  // namespace

cudaError_t launch_slot_mapping(const PoolView& pool, const int32_t* cu_seqlens_q, const int32_t* context_lens,
                                const int32_t* block_tables, int32_t max_blocks, int32_t B, int32_t total_q,
                                int64_t* slot_mapping, cudaStream_t stream) {
    if (total_q <= 0) return cudaSuccess;
    return launch_k(slot_mapping_kernel, grid_for(total_q, kThreads), kThreads, 0, stream, pool, cu_seqlens_q,
                    context_lens, block_tables, max_blocks, B, total_q, slot_mapping);
}

cudaError_t launch_cache_append(const PoolView& pool, void* k_pool, void* v_pool, const void* k_new,
                                const void* v_new, const int64_t* slot_mapping, int32_t T, cudaStream_t stream) {
    if (T <= 0) return cudaSuccess;
    const int32_t vpt = pool.num_kv_heads * (pool.head_dim / 8);
    const int32_t tpb = vpt >= kThreads ? 1 : kThreads / vpt;
    const int64_t steps = (static_cast<int64_t>(T) + tpb - 1) / tpb;
    // kUnroll steps per block, so that every thread has kUnroll tokens' rows
    // in flight; a block loops only once the steps outnumber the blocks the
    // GPU holds.
    return launch_k(append_kernel, grid_for(steps, kUnroll), kThreads, 0, stream, pool, static_cast<uint4*>(k_pool),
                    static_cast<uint4*>(v_pool), static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
                    slot_mapping, T, vpt, tpb);
}

cudaError_t launch_block_copy(const PoolView& pool, void* k_pool, void* v_pool, const int32_t* pairs, int32_t n,
                              cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    const int32_t vpb = pool.num_kv_heads * pool.block_size * (pool.head_dim / 8);
    if (n > 65535) return cudaErrorInvalidValue;
    const dim3 grid((vpb + 2 * kThreads - 1) / (2 * kThreads), n);
    return launch_k(block_move_kernel, grid, kThreads, 0, stream, static_cast<const uint4*>(k_pool),
                    static_cast<const uint4*>(v_pool), pool.num_blocks, static_cast<uint4*>(k_pool),
                    static_cast<uint4*>(v_pool), pool.num_blocks, pairs, vpb, pool.err_word);
}

cudaError_t launch_block_swap(const PoolView& pool, void* k_pool, void* v_pool, void* host_k, void* host_v,
                              int64_t host_blocks, const int32_t* pairs, int32_t n, bool to_host,
                              cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    const int32_t vpb = pool.num_kv_heads * pool.block_size * (pool.head_dim / 8);
    if (n > 65535) return cudaErrorInvalidValue;
    const dim3 grid((vpb + 2 * kThreads - 1) / (2 * kThreads), n);
    if (to_host)
        return launch_k(block_move_kernel, grid, kThreads, 0, stream, static_cast<const uint4*>(k_pool),
                        static_cast<const uint4*>(v_pool), pool.num_blocks, static_cast<uint4*>(host_k),
                        static_cast<uint4*>(host_v), host_blocks, pairs, vpb, pool.err_word);
    return launch_k(block_move_kernel, grid, kThreads, 0, stream, static_cast<const uint4*>(host_k),
                    static_cast<const uint4*>(host_v), host_blocks, static_cast<uint4*>(k_pool),
                    static_cast<uint4*>(v_pool), pool.num_blocks, pairs, vpb, pool.err_word);
}

}  // namespace kvp
