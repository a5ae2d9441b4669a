// kvp_cacheblend.cu -- CacheBlend recompute selection (kvboost 0.6.0, "How
// it works" > "4. Seam repair": one forward pass measures per-token cosine
// deviation between the cached K/V and the K/V with full context, and only
// the ~15% most-deviated tokens are recomputed; approximate, content-hash
// matches always take this path).
//
//  * deviation_kernel: one warp per token; its K and V for every kv head are
//    read from the pool slot and from the fresh buffer with 16-byte loads,
//    deviation = 1 - cos([K;V] cached, [K;V] fresh) in fp32.  HBM-bound.
//  * select_kernel: one CTA per sequence selects k = ceil(n * permille /
//    1000) tokens, the largest deviations first, ties to the lower position:
//    an MSB-first radix select over order-preserving 32-bit keys finds the
//    k-th largest key, then a block-wide scan in position order takes the
//    ties.  It writes the selected tokens' slots (-1 elsewhere), which
//    kvp_cache_append then overwrites with the fresh K/V.
#include "kvp_internal.cuh"

namespace kvp {
namespace {

constexpr int kDevThreads = 256;
constexpr int kSelThreads = 1024;

__device__ __forceinline__ void acc_unit(uint4 a, uint4 b, float& dot, float& na, float& nb, bool bf) {
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 x = bf ? unpack2<true>(aw[j]) : unpack2<false>(aw[j]);
        const float2 y = bf ? unpack2<true>(bw[j]) : unpack2<false>(bw[j]);
        dot = fmaf(x.x, y.x, fmaf(x.y, y.y, dot));
        na = fmaf(x.x, x.x, fmaf(x.y, x.y, na));
        nb = fmaf(y.x, y.x, fmaf(y.y, y.y, nb));
    }
}

template <bool kBF16>
__global__ void __launch_bounds__(kDevThreads) deviation_kernel(PoolView pool, const uint4* __restrict__ k_pool,
                                                                const uint4* __restrict__ v_pool,
                                                                const uint4* __restrict__ k_fresh,
                                                                const uint4* __restrict__ v_fresh,
                                                                const int64_t* __restrict__ slots, int32_t T,
                                                                float* __restrict__ dev) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int vph = pool.head_dim / 8;             // 16-byte units per (token, head)
    const int vpt = pool.num_kv_heads * vph;       // per token
    const int64_t num_slots = pool.num_blocks * pool.block_size;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (kDevThreads / 32);
    for (int64_t t = blockIdx.x * static_cast<int64_t>(kDevThreads / 32) + (threadIdx.x >> 5); t < T; t += warps) {
        const int64_t slot = __ldg(slots + t);
        if (slot < 0 || slot >= num_slots) {
            if (lane == 0) {
                report(pool.err_word, KVP_DEVERR_BAD_SLOT);
                dev[t] = -1.f;
            }
            continue;
        }
        const int64_t blk = slot / pool.block_size, row = slot - blk * pool.block_size;
        float dot = 0.f, na = 0.f, nb = 0.f;
        for (int u = lane; u < vpt; u += 32) {
            const int h = u / vph, c = u - h * vph;
            const int64_t src = ((blk * pool.num_kv_heads + h) * pool.block_size + row) * vph + c;
            acc_unit(__ldg(k_pool + src), __ldcs(k_fresh + t * vpt + u), dot, na, nb, kBF16);
            acc_unit(__ldg(v_pool + src), __ldcs(v_fresh + t * vpt + u), dot, na, nb, kBF16);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            dot += __shfl_xor_sync(0xffffffffu, dot, o);
            na += __shfl_xor_sync(0xffffffffu, na, o);
            nb += __shfl_xor_sync(0xffffffffu, nb, o);
        }
        if (lane == 0) {
            float d;
            if (na == 0.f && nb == 0.f)
                d = 0.f;
            else if (na == 0.f || nb == 0.f)
                d = 1.f;
            else
                d = fminf(fmaxf(1.f - dot / (sqrtf(na) * sqrtf(nb)), 0.f), 2.f);  // cos is in [-1, 1]
            dev[t] = d;
        }
    }
}

// Order-preserving key: larger float -> larger unsigned key.
__device__ __forceinline__ uint32_t fkey(float f) {
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__global__ void __launch_bounds__(kSelThreads) select_kernel(const float* __restrict__ dev,
                                                             const int64_t* __restrict__ slots,
                                                             const int32_t* __restrict__ cu, int32_t permille,
                                                             int64_t* __restrict__ out_slots,
                                                             int32_t* __restrict__ counts) {
    __shared__ uint32_t hist[256];
    __shared__ uint32_t sh_prefix, sh_need;
    __shared__ uint32_t warp_cnt[kSelThreads / 32];
    __shared__ uint32_t sh_base;
    pdl_trigger();
    pdl_wait();  // the deviations come from the kernel before
    const int s = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int a = __ldg(cu + s), n = __ldg(cu + s + 1) - a;
    const uint32_t k = static_cast<uint32_t>((static_cast<int64_t>(n) * permille + 999) / 1000);
    if (tid == 0) counts[s] = static_cast<int32_t>(k);
    if (k == 0) {
        for (int i = tid; i < n; i += kSelThreads) out_slots[a + i] = -1;
        return;
    }
    // Radix select: the k-th largest key, 8 bits at a time from the top.
    uint32_t prefix = 0, mask = 0, need = k;  // keys matching prefix under mask are the candidates
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += kSelThreads) hist[i] = 0;
        __syncthreads();
        for (int i = tid; i < n; i += kSelThreads) {
            const uint32_t key = fkey(__ldg(dev + a + i));
            if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 0xFFu], 1u);
        }
        __syncthreads();
        if (tid == 0) {
            uint32_t above = 0;
            int dsel = 0;
            for (int dgt = 255; dgt >= 0; --dgt) {
                if (above + hist[dgt] >= need) {
                    dsel = dgt;
                    break;
                }
                above += hist[dgt];
            }
            sh_prefix = prefix | (static_cast<uint32_t>(dsel) << shift);
            sh_need = need - above;  // how many keys equal to the final threshold are taken
        }
        __syncthreads();
        prefix = sh_prefix;
        need = sh_need;
        mask |= 0xFFu << shift;
        __syncthreads();
    }
    // prefix is the k-th largest key; take every larger key and the first
    // `need` equal keys in position order.
    if (tid == 0) sh_base = 0;
    __syncthreads();
    for (int i0 = 0; i0 < n; i0 += kSelThreads) {
        const int i = i0 + tid;
        uint32_t key = 0;
        if (i < n) key = fkey(__ldg(dev + a + i));
        const bool eq = i < n && key == prefix;
        const unsigned bal = __ballot_sync(0xffffffffu, eq);
        if (lane == 0) warp_cnt[warp] = __popc(bal);
        __syncthreads();
        uint32_t before = sh_base;
        for (int w = 0; w < warp; ++w) before += warp_cnt[w];
        before += __popc(bal & ((1u << lane) - 1u));
        if (i < n) {
            const bool sel = key > prefix || (eq && before < need);
            out_slots[a + i] = sel ? __ldg(slots + a + i) : -1;
        }
        __syncthreads();
        if (tid == 0) {
            uint32_t tot = 0;
            for (int w = 0; w < kSelThreads / 32; ++w) tot += warp_cnt[w];
            sh_base += tot;
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_kv_deviation(const PoolView& pool, const void* k_pool, const void* v_pool, const void* k_fresh,
                                const void* v_fresh, const int64_t* slots, int32_t T, float* dev,
                                cudaStream_t stream) {
    if (T <= 0) return cudaSuccess;
    int blocks = (T + kDevThreads / 32 - 1) / (kDevThreads / 32);
    int sms = 148;
    int d = 0;
    cudaGetDevice(&d);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d);
    blocks = blocks < sms * 8 ? blocks : sms * 8;
    const uint4* kp = static_cast<const uint4*>(k_pool);
    const uint4* vp = static_cast<const uint4*>(v_pool);
    const uint4* kf = static_cast<const uint4*>(k_fresh);
    const uint4* vf = static_cast<const uint4*>(v_fresh);
    return pool.dtype == KVP_BF16
               ? launch_k(deviation_kernel<true>, blocks, kDevThreads, 0, stream, pool, kp, vp, kf, vf, slots, T, dev)
               : launch_k(deviation_kernel<false>, blocks, kDevThreads, 0, stream, pool, kp, vp, kf, vf, slots, T,
                          dev);
}

cudaError_t launch_select_recompute(const float* dev, const int64_t* slots, const int32_t* cu, int32_t B,
                                    int32_t permille, int64_t* out_slots, int32_t* counts, cudaStream_t stream) {
    if (B <= 0) return cudaSuccess;
    return launch_k(select_kernel, B, kSelThreads, 0, stream, dev, slots, cu, permille, out_slots, counts);
}

}  // namespace kvp
