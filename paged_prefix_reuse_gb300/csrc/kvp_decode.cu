// kvp_decode.cu -- decode attention for a continuous batch (one new token
// per sequence; kvstream 0.1.0 "Request lifecycle"), split over the key
// range, plus the log-sum-exp merge of split partials shared with the
// prefix kernel.
//
// Decode reads every K/V byte of the context once and does ~g*4 flops per
// byte (g = query heads per kv head), so it is HBM-bound.  Design:
//  * one CTA per (key range, kv head, sequence); the g query heads of the
//    group share each loaded page;
//  * a producer warp streams stages of 16 keys (32 for 32-token blocks): the
//    K and V page-heads of the stage's physical blocks, addressed through the
//    block table, with 2-D TMA loads into a ring of four stage slots (32 KB at
//    head_dim 128), swizzled so that the consumers' ldmatrix reads are
//    conflict-free;
//  * two consumer warps take stages round-robin and run q.K^T and P.V as
//    m16n8k16 tensor-core MMAs (the group padded to 16 rows) with an fp32
//    online softmax; the warps' partial states are merged through shared
//    memory at the end (or written as two partials per split);
//  * 96 threads and 128 registers: five CTAs share an SM, so that about
//    160 KB of loads can be in flight per SM;
//  * with more than one split, each CTA writes a normalised partial (O, lse)
//    and merge_kernel combines them: lse = log2 sum_i 2^lse_i,
//    O = sum_i 2^(lse_i - lse) O_i.
#include "kvp_decode_impl.cuh"

namespace kvp {
namespace {

// One warp per output row: merge `splits` partials (normalised O, log2 lse):
//   lse = log2 sum_i 2^lse_i,  O = sum_i 2^(lse_i - lse) O_i.
// Lane i computes the weight of split i (32 at a time); the weights are
// broadcast by shuffle while each lane accumulates four adjacent columns with
// 16-byte loads, so one split's partial is one coalesced 4*D-byte read.
template <bool kBF16, int D>
__global__ void __launch_bounds__(256) merge_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_lse,
                                                    int32_t rows, int32_t Hq, int32_t max_splits,
                                                    void* __restrict__ out, float* __restrict__ lse,
                                                    int32_t lse_stride, const int32_t* __restrict__ ctx,
                                                    int32_t block_size, int32_t pages_per_split,
                                                    int32_t parts_per_split) {
    pdl_trigger();
    pdl_wait();  // the partials come from the kernel before
    constexpr int V4 = D / 4;  // float4 columns per row: 16, 24 or 32
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= rows) return;
    const int64_t row = warp;
    // max_splits * parts_per_split partials per row; a decode row has only
    // its own sequence's splits.
    int splits = max_splits;
    if (ctx) {
        const int L = __ldg(ctx + row / Hq);
        const int np = (L + block_size - 1) / block_size;
        splits = max(0, min(max_splits, (np + pages_per_split - 1) / pages_per_split));
    }
    splits *= parts_per_split;
    max_splits *= parts_per_split;
    const float* lrow = ws_lse + row * max_splits;
    float M = -INFINITY;
    for (int i = lane; i < splits; i += 32) M = fmaxf(M, __ldg(lrow + i));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float sum = 0.f;
    for (int i = lane; i < splits; i += 32) {
        const float li = __ldg(lrow + i);
        sum += (li == -INFINITY) ? 0.f : fast_exp2(li - M);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float tot = (M == -INFINITY || sum <= 0.f) ? -INFINITY : M + __log2f(sum);

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4* orow = reinterpret_cast<const float4*>(ws_o + row * max_splits * D);
    if (tot != -INFINITY) {
        for (int base = 0; base < splits; base += 32) {
            const int i = base + lane;
            const float li = i < splits ? __ldg(lrow + i) : -INFINITY;
            const float wi = (li == -INFINITY) ? 0.f : fast_exp2(li - tot);
            const int n = min(32, splits - base);
            int k = 0;
            for (; k + 4 <= n; k += 4) {
                float w[4];
                float4 v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    w[u] = __shfl_sync(0xffffffffu, wi, k + u);
                    v[u] = lane < V4 ? __ldg(orow + static_cast<int64_t>(base + k + u) * V4 + lane)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    acc.x = fmaf(w[u], v[u].x, acc.x);
                    acc.y = fmaf(w[u], v[u].y, acc.y);
                    acc.z = fmaf(w[u], v[u].z, acc.z);
                    acc.w = fmaf(w[u], v[u].w, acc.w);
                }
            }
            for (; k < n; ++k) {
                const float w0 = __shfl_sync(0xffffffffu, wi, k);
                if (lane < V4) {
                    const float4 v0 = __ldg(orow + static_cast<int64_t>(base + k) * V4 + lane);
                    acc.x = fmaf(w0, v0.x, acc.x);
                    acc.y = fmaf(w0, v0.y, acc.y);
                    acc.z = fmaf(w0, v0.z, acc.z);
                    acc.w = fmaf(w0, v0.w, acc.w);
                }
            }
        }
    }
    if (lane < V4) {
        uint2 pk;
        pk.x = pack2<kBF16>(acc.x, acc.y);
        pk.y = pack2<kBF16>(acc.z, acc.w);
        reinterpret_cast<uint2*>(static_cast<uint8_t*>(out) + row * D * 2)[lane] = pk;
    }
    if (lane == 0 && lse) lse[(row % Hq) * lse_stride + row / Hq] = tot * 0.69314718055994531f;
}

template <bool kBF16, int D, int SK>
cudaError_t launch_decode_t(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                            cudaStream_t stream) {
    return launch_decode_kernel<kBF16, D, SK, 0>(p, tk, tv, stream);
}

template <bool kBF16, int D>
cudaError_t launch_decode_d(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                            cudaStream_t stream) {
    return p.pool.block_size <= 16 ? launch_decode_t<kBF16, D, 16>(p, tk, tv, stream)
                                   : launch_decode_t<kBF16, D, 32>(p, tk, tv, stream);
}

}  // namespace

cudaError_t launch_decode_attn(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                               cudaStream_t stream) {
    const bool bf = p.pool.dtype == KVP_BF16;
    switch (p.pool.head_dim) {
        case 64: return bf ? launch_decode_d<true, 64>(p, tk, tv, stream) : launch_decode_d<false, 64>(p, tk, tv, stream);
        case 96: return bf ? launch_decode_d<true, 96>(p, tk, tv, stream) : launch_decode_d<false, 96>(p, tk, tv, stream);
        case 128: return bf ? launch_decode_d<true, 128>(p, tk, tv, stream) : launch_decode_d<false, 128>(p, tk, tv, stream);
        default: return cudaErrorInvalidValue;
    }
}

int decode_parts_per_split() { return kConsumerWarps; }

cudaError_t launch_merge(const float* ws_o, const float* ws_lse, int32_t rows, int32_t num_q_heads,
                         int32_t head_dim, int32_t max_splits, int32_t dtype, void* out, float* lse,
                         int32_t lse_stride, const int32_t* context_lens, int32_t block_size,
                         int32_t pages_per_split, int32_t parts_per_split, cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    const int threads = 256;
    const int blocks = (rows * 32 + threads - 1) / threads;
    const bool bf = dtype == KVP_BF16;
#define KVP_MERGE(BF, DD)                                                                                     \
    return launch_k(merge_kernel<BF, DD>, blocks, threads, 0, stream, ws_o, ws_lse, rows, num_q_heads, max_splits, \
                    out, lse, lse_stride, context_lens, block_size, pages_per_split, parts_per_split)
    switch (head_dim) {
        case 64: if (bf) KVP_MERGE(true, 64); else KVP_MERGE(false, 64);
        case 96: if (bf) KVP_MERGE(true, 96); else KVP_MERGE(false, 96);
        case 128: if (bf) KVP_MERGE(true, 128); else KVP_MERGE(false, 128);
        default: return cudaErrorInvalidValue;
    }
#undef KVP_MERGE
    return cudaGetLastError();
}

}  // namespace kvp
