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
// Lane i holds lse of partials i, i + 32, ... (the first 128 in registers);
// each lane owns four adjacent columns of O.  The row's lse loads and the O
// rows of its first kChunk partials are issued together, before any of them
// is used, so a row with up to kChunk partials costs one memory round trip;
// later chunks of O rows are loaded kChunk at a time.  The weights reach the
// lanes by shuffle (past the first 128 partials, from a broadcast load).
template <bool kBF16, int D>
__global__ void __launch_bounds__(256) merge_kernel(const float* ws_o, const float* ws_lse,
                                                    int32_t rows, int32_t Hq, int32_t max_splits,
                                                    void* __restrict__ out, float* __restrict__ lse,
                                                    int32_t lse_stride, const int32_t* __restrict__ ctx,
                                                    int32_t block_size, int32_t pages_per_split,
                                                    int32_t parts_per_split) {
    constexpr int V4 = D / 4;     // float4 columns per row: 16, 24 or 32
    constexpr int kChunk = 16;    // O rows loaded at once
    constexpr int kMaxParts = 128;
    pdl_trigger();
    // The partials come from the kernel before: nothing is read before this
    // wait, and they are read through L2 (ld.global.cg), not the
    // non-coherent path, so no load can be taken ahead of it.
    pdl_wait();
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
    const int nparts = splits * parts_per_split;
    const int stride = max_splits * parts_per_split;
    const float* lrow = ws_lse + row * stride;
    const float4* orow = reinterpret_cast<const float4*>(ws_o + row * stride * D);

    float lv[kMaxParts / 32];
#pragma unroll
    for (int k = 0; k < kMaxParts / 32; ++k) lv[k] = lane + 32 * k < nparts ? __ldcg(lrow + lane + 32 * k) : -INFINITY;
    float4 ov[kChunk];
#pragma unroll
    for (int u = 0; u < kChunk; ++u)
        ov[u] = (u < nparts && lane < V4) ? __ldcg(orow + static_cast<int64_t>(u) * V4 + lane)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);

    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < kMaxParts / 32; ++k) M = fmaxf(M, lv[k]);
    for (int i = kMaxParts + lane; i < nparts; i += 32) M = fmaxf(M, __ldcg(lrow + i));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float sum = 0.f;
#pragma unroll
    for (int k = 0; k < kMaxParts / 32; ++k) sum += (lv[k] == -INFINITY) ? 0.f : fast_exp2(lv[k] - M);
    for (int i = kMaxParts + lane; i < nparts; i += 32) {
        const float li = __ldcg(lrow + i);
        sum += (li == -INFINITY) ? 0.f : fast_exp2(li - M);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float tot = (M == -INFINITY || sum <= 0.f) ? -INFINITY : M + __log2f(sum);
    float wv[kMaxParts / 32];  // lane i: weight of partials i, i + 32, ...
#pragma unroll
    for (int k = 0; k < kMaxParts / 32; ++k)
        wv[k] = (tot == -INFINITY || lv[k] == -INFINITY) ? 0.f : fast_exp2(lv[k] - tot);

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int base = 0; base < nparts; base += kChunk) {
        if (base > 0) {
#pragma unroll
            for (int u = 0; u < kChunk; ++u)
                ov[u] = (base + u < nparts && lane < V4)
                            ? __ldcg(orow + static_cast<int64_t>(base + u) * V4 + lane)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // A chunk lies within one group of 32 partials: its weights sit in
        // wv[base / 32] of lanes base % 32 .. base % 32 + kChunk - 1.
        const int kq = base >> 5;
        float wsrc = 0.f;
#pragma unroll
        for (int k = 0; k < kMaxParts / 32; ++k) wsrc = kq == k ? wv[k] : wsrc;
#pragma unroll
        for (int u = 0; u < kChunk; ++u) {
            const int i = base + u;
            float w = __shfl_sync(0xffffffffu, wsrc, i & 31);
            if (i >= kMaxParts && i < nparts) {
                const float li = __ldcg(lrow + i);
                w = (tot == -INFINITY || li == -INFINITY) ? 0.f : fast_exp2(li - tot);
            }
            acc.x = fmaf(w, ov[u].x, acc.x);
            acc.y = fmaf(w, ov[u].y, acc.y);
            acc.z = fmaf(w, ov[u].z, acc.z);
            acc.w = fmaf(w, ov[u].w, acc.w);
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
    return launch_decode_kernel<kBF16, D, SK>(p, tk, tv, stream);
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
