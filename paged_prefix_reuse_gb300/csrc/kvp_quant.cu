// kvp_quant.cu -- the quantized KV pool: quantization of whole blocks and
// decode attention over a context whose cached prefix is quantized.
//
// Pages: kvboost 0.6.0, "Optional: KV quantization" (cached K/V in 8 or 4
// bits, K per channel and V per token as in KIVI, for ~2x / 4x less memory).
// The format (kvp_qpool in kvp.h): one quantization group per page of one kv
// head -- K per channel over the page's tokens, V per token over the
// channels -- asymmetric min/max codes with an fp16 scale rounded up and an
// fp16 min rounded down, codes computed in fp32 against those stored values.
//
// Decode over the quantized prefix uses the decode kernel of
// kvp_decode_impl.cuh with BITS = 8 or 4: a quantized page arrives as four
// bulk copies (codes and scales, ~57% / ~32% of its 16-bit bytes at d=128)
// and the consumer warp dequantizes it into a 16-bit tile before the same
// tensor-core products; the live suffix's pages take the 16-bit TMA path.
#include "kvp_decode_impl.cuh"

namespace kvp {
namespace {

constexpr int kQThreads = 128;

// Scale and min of one group, as stored (fp16, directed rounding) and as
// used (their fp32 values).  A non-finite result flags KVP_DEVERR_QRANGE.
__device__ __forceinline__ void group_params(float mn, float mx, float levels, __half& sh, __half& zh, float& s,
                                             float& z, uint32_t* err) {
    sh = __float2half_ru(__fdiv_rn(__fsub_rn(mx, mn), levels));
    zh = __float2half_rd(mn);
    s = __half2float(sh);
    z = __half2float(zh);
    if (!isfinite(s) || !isfinite(z)) report(err, KVP_DEVERR_QRANGE);
}

// code = clamp(round_half_even((x - z) / s), 0, levels), each step one fp32
// operation; a zero scale (constant group) gives code 0.
__device__ __forceinline__ uint32_t qcode(float x, float s, float z, int levels) {
    if (!(s > 0.f)) return 0u;
    const int c = __float2int_rn(__fdiv_rn(__fsub_rn(x, z), s));
    return static_cast<uint32_t>(min(max(c, 0), levels));
}

// One CTA per (pair, kv head).  K: thread t handles channels 2t and 2t+1 over
// the block's tokens; V: warp w handles tokens w, w+4, ..., its lanes the
// channel pairs of the token.  Codes of a channel pair are stored together:
// two bytes at 8 bits, one byte (even channel in the low nibble) at 4 bits.
template <bool kBF16, int BITS>
__global__ void __launch_bounds__(kQThreads) quantize_kernel(const uint16_t* __restrict__ kp,
                                                             const uint16_t* __restrict__ vp, PoolView pool,
                                                             QPoolView qp, const int32_t* __restrict__ pairs) {
    constexpr int kLevels = (1 << BITS) - 1;
    pdl_trigger();
    pdl_wait();
    const int i = blockIdx.x, h = blockIdx.y;
    const int64_t src = __ldg(pairs + 2 * i), dst = __ldg(pairs + 2 * i + 1);
    if (src < 0 || src >= pool.num_blocks || dst < 0 || dst >= qp.num_blocks) {
        if (threadIdx.x == 0 && h == 0) report(pool.err_word, KVP_DEVERR_BAD_PAIR);
        return;
    }
    const int BS = pool.block_size, D = pool.head_dim, Hkv = pool.num_kv_heads;
    const int crow = D * BITS / 8;
    const int64_t ps = src * Hkv + h, pd = dst * Hkv + h;
    const uint16_t* K = kp + ps * BS * D;
    const uint16_t* V = vp + ps * BS * D;
    uint8_t* kc = qp.k_codes + pd * BS * crow;
    uint8_t* vc = qp.v_codes + pd * BS * crow;
    __half* km = qp.k_meta + pd * 2 * D;
    __half* vm = qp.v_meta + pd * BS * 2;
    uint32_t* err = pool.err_word;

    for (int c2 = threadIdx.x; c2 < D / 2; c2 += kQThreads) {
        float mn0 = INFINITY, mx0 = -INFINITY, mn1 = INFINITY, mx1 = -INFINITY;
        for (int t = 0; t < BS; ++t) {
            const float2 x = unpack2<kBF16>(*reinterpret_cast<const uint32_t*>(K + t * D + 2 * c2));
            mn0 = fminf(mn0, x.x);
            mx0 = fmaxf(mx0, x.x);
            mn1 = fminf(mn1, x.y);
            mx1 = fmaxf(mx1, x.y);
        }
        __half sh0, zh0, sh1, zh1;
        float s0, z0, s1, z1;
        group_params(mn0, mx0, static_cast<float>(kLevels), sh0, zh0, s0, z0, err);
        group_params(mn1, mx1, static_cast<float>(kLevels), sh1, zh1, s1, z1, err);
        km[2 * c2] = sh0;
        km[2 * c2 + 1] = sh1;
        km[D + 2 * c2] = zh0;
        km[D + 2 * c2 + 1] = zh1;
        for (int t = 0; t < BS; ++t) {
            const float2 x = unpack2<kBF16>(*reinterpret_cast<const uint32_t*>(K + t * D + 2 * c2));
            const uint32_t a = qcode(x.x, s0, z0, kLevels), b = qcode(x.y, s1, z1, kLevels);
            if constexpr (BITS == 8)
                *reinterpret_cast<uint16_t*>(kc + t * crow + 2 * c2) = static_cast<uint16_t>(a | (b << 8));
            else
                kc[t * crow + c2] = static_cast<uint8_t>(a | (b << 4));
        }
    }

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int t = warp; t < BS; t += kQThreads / 32) {
        float mn = INFINITY, mx = -INFINITY;
        for (int c2 = lane; c2 < D / 2; c2 += 32) {
            const float2 x = unpack2<kBF16>(*reinterpret_cast<const uint32_t*>(V + t * D + 2 * c2));
            mn = fminf(mn, fminf(x.x, x.y));
            mx = fmaxf(mx, fmaxf(x.x, x.y));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        }
        __half sh, zh;
        float s, z;
        group_params(mn, mx, static_cast<float>(kLevels), sh, zh, s, z, lane == 0 ? err : nullptr);
        if (lane == 0) {
            vm[2 * t] = sh;
            vm[2 * t + 1] = zh;
        }
        for (int c2 = lane; c2 < D / 2; c2 += 32) {
            const float2 x = unpack2<kBF16>(*reinterpret_cast<const uint32_t*>(V + t * D + 2 * c2));
            const uint32_t a = qcode(x.x, s, z, kLevels), b = qcode(x.y, s, z, kLevels);
            if constexpr (BITS == 8)
                *reinterpret_cast<uint16_t*>(vc + t * crow + 2 * c2) = static_cast<uint16_t>(a | (b << 8));
            else
                vc[t * crow + c2] = static_cast<uint8_t>(a | (b << 4));
        }
    }
}

template <bool kBF16, int D>
cudaError_t launch_decode_q_d(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                              cudaStream_t stream) {
    return p.qpool.bits == 8 ? launch_decode_kernel<kBF16, D, 16, 8>(p, tk, tv, stream)
                             : launch_decode_kernel<kBF16, D, 16, 4>(p, tk, tv, stream);
}

}  // namespace

cudaError_t launch_quantize_blocks(const PoolView& pool, const void* k_pool, const void* v_pool,
                                   const QPoolView& qpool, const int32_t* pairs, int32_t n, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    const dim3 grid(n, pool.num_kv_heads);
    const uint16_t* k = static_cast<const uint16_t*>(k_pool);
    const uint16_t* v = static_cast<const uint16_t*>(v_pool);
    const bool bf = pool.dtype == KVP_BF16;
    if (qpool.bits == 8)
        return bf ? launch_k(quantize_kernel<true, 8>, grid, kQThreads, 0, stream, k, v, pool, qpool, pairs)
                  : launch_k(quantize_kernel<false, 8>, grid, kQThreads, 0, stream, k, v, pool, qpool, pairs);
    return bf ? launch_k(quantize_kernel<true, 4>, grid, kQThreads, 0, stream, k, v, pool, qpool, pairs)
              : launch_k(quantize_kernel<false, 4>, grid, kQThreads, 0, stream, k, v, pool, qpool, pairs);
}

cudaError_t launch_decode_attn_q(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                                 cudaStream_t stream) {
    const bool bf = p.pool.dtype == KVP_BF16;
    switch (p.pool.head_dim) {
        case 64: return bf ? launch_decode_q_d<true, 64>(p, tk, tv, stream) : launch_decode_q_d<false, 64>(p, tk, tv, stream);
        case 96: return bf ? launch_decode_q_d<true, 96>(p, tk, tv, stream) : launch_decode_q_d<false, 96>(p, tk, tv, stream);
        case 128: return bf ? launch_decode_q_d<true, 128>(p, tk, tv, stream) : launch_decode_q_d<false, 128>(p, tk, tv, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kvp
