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
// Computed without a division in the common case.  With r = 1/s
// (correctly rounded), q' = (x - z) * r is within |q| * 1.8e-7 of the
// correctly rounded quotient q = (x - z) / s: within 1e-4 for |q'| < 512.
// So when q' lies farther than 1e-4 from a half-integer, q and q' round to
// the same integer; when |q'| >= 512 both lie far outside [0, levels] and
// clamp alike.  Otherwise (and for a NaN) the exact division decides, so the
// result always equals that of the division.
__device__ __forceinline__ uint32_t qcode_fast(float x, float s, float z, float r, int levels) {
    if (!(s > 0.f)) return 0u;
    const float d = __fsub_rn(x, z);
    const float q = __fmul_rn(d, r);
    const float f = fabsf(q - rintf(q));
    int c;
    if (f < 0.4999f || fabsf(q) >= 512.f)
        c = __float2int_rn(q);
    else
        c = __float2int_rn(__fdiv_rn(d, s));
    return static_cast<uint32_t>(min(max(c, 0), levels));
}

// One warp per (pair, kv head) page-head, four per CTA.  Lane l owns the
// 16-byte unit u = l % SEG (channels 8u .. 8u+7; lanes with u >= D/8 idle)
// of rows r0 = l / SEG, r0 + R, ... (R = 32 / SEG rows per pass), and issues
// all its loads of K (then of V) before any arithmetic.  K: per-channel
// minimum and maximum over the lane's rows, combined across the R lanes that
// share the unit; V: per-row minimum and maximum over the lane's 8 channels,
// combined across the row's lanes.  Codes and scales follow the same fp32
// steps as before, so the result is bit-for-bit the format's.
template <bool kBF16, int BITS, int D, int BS>
__global__ void __launch_bounds__(kQThreads) quantize_kernel(const uint16_t* __restrict__ kp,
                                                             const uint16_t* __restrict__ vp, PoolView pool,
                                                             QPoolView qp, const int32_t* __restrict__ pairs,
                                                             int32_t n) {
    constexpr int kLevels = (1 << BITS) - 1;
    constexpr int U = D / 8;              // 16-byte units per row
    constexpr int SEG = U > 8 ? 16 : 8;   // lanes per row segment
    constexpr int R = 32 / SEG;           // rows per pass
    constexpr int NR = BS / R;            // rows per lane
    constexpr int CROW = D * BITS / 8;    // code bytes per row
    pdl_trigger();
    pdl_wait();
    const int Hkv = pool.num_kv_heads;
    const int wg = blockIdx.x * (kQThreads / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (wg >= n * Hkv) return;
    const int i = wg / Hkv, h = wg - (wg / Hkv) * Hkv;
    const int64_t src = __ldg(pairs + 2 * i), dst = __ldg(pairs + 2 * i + 1);
    if (src < 0 || src >= pool.num_blocks || dst < 0 || dst >= qp.num_blocks) {
        if (lane == 0 && h == 0) report(pool.err_word, KVP_DEVERR_BAD_PAIR);
        return;
    }
    const int64_t ps = src * Hkv + h, pd = dst * Hkv + h;
    const uint4* K = reinterpret_cast<const uint4*>(kp + ps * BS * D);
    const uint4* V = reinterpret_cast<const uint4*>(vp + ps * BS * D);
    uint8_t* kc = qp.k_codes + pd * BS * CROW;
    uint8_t* vc = qp.v_codes + pd * BS * CROW;
    __half* km = qp.k_meta + pd * 2 * D;
    __half* vm = qp.v_meta + pd * BS * 2;
    uint32_t* err = pool.err_word;
    const int u = lane % SEG, r0 = lane / SEG;
    const bool act = u < U;

    // Eight codes of one unit, stored as 8 bytes (8 bits) or 4 (4 bits, the
    // even channel in the low nibble).
    auto store_codes = [&](uint8_t* row, const uint32_t (&c)[8]) {
        if constexpr (BITS == 8) {
            *reinterpret_cast<uint2*>(row + 8 * u) =
                make_uint2(c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24), c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24));
        } else {
            *reinterpret_cast<uint32_t*>(row + 4 * u) = c[0] | (c[1] << 4) | (c[2] << 8) | (c[3] << 12) | (c[4] << 16) |
                                                        (c[5] << 20) | (c[6] << 24) | (c[7] << 28);
        }
    };
    auto unpack8 = [&](uint4 a, float (&x)[8]) {
        const float2 p0 = unpack2<kBF16>(a.x), p1 = unpack2<kBF16>(a.y), p2 = unpack2<kBF16>(a.z),
                     p3 = unpack2<kBF16>(a.w);
        x[0] = p0.x; x[1] = p0.y; x[2] = p1.x; x[3] = p1.y; x[4] = p2.x; x[5] = p2.y; x[6] = p3.x; x[7] = p3.y;
    };

    // ---- K: per channel over the page's tokens ----
    {
        uint4 w[NR];
#pragma unroll
        for (int k = 0; k < NR; ++k) w[k] = act ? __ldg(K + (r0 + R * k) * U + u) : make_uint4(0, 0, 0, 0);
        float mn[8], mx[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            mn[c] = INFINITY;
            mx[c] = -INFINITY;
        }
#pragma unroll
        for (int k = 0; k < NR; ++k) {
            float x[8];
            unpack8(w[k], x);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                mn[c] = fminf(mn[c], x[c]);
                mx[c] = fmaxf(mx[c], x[c]);
            }
        }
#pragma unroll
        for (int o = SEG; o < 32; o <<= 1) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                mn[c] = fminf(mn[c], __shfl_xor_sync(0xffffffffu, mn[c], o));
                mx[c] = fmaxf(mx[c], __shfl_xor_sync(0xffffffffu, mx[c], o));
            }
        }
        if (act) {
            float s[8], z[8];
            __half sh[8], zh[8];
#pragma unroll
            for (int c = 0; c < 8; ++c)
                group_params(mn[c], mx[c], static_cast<float>(kLevels), sh[c], zh[c], s[c], z[c],
                             r0 == 0 ? err : nullptr);
            if (r0 == 0) {
                auto pack_h = [](const __half (&a)[8]) {
                    uint32_t w[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        w[j] = static_cast<uint32_t>(__half_as_ushort(a[2 * j])) |
                               (static_cast<uint32_t>(__half_as_ushort(a[2 * j + 1])) << 16);
                    return make_uint4(w[0], w[1], w[2], w[3]);
                };
                *reinterpret_cast<uint4*>(km + 8 * u) = pack_h(sh);
                *reinterpret_cast<uint4*>(km + D + 8 * u) = pack_h(zh);
            }
            float rs[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) rs[c] = s[c] > 0.f ? __frcp_rn(s[c]) : 0.f;
#pragma unroll
            for (int k = 0; k < NR; ++k) {
                float x[8];
                unpack8(w[k], x);
                uint32_t c8[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) c8[c] = qcode_fast(x[c], s[c], z[c], rs[c], kLevels);
                store_codes(kc + (r0 + R * k) * CROW, c8);
            }
        }
    }
    // ---- V: per token over the channels ----
    {
        uint4 w[NR];
#pragma unroll
        for (int k = 0; k < NR; ++k) w[k] = act ? __ldg(V + (r0 + R * k) * U + u) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int k = 0; k < NR; ++k) {
            float x[8];
            unpack8(w[k], x);
            float mn = INFINITY, mx = -INFINITY;
            if (act) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    mn = fminf(mn, x[c]);
                    mx = fmaxf(mx, x[c]);
                }
            }
#pragma unroll
            for (int o = 1; o < SEG; o <<= 1) {
                mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            }
            const int t = r0 + R * k;
            __half sh, zh;
            float s, z;
            group_params(mn, mx, static_cast<float>(kLevels), sh, zh, s, z, u == 0 ? err : nullptr);
            if (u == 0) {
                vm[2 * t] = sh;
                vm[2 * t + 1] = zh;
            }
            if (act) {
                const float r = s > 0.f ? __frcp_rn(s) : 0.f;
                uint32_t c8[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) c8[c] = qcode_fast(x[c], s, z, r, kLevels);
                store_codes(vc + t * CROW, c8);
            }
        }
    }
}

template <bool kBF16, int D>
cudaError_t launch_decode_q_d(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                              cudaStream_t stream) {
    return p.qpool.bits == 8 ? launch_decode_kernel<kBF16, D, 16, 8>(p, tk, tv, stream)
                             : launch_decode_kernel<kBF16, D, 16, 4>(p, tk, tv, stream);
}

template <bool kBF16, int BITS, int D>
cudaError_t launch_quantize_d(const PoolView& pool, const uint16_t* k, const uint16_t* v, const QPoolView& qpool,
                              const int32_t* pairs, int32_t n, cudaStream_t stream) {
    const int64_t warps = static_cast<int64_t>(n) * pool.num_kv_heads;
    const dim3 grid(static_cast<unsigned>((warps + kQThreads / 32 - 1) / (kQThreads / 32)));
    switch (pool.block_size) {
        case 8: return launch_k(quantize_kernel<kBF16, BITS, D, 8>, grid, kQThreads, 0, stream, k, v, pool, qpool, pairs, n);
        case 16: return launch_k(quantize_kernel<kBF16, BITS, D, 16>, grid, kQThreads, 0, stream, k, v, pool, qpool, pairs, n);
        case 32: return launch_k(quantize_kernel<kBF16, BITS, D, 32>, grid, kQThreads, 0, stream, k, v, pool, qpool, pairs, n);
        default: return cudaErrorInvalidValue;
    }
}

template <bool kBF16, int BITS>
cudaError_t launch_quantize_b(const PoolView& pool, const uint16_t* k, const uint16_t* v, const QPoolView& qpool,
                              const int32_t* pairs, int32_t n, cudaStream_t stream) {
    switch (pool.head_dim) {
        case 64: return launch_quantize_d<kBF16, BITS, 64>(pool, k, v, qpool, pairs, n, stream);
        case 96: return launch_quantize_d<kBF16, BITS, 96>(pool, k, v, qpool, pairs, n, stream);
        case 128: return launch_quantize_d<kBF16, BITS, 128>(pool, k, v, qpool, pairs, n, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_quantize_blocks(const PoolView& pool, const void* k_pool, const void* v_pool,
                                   const QPoolView& qpool, const int32_t* pairs, int32_t n, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    const uint16_t* k = static_cast<const uint16_t*>(k_pool);
    const uint16_t* v = static_cast<const uint16_t*>(v_pool);
    const bool bf = pool.dtype == KVP_BF16;
    if (qpool.bits == 8)
        return bf ? launch_quantize_b<true, 8>(pool, k, v, qpool, pairs, n, stream)
                  : launch_quantize_b<false, 8>(pool, k, v, qpool, pairs, n, stream);
    return bf ? launch_quantize_b<true, 4>(pool, k, v, qpool, pairs, n, stream)
              : launch_quantize_b<false, 4>(pool, k, v, qpool, pairs, n, stream);
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
