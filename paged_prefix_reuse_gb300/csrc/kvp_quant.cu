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
// Decode over the quantized prefix (decode_q_kernel below): a quantized page
// arrives as two TMA code tiles and two bulk copies of scales (~57% / ~32%
// of its 16-bit bytes at d=128), and its codes enter transposed tensor-core
// products straight from registers, the scales folded into q and P; the live
// suffix's pages arrive as 16-bit TMA tiles.  Each warp of a CTA loads and
// consumes its own stages from a shared ring; split partials are merged by
// merge_kernel.
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
// The exact division, out of line: it is rare, and inlined at each of a
// warp's 128 codes per page-head it made the kernel's code too large for the
// instruction cache.
__device__ __noinline__ int qcode_exact(float d, float s) { return __float2int_rn(__fdiv_rn(d, s)); }

__device__ __forceinline__ uint32_t qcode_fast(float x, float s, float z, float r, int levels) {
    if (!(s > 0.f)) return 0u;
    const float d = __fsub_rn(x, z);
    const float q = __fmul_rn(d, r);
    const float f = fabsf(q - rintf(q));
    int c;
    if (f < 0.4999f || fabsf(q) >= 512.f)
        c = __float2int_rn(q);
    else
        c = qcode_exact(d, s);
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

// ---------------------------------------------------------------------------
// Decode over a quantized cached prefix.
//
// The products run transposed: S^T = K q^T (keys as the MMA's M dimension,
// the query heads of the group as N = 8) and O^T = V^T P^T (channels as M),
// so a lane's O accumulators are 32 floats at d = 128 instead of 64, and the
// codes enter the tensor core straight from registers, with no dequantized
// tile in shared memory:
//  * K (per-channel scale s_c and min z_c over the page's tokens):
//      q.k_t = sum_c q_c s_c code_tc + sum_c q_c z_c.
//    The codes become fp16 subnormals (code * 2^-24, exact: the code is the
//    mantissa) by one byte permute per pair; q_c s_c is formed once per page
//    as an unevaluated sum hi + lo of two fp16 values (hi = q s rounded,
//    lo = q s - hi by one fused multiply-add, so the pair carries ~20 bits),
//    each multiplied by the codes; a third product with every key row equal
//    to z gives the sum q.z.  S = 2^24 * (first + second) + (third).
//  * V (per-token scale sv_t and min zv_t):
//      sum_t P_t v_tc = sum_t (P_t sv_t) code_tc + sum_t P_t zv_t.
//    The codes become fp16 1024 + code (one byte permute per pair, exact);
//    P' = P sv is rounded to fp16 for the product, and the row's scalar
//    sum_t (P_t zv_t - 1024 P'_t) is accumulated beside O and added at the end.
//  * The live suffix's 16-bit pages use the same products with s = 1, z = 0
//    and no offset (fp16 operands, a bf16 pool's values converted).
// K's contraction runs over the channels in any order, so each lane takes
// whole runs of channels (8 bits: pairs (c, c+1); 4 bits: pairs (c, c+4),
// which a mask of the code word yields directly); q, s and z are paired
// alike.  The row maximum is exact (no lazy threshold), so P <= 1 and P sv
// stays in fp16 range for any stored scale.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 16-bit matrix held as one row per four lanes (lane l:
// row l / 4, columns 2 (l % 4) and 2 (l % 4) + 1), returned in the same layout.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ uint32_t lds16(uint32_t a) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a) : "memory");
    return v;
}

// Byte offset of byte x of code row r in a tile of code rows written by TMA:
// rows of 128 or 64 bytes carry the matching swizzle (the 16-byte chunks of a
// row permuted), other widths none.
template <int CROW>
__device__ __forceinline__ uint32_t code_off(uint32_t r, uint32_t x) {
    if constexpr (CROW == 128) {
        return r * 128u + ((((x >> 4) ^ (r & 7u)) << 4) | (x & 15u));
    } else if constexpr (CROW == 64) {
        return r * 64u + ((((x >> 4) ^ ((r >> 1) & 3u)) << 4) | (x & 15u));
    } else {
        return r * CROW + x;
    }
}

// NB bytes of code row r from byte x (x a multiple of AL) of the tile at
// shared address a into words, with the widest accesses that AL allows; no
// access crosses a 16-byte chunk.
template <int NB, int AL, int CROW>
__device__ __forceinline__ void lds_code(uint32_t a, int r, int x, uint32_t (&w)[(NB + 3) / 4]) {
    if constexpr (AL >= 16 && NB % 16 == 0) {
#pragma unroll
        for (int i = 0; i < NB / 16; ++i) {
            const uint4 v = lds128(a + code_off<CROW>(r, x + 16 * i));
            w[4 * i] = v.x;
            w[4 * i + 1] = v.y;
            w[4 * i + 2] = v.z;
            w[4 * i + 3] = v.w;
        }
    } else if constexpr (AL >= 8 && NB % 8 == 0) {
#pragma unroll
        for (int i = 0; i < NB / 8; ++i) {
            const uint2 v = lds64(a + code_off<CROW>(r, x + 8 * i));
            w[2 * i] = v.x;
            w[2 * i + 1] = v.y;
        }
    } else if constexpr (AL >= 4 && NB % 4 == 0) {
#pragma unroll
        for (int i = 0; i < NB / 4; ++i) w[i] = lds32(a + code_off<CROW>(r, x + 4 * i));
    } else {
        static_assert(NB % 2 == 0, "whole 16-bit pieces");
#pragma unroll
        for (int i = 0; i < (NB + 3) / 4; ++i) w[i] = 0u;
#pragma unroll
        for (int i = 0; i < NB / 2; ++i) w[i / 2] |= lds16(a + code_off<CROW>(r, x + 2 * i)) << (16 * (i % 2));
    }
}

constexpr int lowest_align(int n) { return (n & -n) >= 16 ? 16 : (n & -n); }

// Two warps per CTA, each loading and consuming its own stages; a ring of as
// many slots as 40 KB holds (eight at int8, ten at int4, d = 128) and five
// CTAs per SM.  Measured on the mixed batch's decode (int8 / int4, eight
// slots): 102 / 111 us; six slots at seven CTAs per SM 111 / 120 us, four
// slots at eight 113 / 119 us -- the stages a warp has in flight matter more
// than the number of warps.
constexpr int kDecodeQWarps = 2;
constexpr int kDecodeQRingBytes = 40 * 1024;
constexpr int kDecodeQCtasPerSm = 5;

template <int D, int BITS>
struct QDec {
    static constexpr int SK = 16;         // keys per stage: one 16-token page
    static constexpr int KS = D / 16;     // k-steps of S^T, m-tiles of O^T
    static constexpr int KCH = D / 4;     // K channels of a lane (quarter lane % 4)
    static constexpr int VCH = D / 8;     // V channels of a lane (eighth lane / 4)
    static constexpr int CROW = D * BITS / 8;
    static constexpr int KCB = KCH * BITS / 8;  // code bytes of a lane's K channels, per key
    static constexpr int VCB = VCH * BITS / 8;  // the same for V
    static constexpr int KAL = lowest_align(KCB), VAL = lowest_align(VCB);
    // A 16-bit stage is half a page (HK keys): K then V, each in the swizzled
    // TMA layout of the 16-bit decode kernel (chunk columns of CW channels).
    static constexpr int HK = kDecodeQHalfRows;
    static constexpr int CW = chunk_elems(D), ROWB = 2 * CW, NCH = D / CW, HREGION = HK * ROWB;
    static constexpr int HKBYTES = HK * D * 2;
    // A quantized stage is one page: K codes, V codes, K meta (scale row, min
    // row), V meta ((scale, min) per token), all meta fp16.
    static constexpr int QCODE = SK * CROW;
    static constexpr int QOFF_V = QCODE, QOFF_KM = 2 * QCODE, QOFF_VM = 2 * QCODE + 4 * D;
    static constexpr int QSTAGE = 2 * QCODE + 4 * D + 4 * SK;
    // Slots hold either kind of stage and start on 1024-byte boundaries (the
    // swizzled TMA tiles need it).
    static constexpr int SLOT = ((QSTAGE > 2 * HKBYTES ? QSTAGE : 2 * HKBYTES) + 1023) / 1024 * 1024;
    // Several slots per warp: a stage's copies are in flight for a
    // microsecond or more, so a warp needs stages ahead.
    static constexpr int NS = (kDecodeQRingBytes / SLOT) & ~1;
    static_assert(NS >= 4, "ring depth");
    static constexpr int QC = kDecodeQWarps;  // warps per CTA, each loading and consuming its own stages
    static constexpr int THREADS = QC * 32;
    static_assert(NS % QC == 0, "every slot has one owner warp");
    static constexpr int RED_FLOATS = 4 * KS + 6;  // per lane: O^T, then (m, l, bias) of its two rows
    static_assert(32 * RED_FLOATS * 4 * (QC - 1) <= NS * SLOT, "the combine fits the ring");
    static constexpr int RING_BYTES = NS * SLOT;
    static constexpr int OFF_BAR = RING_BYTES;
    static constexpr int SMEM_BYTES = OFF_BAR + (NS + 1) * 8 + 16 + 1024;
};

// Pairs of the contraction for the 8 consecutive K channels in w[0..3]
// (16-bit values, two per word): o[e][0] and o[e][1] feed k-step 2u + e as
// the pairs of MMA rows (2t, 2t+1) and (2t+8, 2t+9).  8 bits pair (c, c+1),
// 4 bits pair (c, c+4) (channels relative to the run).
template <int BITS>
__device__ __forceinline__ void pair_words(const uint32_t (&w)[4], uint32_t (&o)[2][2]) {
    if constexpr (BITS == 8) {
        o[0][0] = w[0];
        o[0][1] = w[1];
        o[1][0] = w[2];
        o[1][1] = w[3];
    } else {
        o[0][0] = __byte_perm(w[0], w[2], 0x5410);
        o[0][1] = __byte_perm(w[0], w[2], 0x7632);
        o[1][0] = __byte_perm(w[1], w[3], 0x5410);
        o[1][1] = __byte_perm(w[1], w[3], 0x7632);
    }
}

// The same pairs from codes, as fp16 subnormals code * 2^-24: 8 bits, the
// two code words of the run; 4 bits, its one word of eight nibbles (the even
// channel of a byte in the low nibble).
template <int BITS>
__device__ __forceinline__ void code_pairs(const uint32_t* c, uint32_t (&o)[2][2]) {
    if constexpr (BITS == 8) {
        o[0][0] = __byte_perm(c[0], 0u, 0x4140);
        o[0][1] = __byte_perm(c[0], 0u, 0x4342);
        o[1][0] = __byte_perm(c[1], 0u, 0x4140);
        o[1][1] = __byte_perm(c[1], 0u, 0x4342);
    } else {
        constexpr uint32_t M = 0x000F000Fu;
        o[0][0] = c[0] & M;
        o[0][1] = (c[0] >> 4) & M;
        o[1][0] = (c[0] >> 8) & M;
        o[1][1] = (c[0] >> 12) & M;
    }
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
    const float2 f = unpack2<true>(w);
    return pack2<false>(f.x, f.y);
}

// V^T operand pairs for m-tile mt of keys (A, B) = (2t, 2t+1) or (2t+8, 2t+9):
// (1024 + code_A, 1024 + code_B) at the lane's channels 2 mt and 2 mt + 1.
template <int BITS>
__device__ __forceinline__ void v_code_pairs(const uint32_t* wa, const uint32_t* wb, int mt, uint32_t& lo,
                                             uint32_t& hi) {
    if constexpr (BITS == 8) {
        const int j = mt >> 1;
        const uint32_t t = (mt & 1) ? __byte_perm(wa[j], wb[j], 0x7362) : __byte_perm(wa[j], wb[j], 0x5140);
        lo = magic_pair(t, 0x4140);
        hi = magic_pair(t, 0x4342);
    } else {
        const int j = mt >> 2, i = mt & 3;
        const uint32_t sel = i | (i << 4) | ((4 + i) << 8) | ((4 + i) << 12);
        const uint32_t x = __byte_perm(wa[j], wb[j], sel);
        lo = (x & 0x000F000Fu) | 0x64006400u;
        hi = ((x >> 4) & 0x000F000Fu) | 0x64006400u;
    }
}

template <bool kBF16, int D, int BITS>
__global__ void __launch_bounds__(QDec<D, BITS>::THREADS, kDecodeQCtasPerSm)
    decode_q_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                    const __grid_constant__ CUtensorMap tmap_kc, const __grid_constant__ CUtensorMap tmap_vc,
                    const DecodeParams p) {
    using C = QDec<D, BITS>;
    static_assert(BITS == 4 || BITS == 8, "bits");
    constexpr int KS = C::KS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* stall = full + C::NS;  // nothing arrives on it (KVP_LAUNCH_STALL_TEST)
    volatile int* abort_flag = reinterpret_cast<volatile int*>(stall + 1);

    // blockIdx.x = split * ngrp + row block (8 query heads of the group each).
    const int g = p.group;
    const int ngrp = (g + 7) >> 3;
    const int sp = blockIdx.x / ngrp, r_base = 8 * (blockIdx.x - sp * ngrp);
    const int h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_trigger();
    const int Hkv = p.pool.num_kv_heads;
    uint32_t* err = p.pool.err_word;

    const int L = __ldg(p.context_lens + b);
    const int npages = (L + C::SK - 1) / C::SK;
    if (L < 1 || npages > p.max_blocks) {
        if (sp == 0 && r_base == 0 && tid == 0) report(err, KVP_DEVERR_BAD_LEN);
        pdl_wait();  // every CTA waits, so the grid completes after the one before
        return;
    }
    const int page0 = sp * p.pages_per_split;
    if (page0 >= npages) {
        pdl_wait();
        return;
    }
    const int page1 = min(npages, page0 + p.pages_per_split);
    const int key1 = min(L, page1 * C::SK);
    // Pages [0, qp) of this sequence are quantized blocks.  Stages: one per
    // quantized page of the split ([page0, qend)), then one per half of each
    // 16-bit page that holds keys of the context.
    const int qp = p.qpages ? min(max(__ldg(p.qpages + b), 0), npages) : 0;
    const int qend = min(page1, max(page0, qp));
    const int nq = qend - page0;
    const int nstages = nq + max(0, (key1 - qend * C::SK + C::HK - 1) / C::HK);

    if (tid == 0) {
        for (int i = 0; i < C::NS; ++i) mbar_init(&full[i], 1);
        mbar_init(stall, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    // Lane roles: t = lane % 4 picks the rows 2t, 2t+1 of S^T / O^T (query
    // heads r_base + 2t, + 1), the K channel quarter and the keys 2t, 2t+1,
    // 2t+8, 2t+9 of the V operand; u = lane / 4 picks the keys u, u+8 of the
    // K operand, the query head r_base + u of the q operand and the V channel
    // eighth.
    const int u = lane >> 2, t = lane & 3;
    float o[KS][4];
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};
    float bias[2] = {0.f, 0.f};
#pragma unroll
    for (int i = 0; i < KS; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

    // Every warp loads its own stages: stage i sits in slot i % NS and belongs
    // to warp i % QC (NS is a multiple of QC), so the warp that consumes a
    // slot refills it with its next stage -- no producer warp, no empty
    // barriers.  Warp w's stages are i = w + QC * j, j = 0 .. nmine - 1.
    if (lane == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
        prefetch_tmap(&tmap_kc);
        prefetch_tmap(&tmap_vc);
    }
    pdl_wait();  // pool contents from the kernel before are read from here on
    const int nmine = nstages > warp ? (nstages - warp + C::QC - 1) / C::QC : 0;
    int win = 0;  // block ids of this warp's stages, lane l: local index (base of the window) + l
    // Block ids of the local stages [j0, j0 + 32), one per lane.
    auto load_window = [&](int j0) {
        const int si = warp + C::QC * (j0 + lane);
        const int pg = min(si < nq ? page0 + si : qend + (si - nq) / 2, npages - 1);
        int blk = __ldg(p.block_tables + static_cast<int64_t>(b) * p.max_blocks + pg);
        const int64_t nblk = pg < qp ? p.qpool.num_blocks : p.pool.num_blocks;
        if (blk < 0 || blk >= nblk) {
            report(err, KVP_DEVERR_BAD_BLOCK);
            blk = 0;
        }
        win = blk;
    };
    // The copies of local stage jn (all lanes call; lane 0 issues).
    auto issue = [&](int jn) {
        if ((jn & 31) == 0) load_window(jn);
        const int blk = __shfl_sync(0xffffffffu, win, jn & 31);
        const int i = warp + C::QC * jn;
        const int slot = i % C::NS;
        if (lane == 0) {
            uint8_t* st = smem + slot * C::SLOT;
            if (i < nq) {
                // A quantized page: the code tiles by TMA (swizzled), the scale
                // and min rows by bulk copies.
                const int64_t ph = static_cast<int64_t>(blk) * Hkv + h;
                mbar_expect_tx(&full[slot], C::QSTAGE);
                tma_load_2d(st, &tmap_kc, 0, static_cast<int32_t>(ph) * C::SK, &full[slot]);
                tma_load_2d(st + C::QOFF_V, &tmap_vc, 0, static_cast<int32_t>(ph) * C::SK, &full[slot]);
                bulk_load(st + C::QOFF_KM, p.qpool.k_meta + ph * 2 * D, 4 * D, &full[slot]);
                bulk_load(st + C::QOFF_VM, p.qpool.v_meta + ph * 2 * C::SK, 4 * C::SK, &full[slot]);
            } else {
                // Half (i - nq) % 2 of a 16-bit page: rows of HK keys.
                const int32_t y = (blk * Hkv + h) * C::SK + ((i - nq) & 1) * C::HK;
                mbar_expect_tx(&full[slot], 2 * C::HKBYTES);
#pragma unroll
                for (int c = 0; c < C::NCH; ++c) {
                    tma_load_2d(st + c * C::HREGION, &tmap_k, c * C::CW, y, &full[slot]);
                    tma_load_2d(st + C::HKBYTES + c * C::HREGION, &tmap_v, c * C::CW, y, &full[slot]);
                }
            }
        }
    };
    // Test of the failure path: before any copy is issued, warp 0 waits on a
    // barrier nothing arrives on until the limit runs out.
    const bool stalled = p.stall_test && warp == 0 && !stall_wait(stall, abort_flag, err, p.wait_limit_ns);
    int issued = 0;
    if (!stalled)
        for (; issued < min(C::NS / C::QC, nmine); ++issued) issue(issued);
    int jdone = 0;
    {
        // ------------------------------ consumers ------------------------------
        // q operand: query head r_base + u (zero past the group), the lane's
        // K channel quarter, paired as the codes are; fp16 whatever the pool.
        uint32_t qb[KS][2];
        {
            const int r = r_base + u;
            const bool live = r < g;
            const uint4* qrow = reinterpret_cast<const uint4*>(
                static_cast<const uint8_t*>(p.q) +
                ((static_cast<int64_t>(b) * p.num_q_heads + h * g + (live ? r : 0)) * D + t * C::KCH) * 2);
#pragma unroll
            for (int k = 0; k < C::KCH / 8; ++k) {
                const uint4 v = live ? __ldg(qrow + k) : make_uint4(0u, 0u, 0u, 0u);
                uint32_t w[4] = {v.x, v.y, v.z, v.w};
                if constexpr (kBF16) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) w[j] = bf16x2_to_f16x2(w[j]);
                }
                uint32_t pr[2][2];
                pair_words<BITS>(w, pr);
                qb[2 * k][0] = pr[0][0];
                qb[2 * k][1] = pr[0][1];
                qb[2 * k + 1][0] = pr[1][0];
                qb[2 * k + 1][1] = pr[1][1];
            }
        }
        const float sl2 = p.scale_log2;

        for (; jdone < nmine && !stalled; ++jdone) {
            const int i = warp + C::QC * jdone;
            const int slot = i % C::NS;
            if (!mbar_wait(&full[slot], (i / C::NS) & 1, abort_flag, err, p.wait_limit_ns)) break;
            const uint32_t sb = smem_u32(smem + slot * C::SLOT);
            const bool qst = i < nq;
            const int kb = qst ? (page0 + i) * C::SK : qend * C::SK + (i - nq) * C::HK;  // first key
            const int nvalid = min(qst ? C::SK : C::HK, key1 - kb);  // >= 1

            // ---- S^T = K q^T (rows: keys u, u+8; columns: query heads 2t, 2t+1) ----
            float s[4] = {0.f, 0.f, 0.f, 0.f};
            if (qst) {
                constexpr int KW = (C::KCB + 3) / 4;
                uint32_t c0[KW], c1[KW];
                lds_code<C::KCB, C::KAL, C::CROW>(sb, u, t * C::KCB, c0);
                lds_code<C::KCB, C::KAL, C::CROW>(sb, u + 8, t * C::KCB, c1);
                uint32_t sw[C::KCH / 2], zw[C::KCH / 2];  // the fp16 scale and min rows, unswizzled
                lds_code<C::KCH * 2, 16, 4 * D>(sb + C::QOFF_KM, 0, t * C::KCH * 2, sw);
                lds_code<C::KCH * 2, 16, 4 * D>(sb + C::QOFF_KM, 0, 2 * D + t * C::KCH * 2, zw);
                float sl[4] = {0.f, 0.f, 0.f, 0.f}, sz[4] = {0.f, 0.f, 0.f, 0.f};
                constexpr int CWU = BITS == 8 ? 2 : 1;  // code words per 8-channel run
#pragma unroll
                for (int k = 0; k < C::KCH / 8; ++k) {
                    uint32_t a0[2][2], a1[2][2], sp2[2][2], zp2[2][2];
                    code_pairs<BITS>(c0 + CWU * k, a0);
                    code_pairs<BITS>(c1 + CWU * k, a1);
                    const uint32_t s4[4] = {sw[4 * k], sw[4 * k + 1], sw[4 * k + 2], sw[4 * k + 3]};
                    const uint32_t z4[4] = {zw[4 * k], zw[4 * k + 1], zw[4 * k + 2], zw[4 * k + 3]};
                    pair_words<BITS>(s4, sp2);
                    pair_words<BITS>(z4, zp2);
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int ks = 2 * k + e;
                        const __half2 x0 = *reinterpret_cast<const __half2*>(&qb[ks][0]);
                        const __half2 x1 = *reinterpret_cast<const __half2*>(&qb[ks][1]);
                        const __half2 y0 = *reinterpret_cast<const __half2*>(&sp2[e][0]);
                        const __half2 y1 = *reinterpret_cast<const __half2*>(&sp2[e][1]);
                        const __half2 h0 = __hmul2(x0, y0), h1 = __hmul2(x1, y1);
                        const __half2 l0 = __hfma2(x0, y0, __hneg2(h0)), l1 = __hfma2(x1, y1, __hneg2(h1));
                        mma_f16(s, a0[e][0], a1[e][0], a0[e][1], a1[e][1], *reinterpret_cast<const uint32_t*>(&h0),
                                *reinterpret_cast<const uint32_t*>(&h1));
                        mma_f16(sl, a0[e][0], a1[e][0], a0[e][1], a1[e][1], *reinterpret_cast<const uint32_t*>(&l0),
                                *reinterpret_cast<const uint32_t*>(&l1));
                        mma_f16(sz, zp2[e][0], zp2[e][0], zp2[e][1], zp2[e][1], qb[ks][0], qb[ks][1]);
                    }
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) s[e] = fmaf(s[e] + sl[e], 16777216.f, sz[e]);
            } else {
                // Keys u of the half page; MMA rows u + 8 stay zero (masked below).
#pragma unroll
                for (int k = 0; k < C::KCH / 8; ++k) {
                    const int c = t * C::KCH + 8 * k;  // first channel of the run
                    const uint4 x0 = lds128(sb + (c / C::CW) * C::HREGION + swz_offset(u, (c % C::CW) / 8, C::ROWB));
                    uint32_t w0[4] = {x0.x, x0.y, x0.z, x0.w};
                    if constexpr (kBF16) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) w0[j] = bf16x2_to_f16x2(w0[j]);
                    }
                    uint32_t a0[2][2];
                    pair_words<BITS>(w0, a0);
#pragma unroll
                    for (int e = 0; e < 2; ++e)
                        mma_f16(s, a0[e][0], 0u, a0[e][1], 0u, qb[2 * k + e][0], qb[2 * k + e][1]);
                }
            }

            // ---- V operand loads (issued before the softmax) ----
            constexpr int VW = (C::VCB + 3) / 4;
            uint32_t va[VW], vb[VW], vc[VW], vd[VW];  // keys 2t, 2t+1, 2t+8, 2t+9
            uint32_t vm0 = 0u, vm1 = 0u;              // (scale, min) of keys u, u+8
            if (qst) {
                const uint32_t vbase = sb + C::QOFF_V;
                lds_code<C::VCB, C::VAL, C::CROW>(vbase, 2 * t, u * C::VCB, va);
                lds_code<C::VCB, C::VAL, C::CROW>(vbase, 2 * t + 1, u * C::VCB, vb);
                lds_code<C::VCB, C::VAL, C::CROW>(vbase, 2 * t + 8, u * C::VCB, vc);
                lds_code<C::VCB, C::VAL, C::CROW>(vbase, 2 * t + 9, u * C::VCB, vd);
                vm0 = lds32(sb + C::QOFF_VM + 4 * u);
                vm1 = lds32(sb + C::QOFF_VM + 4 * (u + 8));
            }

            // ---- online softmax over the stage's keys (log2 domain) ----
            if (u >= nvalid) s[0] = s[1] = -INFINITY;
            if (u + 8 >= nvalid) s[2] = s[3] = -INFINITY;
            float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
            for (int x = 4; x < 32; x <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, x));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, x));
            }
            const float mx0s = mx0 * sl2, mx1s = mx1 * sl2;
            float a0 = 1.f, a1 = 1.f;
            if (mx0s > m_run[0]) {
                a0 = fast_exp2(m_run[0] - mx0s);
                m_run[0] = mx0s;
            }
            if (mx1s > m_run[1]) {
                a1 = fast_exp2(m_run[1] - mx1s);
                m_run[1] = mx1s;
            }
            if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                    o[mt][0] *= a0;
                    o[mt][2] *= a0;
                    o[mt][1] *= a1;
                    o[mt][3] *= a1;
                }
                l_run[0] *= a0;
                l_run[1] *= a1;
                bias[0] *= a0;
                bias[1] *= a1;
            }
            const float pr0 = fast_exp2(fmaf(s[0], sl2, -m_run[0]));
            const float pr1 = fast_exp2(fmaf(s[1], sl2, -m_run[1]));
            const float pr2 = fast_exp2(fmaf(s[2], sl2, -m_run[0]));
            const float pr3 = fast_exp2(fmaf(s[3], sl2, -m_run[1]));
            l_run[0] += pr0 + pr2;
            l_run[1] += pr1 + pr3;

            // ---- O^T += V^T P^T ----
            uint32_t pk0, pk1;  // (key u | u+8; query heads 2t, 2t+1)
            if (qst) {
                float2 m0 = unpack2<false>(vm0), m1 = unpack2<false>(vm1);  // (scale, min)
                if (u >= nvalid) m0 = make_float2(0.f, 0.f);  // meta past the context is never used
                if (u + 8 >= nvalid) m1 = make_float2(0.f, 0.f);
                pk0 = pack2<false>(pr0 * m0.x, pr1 * m0.x);
                pk1 = pack2<false>(pr2 * m1.x, pr3 * m1.x);
                const float2 r0 = unpack2<false>(pk0), r1 = unpack2<false>(pk1);
                bias[0] += fmaf(pr0, m0.y, pr2 * m1.y) - 1024.f * (r0.x + r1.x);
                bias[1] += fmaf(pr1, m0.y, pr3 * m1.y) - 1024.f * (r0.y + r1.y);
            } else {
                pk0 = pack2<false>(pr0, pr1);
                pk1 = pack2<false>(pr2, pr3);
            }
            const uint32_t pb0 = movmatrix_t(pk0), pb1 = movmatrix_t(pk1);  // P'^T: keys 2t.. / 2t+8..; head u
            if (qst) {
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                    uint32_t x0, x1, x2, x3;
                    v_code_pairs<BITS>(va, vb, mt, x0, x1);
                    v_code_pairs<BITS>(vc, vd, mt, x2, x3);
                    mma_f16(o[mt], x0, x1, x2, x3, pb0, pb1);
                }
            } else {
                // The lane's V channels of keys 2t, 2t+1 of the half page, four
                // at a time; keys past the context (any bytes, even NaN) read as
                // 0, and keys 2t+8, 2t+9 (past the half) are 0.
#pragma unroll
                for (int k = 0; k < C::VCH / 4; ++k) {
                    const int c = u * C::VCH + 4 * k;
                    const uint32_t a = sb + C::HKBYTES + (c / C::CW) * C::HREGION + ((c / 4) & 1) * 8;
                    uint32_t w[2][2];
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        uint2 x = lds64(a + swz_offset(2 * t + j, (c % C::CW) / 8, C::ROWB));
                        if (2 * t + j >= nvalid) x = make_uint2(0u, 0u);
                        if constexpr (kBF16) {
                            x.x = bf16x2_to_f16x2(x.x);
                            x.y = bf16x2_to_f16x2(x.y);
                        }
                        w[j][0] = x.x;
                        w[j][1] = x.y;
                    }
#pragma unroll
                    for (int e = 0; e < 2; ++e)
                        mma_f16(o[2 * k + e], __byte_perm(w[0][e], w[1][e], 0x5410),
                                __byte_perm(w[0][e], w[1][e], 0x7632), 0u, 0u, pb0, pb1);
                }
            }
            // Refill the slot with this warp's stage NS/QC ahead, once every
            // lane's reads of it are done (and ordered before the async copy).
            if (issued < nmine) {
                fence_proxy_async_smem();
                __syncwarp();
                issue(issued);
                ++issued;
            }
        }
        // Do not leave while copies may still land in shared memory.
        if (lane == 0) {
            for (int jj = jdone; jj < issued; ++jj) {
                const int i = warp + C::QC * jj;
                volatile int no_abort = 0;
                mbar_wait(&full[i % C::NS], (i / C::NS) & 1, &no_abort, err);
            }
        }
        __syncwarp();
        // Row sums and offsets were accumulated per lane over its keys.
#pragma unroll
        for (int x = 4; x < 32; x <<= 1) {
            l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], x);
            l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], x);
            bias[0] += __shfl_xor_sync(0xffffffffu, bias[0], x);
            bias[1] += __shfl_xor_sync(0xffffffffu, bias[1], x);
        }
    }

    // ------------------------------ epilogue ------------------------------
    // Lane: query heads r_base + 2t + j (j = 0, 1); channels u*VCH + 2 mt and
    // + 1 in o[mt][j] and o[mt][j + 2].  The consumer warps combine through
    // shared memory (all stages are consumed once every consumer passes the
    // first barrier, so the ring is free); warp 0 writes the CTA's result:
    // the output rows, or with splits one normalised partial (O, log2 lse).
    float* red = reinterpret_cast<float*>(smem);  // [QC - 1][RED_FLOATS][32 lanes]
    asm volatile("bar.sync 1, %0;" ::"r"(C::QC * 32) : "memory");
    if (warp > 0) {
        float* w = red + (warp - 1) * C::RED_FLOATS * 32 + lane;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) w[(4 * mt + e) * 32] = o[mt][e];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            w[(4 * KS + 3 * j) * 32] = m_run[j];
            w[(4 * KS + 3 * j + 1) * 32] = l_run[j];
            w[(4 * KS + 3 * j + 2) * 32] = bias[j];
        }
    }
    // Every consumer warp always reaches both barriers (even after a
    // timed-out wait), so none can be left waiting for another.
    asm volatile("bar.sync 1, %0;" ::"r"(C::QC * 32) : "memory");
    if (warp != 0 || *abort_flag) return;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int r = r_base + 2 * t + j;
        if (r >= g) continue;
        float M = m_run[j];
#pragma unroll
        for (int w = 1; w < C::QC; ++w) M = fmaxf(M, red[((w - 1) * C::RED_FLOATS + 4 * KS + 3 * j) * 32 + lane]);
        float f[C::QC];
        float lsum = 0.f;
#pragma unroll
        for (int w = 0; w < C::QC; ++w) {
            const float mw = w == 0 ? m_run[j] : red[((w - 1) * C::RED_FLOATS + 4 * KS + 3 * j) * 32 + lane];
            const float lw = w == 0 ? l_run[j] : red[((w - 1) * C::RED_FLOATS + 4 * KS + 3 * j + 1) * 32 + lane];
            f[w] = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
            lsum = fmaf(lw, f[w], lsum);
        }
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        const float lse2 = lsum > 0.f ? M + __log2f(lsum) : -INFINITY;
        float x[KS][2];
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            x[mt][0] = (o[mt][j] + bias[j]) * f[0];
            x[mt][1] = (o[mt][j + 2] + bias[j]) * f[0];
        }
#pragma unroll
        for (int w = 1; w < C::QC; ++w) {
            const float* rw = red + (w - 1) * C::RED_FLOATS * 32 + lane;
            const float bw = rw[(4 * KS + 3 * j + 2) * 32];
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                x[mt][0] = fmaf(rw[(4 * mt + j) * 32] + bw, f[w], x[mt][0]);
                x[mt][1] = fmaf(rw[(4 * mt + j + 2) * 32] + bw, f[w], x[mt][1]);
            }
        }
        const int64_t row = static_cast<int64_t>(b) * p.num_q_heads + h * g + r;
        if (p.max_splits > 1) {
            float4* dst = reinterpret_cast<float4*>(p.ws_o + (row * p.max_splits + sp) * D + u * C::VCH);
#pragma unroll
            for (int k = 0; k < KS / 2; ++k)
                dst[k] = make_float4(x[2 * k][0] * inv, x[2 * k][1] * inv, x[2 * k + 1][0] * inv,
                                     x[2 * k + 1][1] * inv);
            if (u == 0) p.ws_lse[row * p.max_splits + sp] = lse2;
            continue;
        }
        uint32_t wv[KS];
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) wv[mt] = pack2<kBF16>(x[mt][0] * inv, x[mt][1] * inv);
        uint8_t* dst = static_cast<uint8_t*>(p.out) + (row * D + u * C::VCH) * 2;
        if constexpr (KS % 4 == 0) {
#pragma unroll
            for (int k = 0; k < KS / 4; ++k)
                reinterpret_cast<uint4*>(dst)[k] = make_uint4(wv[4 * k], wv[4 * k + 1], wv[4 * k + 2], wv[4 * k + 3]);
        } else {
#pragma unroll
            for (int k = 0; k < KS / 2; ++k) reinterpret_cast<uint2*>(dst)[k] = make_uint2(wv[2 * k], wv[2 * k + 1]);
        }
        if (u == 0 && p.lse) p.lse[static_cast<int64_t>(h * g + r) * p.B + b] = lse2 * 0.69314718055994531f;
    }
}

template <bool kBF16, int D, int BITS>
cudaError_t launch_decode_q(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tkc, const CUtensorMap& tvc, cudaStream_t stream) {
    using C = QDec<D, BITS>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(decode_q_kernel<kBF16, D, BITS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int ngrp = (p.group + 7) / 8;
    dim3 grid(p.max_splits * ngrp, p.pool.num_kv_heads, p.B);
    return launch_k(decode_q_kernel<kBF16, D, BITS>, grid, C::THREADS, C::SMEM_BYTES, stream, tk, tv, tkc, tvc, p);
}

template <bool kBF16, int D>
cudaError_t launch_decode_q_d(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& tkc, const CUtensorMap& tvc, cudaStream_t stream) {
    return p.qpool.bits == 8 ? launch_decode_q<kBF16, D, 8>(p, tk, tv, tkc, tvc, stream)
                             : launch_decode_q<kBF16, D, 4>(p, tk, tv, tkc, tvc, stream);
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
                                 const CUtensorMap& tkc, const CUtensorMap& tvc, cudaStream_t stream) {
    const bool bf = p.pool.dtype == KVP_BF16;
#define KVP_DQ(DD) \
    return bf ? launch_decode_q_d<true, DD>(p, tk, tv, tkc, tvc, stream) : launch_decode_q_d<false, DD>(p, tk, tv, tkc, tvc, stream)
    switch (p.pool.head_dim) {
        case 64: KVP_DQ(64);
        case 96: KVP_DQ(96);
        case 128: KVP_DQ(128);
        default: return cudaErrorInvalidValue;
    }
#undef KVP_DQ
}

}  // namespace kvp
