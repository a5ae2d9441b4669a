// kvp_decode.cu -- decode attention for a continuous batch (one new token
// per sequence; kvstream 0.1.0 "Request lifecycle"), split over the key
// range, plus the log-sum-exp merge of split partials shared with the
// prefix kernel.
//
// Decode reads every K/V byte of the context once and does ~g*4 flops per
// byte (g = query heads per kv head), so it is HBM-bound.  Design:
//  * one CTA per (key range, kv head, sequence); the g query heads of the
//    group share each loaded page;
//  * a producer warp streams 32-key stages (K and V page-heads of one or more
//    physical blocks, addressed through the block table) with 2-D TMA loads
//    into a ring of 96 KB of shared memory, swizzled so that the consumers'
//    ldmatrix reads are conflict-free;
//  * four consumer warps take stages round-robin and run q.K^T and P.V as
//    m16n8k16 tensor-core MMAs (the group padded to 16 rows) with an fp32
//    online softmax; the warps' partial states are merged through shared
//    memory at the end;
//  * with more than one split, each CTA writes a normalised partial (O, lse)
//    and merge_kernel combines them: lse = log2 sum_i 2^lse_i,
//    O = sum_i 2^(lse_i - lse) O_i.
#include "kvp_internal.cuh"

namespace kvp {
namespace {

constexpr int kConsumerWarps = 2;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;
constexpr int kRingSlots = 2 * kConsumerWarps;  // two slots per consumer warp: one computing, one loading

// SK keys per stage: 16 (one 16-token block) when blocks hold <= 16 tokens,
// else 32 (one 32-token block).
template <int D, int SK>
struct DecodeCfg {
    static constexpr int CW = chunk_elems(D);
    static constexpr int ROWB = CW * 2;
    static constexpr int NCH = D / CW;
    static constexpr int REGION = SK * ROWB;  // one chunk column of a stage's K (or V)
    static constexpr int KBYTES = SK * D * 2;
    static constexpr int STAGE_BYTES = 2 * KBYTES;
    // Stage i sits in slot i % NS and is consumed by warp i % 4.  NS is a
    // multiple of the consumer count, so every slot has one owner warp that
    // consumes its phases in order: a waiter can never be two phases behind,
    // which a parity wait could not tell apart from the phase it wants.
    static constexpr int NS = kRingSlots;
    static_assert(NS % kConsumerWarps == 0, "ring depth");
    static constexpr int RED_BYTES = (D / 8) * 32 * 16 + 32 * 8;  // one warp's fragments + row stats
    static constexpr int RING_BYTES = NS * STAGE_BYTES > RED_BYTES ? NS * STAGE_BYTES : RED_BYTES;
    static constexpr int SMEM_BYTES = RING_BYTES + 2 * NS * 8 + 16 + 1024;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

template <bool kBF16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    if constexpr (kBF16) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    const uint32_t a = smem_u32(p);
    return p + (((a + 1023u) & ~1023u) - a);
}

template <bool kBF16, int D, int SK>
__global__ void __launch_bounds__(kDecodeThreads, 4)
    decode_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                  const DecodeParams p) {
    using C = DecodeCfg<D, SK>;
    constexpr int kStageKeys = SK;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::RING_BYTES);
    uint64_t* empty = full + C::NS;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + C::NS);

    const int sp = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int BS = p.pool.block_size;
    const int Hkv = p.pool.num_kv_heads;
    const int g = p.group;
    uint32_t* err = p.pool.err_word;

    const int L = __ldg(p.context_lens + b);
    const int npages = (L + BS - 1) / BS;
    if (L < 1 || npages > p.max_blocks) {
        if (sp == 0 && tid == 0) report(err, KVP_DEVERR_BAD_LEN);
        return;
    }
    const int page0 = sp * p.pages_per_split;
    if (page0 >= npages) return;
    const int page1 = min(npages, page0 + p.pages_per_split);
    const int key0 = page0 * BS;
    const int key1 = min(L, page1 * BS);
    const int nstages = (key1 - key0 + kStageKeys - 1) / kStageKeys;
    const int pps = kStageKeys / BS;  // physical pages per stage

    if (tid == 0) {
        for (int i = 0; i < C::NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    // Per-warp online-softmax state for rows r0 = lane/4 and r1 = r0 + 8.
    float o[D / 8][4];
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

    if (warp == kConsumerWarps) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            prefetch_tmap(&tmap_k);
            prefetch_tmap(&tmap_v);
        }
        int my_blk = 0;
        int issued = 0;
        for (int i = 0; i < nstages; ++i) {
            const int slot = i % C::NS;
            const int rel = (i * pps) & 31;
            if (rel == 0) {
                int pg = min(page0 + i * pps + lane, npages - 1);
                int blk = __ldg(p.block_tables + static_cast<int64_t>(b) * p.max_blocks + pg);
                if (blk < 0 || blk >= p.pool.num_blocks) {
                    report(err, KVP_DEVERR_BAD_BLOCK);
                    blk = 0;
                }
                my_blk = blk;
            }
            int ok = 1;
            if (lane == 0 && i >= C::NS) ok = mbar_wait(&empty[slot], ((i / C::NS) - 1) & 1, abort_flag, err);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if (lane == 0) mbar_expect_tx(&full[slot], C::STAGE_BYTES);
            __syncwarp();
            // One lane per physical page of the stage issues that page's boxes.
            const int blk = __shfl_sync(0xffffffffu, my_blk, (rel + lane) & 31);
            uint8_t* kst = smem + slot * C::STAGE_BYTES;
            uint8_t* vst = kst + C::KBYTES;
            if (lane < pps) {
                const int32_t y = (blk * Hkv + h) * BS;
#pragma unroll
                for (int c = 0; c < C::NCH; ++c) {
                    tma_load_2d(kst + c * C::REGION + lane * BS * C::ROWB, &tmap_k, c * C::CW, y, &full[slot]);
                    tma_load_2d(vst + c * C::REGION + lane * BS * C::ROWB, &tmap_v, c * C::CW, y, &full[slot]);
                }
            }
            issued = i + 1;
        }
        // Do not leave while copies may still land in shared memory.
        if (lane == 0) {
            for (int i = max(0, issued - C::NS); i < issued; ++i) {
                volatile int no_abort = 0;
                mbar_wait(&full[i % C::NS], (i / C::NS) & 1, &no_abort, err);
            }
        }
    } else {
        // ------------------------------ consumers ------------------------------
        const int r0 = lane >> 2, r1 = r0 + 8;
        const int cq = 2 * (lane & 3);
        const uint32_t* q32 = static_cast<const uint32_t*>(p.q);
        const int64_t qrow0 = (static_cast<int64_t>(b) * p.num_q_heads + h * g + r0) * D;
        const int64_t qrow1 = (static_cast<int64_t>(b) * p.num_q_heads + h * g + r1) * D;
        uint32_t qa[D / 16][4];
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            qa[ks][0] = r0 < g ? __ldg(q32 + (qrow0 + ks * 16 + cq) / 2) : 0u;
            qa[ks][1] = r1 < g ? __ldg(q32 + (qrow1 + ks * 16 + cq) / 2) : 0u;
            qa[ks][2] = r0 < g ? __ldg(q32 + (qrow0 + ks * 16 + cq + 8) / 2) : 0u;
            qa[ks][3] = r1 < g ? __ldg(q32 + (qrow1 + ks * 16 + cq + 8) / 2) : 0u;
        }
        const float sl2 = p.scale_log2;

        for (int i = warp; i < nstages; i += kConsumerWarps) {
            const int slot = i % C::NS;
            if (!mbar_wait(&full[slot], (i / C::NS) & 1, abort_flag, err)) break;
            uint8_t* kst = smem + slot * C::STAGE_BYTES;
            uint8_t* vst = kst + C::KBYTES;
            const int kbeg = key0 + i * kStageKeys;
            const int nvalid = min(kStageKeys, key1 - kbeg);
            if (nvalid < kStageKeys) {
                // Rows past the context may hold any bytes (even NaN); P is 0
                // there, but 0 * NaN is NaN, so clear those V rows.
                const int vecs_per_row = C::ROWB / 16;
                const int nvec = (kStageKeys - nvalid) * vecs_per_row * C::NCH;
                for (int e = lane; e < nvec; e += 32) {
                    const int c = e / ((kStageKeys - nvalid) * vecs_per_row);
                    const int rem = e - c * (kStageKeys - nvalid) * vecs_per_row;
                    const int row = nvalid + rem / vecs_per_row;
                    const int v16 = rem % vecs_per_row;
                    *reinterpret_cast<uint4*>(vst + c * C::REGION + row * C::ROWB + v16 * 16) =
                        make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
            }
            const uint32_t kbase = smem_u32(kst), vbase = smem_u32(vst);

            // S = q K^T for SK keys: SK/8 n-tiles of 8 keys.
            constexpr int NT = SK / 8;
            float s[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
                for (int np = 0; np < NT / 2; ++np) {
                    const uint32_t key = np * 16 + (lane & 7) + ((lane >> 4) << 3);
                    const uint32_t c16 = ks * 2 + ((lane >> 3) & 1);
                    const uint32_t addr = kbase + (c16 / (C::CW / 8)) * C::REGION +
                                          swz_offset(key, c16 % (C::CW / 8), C::ROWB);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(addr, b0, b1, b2, b3);
                    mma16816<kBF16>(s[2 * np], qa[ks], b0, b1);
                    mma16816<kBF16>(s[2 * np + 1], qa[ks], b2, b3);
                }
            }
            if (nvalid < kStageKeys) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (nt * 8 + cq + (e & 1) >= nvalid) s[nt][e] = -INFINITY;
            }
            // Online softmax (log2 domain; the scale is folded into the exponent).
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
                mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
            }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float mn0 = fmaxf(m_run[0], mx0 * sl2);
            const float mn1 = fmaxf(m_run[1], mx1 * sl2);
            const float a0 = fast_exp2(m_run[0] - mn0);
            const float a1 = fast_exp2(m_run[1] - mn1);
            m_run[0] = mn0;
            m_run[1] = mn1;
            float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                s[nt][0] = fast_exp2(fmaf(s[nt][0], sl2, -mn0));
                s[nt][1] = fast_exp2(fmaf(s[nt][1], sl2, -mn0));
                s[nt][2] = fast_exp2(fmaf(s[nt][2], sl2, -mn1));
                s[nt][3] = fast_exp2(fmaf(s[nt][3], sl2, -mn1));
                ps0 += s[nt][0] + s[nt][1];
                ps1 += s[nt][2] + s[nt][3];
            }
            l_run[0] = l_run[0] * a0 + ps0;
            l_run[1] = l_run[1] * a1 + ps1;
#pragma unroll
            for (int nd = 0; nd < D / 8; ++nd) {
                o[nd][0] *= a0;
                o[nd][1] *= a0;
                o[nd][2] *= a1;
                o[nd][3] *= a1;
            }
            uint32_t pa[SK / 16][4];
#pragma unroll
            for (int kk = 0; kk < SK / 16; ++kk) {
                pa[kk][0] = pack2<kBF16>(s[2 * kk][0], s[2 * kk][1]);
                pa[kk][1] = pack2<kBF16>(s[2 * kk][2], s[2 * kk][3]);
                pa[kk][2] = pack2<kBF16>(s[2 * kk + 1][0], s[2 * kk + 1][1]);
                pa[kk][3] = pack2<kBF16>(s[2 * kk + 1][2], s[2 * kk + 1][3]);
            }
            // O += P V: V is [key][dim] in shared memory, loaded transposed.
#pragma unroll
            for (int kk = 0; kk < SK / 16; ++kk) {
#pragma unroll
                for (int nd2 = 0; nd2 < D / 16; ++nd2) {
                    const uint32_t key = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                    const uint32_t c16 = nd2 * 2 + (lane >> 4);
                    const uint32_t addr = vbase + (c16 / (C::CW / 8)) * C::REGION +
                                          swz_offset(key, c16 % (C::CW / 8), C::ROWB);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(addr, b0, b1, b2, b3);
                    mma16816<kBF16>(o[2 * nd2], pa[kk], b0, b1);
                    mma16816<kBF16>(o[2 * nd2 + 1], pa[kk], b2, b3);
                }
            }
            if (nvalid < kStageKeys) fence_proxy_async_smem();  // generic zeroing before the next TMA write
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
        // Row sums were accumulated per thread over its own columns.
        l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], 1);
        l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], 2);
        l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], 1);
        l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], 2);
    }

    if (warp == kConsumerWarps) return;

    // ------------------------------ epilogue ------------------------------
    const int r0 = lane >> 2, r1 = r0 + 8, cq = 2 * (lane & 3);
    if (p.max_splits > 1) {
        if (*abort_flag) return;
        // Each consumer warp writes its own partial (normalised O, log2 lse):
        // part = split * kConsumerWarps + warp; merge_kernel combines them.
        const int parts = p.max_splits * kConsumerWarps;
        const int part = sp * kConsumerWarps + warp;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int r = half ? r1 : r0;
            if (r >= g) continue;
            const float lsum = l_run[half];
            const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
            const int64_t row = static_cast<int64_t>(b) * p.num_q_heads + h * g + r;
            float* dst = p.ws_o + (row * parts + part) * D;
#pragma unroll
            for (int nd = 0; nd < D / 8; ++nd)
                *reinterpret_cast<float2*>(dst + nd * 8 + cq) =
                    make_float2(o[nd][2 * half] * inv, o[nd][2 * half + 1] * inv);
            if ((lane & 3) == 0)
                p.ws_lse[row * parts + part] = lsum > 0.f ? m_run[half] + __log2f(lsum) : -INFINITY;
        }
        return;
    }
    // One split: combine the consumer warps through shared memory (all stages
    // are consumed once both warps pass the barrier, so the ring is free).
    float4* red = reinterpret_cast<float4*>(smem);                       // [D/8][32 lanes]
    float2* stat = reinterpret_cast<float2*>(smem + (D / 8) * 32 * 16);  // [32 lanes] (m, l) x 2 rows
    asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
    if (warp == 1) {
#pragma unroll
        for (int nd = 0; nd < D / 8; ++nd) red[nd * 32 + lane] = make_float4(o[nd][0], o[nd][1], o[nd][2], o[nd][3]);
        stat[2 * lane] = make_float2(m_run[0], l_run[0]);
        stat[2 * lane + 1] = make_float2(m_run[1], l_run[1]);
    }
    // Both consumer warps always reach both barriers (even after a timed-out
    // wait), so neither can be left waiting for the other.
    asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
    if (warp != 0 || *abort_flag) return;
    float f0[2], f1[2], inv[2], lse2[2];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const float2 st1 = stat[2 * lane + half];
        const float M = fmaxf(m_run[half], st1.x);
        f0[half] = m_run[half] == -INFINITY ? 0.f : fast_exp2(m_run[half] - M);
        f1[half] = st1.x == -INFINITY ? 0.f : fast_exp2(st1.x - M);
        const float lsum = l_run[half] * f0[half] + st1.y * f1[half];
        inv[half] = lsum > 0.f ? 1.f / lsum : 0.f;
        lse2[half] = lsum > 0.f ? M + __log2f(lsum) : -INFINITY;
    }
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int r = half ? r1 : r0;
        if (r >= g) continue;
        const int64_t row = static_cast<int64_t>(b) * p.num_q_heads + h * g + r;
        uint32_t* dst = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(p.out) + row * D * 2);
#pragma unroll
        for (int nd = 0; nd < D / 8; ++nd) {
            const float4 w1 = red[nd * 32 + lane];
            const float a0 = (o[nd][2 * half] * f0[half] + (half ? w1.z : w1.x) * f1[half]) * inv[half];
            const float a1 = (o[nd][2 * half + 1] * f0[half] + (half ? w1.w : w1.y) * f1[half]) * inv[half];
            dst[(nd * 8 + cq) / 2] = pack2<kBF16>(a0, a1);
        }
        if ((lane & 3) == 0 && p.lse)
            p.lse[static_cast<int64_t>(h * g + r) * p.B + b] = lse2[half] * 0.69314718055994531f;
    }
}

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
    using C = DecodeCfg<D, SK>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<kBF16, D, SK>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    dim3 grid(p.max_splits, p.pool.num_kv_heads, p.B);
    decode_kernel<kBF16, D, SK><<<grid, kDecodeThreads, C::SMEM_BYTES, stream>>>(tk, tv, p);
    return cudaGetLastError();
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
#define KVP_MERGE(BF, DD)                                                                                      \
    merge_kernel<BF, DD><<<blocks, threads, 0, stream>>>(ws_o, ws_lse, rows, num_q_heads, max_splits, out, lse, \
                                                        lse_stride, context_lens, block_size, pages_per_split,     \
                                                        parts_per_split)
    switch (head_dim) {
        case 64: if (bf) KVP_MERGE(true, 64); else KVP_MERGE(false, 64); break;
        case 96: if (bf) KVP_MERGE(true, 96); else KVP_MERGE(false, 96); break;
        case 128: if (bf) KVP_MERGE(true, 128); else KVP_MERGE(false, 128); break;
        default: return cudaErrorInvalidValue;
    }
#undef KVP_MERGE
    return cudaGetLastError();
}

}  // namespace kvp
