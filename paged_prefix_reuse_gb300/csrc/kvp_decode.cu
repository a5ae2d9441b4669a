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

constexpr int kStageKeys = 32;
constexpr int kConsumerWarps = 4;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;
constexpr int kRingBytes = 96 * 1024;

template <int D>
struct DecodeCfg {
    static constexpr int CW = chunk_elems(D);
    static constexpr int ROWB = CW * 2;
    static constexpr int NCH = D / CW;
    static constexpr int REGION = kStageKeys * ROWB;  // one chunk column of a stage's K (or V)
    static constexpr int KBYTES = kStageKeys * D * 2;
    static constexpr int STAGE_BYTES = 2 * KBYTES;
    // Stage i sits in slot i % NS and is consumed by warp i % 4.  NS is a
    // multiple of the consumer count, so every slot has one owner warp that
    // consumes its phases in order: a waiter can never be two phases behind,
    // which a parity wait could not tell apart from the phase it wants.
    static constexpr int NS = kConsumerWarps * (kRingBytes / (kConsumerWarps * STAGE_BYTES));
    static_assert(NS >= kConsumerWarps && NS % kConsumerWarps == 0, "ring depth");
    static constexpr int RED_BYTES = kConsumerWarps * 16 * D * 4 + 2 * kConsumerWarps * 16 * 4;
    static constexpr int SMEM_BYTES = NS * STAGE_BYTES + 2 * NS * 8 + 16 + 1024;
    static_assert(RED_BYTES <= NS * STAGE_BYTES, "reduction area reuses the ring");
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

template <bool kBF16, int D>
__global__ void __launch_bounds__(kDecodeThreads, 2)
    decode_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                  const DecodeParams p) {
    using C = DecodeCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::NS * C::STAGE_BYTES);
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

            // S = q K^T for 32 keys: 4 n-tiles of 8 keys.
            float s[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
                for (int np = 0; np < 2; ++np) {
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
                for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (nt * 8 + cq + (e & 1) >= nvalid) s[nt][e] = -INFINITY;
            }
            // Online softmax (log2 domain; the scale is folded into the exponent).
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
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
            for (int nt = 0; nt < 4; ++nt) {
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
            uint32_t pa[2][4];
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                pa[kk][0] = pack2<kBF16>(s[2 * kk][0], s[2 * kk][1]);
                pa[kk][1] = pack2<kBF16>(s[2 * kk][2], s[2 * kk][3]);
                pa[kk][2] = pack2<kBF16>(s[2 * kk + 1][0], s[2 * kk + 1][1]);
                pa[kk][3] = pack2<kBF16>(s[2 * kk + 1][2], s[2 * kk + 1][3]);
            }
            // O += P V: V is [key][dim] in shared memory, loaded transposed.
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
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

    // ------------------- merge the four warps' states -------------------------
    __syncthreads();  // every stage consumed and every copy landed: the ring is free
    float* red_o = reinterpret_cast<float*>(smem);                   // [4][16][D]
    float* red_m = red_o + kConsumerWarps * 16 * D;                  // [4][16]
    float* red_l = red_m + kConsumerWarps * 16;                      // [4][16]
    if (warp < kConsumerWarps) {
        const int r0 = lane >> 2, r1 = r0 + 8, cq = 2 * (lane & 3);
        float* wo = red_o + warp * 16 * D;
#pragma unroll
        for (int nd = 0; nd < D / 8; ++nd) {
            wo[r0 * D + nd * 8 + cq] = o[nd][0];
            wo[r0 * D + nd * 8 + cq + 1] = o[nd][1];
            wo[r1 * D + nd * 8 + cq] = o[nd][2];
            wo[r1 * D + nd * 8 + cq + 1] = o[nd][3];
        }
        if ((lane & 3) == 0) {
            red_m[warp * 16 + r0] = m_run[0];
            red_m[warp * 16 + r1] = m_run[1];
            red_l[warp * 16 + r0] = l_run[0];
            red_l[warp * 16 + r1] = l_run[1];
        }
    }
    __syncthreads();
    if (warp < kConsumerWarps && !*abort_flag) {
        for (int e = tid; e < g * D; e += kConsumerWarps * 32) {
            const int r = e / D, c = e - (e / D) * D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, red_m[w * 16 + r]);
            float lsum = 0.f, acc = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float mw = red_m[w * 16 + r];
                const float f = (mw == -INFINITY) ? 0.f : fast_exp2(mw - M);
                lsum += red_l[w * 16 + r] * f;
                acc += red_o[(w * 16 + r) * D + c] * f;
            }
            const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
            const float lse2 = lsum > 0.f ? M + __log2f(lsum) : -INFINITY;
            const int64_t row = static_cast<int64_t>(b) * p.num_q_heads + h * g + r;
            if (p.max_splits == 1) {
                if constexpr (kBF16)
                    static_cast<__nv_bfloat16*>(p.out)[row * D + c] = __float2bfloat16_rn(acc * inv);
                else
                    static_cast<__half*>(p.out)[row * D + c] = __float2half_rn(acc * inv);
                if (c == 0 && p.lse) p.lse[static_cast<int64_t>(h * g + r) * p.B + b] = lse2 * 0.69314718055994531f;
            } else {
                p.ws_o[(row * p.max_splits + sp) * D + c] = acc * inv;
                if (c == 0) p.ws_lse[row * p.max_splits + sp] = lse2;
            }
        }
    }
}

// One warp per output row: merge `splits` partials (normalised O, log2 lse).
template <bool kBF16>
__global__ void merge_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_lse, int32_t rows,
                             int32_t Hq, int32_t D, int32_t max_splits, void* __restrict__ out,
                             float* __restrict__ lse, int32_t lse_stride, const int32_t* __restrict__ ctx,
                             int32_t block_size, int32_t pages_per_split) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= rows) return;
    const int64_t row = warp;
    int splits = max_splits;
    if (ctx) {  // decode: the sequence's own split count
        const int L = __ldg(ctx + row / Hq);
        const int np = (L + block_size - 1) / block_size;
        splits = max(0, min(max_splits, (np + pages_per_split - 1) / pages_per_split));
    }
    float M = -INFINITY;
    for (int i = lane; i < splits; i += 32) M = fmaxf(M, ws_lse[row * max_splits + i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float sum = 0.f;
    for (int i = lane; i < splits; i += 32) {
        const float li = ws_lse[row * max_splits + i];
        sum += (li == -INFINITY) ? 0.f : fast_exp2(li - M);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float tot = (M == -INFINITY || sum <= 0.f) ? -INFINITY : M + __log2f(sum);
    for (int c = lane; c < D; c += 32) {
        float acc = 0.f;
        if (tot != -INFINITY) {
            for (int i = 0; i < splits; ++i) {
                const float li = ws_lse[row * max_splits + i];
                if (li != -INFINITY) acc += fast_exp2(li - tot) * ws_o[(row * max_splits + i) * D + c];
            }
        }
        if constexpr (kBF16)
            static_cast<__nv_bfloat16*>(out)[row * D + c] = __float2bfloat16_rn(acc);
        else
            static_cast<__half*>(out)[row * D + c] = __float2half_rn(acc);
    }
    if (lane == 0 && lse) lse[(row % Hq) * lse_stride + row / Hq] = tot * 0.69314718055994531f;
}

template <bool kBF16, int D>
cudaError_t launch_decode_t(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                            cudaStream_t stream) {
    using C = DecodeCfg<D>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<kBF16, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    dim3 grid(p.max_splits, p.pool.num_kv_heads, p.B);
    decode_kernel<kBF16, D><<<grid, kDecodeThreads, C::SMEM_BYTES, stream>>>(tk, tv, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_attn(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                               cudaStream_t stream) {
    const bool bf = p.pool.dtype == KVP_BF16;
    switch (p.pool.head_dim) {
        case 64: return bf ? launch_decode_t<true, 64>(p, tk, tv, stream) : launch_decode_t<false, 64>(p, tk, tv, stream);
        case 96: return bf ? launch_decode_t<true, 96>(p, tk, tv, stream) : launch_decode_t<false, 96>(p, tk, tv, stream);
        case 128: return bf ? launch_decode_t<true, 128>(p, tk, tv, stream) : launch_decode_t<false, 128>(p, tk, tv, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_merge(const float* ws_o, const float* ws_lse, int32_t rows, int32_t num_q_heads,
                         int32_t head_dim, int32_t max_splits, int32_t dtype, void* out, float* lse,
                         int32_t lse_stride, const int32_t* context_lens, int32_t block_size,
                         int32_t pages_per_split, cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    const int threads = 256;
    const int blocks = (rows * 32 + threads - 1) / threads;
    if (dtype == KVP_BF16)
        merge_kernel<true><<<blocks, threads, 0, stream>>>(ws_o, ws_lse, rows, num_q_heads, head_dim, max_splits,
                                                           out, lse, lse_stride, context_lens, block_size,
                                                           pages_per_split);
    else
        merge_kernel<false><<<blocks, threads, 0, stream>>>(ws_o, ws_lse, rows, num_q_heads, head_dim,
                                                            max_splits, out, lse, lse_stride, context_lens,
                                                            block_size, pages_per_split);
    return cudaGetLastError();
}

}  // namespace kvp
