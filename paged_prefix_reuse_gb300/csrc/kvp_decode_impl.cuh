// kvp_decode_impl.cuh -- the 16-bit decode-attention kernel template
// (instantiated by kvp_decode.cu; see there for the design) and the small
// shared-memory helpers (align1024) that the decode over a quantized cached
// prefix (kvp_quant.cu) uses too.
#pragma once
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
    static constexpr int OFF_BAR = RING_BYTES;
    static constexpr int SMEM_BYTES = OFF_BAR + (2 * NS + 1) * 8 + 16 + 1024;
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
__global__ void __launch_bounds__(kDecodeThreads, 5)
    decode_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                  const DecodeParams p) {
    using C = DecodeCfg<D, SK>;
    constexpr int kStageKeys = SK;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* empty = full + C::NS;
    uint64_t* stall = empty + C::NS;  // nothing arrives on it (KVP_LAUNCH_STALL_TEST)
    volatile int* abort_flag = reinterpret_cast<volatile int*>(stall + 1);

    const int sp = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_trigger();
    const int BS = p.pool.block_size;
    const int Hkv = p.pool.num_kv_heads;
    const int g = p.group;
    uint32_t* err = p.pool.err_word;

    const int L = __ldg(p.context_lens + b);
    const int npages = (L + BS - 1) / BS;
    if (L < 1 || npages > p.max_blocks) {
        if (sp == 0 && tid == 0) report(err, KVP_DEVERR_BAD_LEN);
        pdl_wait();  // every CTA waits, so the grid completes after the one before
        return;
    }
    const int page0 = sp * p.pages_per_split;
    if (page0 >= npages) {
        pdl_wait();
        return;
    }
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
        mbar_init(stall, 1);
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
        pdl_wait();  // pool contents from the kernel before are read from here on
        // Test of the failure path: before any copy is issued, wait on a
        // barrier nothing arrives on until the limit runs out.
        const bool stalled = p.stall_test && !stall_wait(stall, abort_flag, err, p.wait_limit_ns);
        int my_blk = 0;
        int issued = 0;
        for (int i = 0; i < nstages && !stalled; ++i) {
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
            if (lane == 0 && i >= C::NS)
                ok = mbar_wait(&empty[slot], ((i / C::NS) - 1) & 1, abort_flag, err, p.wait_limit_ns);
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
            if (!mbar_wait(&full[slot], (i / C::NS) & 1, abort_flag, err, p.wait_limit_ns)) break;
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
            // Lazy reference maximum: it moves (and O, l are rescaled) only
            // when a row maximum grows by more than 2^8; exps against a stale
            // reference stay <= 2^8, and the final 1/l uses the same one.
            const float mx0s = mx0 * sl2, mx1s = mx1 * sl2;
            float a0 = 1.f, a1 = 1.f;
            if (mx0s > m_run[0] + 8.f) {
                a0 = fast_exp2(m_run[0] - mx0s);
                m_run[0] = mx0s;
                l_run[0] *= a0;
            }
            if (mx1s > m_run[1] + 8.f) {
                a1 = fast_exp2(m_run[1] - mx1s);
                m_run[1] = mx1s;
                l_run[1] *= a1;
            }
            const float mn0 = m_run[0] == -INFINITY ? 0.f : m_run[0];
            const float mn1 = m_run[1] == -INFINITY ? 0.f : m_run[1];
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
            l_run[0] += ps0;
            l_run[1] += ps1;
            if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
                for (int nd = 0; nd < D / 8; ++nd) {
                    o[nd][0] *= a0;
                    o[nd][1] *= a0;
                    o[nd][2] *= a1;
                    o[nd][3] *= a1;
                }
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

template <bool kBF16, int D, int SK>
cudaError_t launch_decode_kernel(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
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
    return launch_k(decode_kernel<kBF16, D, SK>, grid, kDecodeThreads, C::SMEM_BYTES, stream, tk, tv, p);
}

}  // namespace
}  // namespace kvp
