// kvp_decode_impl.cuh -- the decode-attention kernel template, shared by
// the 16-bit decode (kvp_decode.cu) and the decode over a quantized cached
// prefix (kvp_quant.cu), each translation unit instantiating its own
// variants.  See kvp_decode.cu for the design.
#pragma once
#include "kvp_internal.cuh"

namespace kvp {
namespace {

constexpr int kConsumerWarps = 2;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;
constexpr int kRingSlots = 2 * kConsumerWarps;  // two slots per consumer warp: one computing, one loading

// SK keys per stage: 16 (one 16-token block) when blocks hold <= 16 tokens,
// else 32 (one 32-token block).  BITS 8 or 4: stages of the quantized cached
// prefix arrive as codes and scales (one 16-token block per stage) and each
// consumer warp dequantizes its stage into a private 16-bit tile.
template <int D, int SK, int BITS = 0>
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
    // Quantized stage inside a slot: K codes, V codes, K meta (scale row, min
    // row, fp16), V meta ((scale, min) per token, fp16).
    static constexpr int QCODE = SK * D * BITS / 8;
    static constexpr int QOFF_V = QCODE, QOFF_KM = 2 * QCODE, QOFF_VM = 2 * QCODE + 4 * D;
    static constexpr int QSTAGE = 2 * QCODE + 4 * D + 4 * SK;
    static_assert(BITS == 0 || QSTAGE <= STAGE_BYTES, "quantized stage fits a slot");
    static constexpr int STG_BYTES = BITS ? STAGE_BYTES : 0;  // per consumer warp: dequantized K and V
    static constexpr int OFF_STG = RING_BYTES;
    static constexpr int OFF_BAR = RING_BYTES + kConsumerWarps * STG_BYTES;
    static constexpr int SMEM_BYTES = OFF_BAR + (2 * NS + 1) * 8 + 16 + 1024;
};

// Dequantize one quantized stage (SK keys of one kv head) into the warp's
// fp16 K and V tiles, in the chunked, swizzled layout the TMA path gives.
// K scale/min are per channel (a lane's channels are fixed across its keys
// when 32 is a multiple of the units per row), V's per token.  Keys at or
// past nvalid become zeros.  All addresses are shared-memory addresses; the
// accesses are explicit shared loads and stores, and each half of the
// lane's units has all its code and scale loads issued before its
// arithmetic and stores.
template <int D, int SK, int BITS>
__device__ __forceinline__ void dequant_stage(uint32_t qs, uint32_t stk, uint32_t stv, int nvalid, int lane) {
    using C = DecodeCfg<D, SK, BITS>;
    constexpr int U = D / 8;            // 16-byte output units per row
    constexpr int CROW = D * BITS / 8;  // code bytes per row
    constexpr int IT = SK * U / 32;     // units per lane
    constexpr int H = IT % 2 == 0 ? IT / 2 : IT;  // units per batch of loads
    static_assert((SK * U) % 32 == 0, "whole units per lane");
    const uint32_t kc = qs, vc = qs + C::QOFF_V, km = qs + C::QOFF_KM, vm = qs + C::QOFF_VM;
    constexpr bool kFixedUnit = (32 % U) == 0;
    uint32_t ks[4], kz[4];
    auto load_kmeta = [&](int u) {
        const uint4 a = lds128(km + u * 16);
        const uint4 b = lds128(km + 2 * D + u * 16);
        ks[0] = a.x; ks[1] = a.y; ks[2] = a.z; ks[3] = a.w;
        kz[0] = b.x; kz[1] = b.y; kz[2] = b.z; kz[3] = b.w;
    };
    if constexpr (kFixedUnit) load_kmeta(lane % U);
#pragma unroll
    for (int h0 = 0; h0 < IT; h0 += H) {
        uint2 kw[H], vw[H];
        uint32_t sz[H];
#pragma unroll
        for (int k = 0; k < H; ++k) {
            const int e = lane + 32 * (h0 + k);
            const int key = e / U, u = e - (e / U) * U;
            const uint32_t off = key * CROW + u * BITS;
            if constexpr (BITS == 8) {
                kw[k] = lds64(kc + off);
                vw[k] = lds64(vc + off);
            } else {
                kw[k] = make_uint2(lds32(kc + off), 0u);
                vw[k] = make_uint2(lds32(vc + off), 0u);
            }
            sz[k] = lds32(vm + 4 * key);  // (scale, min) of this token
        }
#pragma unroll
        for (int k = 0; k < H; ++k) {
            const int e = lane + 32 * (h0 + k);
            const int key = e / U, u = e - (e / U) * U;
            if constexpr (!kFixedUnit) load_kmeta(u);
            uint4 ko = make_uint4(0, 0, 0, 0), vo = make_uint4(0, 0, 0, 0);
            if (key < nvalid) {
                ko = dequant_words<BITS>(kw[k], ks, kz);
                const uint32_t s1 = __byte_perm(sz[k], 0, 0x1010), z1 = __byte_perm(sz[k], 0, 0x3232);
                const uint32_t vs[4] = {s1, s1, s1, s1}, vz[4] = {z1, z1, z1, z1};
                vo = dequant_words<BITS>(vw[k], vs, vz);
            }
            const uint32_t off = (u / (C::CW / 8)) * C::REGION + swz_offset(key, u % (C::CW / 8), C::ROWB);
            sts128(stk + off, ko);
            sts128(stv + off, vo);
        }
    }
}

// A 16-bit bf16 stage (the live suffix of a bf16 pool) converted to fp16 for
// the fp16 products of the quantized-prefix kernel; keys at or past nvalid
// become zeros.  Same swizzled layout in and out; shared-memory addresses.
template <int D, int SK, int BITS>
__device__ __forceinline__ void bf16_stage_to_f16(uint32_t kin, uint32_t vin, uint32_t stk, uint32_t stv,
                                                  int nvalid, int lane) {
    using C = DecodeCfg<D, SK, BITS>;
    constexpr int U = D / 8;
#pragma unroll
    for (int it = 0; it < SK * U / 32; ++it) {
        const int e = lane + 32 * it;
        const int key = e / U, u = e - (e / U) * U;
        const uint32_t off = (u / (C::CW / 8)) * C::REGION + swz_offset(key, u % (C::CW / 8), C::ROWB);
        uint4 ko = make_uint4(0, 0, 0, 0), vo = make_uint4(0, 0, 0, 0);
        if (key < nvalid) {
            const uint4 a = lds128(kin + off), b = lds128(vin + off);
            ko = make_uint4(pack2<false>(unpack2<true>(a.x).x, unpack2<true>(a.x).y),
                            pack2<false>(unpack2<true>(a.y).x, unpack2<true>(a.y).y),
                            pack2<false>(unpack2<true>(a.z).x, unpack2<true>(a.z).y),
                            pack2<false>(unpack2<true>(a.w).x, unpack2<true>(a.w).y));
            vo = make_uint4(pack2<false>(unpack2<true>(b.x).x, unpack2<true>(b.x).y),
                            pack2<false>(unpack2<true>(b.y).x, unpack2<true>(b.y).y),
                            pack2<false>(unpack2<true>(b.z).x, unpack2<true>(b.z).y),
                            pack2<false>(unpack2<true>(b.w).x, unpack2<true>(b.w).y));
        }
        sts128(stk + off, ko);
        sts128(stv + off, vo);
    }
}

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

template <bool kBF16, int D, int SK, int BITS>
__global__ void __launch_bounds__(kDecodeThreads, BITS ? 4 : 5)
    decode_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                  const DecodeParams p) {
    using C = DecodeCfg<D, SK, BITS>;
    static_assert(BITS == 0 || BITS == 4 || BITS == 8, "bits");
    // The quantized-prefix kernel runs its tensor-core products in fp16
    // whatever the pool dtype (fp16 holds the dequantized values and a bf16
    // pool's values more closely than bf16); the output keeps the pool dtype.
    constexpr bool kMma = BITS ? false : kBF16;
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
    // Pages [0, qp) of this sequence are quantized blocks (one page per stage
    // then: the quantized path runs with block_size == SK == 16).
    const int qp = (BITS > 0 && p.qpages) ? min(max(__ldg(p.qpages + b), 0), npages) : 0;

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
                const int64_t nblk = (BITS > 0 && pg < qp) ? p.qpool.num_blocks : p.pool.num_blocks;
                if (blk < 0 || blk >= nblk) {
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
            const bool qst = BITS > 0 && page0 + i < qp;
            if (lane == 0) mbar_expect_tx(&full[slot], qst ? C::QSTAGE : C::STAGE_BYTES);
            __syncwarp();
            // One lane per physical page of the stage issues that page's boxes.
            const int blk = __shfl_sync(0xffffffffu, my_blk, (rel + lane) & 31);
            uint8_t* kst = smem + slot * C::STAGE_BYTES;
            uint8_t* vst = kst + C::KBYTES;
            if constexpr (BITS > 0) {
                if (qst) {
                    // A quantized page: codes and scales, four contiguous pieces.
                    if (lane == 0) {
                        const int64_t ph = static_cast<int64_t>(blk) * Hkv + h;
                        bulk_load(kst, p.qpool.k_codes + ph * C::QCODE, C::QCODE, &full[slot]);
                        bulk_load(kst + C::QOFF_V, p.qpool.v_codes + ph * C::QCODE, C::QCODE, &full[slot]);
                        bulk_load(kst + C::QOFF_KM, p.qpool.k_meta + ph * 2 * D, 4 * D, &full[slot]);
                        bulk_load(kst + C::QOFF_VM, p.qpool.v_meta + ph * 2 * SK, 4 * SK, &full[slot]);
                    }
                    issued = i + 1;
                    continue;
                }
            }
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
            if constexpr (kMma != kBF16) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 f = unpack2<kBF16>(qa[ks][j]);
                    qa[ks][j] = pack2<kMma>(f.x, f.y);
                }
            }
        }
        const float sl2 = p.scale_log2;

        for (int i = warp; i < nstages; i += kConsumerWarps) {
            const int slot = i % C::NS;
            if (!mbar_wait(&full[slot], (i / C::NS) & 1, abort_flag, err, p.wait_limit_ns)) break;
            uint8_t* kst = smem + slot * C::STAGE_BYTES;
            uint8_t* vst = kst + C::KBYTES;
            const int kbeg = key0 + i * kStageKeys;
            const int nvalid = min(kStageKeys, key1 - kbeg);
            const bool qst = BITS > 0 && page0 + i < qp;
            // Staged: dequantized (or converted to fp16) into this warp's own
            // tile, after which the slot goes back at once.
            const bool staged = BITS > 0 && (qst || kBF16);
            if constexpr (BITS > 0) {
                if (staged) {
                    uint8_t* stk = smem + C::OFF_STG + warp * C::STG_BYTES;
                    const uint32_t stk_a = smem_u32(stk);
                    if (qst)
                        dequant_stage<D, SK, BITS>(smem_u32(kst), stk_a, stk_a + C::KBYTES, nvalid, lane);
                    else
                        bf16_stage_to_f16<D, SK, BITS>(smem_u32(kst), smem_u32(vst), stk_a, stk_a + C::KBYTES, nvalid,
                                                       lane);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[slot]);
                    kst = stk;
                    vst = stk + C::KBYTES;
                }
            }
            if (!staged && nvalid < kStageKeys) {
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
                    mma16816<kMma>(s[2 * np], qa[ks], b0, b1);
                    mma16816<kMma>(s[2 * np + 1], qa[ks], b2, b3);
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
                pa[kk][0] = pack2<kMma>(s[2 * kk][0], s[2 * kk][1]);
                pa[kk][1] = pack2<kMma>(s[2 * kk][2], s[2 * kk][3]);
                pa[kk][2] = pack2<kMma>(s[2 * kk + 1][0], s[2 * kk + 1][1]);
                pa[kk][3] = pack2<kMma>(s[2 * kk + 1][2], s[2 * kk + 1][3]);
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
                    mma16816<kMma>(o[2 * nd2], pa[kk], b0, b1);
                    mma16816<kMma>(o[2 * nd2 + 1], pa[kk], b2, b3);
                }
            }
            if (!staged) {
                if (nvalid < kStageKeys) fence_proxy_async_smem();  // generic zeroing before the next TMA write
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[slot]);
            } else {
                __syncwarp();  // the tile is rewritten by the next stage's dequantization
            }
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

template <bool kBF16, int D, int SK, int BITS>
cudaError_t launch_decode_kernel(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                                 cudaStream_t stream) {
    using C = DecodeCfg<D, SK, BITS>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<kBF16, D, SK, BITS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    dim3 grid(p.max_splits, p.pool.num_kv_heads, p.B);
    return launch_k(decode_kernel<kBF16, D, SK, BITS>, grid, kDecodeThreads, C::SMEM_BYTES, stream, tk, tv, p);
}

}  // namespace
}  // namespace kvp
