// kvp_internal.cuh -- shared pieces of libkvp's sm_103a kernels: inline-PTX
// wrappers (mbarrier, TMA, tcgen05/TMEM), bounded waits, swizzle addressing,
// and the launch functions each .cu file provides to the C-ABI layer.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvp.h"

namespace kvp {

// ---------------------------------------------------------------------------
// Launch parameters shared between host and device.
// ---------------------------------------------------------------------------
struct PoolView {
    int64_t num_blocks;
    int32_t block_size, num_kv_heads, head_dim, dtype;
    uint32_t* err_word;
};

// ---- programmatic dependent launch (KVP_LAUNCH_PDL) -------------------------
// Both are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

uint32_t launch_flags();      // kvp_set_launch_options
uint64_t wait_limit_ns();     // kvp_set_wait_limit_ns (pipeline waits)

// Launch with the programmatic-stream-serialization attribute when
// KVP_LAUNCH_PDL is set, a plain launch otherwise.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                     Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (launch_flags() & KVP_LAUNCH_PDL) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// A quantized pool (see kvp_qpool in kvp.h).  bits == 0: none.
struct QPoolView {
    uint8_t* k_codes;
    uint8_t* v_codes;
    __half* k_meta;
    __half* v_meta;
    int64_t num_blocks;
    int32_t bits;
};

struct PrefixParams {
    PoolView pool;
    const void* q;
    void* out;
    float* lse;
    const int32_t* cu_seqlens_q;
    const int32_t* context_lens;
    const int32_t* block_tables;
    int32_t max_blocks, B, total_q, num_q_heads, group;  // group = Hq / Hkv
    uint64_t group_mul;  // ceil(2^32 / group): n / group = (n * group_mul) >> 32 for n < 2^24
    int32_t q_tiles;     // CTA row tiles per (sequence, kv head)
    int32_t num_splits;
    float scale_log2;  // softmax_scale * log2(e)
    float* ws_o;       // [total_q * Hq][num_splits][head_dim] fp32 (splits > 1)
    float* ws_lse;     // [total_q * Hq][num_splits] fp32, log2 domain
    uint64_t wait_limit_ns;  // limit of the pipeline waits
    int32_t stall_test;      // KVP_LAUNCH_STALL_TEST: wait on a barrier nothing arrives on
    QPoolView qpool;         // quantized prefix pages (bits 0: none)
    const int32_t* qpages;   // [B]: leading table entries that name qpool blocks
};

struct DecodeParams {
    PoolView pool;
    const void* q;
    void* out;
    float* lse;
    const int32_t* context_lens;
    const int32_t* block_tables;
    int32_t max_blocks, B, num_q_heads, group;
    int32_t pages_per_split;  // multiple of the pages in one stage
    int32_t max_splits;
    float scale_log2;
    float* ws_o;    // [B * Hq][max_splits * parts][head_dim]
    float* ws_lse;  // [B * Hq][max_splits * parts], log2 domain
    QPoolView qpool;         // quantized prefix pages (bits 0: none)
    const int32_t* qpages;   // [B]: leading table entries that name qpool blocks
    uint64_t wait_limit_ns;  // limit of the pipeline waits
    int32_t stall_test;      // KVP_LAUNCH_STALL_TEST: wait on a barrier nothing arrives on
};

// Host-side launchers (defined in the kernel .cu files).
cudaError_t launch_slot_mapping(const PoolView& pool, const int32_t* cu_seqlens_q, const int32_t* context_lens,
                                const int32_t* block_tables, int32_t max_blocks, int32_t B, int32_t total_q,
                                int64_t* slot_mapping, cudaStream_t stream);
cudaError_t launch_cache_append(const PoolView& pool, void* k_pool, void* v_pool, const void* k_new,
                                const void* v_new, const int64_t* slot_mapping, int32_t T, cudaStream_t stream);
cudaError_t launch_block_copy(const PoolView& pool, void* k_pool, void* v_pool, const int32_t* pairs, int32_t n,
                              cudaStream_t stream);
cudaError_t launch_quantize_blocks(const PoolView& pool, const void* k_pool, const void* v_pool,
                                   const QPoolView& qpool, const int32_t* pairs, int32_t n, cudaStream_t stream);
// tk, tv: boxes of kDecodeQHalfRows rows (half a 16-token block) of the
// 16-bit pool; tkc, tvc: the quantized pool's code arrays, boxes of one
// page-head of code rows.
cudaError_t launch_decode_attn_q(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const CUtensorMap& tkc, const CUtensorMap& tvc, cudaStream_t stream);
constexpr int kDecodeQHalfRows = 8;
cudaError_t launch_kv_deviation(const PoolView& pool, const void* k_pool, const void* v_pool, const void* k_fresh,
                                const void* v_fresh, const int64_t* slots, int32_t T, float* dev, cudaStream_t stream);
cudaError_t launch_select_recompute(const float* dev, const int64_t* slots, const int32_t* cu, int32_t B,
                                    int32_t permille, int64_t* out_slots, int32_t* counts, cudaStream_t stream);
cudaError_t launch_block_swap(const PoolView& pool, void* k_pool, void* v_pool, void* host_k, void* host_v,
                              int64_t host_blocks, const int32_t* pairs, int32_t n, bool to_host,
                              cudaStream_t stream);
cudaError_t launch_prefix_attn(const PrefixParams& p, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                               cudaStream_t stream);
// The same over a partly quantized context (p.qpool, p.qpages; block_size 16).
cudaError_t launch_prefix_attn_q(const PrefixParams& p, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                 cudaStream_t stream);
// Query rows (token, head-of-group pairs) one prefix CTA covers.
int prefix_rows_per_cta();
// Columns of one TMA box of the prefix kernel's K/V tiles (64 at head_dim 96:
// that kernel runs head_dim 96 padded to 128).
int prefix_chunk_elems(int head_dim);
cudaError_t launch_decode_attn(const DecodeParams& p, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                               cudaStream_t stream);
// Merge of split partials: rows = total_q*Hq (prefix) or B*Hq (decode), with
// max_splits * parts_per_split partials per row.  For decode, each row's
// split count derives from its sequence's context length.
cudaError_t launch_merge(const float* ws_o, const float* ws_lse, int32_t rows, int32_t num_q_heads,
                         int32_t head_dim, int32_t max_splits, int32_t dtype, void* out, float* lse,
                         int32_t lse_stride, const int32_t* context_lens, int32_t block_size,
                         int32_t pages_per_split, int32_t parts_per_split, cudaStream_t stream);
// Partials one decode split writes (one per consumer warp).
int decode_parts_per_split();
// Validates a decode call's arguments exactly as kvp_decode_attn does and
// sets *need to the workspace bytes of the split count that call would
// resolve (split geometry included; 0 for one split or an empty batch).
kvp_status decode_workspace_need(const kvp_pool* pool, const void* q, void* out, float* lse,
                                 const int32_t* context_lens, const int32_t* block_tables, int32_t max_blocks,
                                 int32_t B, int32_t num_q_heads, int32_t max_context_len, float softmax_scale,
                                 int32_t num_splits, size_t* need);

// Give up on any single wait after this long by default; a healthy wait
// lasts microseconds.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Swizzle chunk width (elements of one TMA box row) for a head dimension:
// 64 elements (128-byte rows, 128B swizzle) when head_dim is a multiple of
// 64, else 32 elements (64-byte rows, 64B swizzle).
__host__ __device__ constexpr int chunk_elems(int head_dim) { return (head_dim % 64 == 0) ? 64 : 32; }

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------
#if defined(__CUDACC__)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void report(uint32_t* err_word, uint32_t bits) {
    if (err_word) atomicOr(err_word, bits);
}

// ---- mbarrier ----
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// The same test, but a thread whose phase is not complete sleeps in hardware
// until the phase completes (or the hint, in ns, runs out) instead of
// returning at once: a waiting warp then takes no issue slots from the warps
// that share its scheduler.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(100000u)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity.  Returns false when the
// wait gave up (limit reached, or another thread of the CTA already gave up
// and raised *abort); the caller must then wind down.  Pipeline waits take
// the call's limit (kvp_set_wait_limit_ns); the drain waits of a CTA that is
// winding down -- copies in flight, the last tensor-core commit -- keep the
// default, so that nothing can land in shared or tensor memory after exit.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint32_t* err_word, uint64_t limit_ns = kWaitLimitNs) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_sleep(a, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > limit_ns) {
                *abort = 1;
                report(err_word, KVP_DEVERR_TIMEOUT);
                return false;
            }
        }
    }
}

// KVP_LAUNCH_STALL_TEST: the calling threads wait on `bar`, which nothing
// arrives on, until the pipeline limit runs out; the wait gives up, raises
// *abort and reports KVP_DEVERR_TIMEOUT, and the CTA winds down along the
// same paths as after any timed-out wait.  Returns false.
__device__ __forceinline__ bool stall_wait(uint64_t* bar, volatile int* abort, uint32_t* err_word,
                                           uint64_t limit_ns) {
    // test_wait never suspends the thread, and the clock is read on every
    // pass, so the give-up time is the limit itself.
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], 0;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(a)
            : "memory");
        if (done) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > limit_ns) {
            *abort = 1;
            report(err_word, KVP_DEVERR_TIMEOUT);
            return false;
        }
    }
}

// ---- proxy fences ----
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- TMA: 2-D tiled load into shared memory, completion on an mbarrier ----
__device__ __forceinline__ void tma_load_2d(void* dst_smem, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_u32(dst_smem)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// 1-D bulk copy global -> shared, completion on an mbarrier (both addresses
// 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst_smem)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- swizzled shared-memory addressing --------------------------------------
// Byte offset of the 16-byte chunk `c16` of row `row` in a tile whose rows are
// `row_bytes` (128 or 64) long, written by TMA with the matching swizzle mode
// (128B: chunk ^= row % 8; 64B: chunk ^= (row / 2) % 4).  The tile must start
// on a 1024-byte boundary.
__device__ __forceinline__ uint32_t swz_offset(uint32_t row, uint32_t c16, uint32_t row_bytes) {
    if (row_bytes == 128) return row * 128u + ((c16 ^ (row & 7u)) << 4);
    return row * 64u + ((c16 ^ ((row >> 1) & 3u)) << 4);
}

// ---- tcgen05 / TMEM ---------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (fp16/bf16 in, fp32 accumulate).
// The tcgen05.mma / tcgen05.commit wrappers below are warp-collective: all
// 32 lanes of the issuing warp call them together (converged) and one lane,
// chosen by elect.sync inside the same asm block, issues the instruction.
// Issuing from a lane-0 branch instead leaves the warp diverged, and a
// diverged issuer that shares its SM sub-partition with busy softmax warps
// issues MMAs up to 3x slower than the tensor core executes them (measured
// on GB300); the converged, predicated form is unaffected.
__device__ __forceinline__ void tc_mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on an mbarrier once all previously issued tcgen05 ops of the
// issuing thread complete (warp-collective, one elected lane commits).
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
            smem_u32(bar))
        : "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (>> 4), version 1 at bits 46-47, swizzle mode at
// bits 61-63 (0 none, 2 = 128B, 4 = 64B, 6 = 32B).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swz) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(swz & 7u) << 61;
    return d;
}

// Instruction descriptor for kind::f16: fp32 accumulator, A/B fp16 or bf16,
// A K-major, B K-major (b_mn_major = 0) or MN-major (1), shape M x N.
__host__ __device__ constexpr uint32_t instr_desc_f16(bool bf16, int M, int N, bool b_mn_major) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// 32 lanes x 32 bits, 32 consecutive columns: thread i of the warp receives
// columns [col, col+32) of TMEM lane (warp's lane quarter base + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }


// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16; A is M x K with row i in TMEM
// lane i and two 16-bit elements per 32-bit column (lower K index in the low half).
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 32 lanes x 32 bits, 64 consecutive columns starting at taddr.
__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]), "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]), "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]), "r"(r[40]), "r"(r[41]), "r"(r[42]), "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]), "r"(r[48]), "r"(r[49]), "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]), "r"(r[56]), "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63])
        : "memory");
}

// Blackwell packed-fp32 arithmetic and the 3-input maximum.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(d)
        : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)),
          "l"(*reinterpret_cast<uint64_t*>(&c)));
    return *reinterpret_cast<float2*>(&d);
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    uint64_t d;
    asm("add.f32x2 %0, %1, %2;"
        : "=l"(d)
        : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
    return *reinterpret_cast<float2*>(&d);
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// ---- small numeric helpers ----
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---- dequantization of 8/4-bit codes (the quantized pool) ----
// Two codes -> half2 (1024 + c0, 1024 + c1): exact, since fp16 has unit
// spacing on [1024, 2048).  The codes sit in bytes i and j of w; every byte
// of the constant source is 0x64, the high byte of 1024.0 in fp16.
__device__ __forceinline__ uint32_t magic_pair(uint32_t w, uint32_t sel) {
    return __byte_perm(w, 0x64646464u, sel);
}

// Dequantize one 8-channel unit: codes -> fp16 (1024 + c) - 1024, then
// c * s + z in one fp16 fused multiply-add per pair (a single rounding).
// 8 bits: 8 code bytes in w.x, w.y; 4 bits: 8 nibbles in w.x, the even
// channel in the low one.
template <int BITS>
__device__ __forceinline__ uint4 dequant_words(uint2 w, const uint32_t (&s2)[4], const uint32_t (&z2)[4]) {
    uint32_t h[4];
    if constexpr (BITS == 8) {
        h[0] = magic_pair(w.x, 0x4140);
        h[1] = magic_pair(w.x, 0x4342);
        h[2] = magic_pair(w.y, 0x4140);
        h[3] = magic_pair(w.y, 0x4342);
    } else {
        const uint32_t lo = w.x & 0x0F0F0F0Fu, hi = (w.x >> 4) & 0x0F0F0F0Fu;  // even / odd channels
        const uint32_t t = __byte_perm(lo, hi, 0x5140), u = __byte_perm(lo, hi, 0x7362);  // c0..c3, c4..c7
        h[0] = magic_pair(t, 0x4140);
        h[1] = magic_pair(t, 0x4342);
        h[2] = magic_pair(u, 0x4140);
        h[3] = magic_pair(u, 0x4342);
    }
    const __half2 k1024 = __float2half2_rn(1024.f);
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const __half2 c = __hsub2(*reinterpret_cast<const __half2*>(&h[j]), k1024);
        const __half2 x = __hfma2(c, *reinterpret_cast<const __half2*>(&s2[j]), *reinterpret_cast<const __half2*>(&z2[j]));
        o[j] = *reinterpret_cast<const uint32_t*>(&x);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// The same, reading the unit's codes through a pointer.
template <int BITS>
__device__ __forceinline__ uint4 dequant_unit(const uint8_t* codes, const uint32_t (&s2)[4], const uint32_t (&z2)[4]) {
    uint2 w;
    if constexpr (BITS == 8) {
        w = *reinterpret_cast<const uint2*>(codes);
    } else {
        w = make_uint2(*reinterpret_cast<const uint32_t*>(codes), 0u);
    }
    return dequant_words<BITS>(w, s2, z2);
}

// ---- explicit shared-memory accesses (32-bit shared addresses) ----
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a)
                 : "memory");
    return v;
}
__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

template <bool kBF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    if constexpr (kBF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&v);
    } else {
        __half2 v = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&v);
    }
}

template <bool kBF16>
__device__ __forceinline__ float2 unpack2(uint32_t u) {
    if constexpr (kBF16) {
        __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
        return __bfloat1622float2(v);
    } else {
        __half2 v = *reinterpret_cast<__half2*>(&u);
        return __half22float2(v);
    }
}

#endif  // __CUDACC__

}  // namespace kvp
