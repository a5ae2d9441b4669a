// kvp_api.cu -- the extern "C" entry points of libkvp: host-side argument
// validation, TMA tensor-map construction for the pools, split-count
// heuristics, workspace carving, and kernel launches on the caller's stream.
#include <math.h>
#include <string.h>

#include <atomic>

#include "kvp_internal.cuh"

namespace kvp {

std::atomic<uint32_t> g_launch_flags{0};
uint32_t launch_flags() { return g_launch_flags.load(std::memory_order_relaxed); }
std::atomic<uint64_t> g_wait_limit_ns{kWaitLimitNs};
uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }
namespace {

constexpr int kNumSMs = 152;  // GB300; used only by the split heuristics

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The pool viewed as a 2-D tensor of rows (block, kv head, slot) x head_dim;
// one TMA box is one block of one kv head, `chunk_elems` columns wide.
// Boxes of CW columns (0: the head dim's chunk) by box_rows rows (0: one
// block); a box wider than the row reads zeros past it.
kvp_status make_pool_map(CUtensorMap* map, void* base, const kvp_pool* pool, int CW = 0, int box_rows = 0) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return KVP_ERR_CUDA;
    const int D = pool->head_dim;
    if (CW == 0) CW = chunk_elems(D);
    if (box_rows == 0) box_rows = pool->block_size;
    const cuuint64_t rows = static_cast<cuuint64_t>(pool->num_blocks) * pool->num_kv_heads * pool->block_size;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), rows};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(CW), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt =
        pool->dtype == KVP_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const CUtensorMapSwizzle swz = CW == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    CUresult r = enc(map, dt, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? KVP_OK : KVP_ERR_CUDA;
}

// A code array of a quantized pool as a 2-D tensor of one row of codes per
// token (head_dim * bits / 8 bytes), boxes of one page-head.  Rows of 128 or
// 64 bytes land with the matching swizzle, other widths unswizzled.
kvp_status make_code_map(CUtensorMap* map, void* base, const kvp_qpool* qp) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return KVP_ERR_CUDA;
    const int crow = qp->head_dim * qp->bits / 8;
    const cuuint64_t rows = static_cast<cuuint64_t>(qp->num_blocks) * qp->num_kv_heads * qp->block_size;
    if (rows >= (cuuint64_t(1) << 31)) return KVP_ERR_INVALID_ARG;  // TMA row coordinates are int32
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(crow), rows};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(crow)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(crow), static_cast<cuuint32_t>(qp->block_size)};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle swz = crow == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                   : crow == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                : CU_TENSOR_MAP_SWIZZLE_NONE;
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? KVP_OK : KVP_ERR_CUDA;
}

kvp_status check_pool(const kvp_pool* pool) {
    if (!pool || !pool->k_pool || !pool->v_pool) return KVP_ERR_INVALID_ARG;
    if (!aligned16(pool->k_pool) || !aligned16(pool->v_pool)) return KVP_ERR_INVALID_ARG;
    if (pool->num_blocks < 1 || pool->num_kv_heads < 1) return KVP_ERR_INVALID_ARG;
    if (pool->dtype != KVP_F16 && pool->dtype != KVP_BF16) return KVP_ERR_UNSUPPORTED;
    if (pool->head_dim != 64 && pool->head_dim != 96 && pool->head_dim != 128) return KVP_ERR_UNSUPPORTED;
    if (pool->block_size != 8 && pool->block_size != 16 && pool->block_size != 32) return KVP_ERR_UNSUPPORTED;
    // TMA row coordinates are int32.
    const int64_t rows = pool->num_blocks * pool->num_kv_heads * static_cast<int64_t>(pool->block_size);
    if (rows <= 0 || rows >= (int64_t(1) << 31)) return KVP_ERR_INVALID_ARG;
    return KVP_OK;
}

PoolView view_of(const kvp_pool* pool) {
    PoolView v;
    v.num_blocks = pool->num_blocks;
    v.block_size = pool->block_size;
    v.num_kv_heads = pool->num_kv_heads;
    v.head_dim = pool->head_dim;
    v.dtype = pool->dtype;
    v.err_word = pool->err_word;
    return v;
}

kvp_status from_cuda(cudaError_t e) { return e == cudaSuccess ? KVP_OK : KVP_ERR_CUDA; }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

int32_t ceil_div(int64_t a, int64_t b) { return static_cast<int32_t>((a + b - 1) / b); }

// Decode split geometry: pages per split (a multiple of the pages in one
// 32-key stage) and the resulting split count of the longest context.
void decode_geometry(int32_t block_size, int32_t max_context_len, int32_t num_splits, int32_t* pages_per_split,
                     int32_t* max_splits) {
    const int32_t max_pages = ceil_div(max_context_len, block_size);
    const int32_t stage_pages = 32 / block_size;
    int32_t pps = ceil_div(max_pages, num_splits < 1 ? 1 : num_splits);
    pps = ceil_div(pps, stage_pages) * stage_pages;
    *pages_per_split = pps;
    *max_splits = ceil_div(max_pages, pps);
}

}  // namespace
}  // namespace kvp

using namespace kvp;

extern "C" {

int32_t kvp_version(void) { return 100; }

void kvp_set_launch_options(uint32_t flags) { kvp::g_launch_flags.store(flags, std::memory_order_relaxed); }
uint32_t kvp_get_launch_options(void) { return kvp::g_launch_flags.load(std::memory_order_relaxed); }

void kvp_set_wait_limit_ns(uint64_t ns) {
    kvp::g_wait_limit_ns.store(ns == 0 ? kWaitLimitNs : ns, std::memory_order_relaxed);
}
uint64_t kvp_get_wait_limit_ns(void) { return kvp::g_wait_limit_ns.load(std::memory_order_relaxed); }

kvp_status kvp_pool_errors(const kvp_pool* pool, uint32_t* bits, void* stream) {
    if (!pool || !bits) return KVP_ERR_INVALID_ARG;
    *bits = 0;
    if (!pool->err_word) return KVP_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t host = 0;
    if (cudaMemcpyAsync(&host, pool->err_word, sizeof(host), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return KVP_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KVP_ERR_CUDA;
    *bits = host;
    return (host & KVP_DEVERR_TIMEOUT) ? KVP_ERR_TIMEOUT : KVP_OK;
}

const char* kvp_status_string(kvp_status status) {
    switch (status) {
        case KVP_OK: return "ok";
        case KVP_ERR_INVALID_ARG: return "invalid argument";
        case KVP_ERR_UNSUPPORTED: return "unsupported dtype, head_dim or block_size";
        case KVP_ERR_WORKSPACE: return "workspace missing or too small";
        case KVP_ERR_CUDA: return "CUDA error";
        case KVP_ERR_TIMEOUT: return "an in-kernel wait timed out";
        case KVP_ERR_NO_BLOCKS: return "too few free or evictable blocks";
        default: return "unknown status";
    }
}

int32_t kvp_prefix_num_splits(int32_t B, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                              int32_t max_q_len, int32_t max_context_len) {
    (void)head_dim;
    if (B <= 0 || num_kv_heads <= 0 || num_q_heads <= 0 || max_q_len <= 0) return 1;
    const int64_t g = num_q_heads / num_kv_heads;
    const int64_t rows = prefix_rows_per_cta();
    const int64_t q_tiles = (static_cast<int64_t>(max_q_len) * g + rows - 1) / rows;
    const int64_t ctas = q_tiles * num_kv_heads * B;
    const int64_t key_tiles = (static_cast<int64_t>(max_context_len) + 127) / 128;
    // Split only when the CTAs would leave most of the GPU idle and each has a
    // long key range: split partials cost an fp32 round trip and a merge
    // launch.  (Measured on GB300: 128 CTAs over ~10 key tiles ran 2.3x slower
    // split in two than unsplit.)
    if (ctas > kNumSMs / 4 || key_tiles < 16) return 1;
    int64_t splits = kNumSMs / ctas;
    if (splits > key_tiles / 8) splits = key_tiles / 8;
    if (splits > 16) splits = 16;
    return splits < 1 ? 1 : static_cast<int32_t>(splits);
}

int32_t kvp_decode_num_splits(int32_t B, int32_t num_kv_heads, int32_t block_size, int32_t max_context_len) {
    if (B <= 0 || num_kv_heads <= 0 || max_context_len <= 0) return 1;
    (void)block_size;
    // About 1024 keys per CTA: on the mixed batch (64 sequences, 8 kv heads,
    // contexts 512..8192) 8 splits decoded in 111 us against 115 us at 512
    // keys per CTA and 131 us at 256; fewer splits mean fewer partials to merge.
    int64_t splits = (static_cast<int64_t>(max_context_len) + 1023) / 1024;
    const int64_t pairs = static_cast<int64_t>(B) * num_kv_heads;
    const int64_t target = 2 * kNumSMs;
    if (pairs * splits < target) {
        int64_t want = (target + pairs - 1) / pairs;
        const int64_t cap = (static_cast<int64_t>(max_context_len) + 127) / 128;  // >= 128 keys per CTA
        splits = want < cap ? want : cap;
    }
    if (splits > 64) splits = 64;
    return splits < 1 ? 1 : static_cast<int32_t>(splits);
}

size_t kvp_workspace_size(int32_t op, int32_t rows, int32_t num_q_heads, int32_t head_dim, int32_t num_splits) {
    if (num_splits <= 1 || rows <= 0 || num_q_heads <= 0 || head_dim <= 0) return 0;
    const size_t parts = op == 1 ? static_cast<size_t>(decode_parts_per_split()) : 1;
    const size_t r = static_cast<size_t>(rows) * num_q_heads * num_splits * parts;
    return align256(r * head_dim * sizeof(float)) + align256(r * sizeof(float));
}

kvp_status kvp_slot_mapping(const kvp_pool* pool, const int32_t* cu_seqlens_q, const int32_t* context_lens,
                            const int32_t* block_tables, int32_t max_blocks, int32_t B, int32_t total_q,
                            int64_t* slot_mapping, void* stream) {
    kvp_status st = check_pool(pool);
    if (st != KVP_OK) return st;
    if (B < 0 || total_q < 0 || max_blocks < 0) return KVP_ERR_INVALID_ARG;
    if (total_q == 0) return KVP_OK;
    if (B == 0 || max_blocks == 0 || !cu_seqlens_q || !context_lens || !block_tables || !slot_mapping)
        return KVP_ERR_INVALID_ARG;
    return from_cuda(launch_slot_mapping(view_of(pool), cu_seqlens_q, context_lens, block_tables, max_blocks, B,
                                         total_q, slot_mapping, static_cast<cudaStream_t>(stream)));
}

kvp_status kvp_cache_append(const kvp_pool* pool, const void* k_new, const void* v_new,
                            const int64_t* slot_mapping, int32_t T, void* stream) {
    kvp_status st = check_pool(pool);
    if (st != KVP_OK) return st;
    if (T < 0) return KVP_ERR_INVALID_ARG;
    if (T == 0) return KVP_OK;
    if (!k_new || !v_new || !slot_mapping || !aligned16(k_new) || !aligned16(v_new)) return KVP_ERR_INVALID_ARG;
    return from_cuda(launch_cache_append(view_of(pool), pool->k_pool, pool->v_pool, k_new, v_new, slot_mapping, T,
                                         static_cast<cudaStream_t>(stream)));
}

kvp_status kvp_block_copy(const kvp_pool* pool, const int32_t* pairs, int32_t n, void* stream) {
    kvp_status st = check_pool(pool);
    if (st != KVP_OK) return st;
    if (n < 0 || n > 65535) return KVP_ERR_INVALID_ARG;
    if (n == 0) return KVP_OK;
    if (!pairs) return KVP_ERR_INVALID_ARG;
    return from_cuda(
        launch_block_copy(view_of(pool), pool->k_pool, pool->v_pool, pairs, n, static_cast<cudaStream_t>(stream)));
}

kvp_status kvp_block_swap(const kvp_pool* pool, const kvp_host_pool* host, const int32_t* pairs, int32_t n,
                          int32_t direction, void* stream) {
    kvp_status st = check_pool(pool);
    if (st != KVP_OK) return st;
    if (!host || n < 0 || n > 65535) return KVP_ERR_INVALID_ARG;
    if (direction != KVP_SWAP_OUT && direction != KVP_SWAP_IN) return KVP_ERR_INVALID_ARG;
    if (!host->k_pool || !host->v_pool || host->num_blocks < 1) return KVP_ERR_INVALID_ARG;
    if (!aligned16(host->k_pool) || !aligned16(host->v_pool)) return KVP_ERR_INVALID_ARG;
    if (n == 0) return KVP_OK;
    if (!pairs) return KVP_ERR_INVALID_ARG;
    return from_cuda(launch_block_swap(view_of(pool), pool->k_pool, pool->v_pool, host->k_pool, host->v_pool,
                                       host->num_blocks, pairs, n, direction == KVP_SWAP_OUT,
                                       static_cast<cudaStream_t>(stream)));
}

kvp_status kvp_kv_deviation(const kvp_pool* pool, const void* k_fresh, const void* v_fresh, const int64_t* slots,
                            int32_t T, float* deviation, void* stream) {
    kvp_status st = check_pool(pool);
    if (st != KVP_OK) return st;
    if (T < 0) return KVP_ERR_INVALID_ARG;
    if (T == 0) return KVP_OK;
    if (!k_fresh || !v_fresh || !slots || !deviation || !aligned16(k_fresh) || !aligned16(v_fresh))
        return KVP_ERR_INVALID_ARG;
    return from_cuda(launch_kv_deviation(view_of(pool), pool->k_pool, pool->v_pool, k_fresh, v_fresh, slots, T,
                                         deviation, static_cast<cudaStream_t>(stream)));
}

kvp_status kvp_select_recompute(const float* deviation, const int64_t* slots, const int32_t* cu_seqlens, int32_t B,
                                int32_t permille, int64_t* recompute_slots, int32_t* counts, void* stream) {
    if (B < 0 || permille < 0 || permille > 1000) return KVP_ERR_INVALID_ARG;
    if (B == 0) return KVP_OK;
    if (!deviation || !slots || !cu_seqlens || !recompute_slots || !counts) return KVP_ERR_INVALID_ARG;
    return from_cuda(launch_select_recompute(deviation, slots, cu_seqlens, B, permille, recompute_slots, counts,
                                             static_cast<cudaStream_t>(stream)));
}

static kvp_status check_qpool(const kvp_pool* pool, const kvp_qpool* qp);
static QPoolView qview_of(const kvp_qpool* qp);

// Prefix attention, with (qpool != nullptr) or without a quantized prefix.
static kvp_status prefix_common(const kvp_pool* pool, const kvp_qpool* qpool, const int32_t* qpages, const void* q,
                                void* out, float* lse, const int32_t* cu_seqlens_q, const int32_t* context_lens,
                                const int32_t* block_tables, int32_t max_blocks, int32_t B, int32_t total_q,
                                int32_t num_q_heads, int32_t max_q_len, int32_t max_context_len, float softmax_scale,
                                int32_t num_splits, void* workspace, size_t workspace_bytes, void* stream) {
    kvp_status st = check_pool(pool);
    if (st != KVP_OK) return st;
    if (qpool) {
        if ((st = check_qpool(pool, qpool)) != KVP_OK) return st;
        if (pool->block_size != 16) return KVP_ERR_UNSUPPORTED;
    }
    if (B < 0 || total_q < 0 || max_blocks < 0 || num_splits < 0 || max_q_len < 0 || max_context_len < 0)
        return KVP_ERR_INVALID_ARG;
    if (B == 0 || total_q == 0) return KVP_OK;
    if (!q || !out || !cu_seqlens_q || !context_lens || !block_tables || max_blocks == 0) return KVP_ERR_INVALID_ARG;
    if (qpool && !qpages) return KVP_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out)) return KVP_ERR_INVALID_ARG;
    if (num_q_heads < 1 || num_q_heads % pool->num_kv_heads != 0) return KVP_ERR_INVALID_ARG;
    if (max_q_len < 1 || max_context_len < 1) return KVP_ERR_INVALID_ARG;
    if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return KVP_ERR_INVALID_ARG;
    if (pool->num_kv_heads > 65535 || B > 65535) return KVP_ERR_INVALID_ARG;
    const int32_t g = num_q_heads / pool->num_kv_heads;
    const int64_t rows_per_cta = prefix_rows_per_cta();
    const int64_t q_tiles = (static_cast<int64_t>(max_q_len) * g + rows_per_cta - 1) / rows_per_cta;
    int32_t splits = num_splits > 0 ? num_splits
                                    : kvp_prefix_num_splits(B, num_q_heads, pool->num_kv_heads, pool->head_dim,
                                                            max_q_len, max_context_len);
    if (q_tiles * splits >= (int64_t(1) << 31)) return KVP_ERR_INVALID_ARG;
    PrefixParams p;
    p.pool = view_of(pool);
    p.q = q;
    p.out = out;
    p.lse = lse;
    p.cu_seqlens_q = cu_seqlens_q;
    p.context_lens = context_lens;
    p.block_tables = block_tables;
    p.max_blocks = max_blocks;
    p.B = B;
    p.total_q = total_q;
    p.num_q_heads = num_q_heads;
    p.group = g;
    p.group_mul = ((uint64_t(1) << 32) + g - 1) / g;
    p.q_tiles = static_cast<int32_t>(q_tiles);
    p.num_splits = splits;
    p.wait_limit_ns = wait_limit_ns();
    p.stall_test = (launch_flags() & KVP_LAUNCH_STALL_TEST) ? 1 : 0;
    p.qpool = qpool ? qview_of(qpool) : QPoolView{nullptr, nullptr, nullptr, nullptr, 0, 0};
    p.qpages = qpool ? qpages : nullptr;
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.ws_o = nullptr;
    p.ws_lse = nullptr;
    if (splits > 1) {
        const size_t need = kvp_workspace_size(0, total_q, num_q_heads, pool->head_dim, splits);
        if (!workspace || workspace_bytes < need || !aligned16(workspace)) return KVP_ERR_WORKSPACE;
        const size_t r = static_cast<size_t>(total_q) * num_q_heads * splits;
        p.ws_o = static_cast<float*>(workspace);
        p.ws_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + align256(r * pool->head_dim * 4));
    }
    CUtensorMap tk, tv;
    const int pcw = prefix_chunk_elems(pool->head_dim);
    if ((st = make_pool_map(&tk, pool->k_pool, pool, pcw)) != KVP_OK) return st;
    if ((st = make_pool_map(&tv, pool->v_pool, pool, pcw)) != KVP_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = qpool ? launch_prefix_attn_q(p, tk, tv, s) : launch_prefix_attn(p, tk, tv, s);
    if (e != cudaSuccess) return KVP_ERR_CUDA;
    if (splits > 1)
        e = launch_merge(p.ws_o, p.ws_lse, total_q * num_q_heads, num_q_heads, pool->head_dim, splits, pool->dtype,
                         out, lse, total_q, nullptr, pool->block_size, 0, 1, s);
    return from_cuda(e);
}

kvp_status kvp_prefix_attn(const kvp_pool* pool, const void* q, void* out, float* lse, const int32_t* cu_seqlens_q,
                           const int32_t* context_lens, const int32_t* block_tables, int32_t max_blocks, int32_t B,
                           int32_t total_q, int32_t num_q_heads, int32_t max_q_len, int32_t max_context_len,
                           float softmax_scale, int32_t num_splits, void* workspace, size_t workspace_bytes,
                           void* stream) {
    return prefix_common(pool, nullptr, nullptr, q, out, lse, cu_seqlens_q, context_lens, block_tables, max_blocks, B,
                         total_q, num_q_heads, max_q_len, max_context_len, softmax_scale, num_splits, workspace,
                         workspace_bytes, stream);
}

kvp_status kvp_prefix_attn_q(const kvp_pool* pool, const kvp_qpool* qpool, const int32_t* qpages, const void* q,
                             void* out, float* lse, const int32_t* cu_seqlens_q, const int32_t* context_lens,
                             const int32_t* block_tables, int32_t max_blocks, int32_t B, int32_t total_q,
                             int32_t num_q_heads, int32_t max_q_len, int32_t max_context_len, float softmax_scale,
                             int32_t num_splits, void* workspace, size_t workspace_bytes, void* stream) {
    if (!qpool) return KVP_ERR_INVALID_ARG;
    return prefix_common(pool, qpool, qpages, q, out, lse, cu_seqlens_q, context_lens, block_tables, max_blocks, B,
                         total_q, num_q_heads, max_q_len, max_context_len, softmax_scale, num_splits, workspace,
                         workspace_bytes, stream);
}

static kvp_status check_qpool(const kvp_pool* pool, const kvp_qpool* qp) {
    if (!qp || !qp->k_codes || !qp->v_codes || !qp->k_meta || !qp->v_meta || qp->num_blocks < 1)
        return KVP_ERR_INVALID_ARG;
    if (!aligned16(qp->k_codes) || !aligned16(qp->v_codes) || !aligned16(qp->k_meta) || !aligned16(qp->v_meta))
        return KVP_ERR_INVALID_ARG;
    if (qp->bits != 8 && qp->bits != 4) return KVP_ERR_UNSUPPORTED;
    if (qp->block_size != pool->block_size || qp->num_kv_heads != pool->num_kv_heads ||
        qp->head_dim != pool->head_dim)
        return KVP_ERR_INVALID_ARG;
    return KVP_OK;
}

static QPoolView qview_of(const kvp_qpool* qp) {
    QPoolView v;
    v.k_codes = static_cast<uint8_t*>(qp->k_codes);
    v.v_codes = static_cast<uint8_t*>(qp->v_codes);
    v.k_meta = static_cast<__half*>(qp->k_meta);
    v.v_meta = static_cast<__half*>(qp->v_meta);
    v.num_blocks = qp->num_blocks;
    v.bits = qp->bits;
    return v;
}

kvp_status kvp_quantize_blocks(const kvp_pool* pool, const kvp_qpool* qpool, const int32_t* pairs, int32_t n,
                               void* stream) {
    kvp_status st = check_pool(pool);
    if (st != KVP_OK) return st;
    if ((st = check_qpool(pool, qpool)) != KVP_OK) return st;
    if (n < 0 || n > 65535) return KVP_ERR_INVALID_ARG;
    if (n == 0) return KVP_OK;
    if (!pairs) return KVP_ERR_INVALID_ARG;
    return from_cuda(launch_quantize_blocks(view_of(pool), pool->k_pool, pool->v_pool, qview_of(qpool), pairs, n,
                                            static_cast<cudaStream_t>(stream)));
}

// Host-side validation of a decode call and its launch parameters (without
// workspace).  Returns KVP_OK with *empty set when there is nothing to do.
static kvp_status decode_prepare(const kvp_pool* pool, const kvp_qpool* qpool, const int32_t* qpages, const void* q,
                                 void* out, float* lse, const int32_t* context_lens, const int32_t* block_tables,
                                 int32_t max_blocks, int32_t B, int32_t num_q_heads, int32_t max_context_len,
                                 float softmax_scale, int32_t num_splits, DecodeParams* pp, bool* empty) {
    *empty = false;
    kvp_status st = check_pool(pool);
    if (st != KVP_OK) return st;
    if (qpool) {
        if ((st = check_qpool(pool, qpool)) != KVP_OK) return st;
        if (pool->block_size != 16) return KVP_ERR_UNSUPPORTED;
    }
    if (B < 0 || max_blocks < 0 || num_splits < 0 || max_context_len < 0) return KVP_ERR_INVALID_ARG;
    if (B == 0) {
        *empty = true;
        return KVP_OK;
    }
    if (!q || !out || !context_lens || !block_tables || max_blocks == 0) return KVP_ERR_INVALID_ARG;
    if (qpool && !qpages) return KVP_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out)) return KVP_ERR_INVALID_ARG;
    if (num_q_heads < 1 || num_q_heads % pool->num_kv_heads != 0) return KVP_ERR_INVALID_ARG;
    const int32_t g = num_q_heads / pool->num_kv_heads;
    if (g > 16) return KVP_ERR_UNSUPPORTED;
    if (max_context_len < 1) return KVP_ERR_INVALID_ARG;
    if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return KVP_ERR_INVALID_ARG;
    if (pool->num_kv_heads > 65535 || B > 65535) return KVP_ERR_INVALID_ARG;
    const int32_t req = num_splits > 0
                            ? num_splits
                            : kvp_decode_num_splits(B, pool->num_kv_heads, pool->block_size, max_context_len);
    DecodeParams p;
    p.pool = view_of(pool);
    p.q = q;
    p.out = out;
    p.lse = lse;
    p.context_lens = context_lens;
    p.block_tables = block_tables;
    p.max_blocks = max_blocks;
    p.B = B;
    p.num_q_heads = num_q_heads;
    p.group = g;
    decode_geometry(pool->block_size, max_context_len, req, &p.pages_per_split, &p.max_splits);
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.ws_o = nullptr;
    p.ws_lse = nullptr;
    p.qpool = qpool ? qview_of(qpool) : QPoolView{nullptr, nullptr, nullptr, nullptr, 0, 0};
    p.qpages = qpool ? qpages : nullptr;
    p.wait_limit_ns = wait_limit_ns();
    p.stall_test = (launch_flags() & KVP_LAUNCH_STALL_TEST) ? 1 : 0;
    *pp = p;
    return KVP_OK;
}

// Decode attention, with (qpool != nullptr) or without a quantized prefix.
static kvp_status decode_common(const kvp_pool* pool, const kvp_qpool* qpool, const int32_t* qpages, const void* q,
                                void* out, float* lse, const int32_t* context_lens, const int32_t* block_tables,
                                int32_t max_blocks, int32_t B, int32_t num_q_heads, int32_t max_context_len,
                                float softmax_scale, int32_t num_splits, void* workspace, size_t workspace_bytes,
                                void* stream) {
    DecodeParams p;
    bool empty = false;
    kvp_status st = decode_prepare(pool, qpool, qpages, q, out, lse, context_lens, block_tables, max_blocks, B,
                                   num_q_heads, max_context_len, softmax_scale, num_splits, &p, &empty);
    if (st != KVP_OK || empty) return st;
    if (p.max_splits > 1) {
        const size_t need = kvp_workspace_size(1, B, num_q_heads, pool->head_dim, p.max_splits);
        if (!workspace || workspace_bytes < need || !aligned16(workspace)) return KVP_ERR_WORKSPACE;
        // The 16-bit kernel writes a partial per consumer warp and split, the
        // quantized-prefix kernel one per split; the workspace fits either.
        const size_t r = static_cast<size_t>(B) * num_q_heads * p.max_splits * (qpool ? 1 : decode_parts_per_split());
        p.ws_o = static_cast<float*>(workspace);
        p.ws_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + align256(r * pool->head_dim * 4));
    }
    // The quantized-prefix kernel takes its 16-bit pages in halves of 8 rows.
    CUtensorMap tk, tv;
    const int rows = qpool ? kDecodeQHalfRows : 0;
    if ((st = make_pool_map(&tk, pool->k_pool, pool, 0, rows)) != KVP_OK) return st;
    if ((st = make_pool_map(&tv, pool->v_pool, pool, 0, rows)) != KVP_OK) return st;
    CUtensorMap tkc, tvc;
    if (qpool) {
        if ((st = make_code_map(&tkc, qpool->k_codes, qpool)) != KVP_OK) return st;
        if ((st = make_code_map(&tvc, qpool->v_codes, qpool)) != KVP_OK) return st;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = qpool ? launch_decode_attn_q(p, tk, tv, tkc, tvc, s) : launch_decode_attn(p, tk, tv, s);
    if (e != cudaSuccess) return KVP_ERR_CUDA;
    if (p.max_splits > 1)
        e = launch_merge(p.ws_o, p.ws_lse, B * num_q_heads, num_q_heads, pool->head_dim, p.max_splits, pool->dtype,
                         out, lse, B, context_lens, pool->block_size, p.pages_per_split,
                         qpool ? 1 : decode_parts_per_split(), s);
    return from_cuda(e);
}

kvp_status kvp_decode_attn(const kvp_pool* pool, const void* q, void* out, float* lse, const int32_t* context_lens,
                           const int32_t* block_tables, int32_t max_blocks, int32_t B, int32_t num_q_heads,
                           int32_t max_context_len, float softmax_scale, int32_t num_splits, void* workspace,
                           size_t workspace_bytes, void* stream) {
    return decode_common(pool, nullptr, nullptr, q, out, lse, context_lens, block_tables, max_blocks, B, num_q_heads,
                         max_context_len, softmax_scale, num_splits, workspace, workspace_bytes, stream);
}

kvp_status kvp_decode_attn_q(const kvp_pool* pool, const kvp_qpool* qpool, const int32_t* qpages, const void* q,
                             void* out, float* lse, const int32_t* context_lens, const int32_t* block_tables,
                             int32_t max_blocks, int32_t B, int32_t num_q_heads, int32_t max_context_len,
                             float softmax_scale, int32_t num_splits, void* workspace, size_t workspace_bytes,
                             void* stream) {
    if (!qpool) return KVP_ERR_INVALID_ARG;
    return decode_common(pool, qpool, qpages, q, out, lse, context_lens, block_tables, max_blocks, B, num_q_heads,
                         max_context_len, softmax_scale, num_splits, workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace kvp {

kvp_status decode_workspace_need(const kvp_pool* pool, const void* q, void* out, float* lse,
                                 const int32_t* context_lens, const int32_t* block_tables, int32_t max_blocks,
                                 int32_t B, int32_t num_q_heads, int32_t max_context_len, float softmax_scale,
                                 int32_t num_splits, size_t* need) {
    *need = 0;
    DecodeParams p;
    bool empty = false;
    kvp_status st = decode_prepare(pool, nullptr, nullptr, q, out, lse, context_lens, block_tables, max_blocks, B,
                                   num_q_heads, max_context_len, softmax_scale, num_splits, &p, &empty);
    if (st != KVP_OK || empty) return st;
    *need = kvp_workspace_size(1, B, num_q_heads, pool->head_dim, p.max_splits);
    return KVP_OK;
}

}  // namespace kvp
