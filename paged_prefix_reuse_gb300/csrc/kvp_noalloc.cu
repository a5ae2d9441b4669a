// kvp_noalloc.cu -- decode attention for callers that cannot allocate device
// memory.  The split partials live in one fixed array that is part of the
// library's device image instead of a caller-supplied workspace.
//
// The array is file-scope device memory: every GPU that loads the library
// holds KVP_DECODE_NOALLOC_SCRATCH_BYTES of it until the process exits.  Host
// code cannot use the array's name as a device address (on the host it is a
// stand-in), so the device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, and cached.
#include <atomic>
#include <mutex>

#include "kvp_internal.cuh"

namespace {

constexpr size_t kScratchBytes = KVP_DECODE_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size");

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device (set-up on the
// first call per device).  Returns nullptr and sets *err on failure.
void* scratch_address(cudaError_t* err) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *err = e != cudaSuccess ? e : cudaErrorInvalidDevice;
        return nullptr;
    }
    void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
    if (p) return p;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
    if (!p) {
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess || !p) {
            *err = e != cudaSuccess ? e : cudaErrorInvalidSymbol;
            return nullptr;
        }
        g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
    return p;
}

}  // namespace

extern "C" kvp_status kvp_decode_attn_noalloc(const kvp_pool* pool, const void* q, void* out, float* lse,
                                              const int32_t* context_lens, const int32_t* block_tables,
                                              int32_t max_blocks, int32_t B, int32_t num_q_heads,
                                              int32_t max_context_len, float softmax_scale, int32_t num_splits,
                                              void* stream) {
    // Validate exactly as kvp_decode_attn does (so its error codes come
    // first), then size the request by the split count that call resolves --
    // the geometry rounds pages per split up to whole stages, so it may be
    // smaller than num_splits -- and refuse it if its partials do not fit.
    size_t need = 0;
    kvp_status st = kvp::decode_workspace_need(pool, q, out, lse, context_lens, block_tables, max_blocks, B,
                                               num_q_heads, max_context_len, softmax_scale, num_splits, &need);
    if (st != KVP_OK) return st;
    if (B == 0) return KVP_OK;
    if (need > kScratchBytes) return KVP_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (need > 0) {
        cudaError_t e = cudaSuccess;
        scratch = scratch_address(&e);
        if (!scratch) return KVP_ERR_CUDA;
    }
    return kvp_decode_attn(pool, q, out, lse, context_lens, block_tables, max_blocks, B, num_q_heads,
                           max_context_len, softmax_scale, num_splits, scratch, need > 0 ? kScratchBytes : 0,
                           stream);
}
