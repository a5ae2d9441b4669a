// kvp_prefix_q.cu -- prefix attention over a context whose cached prefix is
// held in the quantized pool (kvboost 0.6.0, "Optional: KV quantization":
// cached K per channel and V per token, 8 or 4 bits): the tcgen05 prefix
// kernel (kvp_prefix_impl.cuh) with its eight dequantizing warps, for
// fp16/bf16 pools and head_dim 64/96/128 at block_size 16.
#include "kvp_prefix_impl.cuh"

namespace kvp {

namespace {
template <int BITS>
cudaError_t launch_prefix_q_bits(const PrefixParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                                 cudaStream_t stream) {
    const bool bf = p.pool.dtype == KVP_BF16;
    switch (p.pool.head_dim) {
        case 64: return bf ? launch_prefix_t<true, 64, BITS>(p, tk, tv, stream) : launch_prefix_t<false, 64, BITS>(p, tk, tv, stream);
        case 96: return bf ? launch_prefix_t<true, 96, BITS>(p, tk, tv, stream) : launch_prefix_t<false, 96, BITS>(p, tk, tv, stream);
        case 128: return bf ? launch_prefix_t<true, 128, BITS>(p, tk, tv, stream) : launch_prefix_t<false, 128, BITS>(p, tk, tv, stream);
        default: return cudaErrorInvalidValue;
    }
}
}  // namespace

cudaError_t launch_prefix_attn_q(const PrefixParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                                 cudaStream_t stream) {
    if (p.pool.block_size != 16) return cudaErrorInvalidValue;
    return p.qpool.bits == 8 ? launch_prefix_q_bits<8>(p, tk, tv, stream) : launch_prefix_q_bits<4>(p, tk, tv, stream);
}

}  // namespace kvp
