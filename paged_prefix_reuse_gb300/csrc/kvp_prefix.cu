// kvp_prefix.cu -- prefix attention over the 16-bit pool: instantiations of
// the tcgen05 prefix kernel (kvp_prefix_impl.cuh, where the design is
// described) for fp16/bf16 and head_dim 64/96/128.
#include "kvp_prefix_impl.cuh"

namespace kvp {
int prefix_rows_per_cta() { return kRowsPerCta; }

int prefix_chunk_elems(int head_dim) { return chunk_elems(prefix_width(head_dim)); }

cudaError_t launch_prefix_attn(const PrefixParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                               cudaStream_t stream) {
    const bool bf = p.pool.dtype == KVP_BF16;
    switch (p.pool.head_dim) {
        case 64: return bf ? launch_prefix_t<true, 64, 0>(p, tk, tv, stream) : launch_prefix_t<false, 64, 0>(p, tk, tv, stream);
        case 96: return bf ? launch_prefix_t<true, 96, 0>(p, tk, tv, stream) : launch_prefix_t<false, 96, 0>(p, tk, tv, stream);
        case 128: return bf ? launch_prefix_t<true, 128, 0>(p, tk, tv, stream) : launch_prefix_t<false, 128, 0>(p, tk, tv, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kvp
