// kvp_prefix_impl.cuh -- causal attention of a chunk of new tokens over a
// paged KV cache (cached prefix + the chunk's own K/V), on the 5th-generation
// tensor cores (tcgen05, operands and accumulators in tensor memory).  The
// kernel template is shared by the 16-bit prefix attention (kvp_prefix.cu)
// and the prefix attention over a quantized cached prefix (kvp_prefix_q.cu),
// each translation unit instantiating its own variants.
//
// What it computes (kvboost 0.6.0, "How it works" step 5: the live suffix
// attends to the cached prefix in one forward; "Flash Attention (CUDA)":
// tiled online softmax with causal masking that skips future K/V tiles,
// fp16/bf16, head_dim 64/96/128, any length): for every new token t of
// sequence s and query head h,
//     out[t][h] = softmax_j(scale * q[t][h] . K[j]) . V[j],  j <= P_s + i_t,
// K/V read through the block table (kvboost "CPU paged attention").
//
// Design for sm_103a.  One CTA handles two 128-row query tiles (256 rows) of
// one kv head of one sequence [and one share of its key tiles when split].
// Rows are (token, query head of the GQA group) pairs, so every query head
// that shares a kv head consumes each K/V tile once, and the two query tiles
// halve the K/V bytes each MMA flop needs.  320 threads:
//  * warp 8 (producer) gathers 128-key K and V tiles into a ring of shared
//    memory slots with 2-D TMA boxes, one box per (physical block, 64-column
//    chunk) found through the block table, one lane per block; 128B-swizzled
//    to match the UMMA descriptors (head_dim 96 runs 128 wide: see
//    prefix_width);
//  * warp 9 (MMA) runs converged and elects one lane to issue each
//    tcgen05.mma: S_i = Q_i K^T (SS, M=128, N=128) into TMEM, and
//    O_i += P_i V (TS: P_i read from TMEM, M=128, N = the tile width).  The
//    two query tiles alternate on the tensor core --
//    PV_0, S_0, PV_1, S_1 -- so each softmax warpgroup works while the tensor
//    core serves the other;
//  * warps 0-3 and 4-7 (softmax warpgroups, one per query tile; thread i
//    owns row i = TMEM lane i) read S with one 128-column tcgen05.ld, mask
//    the causal diagonal, run the online softmax in fp32 (log2 domain,
//    packed f32x2 arithmetic, ex2.approx), write P as 16-bit pairs back over
//    S in TMEM (tcgen05.st), and rescale O in TMEM only when a row maximum
//    grew by more than 2^8 (exact: the final 1/l uses the same reference);
//  * the commit that signals S_i(j+1) also covers PV_i(j), so when a
//    warpgroup sees S it may touch O_i and overwrite the P columns freely;
//  * key tiles past the last query's position are never loaded; pages of a
//    loaded tile that lie past the context arrive as out-of-bounds TMA boxes
//    (zeros, no memory read), and the rows of the last page past the context
//    are zeroed in shared memory before P.V (0 * NaN = NaN);
//  * the grid is (query-tile pairs x splits, sequences, kv heads), so the CTAs
//    of all sequences of one kv head run together and blocks that several
//    sequences share are re-read from L2.
//
// TMEM columns: S_0/P_0 [0,128), S_1/P_1 [128,256), O_0 [256,256+d),
// O_1 [256+d, 256+2d) -- 512 columns, one CTA per SM.
//
// Over a quantized cached prefix (BITS 8 or 4; kvboost "Optional: KV
// quantization": cached K per channel, V per token, 8 or 4 bits), four more
// warps (10 to 13) turn codes into the fp16 tiles tcgen05 reads:
//  * for a K or V half-tile holding quantized pages, the producer first
//    stages those pages' codes and scales (bulk copies, a few hundred bytes
//    to 2 KB each) in a ring of its own, then TMA-loads the half-tile's
//    16-bit pages (the live suffix) straight into the K/V ring slot;
//  * each dequantizing warp owns a quarter of the slot's rows: quantized pages
//    become code * s + z in fp16 (one fused multiply-add per pair), written
//    in the same 128B-swizzled layout TMA gives; a bf16 pool's 16-bit pages
//    are converted to fp16 in place; then the slot goes to the MMA warp;
//  * the products run in fp16 whatever the pool dtype (Q is converted when
//    it is staged, P is written as fp16), as in the quantized decode.
//  * fourteen warps leave 128 registers a thread (registers are allocated per
//    SM sub-partition, and two of them hold four warps), so this kernel's
//    softmax reads S in two halves of 64 columns, twice each.

#pragma once
#include "kvp_internal.cuh"

namespace kvp {
namespace {

constexpr int kSoftmaxWarps = 8;                    // two warpgroups, one per query tile
constexpr int kProducerWarp = kSoftmaxWarps;        // warp 8
constexpr int kMmaWarp = kSoftmaxWarps + 1;         // warp 9
constexpr int kThreads = (kSoftmaxWarps + 2) * 32;  // 320
constexpr int kDequantWarp0 = kSoftmaxWarps + 2;    // warps 10-17 (quantized prefix only)
// One dequantizing warp per page of a 128-key tile.  Measured on the long
// context: four warps (two pages each) ran int8 at the same speed but int4
// 12% slower.
constexpr int kDequantWarps = 8;
__host__ __device__ constexpr int prefix_threads(int bits) { return kThreads + (bits ? kDequantWarps * 32 : 0); }
constexpr int kBM = 128;                            // rows per query tile (TMEM lanes)
constexpr int kRowsPerCta = 2 * kBM;
constexpr int kBN = 128;  // keys per K/V tile
constexpr uint32_t kTmemCols = 512;
constexpr int kSmemBudget = 227 * 1024 - 2048;

// Width of the shared-memory tiles and of the products: head_dim 96 runs as
// 128 with zero columns, because a 96-column page needs three 32-column TMA
// boxes (64B swizzle) where 128 takes two 64-column ones (128B swizzle; the
// second box's columns past 96 are out of the tensor and arrive as zeros).
// At d = 96 the kernel is bound by its TMA box rate, not by its products.
__host__ __device__ constexpr int prefix_width(int head_dim) { return head_dim == 96 ? 128 : head_dim; }

// Staging of a quantized K or V half-tile (the kBN/16 pages of 16 tokens of
// one K/V tile): codes of each page, then each page's scales and minima.
// DH is the head dimension of the pool (the tile width may be larger).
template <int DH, int BITS>
struct PrefixQCfg {
    static constexpr int PAGES = kBN / 16;
    static constexpr int CODE = 16 * DH * BITS / 8;  // codes of one page of one kv head
    static constexpr int KMETA = 4 * DH;             // fp16 scale row + min row (per channel)
    static constexpr int VMETA = 4 * 16;             // fp16 (scale, min) per token
    static constexpr int OFF_META = PAGES * CODE;
    static constexpr int SLOT = BITS ? PAGES * (CODE + KMETA) : 0;  // sized for K, the larger
    static constexpr int NQS = BITS == 0 ? 0 : (BITS == 8 ? 3 : 4);  // staging slots
    static constexpr int BYTES = NQS * SLOT;
    static_assert(BITS == 0 || (CODE % 16 == 0 && KMETA % 16 == 0), "bulk copies of 16-byte multiples");
};

template <int D, int QBYTES = 0, int NQS = 0>
struct PrefixCfg {
    static constexpr int CW = chunk_elems(D);
    static constexpr int ROWB = CW * 2;
    static constexpr int NCH = D / CW;
    static constexpr uint32_t SWZ = ROWB == 128 ? 2u : 4u;  // descriptor swizzle code: 128B or 64B
    static constexpr int CHUNK_BYTES = kBM * ROWB;          // one chunk column of a 128-row tile
    static constexpr int TILE_BYTES = kBM * D * 2;          // a Q tile, or a K or V tile of 128 keys
    static constexpr int NSLOT_FIT = (kSmemBudget - 2 * TILE_BYTES - QBYTES) / TILE_BYTES;
    static constexpr int NSLOT = NSLOT_FIT < 8 ? NSLOT_FIT : 8;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_RING = 2 * TILE_BYTES;
    static constexpr int OFF_QST = OFF_RING + NSLOT * TILE_BYTES;  // quantized staging ring
    static constexpr int OFF_BAR = OFF_QST + QBYTES;
    // q_full, s_full, p_full, o_done (2 each), slot_full, slot_empty, the
    // stall barrier; quantized: tfull per ring slot, qfull, qempty per stage.
    static constexpr int NBARS = 9 + 2 * NSLOT + (QBYTES ? NSLOT + 2 * NQS : 0);
    static constexpr int SMEM_BYTES = OFF_BAR + NBARS * 8 + 16 + 1024;
    static constexpr uint32_t S_COL0 = 0, S_COL1 = 128;
    static constexpr uint32_t O_COL0 = 256, O_COL1 = 256 + D;
    static_assert(NSLOT >= (QBYTES ? 3 : 4), "K/V ring too shallow");
    static_assert(SMEM_BYTES <= 232448, "shared memory");
    static_assert(256 + 2 * D <= (int)kTmemCols, "tensor memory");
};

// Named barrier `id` over the 128 threads of a warpgroup that also returns,
// to every one of them, whether v held in all of them (bar.red.and).
__device__ __forceinline__ bool warpgroup_all(int id, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(id)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    const uint32_t a = smem_u32(p);
    return p + (((a + 1023u) & ~1023u) - a);
}

// tcgen05.ld of 128 columns followed by its wait, in one statement so that no
// use of the registers can be scheduled before the data has arrived.
__device__ __forceinline__ void tmem_ld128_sync(uint32_t taddr, uint32_t (&r)[128]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x128.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,"
        "%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,"
        "%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,"
        "%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,"
        "%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,"
        "%126,%127}, [%128];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]),
          "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]),
          "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]),
          "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]),
          "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]),
          "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]),
          "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]),
          "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]),
          "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]),
          "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]),
          "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]),
          "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]),
          "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]),
          "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld16_sync(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld32_sync(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// Row rg of a (sequence, kv head) problem is (token rg / g, query head h g +
// rg % g); the quotient by multiply-shift, exact for rg < 2^24 (checked).
__device__ __forceinline__ int64_t out_row(const PrefixParams& p, int cu0, int h, int rg) {
    const int t = static_cast<int>((static_cast<uint64_t>(static_cast<uint32_t>(rg)) * p.group_mul) >> 32);
    return static_cast<int64_t>(cu0 + t) * p.num_q_heads + h * p.group + (rg - t * p.group);
}

__device__ __forceinline__ void tmem_ld64_sync(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,"
        "%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,"
        "%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]),
          "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]),
          "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]),
          "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]),
          "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,"
        "%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// Eight bf16 values -> eight fp16 values (round to nearest).
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 a) {
    const float2 x = unpack2<true>(a.x), y = unpack2<true>(a.y), z = unpack2<true>(a.z), w = unpack2<true>(a.w);
    return make_uint4(pack2<false>(x.x, x.y), pack2<false>(y.x, y.y), pack2<false>(z.x, z.y), pack2<false>(w.x, w.y));
}

// One dequantizing warp's share of a K (kv 0) or V (kv 1) ring slot: the
// rows of pages kPagesPerWarp * dw .. kPagesPerWarp * (dw + 1) - 1 of the
// tile (one page each with eight warps), written as fp16 in the slot's
// chunked, 128B-swizzled layout.  Pages i < nq come from
// the staged codes: K[t][c] = code * s_c + z_c (per channel of the page),
// V[t][c] = code * s_t + z_t (per token), one fp16 fused multiply-add per
// pair; columns past the head dimension are zeros.  The other pages already
// hold 16-bit values from TMA and, for a bf16 pool, are converted in place.
// stage and dst are shared-memory addresses.  Per page, every code and scale
// load is issued before the page's arithmetic and stores.
template <bool kBF16, int D, int BITS>
__device__ __forceinline__ void prefix_fill_rows(uint32_t stage, uint32_t dst, int kv, int dw, int nq, int lane) {
    constexpr int DP = prefix_width(D);
    using QC = PrefixQCfg<D, BITS>;
    using L = PrefixCfg<DP>;         // layout of a slot (chunks of CW columns)
    constexpr int U = DP / 8;        // 16-byte units per row of the slot
    constexpr int UD = D / 8;        // units that hold data
    constexpr int RPP = 32 / U;      // rows per pass of the warp
    constexpr int IT = 16 / RPP;     // passes per page
    constexpr int CROW = D * BITS / 8;
    const int u = lane % U;
    const int r_in = lane / U;
    const bool has = u < UD;
    const int uc = u % (L::CW / 8);
    const uint32_t ubase = dst + (u / (L::CW / 8)) * L::CHUNK_BYTES;
    constexpr int kPagesPerWarp = QC::PAGES / kDequantWarps;
    const int i0 = kPagesPerWarp * dw;
    const int nmine = min(max(nq - i0, 0), kPagesPerWarp);  // quantized pages among this warp's
#pragma unroll 1
    for (int pg = 0; pg < nmine; ++pg) {
        const int i = i0 + pg;
        const uint32_t codes = stage + i * QC::CODE + u * BITS + r_in * CROW;
        const uint32_t meta = stage + QC::OFF_META + i * (kv ? QC::VMETA : QC::KMETA);
        uint2 c[IT];
        uint32_t sz[IT];
#pragma unroll
        for (int it = 0; it < IT; ++it) {
            const uint32_t a = codes + it * RPP * CROW;
            c[it] = has ? (BITS == 8 ? lds64(a) : make_uint2(lds32(a), 0u)) : make_uint2(0u, 0u);
        }
        uint32_t ks[4], kz[4];
        if (kv == 0) {
            const uint4 a = has ? lds128(meta + u * 16) : make_uint4(0, 0, 0, 0);
            const uint4 z = has ? lds128(meta + 2 * D + u * 16) : make_uint4(0, 0, 0, 0);
            ks[0] = a.x; ks[1] = a.y; ks[2] = a.z; ks[3] = a.w;
            kz[0] = z.x; kz[1] = z.y; kz[2] = z.z; kz[3] = z.w;
        } else {
#pragma unroll
            for (int it = 0; it < IT; ++it) sz[it] = lds32(meta + 4 * (it * RPP + r_in));  // (s_t, z_t)
        }
#pragma unroll
        for (int it = 0; it < IT; ++it) {
            uint4 v;
            if (kv == 0) {
                v = dequant_words<BITS>(c[it], ks, kz);
            } else {
                const uint32_t s1 = __byte_perm(sz[it], 0, 0x1010), z1 = __byte_perm(sz[it], 0, 0x3232);
                const uint32_t vs[4] = {s1, s1, s1, s1}, vz[4] = {z1, z1, z1, z1};
                v = dequant_words<BITS>(c[it], vs, vz);
            }
            if (!has) v = make_uint4(0, 0, 0, 0);
            sts128(ubase + swz_offset(16 * i + it * RPP + r_in, uc, L::ROWB), v);
        }
    }
    if constexpr (kBF16) {
        // This warp's 16-bit pages (the live suffix): bf16 -> fp16 in place.
#pragma unroll 1
        for (int pg = nmine; pg < kPagesPerWarp; ++pg) {
            uint4 a[IT];
#pragma unroll
            for (int it = 0; it < IT; ++it) a[it] = lds128(ubase + swz_offset(16 * (i0 + pg) + it * RPP + r_in, uc, L::ROWB));
#pragma unroll
            for (int it = 0; it < IT; ++it)
                sts128(ubase + swz_offset(16 * (i0 + pg) + it * RPP + r_in, uc, L::ROWB), bf16x8_to_f16x8(a[it]));
        }
    }
}

template <bool kBF16, int D, int BITS>
__global__ void __launch_bounds__(prefix_threads(BITS), 1)
    prefix_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                  const PrefixParams p) {
    constexpr int DP = prefix_width(D);  // tile and product width (>= D; the extra columns are zeros)
    using QC = PrefixQCfg<D, BITS>;
    using C = PrefixCfg<DP, QC::BYTES, QC::NQS>;
    // Operand type of the products: the pool's, or fp16 over a quantized prefix.
    constexpr bool kMma = BITS ? false : kBF16;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* q_full = bars + 0;                 // [2] Q tile i in shared memory (128 arrivals)
    uint64_t* s_full = bars + 2;                 // [2] S_i in TMEM (commit)
    uint64_t* p_full = bars + 4;                 // [2] P_i in TMEM (4 warp arrivals)
    uint64_t* o_done = bars + 6;                 // [2] last PV_i complete (commit)
    uint64_t* slot_full = bars + 8;              // [NSLOT] ring slot loaded (TMA bytes)
    uint64_t* slot_empty = bars + 8 + C::NSLOT;  // [NSLOT] ring slot released (commit)
    uint64_t* stall = bars + 8 + 2 * C::NSLOT;   // nothing arrives on it (KVP_LAUNCH_STALL_TEST)
    uint64_t* tfull = stall + 1;                 // [NSLOT] quantized: the slot's 16-bit pages landed
    uint64_t* qfull = tfull + C::NSLOT;          // [NQS] staged codes and scales landed
    uint64_t* qempty = qfull + QC::NQS;          // [NQS] staging slot dequantized (2 warp arrivals)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_trigger();
    const int split = blockIdx.x % p.num_splits;
    const int ct = p.q_tiles - 1 - static_cast<int>(blockIdx.x) / p.num_splits;  // heavy tiles first
    // Head-major order: the CTAs of all sequences of one kv head run together,
    // so K/V blocks that several sequences share are re-read from L2.
    const int s = blockIdx.y, h = blockIdx.z;
    const int g = p.group, BS = p.pool.block_size, Hkv = p.pool.num_kv_heads;
    uint32_t* err = p.pool.err_word;

    // The metadata loads, and the producer's first 32 block-table entries
    // (the key range of split 0 starts at page 0), in one memory round trip.
    const int pre_blk = (warp == kProducerWarp && split == 0)
                            ? __ldg(p.block_tables + static_cast<int64_t>(s) * p.max_blocks + min(lane, p.max_blocks - 1))
                            : 0;
    const int cu0 = __ldg(p.cu_seqlens_q + s);
    const int cu1 = __ldg(p.cu_seqlens_q + s + 1);
    const int L = __ldg(p.context_lens + s);
    const int qp_raw = BITS ? __ldg(p.qpages + s) : 0;
    const int N = cu1 - cu0;
    const int rows_total = N * g;
    const int r0 = ct * kRowsPerCta;
    if (r0 >= rows_total) {
        pdl_wait();  // every CTA waits, so the grid completes after the one before
        return;
    }
    const int P = L - N;
    const int npages = (L + BS - 1) / BS;
    const int qp = min(max(qp_raw, 0), npages);  // pages read from the quantized pool
    if (P < 0 || npages > p.max_blocks || rows_total >= (1 << 24)) {
        if (tid == 0 && split == 0) report(err, KVP_DEVERR_BAD_LEN);
        pdl_wait();
        return;
    }
    const bool has1 = r0 + kBM < rows_total;  // is the second query tile non-empty?
    const int r_last = min(rows_total, r0 + kRowsPerCta) - 1;
    const int qpos_max = P + r_last / g;
    const int n_tiles = qpos_max / kBN + 1;
    const int per = (n_tiles + p.num_splits - 1) / p.num_splits;
    const int j_begin = min(n_tiles, split * per);
    const int n_local = min(n_tiles, j_begin + per) - j_begin;

    if (n_local <= 0) {
        // This split's key range is empty for the whole CTA: empty partials.
        pdl_wait();
        if (tid < kRowsPerCta && r0 + tid < rows_total) {
            const int rg = r0 + tid;
            const int64_t wrow = static_cast<int64_t>(cu0 + rg / g) * p.num_q_heads + h * g + rg % g;
            p.ws_lse[wrow * p.num_splits + split] = -INFINITY;
            for (int c = 0; c < D; ++c) p.ws_o[(wrow * p.num_splits + split) * D + c] = 0.f;
        }
        return;
    }

    // Softmax warps: issue the global loads of their Q tile now, so their
    // latency overlaps the barrier initialisation and the TMEM allocation.
    constexpr int V16 = D / 8;
    const int wg = warp >> 2;
    const int row = tid & (kBM - 1);
    const bool q_mine = warp < kSoftmaxWarps && (wg == 0 || has1);
    uint4 qv[V16];
    if (q_mine) {
        const uint4* q4 = static_cast<const uint4*>(p.q);
#pragma unroll
        for (int k = 0; k < V16; ++k) {
            const int e = row + k * kBM;
            const int rr = e / V16, c16 = e % V16;
            const int rgl = r0 + wg * kBM + rr;
            qv[k] = make_uint4(0, 0, 0, 0);
            if (rgl < rows_total) qv[k] = __ldg(q4 + out_row(p, cu0, h, rgl) * V16 + c16);
        }
    }

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&q_full[i], kBM);
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 4);
            mbar_init(&o_done[i], 1);
        }
        for (int i = 0; i < C::NSLOT; ++i) {
            mbar_init(&slot_full[i], BITS ? kDequantWarps : 1);
            mbar_init(&slot_empty[i], 1);
            if (BITS) mbar_init(&tfull[i], 1);
        }
        for (int i = 0; i < QC::NQS; ++i) {
            mbar_init(&qfull[i], 1);
            mbar_init(&qempty[i], kDequantWarps);
        }
        mbar_init(stall, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < kSoftmaxWarps) {
        // =========================== softmax warpgroups ===========================
        if (q_mine) {
            const int rg = r0 + wg * kBM + row;
            const bool valid = rg < rows_total;
            const int tq = static_cast<int>((static_cast<uint64_t>(static_cast<uint32_t>(rg)) * p.group_mul) >> 32);
            const int token = valid ? tq : 0;
            const int head = h * g + (valid ? rg - tq * g : 0);
            const int qpos = valid ? P + token : L - 1;

            {  // Q tile wg (loaded above) -> swizzled shared memory (K-major A operand)
                uint8_t* qt = smem + C::OFF_Q + wg * C::TILE_BYTES;
#pragma unroll
                for (int k = 0; k < V16; ++k) {
                    const int e = row + k * kBM;
                    const int rr = e / V16, c16 = e % V16;
                    const int ch = c16 / (C::CW / 8), ci = c16 % (C::CW / 8);
                    uint4 v = qv[k];
                    if constexpr (kMma != kBF16) v = bf16x8_to_f16x8(v);
                    *reinterpret_cast<uint4*>(qt + ch * C::CHUNK_BYTES + swz_offset(rr, ci, C::ROWB)) = v;
                }
#pragma unroll
                for (int c16 = V16; c16 < DP / 8; ++c16) {  // padded columns of this thread's row: zeros
                    const int ch = c16 / (C::CW / 8), ci = c16 % (C::CW / 8);
                    *reinterpret_cast<uint4*>(qt + ch * C::CHUNK_BYTES + swz_offset(row, ci, C::ROWB)) =
                        make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                mbar_arrive(&q_full[wg]);
            }

            const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
            const uint32_t scol = wg ? C::S_COL1 : C::S_COL0;
            const uint32_t ocol = wg ? C::O_COL1 : C::O_COL0;
            const float sl2 = p.scale_log2;
            float m = -INFINITY, l = 0.f;
            bool ok = true;
            for (int jj = 0; jj < n_local; ++jj) {
                const int j = j_begin + jj;
                if (!mbar_wait(&s_full[wg], jj & 1, abort_flag, err, p.wait_limit_ns)) { ok = false; break; }
                tc_fence_after();
                if constexpr (BITS == 0) {
                    float x[kBN];
                    {
                        uint32_t r[kBN];
                        tmem_ld128_sync(lane_base + scol, r);
#pragma unroll
                        for (int i = 0; i < kBN; ++i) x[i] = __uint_as_float(r[i]);
                    }
                    const int lim = qpos - j * kBN;  // last visible column of this tile
                    if (lim < kBN - 1) {
#pragma unroll
                        for (int c = 0; c < kBN; ++c)
                            if (c > lim) x[c] = -INFINITY;
                    }
                    // Row maximum: 3-input max in eight independent chains.
                    float mx8[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) mx8[i] = x[i];
#pragma unroll
                    for (int c = 8; c < kBN - 8; c += 16) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) mx8[i] = fmax3(mx8[i], x[c + i], x[c + 8 + i]);
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(mx8[i], x[kBN - 8 + i]);
                    const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                                           fmaxf(mx8[6], mx8[7]));
                    const float m_new = fmaxf(m, mx * sl2);
                    const bool need = m_new > m + 8.0f;
                    float alpha = 1.f;
                    if (need) {
                        alpha = fast_exp2(m - m_new);
                        m = m_new;
                        l *= alpha;
                    }
                    const float mref = (m == -INFINITY) ? 0.f : m;
                    // p = 2^(x * scale * log2 e - m), pairs on the packed fp32 pipe.
                    const float2 sc = make_float2(sl2, sl2), nb = make_float2(-mref, -mref);
                    float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                     make_float2(0.f, 0.f)};
                    uint32_t pk[kBN / 2];
#pragma unroll
                    for (int c = 0; c < kBN; c += 2) {
                        const float2 t = ffma2(make_float2(x[c], x[c + 1]), sc, nb);
                        const float2 e = make_float2(fast_exp2(t.x), fast_exp2(t.y));
                        acc[(c >> 1) & 3] = fadd2(acc[(c >> 1) & 3], e);
                        pk[c >> 1] = pack2<kMma>(e.x, e.y);
                    }
                    const float2 a = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
                    l += a.x + a.y;

                    if (jj > 0 && __any_sync(0xffffffffu, need)) {
                        // O_wg holds PV_0 .. PV_{jj-1} (the commit that signalled S
                        // covered them) at the old reference maximum: rescale it.
#pragma unroll
                        for (int cb = 0; cb < D / 16; ++cb) {
                            uint32_t r[16];
                            tmem_ld16_sync(lane_base + ocol + 16 * cb, r);
#pragma unroll
                            for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                            tmem_st16(lane_base + ocol + 16 * cb, r);
                        }
                    }
                    tmem_st64(lane_base + scol, pk);  // P over the first 64 columns of S
                } else {
                    // Eighteen warps leave 96 registers: S is read in two halves
                    // of 64 columns, twice -- for the row maximum, then for the
                    // exponentials -- and P is stored per half (the half-0 P goes
                    // over S columns already read; half 1's S lies beyond it).
                    // The half loops are not unrolled: with every warp role of
                    // this kernel the unrolled code overflowed the instruction
                    // cache (ncu: 1.5 fetch stalls per issued instruction).
                    const int lim = qpos - j * kBN;  // last visible column of this tile
                    float mx = -INFINITY;
#pragma unroll 1
                    for (int half = 0; half < 2; ++half) {
                        uint32_t r[kBN / 2];
                        tmem_ld64_sync(lane_base + scol + half * (kBN / 2), r);
                        float xh[kBN / 2];
#pragma unroll
                        for (int c = 0; c < kBN / 2; ++c) xh[c] = __uint_as_float(r[c]);
                        if (lim < kBN - 1) {
#pragma unroll
                            for (int c = 0; c < kBN / 2; ++c)
                                if (half * (kBN / 2) + c > lim) xh[c] = -INFINITY;
                        }
                        float mx4[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) mx4[i] = xh[i];
#pragma unroll
                        for (int c = 4; c < kBN / 2 - 4; c += 8) {
#pragma unroll
                            for (int i = 0; i < 4; ++i) mx4[i] = fmax3(mx4[i], xh[c + i], xh[c + 4 + i]);
                        }
#pragma unroll
                        for (int i = 0; i < 4; ++i) mx4[i] = fmaxf(mx4[i], xh[kBN / 2 - 4 + i]);
                        mx = fmaxf(mx, fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])));
                    }
                    const float m_new = fmaxf(m, mx * sl2);
                    const bool need = m_new > m + 8.0f;
                    float alpha = 1.f;
                    if (need) {
                        alpha = fast_exp2(m - m_new);
                        m = m_new;
                        l *= alpha;
                    }
                    const float mref = (m == -INFINITY) ? 0.f : m;
                    if (jj > 0 && __any_sync(0xffffffffu, need)) {
                        // Rescale O (as above) before this tile's P.V adds to it.
#pragma unroll
                        for (int cb = 0; cb < D / 16; ++cb) {
                            uint32_t r[16];
                            tmem_ld16_sync(lane_base + ocol + 16 * cb, r);
#pragma unroll
                            for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                            tmem_st16(lane_base + ocol + 16 * cb, r);
                        }
                    }
                    const float2 sc = make_float2(sl2, sl2), nb = make_float2(-mref, -mref);
                    float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                     make_float2(0.f, 0.f)};
#pragma unroll 1
                    for (int half = 0; half < 2; ++half) {
                        uint32_t r[kBN / 2];
                        tmem_ld64_sync(lane_base + scol + half * (kBN / 2), r);
                        float xh[kBN / 2];
#pragma unroll
                        for (int c = 0; c < kBN / 2; ++c) xh[c] = __uint_as_float(r[c]);
                        if (lim < kBN - 1) {
#pragma unroll
                            for (int c = 0; c < kBN / 2; ++c)
                                if (half * (kBN / 2) + c > lim) xh[c] = -INFINITY;
                        }
                        uint32_t pk[kBN / 4];
#pragma unroll
                        for (int c = 0; c < kBN / 2; c += 2) {
                            const float2 t = ffma2(make_float2(xh[c], xh[c + 1]), sc, nb);
                            const float2 e = make_float2(fast_exp2(t.x), fast_exp2(t.y));
                            acc[(c >> 1) & 3] = fadd2(acc[(c >> 1) & 3], e);
                            pk[c >> 1] = pack2<kMma>(e.x, e.y);
                        }
                        tmem_st32(lane_base + scol + half * (kBN / 4), pk);
                    }
                    const float2 a = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
                    l += a.x + a.y;
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[wg]);
            }

            // ------------------------------ epilogue ------------------------------
            if (ok) ok = mbar_wait(&o_done[wg], 0, abort_flag, err, p.wait_limit_ns);
            // Make the outcome uniform over the warpgroup before its named
            // barrier below (which cannot time out): every warp passes this one,
            // which returns the AND over the warpgroup of "no wait gave up".
            ok = warpgroup_all(wg + 1, ok && !*abort_flag);
            if (ok) {
                tc_fence_after();
                const float inv = l > 0.f ? 1.f / l : 0.f;
                const float lse2 = l > 0.f ? m + __log2f(l) : -INFINITY;
                const int64_t orow = static_cast<int64_t>(cu0 + token) * p.num_q_heads + head;
                if (p.num_splits == 1) {
                    // Stage the bf16/fp16 O tile in this warpgroup's Q region (the
                    // last S_wg that read it has completed), then write whole rows
                    // with coalesced 16-byte stores.  Row rr's 16-byte chunk c
                    // sits at chunk position (c + rr) % (d/8) to spread banks.
                    uint4* stg = reinterpret_cast<uint4*>(smem + C::OFF_Q + wg * C::TILE_BYTES);
#pragma unroll 1
                    for (int cb = 0; cb < D / 32; ++cb) {
                        uint32_t r[32];
                        tmem_ld32_sync(lane_base + ocol + 32 * cb, r);
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            uint4 a;
                            a.x = pack2<kBF16>(__uint_as_float(r[8 * u]) * inv, __uint_as_float(r[8 * u + 1]) * inv);
                            a.y = pack2<kBF16>(__uint_as_float(r[8 * u + 2]) * inv, __uint_as_float(r[8 * u + 3]) * inv);
                            a.z = pack2<kBF16>(__uint_as_float(r[8 * u + 4]) * inv, __uint_as_float(r[8 * u + 5]) * inv);
                            a.w = pack2<kBF16>(__uint_as_float(r[8 * u + 6]) * inv, __uint_as_float(r[8 * u + 7]) * inv);
                            stg[row * V16 + (4 * cb + u + row) % V16] = a;
                        }
                    }
                    if (valid && p.lse)
                        p.lse[static_cast<int64_t>(head) * p.total_q + cu0 + token] = lse2 * 0.69314718055994531f;
                    // Named barrier over this warpgroup's 128 threads (ids 1 and 2).
                    if (wg == 0)
                        asm volatile("bar.sync 1, 128;" ::: "memory");
                    else
                        asm volatile("bar.sync 2, 128;" ::: "memory");
                    // Thread i writes 16-byte chunk (e % (d/8)) of row e / (d/8) for
                    // e = i + 128 k; unrolled by five so that several chunks are
                    // in flight at once.
                    uint4* out4 = static_cast<uint4*>(p.out);
#pragma unroll 5
                    for (int e = row; e < kBM * V16; e += kBM) {
                        const int rr = e / V16, c = e % V16;
                        const int rgl = r0 + wg * kBM + rr;
                        if (rgl < rows_total) out4[out_row(p, cu0, h, rgl) * V16 + c] = stg[rr * V16 + (c + rr) % V16];
                    }
                } else {
                    float* dst = p.ws_o + (orow * p.num_splits + split) * D;
#pragma unroll
                    for (int cb = 0; cb < D / 16; ++cb) {
                        uint32_t r[16];
                        tmem_ld16_sync(lane_base + ocol + 16 * cb, r);
                        if (valid) {
#pragma unroll
                            for (int i = 0; i < 16; i += 4)
                                *reinterpret_cast<float4*>(dst + 16 * cb + i) =
                                    make_float4(__uint_as_float(r[i]) * inv, __uint_as_float(r[i + 1]) * inv,
                                                __uint_as_float(r[i + 2]) * inv, __uint_as_float(r[i + 3]) * inv);
                        }
                    }
                    if (valid) p.ws_lse[orow * p.num_splits + split] = lse2;
                }
            }
        }
    } else if (warp == kProducerWarp) {
        // ============================ TMA producer warp ============================
        if (lane == 0) {
            prefetch_tmap(&tmap_k);
            prefetch_tmap(&tmap_v);
        }
        const int pages_per_tile = kBN / BS;  // 4, 8 or 16: a tile never straddles a 32-page batch
        const int page_first = j_begin * pages_per_tile;
        const int32_t* table = p.block_tables + static_cast<int64_t>(s) * p.max_blocks;
        const int32_t pool_rows = static_cast<int32_t>(p.pool.num_blocks) * Hkv * BS;  // < 2^31 (host check)
        // Lane i holds the block id of page (batch * 32 + i); the next batch is
        // requested 32 pages ahead so its latency hides behind the tiles in flight.
        auto load_batch = [&](int batch) -> int {
            const int pg = min(page_first + batch * 32 + lane, npages - 1);
            return __ldg(table + pg);
        };
        // Split 0's first batch was loaded with the metadata; clamp it the
        // same way (pages past the context repeat the last page).
        int blk_cur = page_first == 0 ? __shfl_sync(0xffffffffu, pre_blk, min(lane, npages - 1)) : load_batch(0);
        int blk_nxt = load_batch(1);
        pdl_wait();  // pool contents from the kernel before (the append) are read from here on
        int loads = 0;   // ring loads issued: K_j is load 2j, V_j is load 2j+1
        int staged = 0;  // quantized half-tiles staged (they come first)
        bool stop = false;
        for (int jj = 0; jj < n_local && !stop; ++jj) {
            const int rel = jj * pages_per_tile;
            if ((rel & 31) == 0 && jj > 0) {
                blk_cur = blk_nxt;
                blk_nxt = load_batch((rel >> 5) + 1);
            }
            int my_blk = blk_cur;
            // Pages before qp name blocks of the quantized pool.
            const int my_pg = min(page_first + (rel & ~31) + lane, npages - 1);
            const int64_t my_lim = (BITS > 0 && my_pg < qp) ? p.qpool.num_blocks : p.pool.num_blocks;
            if (my_blk < 0 || my_blk >= my_lim) {
                report(err, KVP_DEVERR_BAD_BLOCK);
                my_blk = 0;
            }
            // One lane per physical page issues that page's boxes: TMA issue from
            // a single thread is serial, so spread it over the pages of the tile.
            const int blk_q = __shfl_sync(0xffffffffu, my_blk, ((rel & 31) + lane) & 31);
            // A page past the context is fetched as a box below the last row of
            // the pool tensor: TMA fills it with zeros and reads no memory.
            const int32_t y = page_first + rel + lane < npages ? (blk_q * Hkv + h) * BS : pool_rows;
            // Quantized pages of this tile: its first nq pages (BITS > 0: 16-token pages).
            const int nq = BITS ? min(max(qp - (page_first + rel), 0), pages_per_tile) : 0;
            for (int kv = 0; kv < 2; ++kv) {
                const int gl = 2 * jj + kv;
                const int slot = gl % C::NSLOT;
                if constexpr (BITS > 0) {
                    if (nq > 0) {
                        // Stage the quantized pages' codes and scales.  Half-tiles with
                        // quantized pages come first, so the staging index is gl.
                        const int qs = gl % QC::NQS;
                        int okq = 1;
                        if (lane == 0 && gl >= QC::NQS)
                            okq = mbar_wait(&qempty[qs], ((gl / QC::NQS) - 1) & 1, abort_flag, err, p.wait_limit_ns);
                        okq = __shfl_sync(0xffffffffu, okq, 0);
                        if (!okq) {
                            stop = true;
                            break;
                        }
                        const int meta = kv ? QC::VMETA : QC::KMETA;
                        if (lane == 0) mbar_expect_tx(&qfull[qs], nq * (QC::CODE + meta));
                        __syncwarp();
                        if (lane < nq) {
                            const int64_t ph = static_cast<int64_t>(blk_q) * Hkv + h;
                            uint8_t* st = smem + C::OFF_QST + qs * QC::SLOT;
                            bulk_load(st + lane * QC::CODE, (kv ? p.qpool.v_codes : p.qpool.k_codes) + ph * QC::CODE,
                                      QC::CODE, &qfull[qs]);
                            const __half* msrc = kv ? p.qpool.v_meta + ph * 32 : p.qpool.k_meta + ph * 2 * D;
                            bulk_load(st + QC::OFF_META + lane * meta, msrc, meta, &qfull[qs]);
                        }
                        staged = gl + 1;
                    }
                }
                int ok = 1;
                if (lane == 0 && gl >= C::NSLOT)
                    ok = mbar_wait(&slot_empty[slot], ((gl / C::NSLOT) - 1) & 1, abort_flag, err, p.wait_limit_ns);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) {
                    stop = true;
                    break;
                }
                // 16-bit pages land on slot_full directly, or (quantized prefix) on
                // tfull, which hands the slot to the dequantizing warps.
                uint64_t* landed = BITS ? &tfull[slot] : &slot_full[slot];
                const uint32_t tbytes =
                    BITS ? static_cast<uint32_t>((pages_per_tile - nq) * BS * C::ROWB * C::NCH) : C::TILE_BYTES;
                if (lane == 0) {
                    if (tbytes)
                        mbar_expect_tx(landed, tbytes);
                    else
                        mbar_arrive(landed);
                }
                __syncwarp();
                uint8_t* dst = smem + C::OFF_RING + slot * C::TILE_BYTES;
                if (lane >= nq && lane < pages_per_tile) {
#pragma unroll
                    for (int c = 0; c < C::NCH; ++c)
                        tma_load_2d(dst + c * C::CHUNK_BYTES + lane * BS * C::ROWB, kv ? &tmap_v : &tmap_k,
                                    c * C::CW, y, landed);
                }
                loads = gl + 1;
            }
        }
        // Do not leave while copies may still land in shared memory.
        if (lane == 0) {
            volatile int no_abort = 0;
            for (int gl = max(0, loads - C::NSLOT); gl < loads; ++gl)
                mbar_wait(BITS ? &tfull[gl % C::NSLOT] : &slot_full[gl % C::NSLOT], (gl / C::NSLOT) & 1, &no_abort,
                          err);
            if constexpr (BITS > 0) {
                for (int gl = max(0, staged - QC::NQS); gl < staged; ++gl)
                    mbar_wait(&qfull[gl % QC::NQS], (gl / QC::NQS) & 1, &no_abort, err);
            }
        }
    } else if (warp == kMmaWarp) {
        // ============================ MMA issuer warp ============================
        constexpr uint32_t idesc_s = instr_desc_f16(kMma, kBM, kBN, false);
        // The products span the head dimension only: at d = 96 the tiles are
        // 128 wide, but S needs 6 k-steps of 16 (the rest are zero columns)
        // and P.V 96 output columns (N = 96; the 128-byte swizzled V tile is
        // read as one 64-column chunk and half of the next).
        constexpr uint32_t idesc_o = instr_desc_f16(kMma, kBM, D, true);
        const uint32_t ring = smem_u32(smem + C::OFF_RING);
        const uint32_t qb0 = smem_u32(smem + C::OFF_Q), qb1 = qb0 + C::TILE_BYTES;
        uint64_t* last_bar = nullptr;
        uint32_t last_par = 0;
        auto slot_addr = [&](int gl) -> uint32_t { return ring + (gl % C::NSLOT) * C::TILE_BYTES; };
        auto wait_slot = [&](int gl) -> bool {
            return mbar_wait(&slot_full[gl % C::NSLOT], (gl / C::NSLOT) & 1, abort_flag, err, p.wait_limit_ns);
        };
        auto release = [&](int gl) {
            tc_commit(&slot_empty[gl % C::NSLOT]);
            last_bar = &slot_empty[gl % C::NSLOT];
            last_par = (gl / C::NSLOT) & 1;
        };
        // The whole warp runs these (the MMA and commit wrappers elect one lane).
        auto issue_s = [&](int i, uint32_t kbase) {
            const uint32_t qb = i ? qb1 : qb0;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = ((kk * 16) / C::CW) * C::CHUNK_BYTES + ((kk * 16) % C::CW) * 2;
                const uint64_t ad = smem_desc(qb + off, 16, 8 * C::ROWB, C::SWZ);
                const uint64_t bd = smem_desc(kbase + off, 16, 8 * C::ROWB, C::SWZ);
                tc_mma_ss(tmem + (i ? C::S_COL1 : C::S_COL0), ad, bd, idesc_s, kk > 0 ? 1u : 0u);
            }
            tc_commit(&s_full[i]);
        };
        auto issue_pv = [&](int i, uint32_t vbase, bool accumulate) {
            const uint32_t scol = i ? C::S_COL1 : C::S_COL0;
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk) {
                const uint64_t bd = smem_desc(vbase + kk * 16 * C::ROWB, C::CHUNK_BYTES, 8 * C::ROWB, C::SWZ);
                tc_mma_ts(tmem + (i ? C::O_COL1 : C::O_COL0), tmem + scol + kk * 8, bd, idesc_o,
                          (accumulate || kk > 0) ? 1u : 0u);
            }
        };

        // Test of the failure path: before anything is issued to the tensor
        // core, wait on a barrier nothing arrives on until the limit runs out.
        bool ok = p.stall_test ? stall_wait(stall, abort_flag, err, p.wait_limit_ns) : true;
        if (ok) ok = mbar_wait(&q_full[0], 0, abort_flag, err, p.wait_limit_ns);
        if (ok && has1) ok = mbar_wait(&q_full[1], 0, abort_flag, err, p.wait_limit_ns);
        if (ok) ok = wait_slot(0);
        if (ok) {
            tc_fence_after();
            issue_s(0, slot_addr(0));
            if (has1) issue_s(1, slot_addr(0));
            release(0);
            __syncwarp();
        }
        for (int jj = 0; ok && jj < n_local; ++jj) {
            const int gv = 2 * jj + 1, gk = 2 * jj + 2;
            const bool more = jj + 1 < n_local;
            if (!wait_slot(gv)) { ok = false; break; }
            const int nvalid = L - (j_begin + jj) * kBN;
            if (nvalid < kBN && nvalid % BS != 0) {
                // Rows of the last page past the context may hold any bytes
                // (even NaN); P is 0 there, but 0 * NaN is NaN, so clear those V
                // rows.  Whole pages past the context arrived as zeros.
                uint8_t* vt = smem + C::OFF_RING + (gv % C::NSLOT) * C::TILE_BYTES;
                const int first = nvalid;
                const int nbytes = (BS - nvalid % BS) * C::ROWB;  // contiguous in each chunk column
                for (int c = 0; c < C::NCH; ++c)
                    for (int o = 16 * lane; o < nbytes; o += 16 * 32)
                        *reinterpret_cast<uint4*>(vt + c * C::CHUNK_BYTES + first * C::ROWB + o) = make_uint4(0, 0, 0, 0);
                fence_proxy_async_smem();
                __syncwarp();
            }
            // ---- query tile 0: PV_0(jj), then S_0(jj+1)
            if (!mbar_wait(&p_full[0], jj & 1, abort_flag, err, p.wait_limit_ns)) { ok = false; break; }
            tc_fence_after();
            issue_pv(0, slot_addr(gv), jj > 0);
            if (!more) tc_commit(&o_done[0]);
            if (more) {
                if (!wait_slot(gk)) { ok = false; break; }
                tc_fence_after();
                issue_s(0, slot_addr(gk));
            }
            // ---- query tile 1: PV_1(jj), then S_1(jj+1)
            if (has1) {
                if (!mbar_wait(&p_full[1], jj & 1, abort_flag, err, p.wait_limit_ns)) { ok = false; break; }
                tc_fence_after();
                issue_pv(1, slot_addr(gv), jj > 0);
                if (!more) tc_commit(&o_done[1]);
            }
            release(gv);
            if (more) {
                if (has1) issue_s(1, slot_addr(gk));
                release(gk);
            }
            __syncwarp();
        }
        // Let every issued MMA finish before tensor memory is released.
        if (lane == 0 && last_bar) {
            volatile int no_abort = 0;
            mbar_wait(last_bar, last_par, &no_abort, err);
        }
        __syncwarp();
    } else {
        // ====================== dequantizing warps (BITS > 0) ======================
        if constexpr (BITS > 0) {
            const int dw = warp - kDequantWarp0;  // owns page dw's rows of every slot
            for (int gl = 0; gl < 2 * n_local; ++gl) {
                const int slot = gl % C::NSLOT;
                // The slot is ours once the producer has armed it (after the MMA
                // released it) and its 16-bit pages have landed.
                if (!mbar_wait(&tfull[slot], (gl / C::NSLOT) & 1, abort_flag, err, p.wait_limit_ns)) break;
                const int nq = min(max(qp - (j_begin + (gl >> 1)) * QC::PAGES, 0), QC::PAGES);
                uint8_t* dst = smem + C::OFF_RING + slot * C::TILE_BYTES;
                if (nq > 0) {
                    const int qs = gl % QC::NQS;
                    if (!mbar_wait(&qfull[qs], (gl / QC::NQS) & 1, abort_flag, err, p.wait_limit_ns)) break;
                    prefix_fill_rows<kBF16, D, BITS>(smem_u32(smem + C::OFF_QST + qs * QC::SLOT), smem_u32(dst),
                                                     gl & 1, dw, nq, lane);
                } else if constexpr (kBF16) {
                    prefix_fill_rows<kBF16, D, BITS>(0u, smem_u32(dst), gl & 1, dw, 0, lane);
                }
                // Generic-proxy writes, read next by the tensor core (async proxy).
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (nq > 0) mbar_arrive(&qempty[gl % QC::NQS]);
                    mbar_arrive(&slot_full[slot]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <bool kBF16, int D, int BITS>
cudaError_t launch_prefix_t(const PrefixParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                            cudaStream_t stream) {
    using QC = PrefixQCfg<D, BITS>;
    using C = PrefixCfg<prefix_width(D), QC::BYTES, QC::NQS>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(prefix_kernel<kBF16, D, BITS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    dim3 grid(p.q_tiles * p.num_splits, p.B, p.pool.num_kv_heads);
    return launch_k(prefix_kernel<kBF16, D, BITS>, grid, prefix_threads(BITS), C::SMEM_BYTES, stream, tk, tv, p);
}

}  // namespace
}  // namespace kvp
