/*
 * kvp_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU restatement of paged prefix-reuse
 * attention, in fp64.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load it.  It shares no code, header, table or helper
 * with the CUDA library and includes nothing from it.
 *
 * What it follows (pages: "kvboost 0.6.0" on PyPI, "kvstream 0.1.0" on PyPI):
 *  - kvboost, "CPU paged attention": KV lives in a fixed pool of physical
 *    blocks of block_size tokens; shared prefixes share physical blocks
 *    copy-on-write.  Paging changes where bytes live, not the mathematics.
 *  - kvstream, "Request lifecycle" steps 2-3: the page table grows one slot
 *    per new token; a known prefix's block table is forked copy-on-write and
 *    shared pages are never duplicated.
 *  - kvstream.yaml "memory" comment: one page holds block_size x heads x
 *    head_dim x 2 (K and V) x dtype_bytes.
 *  - kvboost, "How it works" step 5: the live suffix attends to the cached
 *    prefix plus itself in one forward; "Flash Attention (CUDA)": tiled
 *    online softmax is exact attention, causal.
 * The pages give no attention formula; the textbook definition is used:
 *   x_j = scale * <q, k_j>, j = 0..p   (p = absolute position of the query)
 *   o   = sum_j exp(x_j - m) v_j / sum_j exp(x_j - m),  m = max_j x_j
 *   lse = m + ln(sum_j exp(x_j - m))
 * computed in two plain passes over the logical key sequence.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - a chunk of N new tokens over a cached prefix is aligned bottom-right:
 *    query i of sequence s sits at position context_len[s] - N + i and sees
 *    keys 0..that position;
 *  - grouped-query heads: query head h reads kv head h / (Hq / Hkv);
 *  - pool layout [num_blocks][Hkv][block_size][head_dim], K and V separate;
 *  - logical token j of sequence s is at block_tables[s][j / bs], row j % bs;
 *  - a slot of -1 means "no write".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- storage formats, decoded from their definitions -------------------- */

/* IEEE 754 binary16: sign bit 15, 5 exponent bits (bias 15), 10 fraction bits. */
static double f16_value(uint16_t h) {
    int sign = h >> 15, e = (h >> 10) & 0x1f, f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24); /* subnormal: f * 2^(1-15-10) */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/2^10) 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: sign bit 15, 8 exponent bits (bias 127), 7 fraction bits. */
static double bf16_value(uint16_t b) {
    int sign = b >> 15, e = (b >> 7) & 0xff, f = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133); /* subnormal: f * 2^(1-127-7) */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + f), e - 134); /* (1 + f/2^7) 2^(e-127) */
    return sign ? -v : v;
}

static double value_of(int dtype, uint16_t bits) {
    return dtype == 0 ? f16_value(bits) : bf16_value(bits);
}

void oracle_decode_bits(int dtype, const uint16_t *in, double *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = value_of(dtype, in[i]);
}

/* ---- slot indexing (one slot per new token) ------------------------------ */

/* For sequence s with N_s = cu[s+1]-cu[s] new tokens and context L_s, new
 * token i sits at position p = L_s - N_s + i and is stored at slot
 * block_tables[s][p / bs] * bs + p % bs.  A table entry outside
 * [0, num_blocks), or a position past the table, gives slot -1.
 * Returns the number of such invalid tokens. */
int64_t oracle_slot_mapping(int32_t B, const int32_t *cu_seqlens_q, const int32_t *context_lens,
                            const int32_t *block_tables, int32_t max_blocks, int32_t bs,
                            int64_t num_blocks, int64_t *slots) {
    int64_t bad = 0;
    for (int32_t s = 0; s < B; ++s) {
        int32_t n = cu_seqlens_q[s + 1] - cu_seqlens_q[s];
        int32_t L = context_lens[s];
        for (int32_t i = 0; i < n; ++i) {
            int64_t p = (int64_t)L - n + i;
            int64_t logical = p / bs;
            int64_t slot = -1;
            if (p >= 0 && logical < max_blocks) {
                int64_t blk = block_tables[(int64_t)s * max_blocks + logical];
                if (blk >= 0 && blk < num_blocks) slot = blk * bs + p % bs;
            }
            if (slot < 0) ++bad;
            slots[cu_seqlens_q[s] + i] = slot;
        }
    }
    return bad;
}

/* ---- append: pool[slot] = new token's K/V for every kv head -------------- */

int64_t oracle_cache_append(uint16_t *k_pool, uint16_t *v_pool, int64_t num_blocks, int32_t Hkv,
                            int32_t bs, int32_t d, const uint16_t *k_new, const uint16_t *v_new,
                            const int64_t *slots, int32_t T) {
    int64_t skipped_bad = 0;
    for (int32_t t = 0; t < T; ++t) {
        int64_t slot = slots[t];
        if (slot == -1) continue;
        if (slot < 0 || slot >= num_blocks * bs) {
            ++skipped_bad;
            continue;
        }
        int64_t blk = slot / bs, row = slot % bs;
        for (int32_t h = 0; h < Hkv; ++h) {
            int64_t dst = ((blk * Hkv + h) * bs + row) * d;
            int64_t src = ((int64_t)t * Hkv + h) * d;
            for (int32_t c = 0; c < d; ++c) {
                k_pool[dst + c] = k_new[src + c];
                v_pool[dst + c] = v_new[src + c];
            }
        }
    }
    return skipped_bad;
}

/* ---- copy-on-write fork: pool'[dst] = pool[src] --------------------------- */

int64_t oracle_block_copy(uint16_t *k_pool, uint16_t *v_pool, int64_t num_blocks, int64_t block_elems,
                          const int32_t *pairs, int32_t n) {
    int64_t bad = 0;
    for (int32_t i = 0; i < n; ++i) {
        int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            ++bad;
            continue;
        }
        for (int64_t e = 0; e < block_elems; ++e) {
            k_pool[dst * block_elems + e] = k_pool[src * block_elems + e];
            v_pool[dst * block_elems + e] = v_pool[src * block_elems + e];
        }
    }
    return bad;
}

/* ---- attention of new tokens over the gathered logical sequence ---------- */

/* rows[r] = t * Hq + h names query token t (packed over all sequences) and
 * query head h; rows == NULL means every row in order.  Writes out[r][0..d)
 * and lse[r] (natural log).  A row whose keys name an invalid block gets NaN
 * and is counted in the return value. */
int64_t oracle_prefix_attn(int32_t dtype, const uint16_t *k_pool, const uint16_t *v_pool,
                           int64_t num_blocks, int32_t Hkv, int32_t bs, int32_t d, const uint16_t *q,
                           int32_t Hq, const int32_t *cu_seqlens_q, const int32_t *context_lens,
                           const int32_t *block_tables, int32_t max_blocks, int32_t B, double scale,
                           const int64_t *rows, int64_t nrows, double *out, double *lse) {
    int64_t bad = 0;
    int32_t group = Hq / Hkv;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t row = rows ? rows[r] : r;
        int64_t t = row / Hq;
        int32_t h = (int32_t)(row % Hq);
        int32_t s = 0;
        while (s < B && !(cu_seqlens_q[s] <= t && t < cu_seqlens_q[s + 1])) ++s;
        double *o = out + r * d;
        if (s == B) {
            for (int32_t c = 0; c < d; ++c) o[c] = NAN;
            lse[r] = NAN;
            ++bad;
            continue;
        }
        int32_t n = cu_seqlens_q[s + 1] - cu_seqlens_q[s];
        int64_t p = (int64_t)context_lens[s] - n + (t - cu_seqlens_q[s]);
        int32_t kvh = h / group;
        int64_t nkeys = p + 1;
        double *qv = (double *)malloc(sizeof(double) * d);
        double *x = (double *)malloc(sizeof(double) * (nkeys > 0 ? nkeys : 1));
        int64_t *base = (int64_t *)malloc(sizeof(int64_t) * (nkeys > 0 ? nkeys : 1));
        int ok = nkeys > 0;
        for (int32_t c = 0; c < d; ++c) qv[c] = value_of(dtype, q[(t * Hq + h) * (int64_t)d + c]);
        /* gather: logical key j -> element offset of its row in the pool */
        for (int64_t j = 0; j < nkeys && ok; ++j) {
            int64_t lb = j / bs;
            int64_t blk = lb < max_blocks ? block_tables[(int64_t)s * max_blocks + lb] : -1;
            if (blk < 0 || blk >= num_blocks) {
                ok = 0;
                break;
            }
            base[j] = ((blk * Hkv + kvh) * bs + j % bs) * d;
        }
        if (!ok) {
            for (int32_t c = 0; c < d; ++c) o[c] = NAN;
            lse[r] = NAN;
            ++bad;
        } else {
            /* pass 1: logits and their maximum */
            double m = -INFINITY;
            for (int64_t j = 0; j < nkeys; ++j) {
                double dot = 0.0;
                for (int32_t c = 0; c < d; ++c) dot += qv[c] * value_of(dtype, k_pool[base[j] + c]);
                x[j] = scale * dot;
                if (x[j] > m) m = x[j];
            }
            /* pass 2: normaliser and weighted sum of values */
            double denom = 0.0;
            for (int32_t c = 0; c < d; ++c) o[c] = 0.0;
            for (int64_t j = 0; j < nkeys; ++j) {
                double w = exp(x[j] - m);
                denom += w;
                for (int32_t c = 0; c < d; ++c) o[c] += w * value_of(dtype, v_pool[base[j] + c]);
            }
            for (int32_t c = 0; c < d; ++c) o[c] /= denom;
            lse[r] = m + log(denom);
        }
        free(qv);
        free(x);
        free(base);
    }
    return bad;
}

/* ---- merge of partial results over disjoint key ranges ------------------- */

/* Given n partials (o_i, lse_i) of one query row over disjoint key sets,
 *   lse = ln(sum_i exp(lse_i)),  o = sum_i exp(lse_i - lse) o_i.
 * A partial with lse_i = -inf (no keys) contributes nothing. */
void oracle_lse_merge(int32_t n, int32_t d, const double *o_parts, const double *lse_parts, double *o,
                      double *lse) {
    double m = -INFINITY;
    for (int32_t i = 0; i < n; ++i)
        if (lse_parts[i] > m) m = lse_parts[i];
    for (int32_t c = 0; c < d; ++c) o[c] = 0.0;
    if (m == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double total = 0.0;
    for (int32_t i = 0; i < n; ++i) total += exp(lse_parts[i] - m);
    *lse = m + log(total);
    for (int32_t i = 0; i < n; ++i) {
        double w = exp(lse_parts[i] - *lse);
        for (int32_t c = 0; c < d; ++c) o[c] += w * o_parts[(int64_t)i * d + c];
    }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
