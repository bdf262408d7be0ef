/*
 * pa_oracle.c -- the oracle: a plain, slow, fp64 CPU statement of the paged-KV
 * decode-step hot path (cache append, FP8 page quantisation, GQA decode).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls this code;
 * only the tests, the smoke check and the benchmark's CPU-baseline leg load
 * it.  It shares no code, header, table or constant with the CUDA path.
 *
 * What each function follows (page title, then section):
 *   - "rvLLM: High-performance LLM inference in Rust", CUDA Kernels table:
 *       "Reshape and Cache" (write the new K/V into the paged cache),
 *       "PagedAttention V2" (attention through a block table, online softmax),
 *       "FP8 KV Cache" (E4M3 quantise / dequantise of the KV cache);
 *     feature list: "FP8 KV cache (E4M3 quantization with per-head scaling)".
 *   - "rvllm - A Small LLM Inference Engine in Rust", How it's put together:
 *       the KV cache is a pool of fixed-size blocks; each step writes the new
 *       K/V at explicit write positions and attends over the read blocks that
 *       the block table lists; grouped-query attention shares each KV head
 *       among a group of query heads.
 *   - "LLM Serving Kernels", Projects table, rows 04 (page tables, GQA/MQA,
 *       online softmax) and 05 (E4M3 storage, page scales, fused dequant).
 *   - E4M3 bit layout: the OCP 8-bit floating point specification (OFP8),
 *       E4M3 format: bias 7, 3 mantissa bits, no infinities, S.1111.111 = NaN,
 *       largest finite 448.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   cache layout [num_blocks][num_kv_heads][block_size][head_dim]; q head hq
 *   reads kv head hq / (Hq/Hkv); a negative slot is padding and is skipped;
 *   context_len 0 gives a zero output; FP8 scale per (physical block, kv head)
 *   = amax/448 in fp32 (1.0 when amax is 0), codes = RNE-saturating E4M3 of
 *   the fp32 quotient x/scale; a page's first appended token (slot %
 *   block_size == 0) sets its scale, later tokens reuse it.
 *
 * Decode is stated as its plain definition: scores in double, a two-pass
 * softmax (max, then exp and sum), and the weighted sum of V, all in double.
 * Online softmax and context partitions reach this same result up to rounding.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- scalars */

/* IEEE 754 binary16 -> double, from the format's definition. */
static double half_bits_to_double(uint16_t h)
{
    int s = h >> 15, e = (h >> 10) & 0x1f, m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);              /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp(1.0 + m / 1024.0, e - 15);
    return s ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double act_to_double(uint16_t h, int is_bf16)
{
    return is_bf16 ? bf16_bits_to_double(h) : half_bits_to_double(h);
}

/* E4M3 code -> value (OFP8 E4M3: bias 7, subnormals when E == 0). */
double oracle_e4m3_value(uint8_t c)
{
    int s = c >> 7, E = (c >> 3) & 15, M = c & 7;
    double v;
    if (E == 15 && M == 7)
        return NAN;
    if (E == 0)
        v = ldexp(M / 8.0, -6);
    else
        v = ldexp(1.0 + M / 8.0, E - 7);
    return s ? -v : v;
}

/*
 * binary32 -> E4M3 code, round to nearest with ties to even, saturating:
 * every magnitude at or above 448 (infinity included) gives +-448 (S.1111.110);
 * NaN gives 0x7F.  The sign of zero is kept.
 *
 * The grid spacing (quantum) of E4M3 is 2^-9 below 2^-6 (subnormals) and
 * 2^(floor(log2|v|) - 3) above, so rounding is: divide by the quantum (exact,
 * a power of two), round to the nearest integer with ties to even, multiply
 * back.  The rounded magnitude is then written as E/M fields.
 */
uint8_t oracle_e4m3_encode(float x)
{
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0)
        return sign | 0x7E;
    double q;
    if (a < ldexp(1.0, -6)) {
        q = ldexp(1.0, -9);
    } else {
        int e;
        frexp(a, &e);                   /* a = f * 2^e, f in [0.5, 1) */
        q = ldexp(1.0, (e - 1) - 3);    /* floor(log2 a) = e - 1 */
    }
    double v = nearbyint(a / q) * q;    /* default rounding: ties to even */
    if (v == 0.0)
        return sign;
    if (v < ldexp(1.0, -6))
        return sign | (uint8_t)(v / ldexp(1.0, -9));      /* E = 0, M = v / 2^-9 */
    int e;
    frexp(v, &e);
    int E = (e - 1) + 7;
    int M = (int)((v / ldexp(1.0, e - 1) - 1.0) * 8.0);
    return sign | (uint8_t)(E << 3) | (uint8_t)M;
}

void oracle_e4m3_encode_array(const float *x, uint8_t *codes, int64_t n)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++)
        codes[i] = oracle_e4m3_encode(x[i]);
}

void oracle_e4m3_value_array(const uint8_t *codes, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = oracle_e4m3_value(codes[i]);
}

/* ------------------------------------------------------------------ append */

/*
 * "Reshape and Cache": for token i with slot s = slot_mapping[i] >= 0, copy
 * its K and V rows for every kv head into cache[s / bs][h][s % bs][:].  A pure
 * byte copy; every other byte of the caches is left as it was.
 */
void oracle_cache_append(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                         const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                         int head_dim, int block_size, int elem_bytes)
{
    size_t row = (size_t)head_dim * elem_bytes;
    for (int i = 0; i < num_tokens; i++) {
        int64_t s = slot_mapping[i];
        if (s < 0)
            continue;
        int64_t blk = s / block_size, off = s % block_size;
        for (int h = 0; h < num_kv_heads; h++) {
            size_t src = ((size_t)i * num_kv_heads + h) * row;
            size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + off) * row;
            memcpy((char *)k_cache + dst, (const char *)k_new + src, row);
            memcpy((char *)v_cache + dst, (const char *)v_new + src, row);
        }
    }
}

/* ------------------------------------------------------------ block copy */

/* rvLLM: High-performance LLM inference in Rust, CUDA Kernels table, "Block
 * Copy" (KV cache block copy for beam search); Architecture, the block
 * manager's copy-on-write.  Pairs (src, dst) are applied in order: the whole
 * physical block src of each pool (block_bytes) is copied to block dst, and
 * with scales given, the block's num_kv_heads scales of each pool too.
 * Pairs naming a block outside [0, num_blocks) are skipped. */
void oracle_copy_blocks(void *k_cache, void *v_cache, float *k_scale, float *v_scale,
                        const int64_t *pairs, int num_pairs, size_t block_bytes,
                        int num_kv_heads, int64_t num_blocks)
{
    for (int i = 0; i < num_pairs; i++) {
        int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks || src == dst)
            continue;
        memcpy((char *)k_cache + (size_t)dst * block_bytes,
               (const char *)k_cache + (size_t)src * block_bytes, block_bytes);
        memcpy((char *)v_cache + (size_t)dst * block_bytes,
               (const char *)v_cache + (size_t)src * block_bytes, block_bytes);
        for (int h = 0; h < num_kv_heads && k_scale && v_scale; h++) {
            k_scale[dst * num_kv_heads + h] = k_scale[src * num_kv_heads + h];
            v_scale[dst * num_kv_heads + h] = v_scale[src * num_kv_heads + h];
        }
    }
}

/* --------------------------------------------------------- FP8 quantise */

static float e4m3_page_scale(float amax)
{
    return amax > 0.0f ? amax / 448.0f : 1.0f;     /* IEEE fp32 division */
}

/*
 * Bulk page quantisation: for every (physical block, kv head) tile of one
 * fp16 pool, amax = max |x| over the tile, scale = amax / 448 (fp32),
 * code = E4M3(x / scale) with the quotient taken in fp32.
 */
void oracle_quantize_fp8(const uint16_t *src, int64_t num_blocks, int num_kv_heads, int block_size,
                         int head_dim, uint8_t *codes, float *scales)
{
    int64_t tiles = num_blocks * num_kv_heads;
    int64_t tile_elems = (int64_t)block_size * head_dim;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < tiles; t++) {
        const uint16_t *x = src + t * tile_elems;
        float amax = 0.0f;
        for (int64_t i = 0; i < tile_elems; i++) {
            float a = fabsf((float)half_bits_to_double(x[i]));
            if (a > amax)
                amax = a;
        }
        float s = e4m3_page_scale(amax);
        scales[t] = s;
        for (int64_t i = 0; i < tile_elems; i++) {
            float xf = (float)half_bits_to_double(x[i]);
            codes[t * tile_elems + i] = oracle_e4m3_encode(xf / s);
        }
    }
}

/*
 * FP8 append: like the plain append, but the token's row (fp16, or bf16 when
 * is_bf16) is encoded, per kv head and separately for K and V.
 *   - A page that receives its first token (slot % block_size == 0) takes the
 *     scale amax(row) / 448 of that row.
 *   - A later token of the page is encoded with the stored scale s when
 *     fl32(amax(row) / s) <= 448, that is when no element saturates.
 *   - Otherwise the page is re-scaled first: s' = amax(row) / 448, each code c
 *     of the page's rows before the new one becomes
 *     E4M3(fl32(fl32(e4m3(c) * s) / s')), and s' is stored.
 * Codes are E4M3_RNE_sat(fl32(x / scale)).  Tokens are taken in order.  (LLM
 * Serving Kernels, Projects table, row 05: E4M3 storage with page scales;
 * rvLLM, CUDA Kernels table, "FP8 KV Cache": quantisation on the cache write.)
 */
static float row_amax(const uint16_t *x, int n, int is_bf16)
{
    float amax = 0.0f;
    for (int d = 0; d < n; d++) {
        float a = fabsf((float)act_to_double(x[d], is_bf16));
        if (a > amax)
            amax = a;
    }
    return amax;
}

void oracle_cache_append_fp8(const uint16_t *k_new, const uint16_t *v_new, uint8_t *k_cache,
                             uint8_t *v_cache, float *k_scale, float *v_scale,
                             const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                             int head_dim, int block_size, int is_bf16)
{
    for (int i = 0; i < num_tokens; i++) {
        int64_t s = slot_mapping[i];
        if (s < 0)
            continue;
        int64_t blk = s / block_size, off = s % block_size;
        for (int h = 0; h < num_kv_heads; h++) {
            int64_t tile = blk * num_kv_heads + h;
            for (int kv = 0; kv < 2; kv++) {
                const uint16_t *x = (kv ? v_new : k_new) + ((size_t)i * num_kv_heads + h) * head_dim;
                uint8_t *page = (kv ? v_cache : k_cache) + tile * block_size * head_dim;
                float *sc = kv ? v_scale : k_scale;
                float amax = row_amax(x, head_dim, is_bf16);
                if (off == 0) {
                    sc[tile] = e4m3_page_scale(amax);
                } else if (amax / sc[tile] > 448.0f) {
                    float s_old = sc[tile], s_new = e4m3_page_scale(amax);
                    for (int64_t j = 0; j < off * head_dim; j++) {
                        float v = (float)oracle_e4m3_value(page[j]) * s_old;
                        page[j] = oracle_e4m3_encode(v / s_new);
                    }
                    sc[tile] = s_new;
                }
                float scale = sc[tile];
                for (int d = 0; d < head_dim; d++)
                    page[off * head_dim + d] =
                        oracle_e4m3_encode((float)act_to_double(x[d], is_bf16) / scale);
            }
        }
    }
}

/* ------------------------------------------------------------------ decode */

/* Where one element of the pool comes from: 16-bit activations or E4M3 codes. */
typedef struct {
    const void *k, *v;                 /* pools [NB][Hkv][bs][D] */
    const float *k_scale, *v_scale;    /* [NB][Hkv] when the pool holds E4M3 codes */
    int is_bf16, is_fp8;
} pool_view;

static double pool_elem(const pool_view *p, int which, size_t tile, size_t idx)
{
    if (p->is_fp8) {
        const uint8_t *c = (const uint8_t *)(which ? p->v : p->k);
        const float *sc = which ? p->v_scale : p->k_scale;
        return oracle_e4m3_value(c[idx]) * (double)sc[tile];
    }
    const uint16_t *h = (const uint16_t *)(which ? p->v : p->k);
    return act_to_double(h[idx], p->is_bf16);
}

/*
 * Query i of sequence b (0 <= i < n_q; n_q = 1 for a plain decode step) sits
 * at position pos = L - n_q + i, where L = context_lens[b] counts every token
 * in the cache, the queries' own included.  It attends positions
 * lo..pos (causal), lo = max(0, pos - window + 1) for a sliding window of
 * `window` tokens, 0 when window is 0:
 *   out[b][i][hq][:] = sum_t softmax_t(scale * q[b][i][hq] . K_t) V_t,
 * token t living in physical block block_tables[b][t / bs] at row t % bs,
 * kv head hq / (Hq / Hkv).  A query with nothing to attend (pos < 0) gets a
 * zero output.  q and out are [B][n_q][Hq][D].  rows (optional, n_rows
 * entries) restricts the work to those sequences; wsum_dev (optional,
 * [B][n_q][Hq]) receives |sum_t w_t / Z - 1| for each output.
 * (rvLLM, CUDA Kernels table, "PagedAttention V2"; feature list, "Sliding
 * window attention"; LLM Serving Kernels, Projects table, row 04.)
 */
static void decode_impl(double *out, const uint16_t *q, int q_is_bf16, const pool_view *pool,
                        const int32_t *block_tables, int max_blocks_per_seq,
                        const int32_t *context_lens, int num_seqs, int num_q_heads,
                        int num_kv_heads, int head_dim, int block_size, float scale, int window,
                        int n_q, const int32_t *rows, int n_rows, double *wsum_dev)
{
    int group = num_q_heads / num_kv_heads;
    int nsel = rows ? n_rows : num_seqs;
    int64_t per_seq = (int64_t)n_q * num_q_heads;
    int64_t work = (int64_t)nsel * per_seq;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t w = 0; w < work; w++) {
        int b = rows ? rows[w / per_seq] : (int)(w / per_seq);
        int i = (int)((w % per_seq) / num_q_heads);
        int hq = (int)(w % num_q_heads);
        int h = hq / group;
        int L = context_lens[b];
        size_t row = ((size_t)b * n_q + i) * num_q_heads + hq;
        double *o = out + row * head_dim;
        for (int d = 0; d < head_dim; d++)
            o[d] = 0.0;
        if (wsum_dev)
            wsum_dev[row] = 0.0;
        int pos = L - n_q + i;
        if (L <= 0 || pos < 0)
            continue;
        int lo = window > 0 && pos - window + 1 > 0 ? pos - window + 1 : 0;
        int n = pos + 1 - lo;

        double qd[256];
        const uint16_t *qr = q + row * head_dim;
        for (int d = 0; d < head_dim; d++)
            qd[d] = act_to_double(qr[d], q_is_bf16);

        double *s = (double *)malloc(sizeof(double) * (size_t)n);
        for (int j = 0; j < n; j++) {
            int t = lo + j;
            size_t blk = (size_t)block_tables[(size_t)b * max_blocks_per_seq + t / block_size];
            size_t tile = blk * num_kv_heads + h;
            size_t base = (tile * block_size + t % block_size) * head_dim;
            double dot = 0.0;
            for (int d = 0; d < head_dim; d++)
                dot += qd[d] * pool_elem(pool, 0, tile, base + d);
            s[j] = (double)scale * dot;
        }
        double m = s[0];
        for (int j = 1; j < n; j++)
            if (s[j] > m)
                m = s[j];
        double Z = 0.0;
        for (int j = 0; j < n; j++) {
            s[j] = exp(s[j] - m);
            Z += s[j];
        }
        double wsum = 0.0;
        for (int j = 0; j < n; j++) {
            int t = lo + j;
            size_t blk = (size_t)block_tables[(size_t)b * max_blocks_per_seq + t / block_size];
            size_t tile = blk * num_kv_heads + h;
            size_t base = (tile * block_size + t % block_size) * head_dim;
            double wt = s[j] / Z;
            wsum += wt;
            for (int d = 0; d < head_dim; d++)
                o[d] += wt * pool_elem(pool, 1, tile, base + d);
        }
        if (wsum_dev)
            wsum_dev[row] = fabs(wsum - 1.0);
        free(s);
    }
}

void oracle_decode(double *out, const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                   int is_bf16, const int32_t *block_tables, int max_blocks_per_seq,
                   const int32_t *context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                   int head_dim, int block_size, float scale, int window, int n_q,
                   const int32_t *rows, int n_rows, double *wsum_dev)
{
    pool_view p = {k_cache, v_cache, 0, 0, is_bf16, 0};
    decode_impl(out, q, is_bf16, &p, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                num_q_heads, num_kv_heads, head_dim, block_size, scale, window, n_q, rows, n_rows,
                wsum_dev);
}

/* FP8 pool: K = e4m3(code) * k_scale[block][kv head] exactly (in double); Q is
 * fp16, or bf16 when q_is_bf16. */
void oracle_decode_fp8(double *out, const uint16_t *q, int q_is_bf16, const uint8_t *k_cache,
                       const uint8_t *v_cache, const float *k_scale, const float *v_scale,
                       const int32_t *block_tables, int max_blocks_per_seq,
                       const int32_t *context_lens, int num_seqs, int num_q_heads,
                       int num_kv_heads, int head_dim, int block_size, float scale, int window,
                       int n_q, const int32_t *rows, int n_rows, double *wsum_dev)
{
    pool_view p = {k_cache, v_cache, k_scale, v_scale, 0, 1};
    decode_impl(out, q, q_is_bf16, &p, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                num_q_heads, num_kv_heads, head_dim, block_size, scale, window, n_q, rows, n_rows,
                wsum_dev);
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads of the parallel loops from now on (n >= 1); a harness setting, used
 * to time the oracle on one core.  Results do not depend on it: every output
 * row is reduced serially by one thread. */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
