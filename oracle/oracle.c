/*
 * oracle.c -- plain, slow, fp64 reference for the paged decode-step hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file; only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark do.  It shares no code, header or constant generator with the CUDA
 * library: every format below is written out here from its definition.
 *
 * What it computes (each function names the passage it follows):
 *
 *   orc_bf16_to_double / orc_double_to_bf16   bfloat16 <-> real, round to
 *        nearest even (the storage type the pages use for K/V, "KV cache
 *        complete guide", FP8 section: FP16/BF16 -> FP8).
 *   orc_e4m3_decode / orc_e4m3_encode         the OCP 8-bit E4M3 ("fn") format:
 *        bias 7, 3 mantissa bits, no infinities, NaN only at S.1111.111,
 *        largest finite 448; encode rounds to nearest even and saturates to
 *        +-448.  The pages ask for an FP8 KV cache with a per-tensor scale
 *        ("KV cache complete guide", section "(1) FP8 quantization") but fix
 *        no format; E4M3 with x/scale is the plainest reading.
 *   orc_append                                 write the new token's K/V at its
 *        slot before attending ("Transformer attention mask and KV cache
 *        inference", section "Prefill and decode phases"; slot =
 *        block_table[pos / 16] * 16 + pos % 16, "KV Cache, Flash Attention and
 *        inference optimization", section "PagedAttention").
 *   orc_paged_attention                        for each sequence gather its
 *        blocks into contiguous K/V, then softmax(q K^T * scale + mask) V with
 *        the mask excluding key positions >= the context length ("KV Cache"
 *        (heepie), core formula; "Transformer attention mask ...", sections
 *        "State of scaled dot-product attention" and "Padding mask and batch
 *        length").  GQA: query head h reads KV head h / G ("KV cache complete
 *        guide", section "(2) GQA").  An empty context yields zeros (the pages
 *        warn that an all-masked row is NaN or uniform; zeros is the defined
 *        reading used here).
 *
 * Cache layout (the pages fix none): per layer k_cache, v_cache are
 * [num_blocks][num_kv_heads][16][head_dim] elements of kv_dtype, i.e. the
 * [batch, heads, seq, head_dim] shape of "KV Cache" (heepie), section
 * "Tensor", taken inside one 16-token block.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_BLOCK 16
#define ORC_BF16 0
#define ORC_FP8_E4M3 1

/* ---------------------------------------------------------------- bfloat16 */

/* bfloat16 is the upper half of an IEEE binary32 word. */
double orc_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round half to even of a non-negative real that is a multiple of 1/2
 * after scaling: r = x / quantum, exact in double for our callers. */
static double rne_int(double r)
{
    double fl = floor(r);
    double frac = r - fl;
    if (frac > 0.5) return fl + 1.0;
    if (frac < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* Nearest bfloat16 to x, ties to even, computed directly from x (no detour
 * through binary32, which could round twice).  bfloat16: 8 exponent bits
 * (bias 127), 7 stored mantissa bits, subnormal quantum 2^-133. */
uint16_t orc_double_to_bf16(double x)
{
    if (isnan(x)) return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80);
    int e;
    frexp(a, &e);                 /* a = f * 2^e, f in [0.5, 1) */
    int ebits = e - 1;            /* a in [2^ebits, 2^(ebits+1)) */
    if (ebits < -126) ebits = -126;  /* subnormal range shares the min quantum */
    double quantum = ldexp(1.0, ebits - 7);
    double r = rne_int(a / quantum) * quantum;
    /* largest finite bf16 = (2 - 2^-7) * 2^127; anything rounding above is inf */
    if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
    float f = (float)r;            /* exact: r is a bf16 value */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (u >> 16));
}

void orc_double_to_bf16_array(const double* x, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_double_to_bf16(x[i]);
}

void orc_bf16_to_double_array(const uint16_t* x, double* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_to_double(x[i]);
}

/* -------------------------------------------------------------- E4M3 (fn) */

double orc_e4m3_decode(uint8_t b)
{
    int s = (b >> 7) & 1;
    int e = (b >> 3) & 0xF;
    int m = b & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);          /* subnormal */
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);          /* normal */
    return s ? -v : v;
}

/* Encode a real (already the quotient x / scale) to E4M3, round to nearest
 * even, saturating finite overflow and infinities to +-448. */
uint8_t orc_e4m3_encode(double x)
{
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs(x);
    double r;
    if (isinf(a)) {
        r = 448.0;
    } else if (a < ldexp(1.0, -6)) {
        /* subnormals: multiples of 2^-9 */
        r = rne_int(a / ldexp(1.0, -9)) * ldexp(1.0, -9);
    } else {
        int e;
        frexp(a, &e);
        int ebits = e - 1;                 /* a in [2^ebits, 2^(ebits+1)) */
        double quantum = ldexp(1.0, ebits - 3);
        r = rne_int(a / quantum) * quantum;
    }
    if (r > 448.0) r = 448.0;
    if (r == 0.0) return sign;
    /* r is now an E4M3 value: find its fields */
    uint8_t code;
    if (r < ldexp(1.0, -6)) {
        code = (uint8_t)(r / ldexp(1.0, -9));          /* e = 0, m = r/2^-9 */
    } else {
        int e;
        double f = frexp(r, &e);                        /* r = f 2^e, f in [.5,1) */
        int ebits = e - 1;
        int mant = (int)((f * 2.0 - 1.0) * 8.0);       /* exact */
        code = (uint8_t)(((ebits + 7) << 3) | mant);
    }
    return (uint8_t)(sign | code);
}

/* The quantised code of one stored element: the quotient x / scale is formed
 * in binary32 (the precision of the kernel that writes the cache; a double
 * quotient rounded once to float is the correctly rounded float quotient),
 * then encoded. */
uint8_t orc_quantize_e4m3(uint16_t x_bf16, float scale)
{
    double x = orc_bf16_to_double(x_bf16);
    float qf = (float)(x / (double)scale);
    return orc_e4m3_encode((double)qf);
}

void orc_quantize_e4m3_array(const uint16_t* x, uint8_t* out, int64_t n, float scale)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_quantize_e4m3(x[i], scale);
}

/* ------------------------------------------------------------------ append */

/* k, v: [num_tokens][num_kv_heads][head_dim] bfloat16 bit patterns.
 * slot_mapping[t] < 0 means "padding token, write nothing".
 * Returns 0, or -1 if a slot lies outside the pool (nothing is written for
 * that token). */
int orc_append(uint8_t* k_cache, uint8_t* v_cache, const uint16_t* k, const uint16_t* v,
               const int64_t* slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
               int64_t num_blocks, int kv_dtype, float k_scale, float v_scale)
{
    int rc = 0;
    int es = (kv_dtype == ORC_FP8_E4M3) ? 1 : 2;
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_blocks * ORC_BLOCK) { rc = -1; continue; }
        int64_t blk = slot / ORC_BLOCK;
        int64_t off = slot % ORC_BLOCK;
        for (int h = 0; h < num_kv_heads; ++h) {
            for (int i = 0; i < head_dim; ++i) {
                int64_t src = ((int64_t)t * num_kv_heads + h) * head_dim + i;
                int64_t dst = ((blk * num_kv_heads + h) * ORC_BLOCK + off) * head_dim + i;
                if (es == 2) {
                    memcpy(k_cache + dst * 2, &k[src], 2);
                    memcpy(v_cache + dst * 2, &v[src], 2);
                } else {
                    k_cache[dst] = orc_quantize_e4m3(k[src], k_scale);
                    v_cache[dst] = orc_quantize_e4m3(v[src], v_scale);
                }
            }
        }
    }
    return rc;
}

/* ------------------------------------------------------- decode attention */

static double cache_elem(const uint8_t* cache, int kv_dtype, int64_t idx, double scale)
{
    if (kv_dtype == ORC_FP8_E4M3) return orc_e4m3_decode(cache[idx]) * scale;
    uint16_t b;
    memcpy(&b, cache + idx * 2, 2);
    return orc_bf16_to_double(b);
}

/* One (sequence, KV head) pair: gather, then plain masked softmax attention
 * for each of the G query heads that share the KV head. */
static int attend_pair(double* out, const double* q, const uint8_t* k_cache,
                       const uint8_t* v_cache, int kv_dtype, double k_scale, double v_scale,
                       const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                       int num_q_heads, int num_kv_heads, int head_dim, int64_t num_blocks,
                       double scale, int s, int hkv)
{
    int G = num_q_heads / num_kv_heads;
    int L = context_lens[s];
    double* outs = out + (int64_t)s * num_q_heads * head_dim;
    if (L <= 0) {
        for (int g = 0; g < G; ++g)
            for (int i = 0; i < head_dim; ++i)
                outs[(int64_t)(hkv * G + g) * head_dim + i] = 0.0;
        return 0;
    }
    if ((L + ORC_BLOCK - 1) / ORC_BLOCK > max_blocks) return -2;

    /* 1. gather the logical sequence into contiguous K, V */
    double* K = (double*)malloc(sizeof(double) * (size_t)L * head_dim);
    double* V = (double*)malloc(sizeof(double) * (size_t)L * head_dim);
    double* z = (double*)malloc(sizeof(double) * (size_t)L);
    if (!K || !V || !z) { free(K); free(V); free(z); return -3; }
    int rc = 0;
    for (int j = 0; j < L; ++j) {
        int32_t blk = block_tables[(int64_t)s * max_blocks + j / ORC_BLOCK];
        if (blk < 0 || blk >= num_blocks) { rc = -4; blk = 0; }
        int64_t base = (((int64_t)blk * num_kv_heads + hkv) * ORC_BLOCK + j % ORC_BLOCK) * head_dim;
        for (int i = 0; i < head_dim; ++i) {
            K[(int64_t)j * head_dim + i] = cache_elem(k_cache, kv_dtype, base + i, k_scale);
            V[(int64_t)j * head_dim + i] = cache_elem(v_cache, kv_dtype, base + i, v_scale);
        }
    }
    /* 2. softmax(q K^T * scale) V for each query head of the group */
    for (int g = 0; g < G; ++g) {
        int h = hkv * G + g;
        const double* qh = q + ((int64_t)s * num_q_heads + h) * head_dim;
        double zmax = -INFINITY;
        for (int j = 0; j < L; ++j) {
            double dot = 0.0;
            for (int i = 0; i < head_dim; ++i) dot += qh[i] * K[(int64_t)j * head_dim + i];
            z[j] = scale * dot;
            if (z[j] > zmax) zmax = z[j];
        }
        double den = 0.0;
        for (int j = 0; j < L; ++j) { z[j] = exp(z[j] - zmax); den += z[j]; }
        double* oh = outs + (int64_t)h * head_dim;
        for (int i = 0; i < head_dim; ++i) {
            double acc = 0.0;
            for (int j = 0; j < L; ++j) acc += z[j] * V[(int64_t)j * head_dim + i];
            oh[i] = acc / den;
        }
    }
    free(K); free(V); free(z);
    return rc;
}

/* q: [num_seqs][num_q_heads][head_dim] reals; out: same shape.
 * pair_select: NULL for every (sequence, KV head) pair, otherwise an array of
 * num_seqs*num_kv_heads flags; unselected pairs are left untouched.
 * nthreads <= 0 uses the OpenMP default.  Returns 0, or a negative code if a
 * context is longer than its block-table row (-2) or names a block outside
 * the pool (-4). */
int orc_paged_attention(double* out, const double* q, const uint8_t* k_cache,
                        const uint8_t* v_cache, int kv_dtype, double k_scale, double v_scale,
                        const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                        int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                        int64_t num_blocks, double scale, const uint8_t* pair_select, int nthreads)
{
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return -1;
    int npairs = num_seqs * num_kv_heads;
    int rc = 0;
#ifdef _OPENMP
    /* a per-call team size; the process-wide default stays as it was */
    const int team = nthreads > 0 ? nthreads : omp_get_max_threads();
#pragma omp parallel for num_threads(team) schedule(dynamic, 1) reduction(min : rc)
#endif
    for (int p = 0; p < npairs; ++p) {
        if (pair_select && !pair_select[p]) continue;
        int r = attend_pair(out, q, k_cache, v_cache, kv_dtype, k_scale, v_scale, block_tables,
                            max_blocks, context_lens, num_q_heads, num_kv_heads, head_dim,
                            num_blocks, scale, p / num_kv_heads, p % num_kv_heads);
        if (r < rc) rc = r;
    }
    return rc;
}

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
