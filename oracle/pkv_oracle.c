/*
 * pkv_oracle.c -- TEST INFRASTRUCTURE ONLY: the CPU oracle for paged decode attention.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference leg may
 * load this library.  It shares no code, header, table or constant with the CUDA library
 * under paged_kv_cache_159_gb300/; it includes only the C standard library.
 *
 * Everything here is plain and slow on purpose: fp64 arithmetic, loops in the order the
 * definitions are written, no blocking, no fusion, no online softmax.
 *
 * Sources (page title, section):
 *   [Attn]   "传统 Attention 的 KV Cache 问题" (pyllm.pages.dev), §1.1: the attention formula
 *            Attention(Q_i,K,V) = sum_j softmax_j(Q_i K_j^T / sqrt(d_k)) V_j.
 *   [Causal] "理解 KV Cache：Attention、P/D 分离与 vLLM 的页式显存管理" (steinslab.io), §1.2:
 *            causal mask (position i sees j <= i), and GQA head sharing.
 *   [Decode] same page, §1.3 and §2.2: a decode step computes only the new token's query and
 *            attends over every cached K/V of its sequence, the new token included.
 *   [Slot]   same page, §3.3-§3.4: logical block = floor(i / bs), offset = i mod bs,
 *            physical = block_table[logical], slot = physical * bs + offset.
 *   [Layout] same page, §3.2: per layer and block, K and V are [num_kv_heads, block_size,
 *            head_dim] (head-first, "HND").
 *   [GQA]    "KV Cache 与推理优化" (note.yj-dis.top), section on the three attention layouts:
 *            query heads share a KV head in contiguous groups (Q1-Q4 -> K1, Q5-Q8 -> K2).
 *   [Quant]  same page, section "KV 量化": K/V may be stored in FP8 (1 byte) while the
 *            arithmetic stays in higher precision.  The FP8 format itself is the OCP "E4M3"
 *            encoding (sign 1, exponent 4 with bias 7, mantissa 3, no infinities, the single
 *            NaN pattern S.1111.111, largest finite value 448).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - the appended token occupies position seq_len-1 and is attended to (causal i <= i);
 *   - K and V live in two tensors key_cache/value_cache, each [num_blocks, Hkv, bs, D];
 *   - FP8 encode is y = fl32(x * fl32(1/scale)) then round-to-nearest-even with saturation
 *     to +-448; decode is value(code) * scale.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_BF16 = 0, ORC_FP8E4M3 = 1 };

/* bf16 is the top 16 bits of an IEEE binary32; widening to double is exact. */
static double orc_bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static float orc_bf16_to_float(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* ---------------------------------------------------------------------------------------
 * FP8 E4M3 (OCP), written from the format definition.
 *   code = s eeee mmm;  e == 0      -> (-1)^s * m * 2^-9          (subnormal)
 *                       e in 1..15  -> (-1)^s * (1 + m/8) * 2^(e-7)
 *                       e == 15, m == 7 -> NaN (no infinities)
 * ------------------------------------------------------------------------------------- */
double oracle_e4m3_decode(uint8_t code)
{
    int s = (code >> 7) & 1;
    int e = (code >> 3) & 15;
    int m = code & 7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);
    else
        mag = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* Round-to-nearest-even onto the E4M3 grid, saturating finite overflow (and infinities)
 * to +-448.  NaN encodes as 0x7F.  The grid spacing in the binade [2^E, 2^(E+1)) is
 * 2^(E-3); below the smallest normal 2^-6 the spacing stays 2^-9. */
uint8_t oracle_e4m3_encode(float x)
{
    double a, quantum, n, r, v;
    int sign, E, e_field, m_field;
    if (isnan(x))
        return 0x7F;
    sign = signbit(x) ? 1 : 0;
    a = fabs((double)x);
    if (a >= 448.0)
        return (uint8_t)((sign << 7) | 0x7E);           /* 0x7E = 1.110b * 2^8 = 448 */
    if (a == 0.0)
        return (uint8_t)(sign << 7);
    (void)frexp(a, &E);                                 /* a = f * 2^E, f in [0.5, 1) */
    E -= 1;                                             /* a in [2^E, 2^(E+1)) */
    if (E < -6)
        E = -6;
    quantum = ldexp(1.0, E - 3);
    n = a / quantum;                                    /* exact: power-of-two divide */
    r = nearbyint(n);                                   /* default mode: ties to even */
    v = r * quantum;
    if (v == 0.0)
        return (uint8_t)(sign << 7);
    (void)frexp(v, &E);
    E -= 1;
    if (E < -6) {                                       /* subnormal: v = m * 2^-9 */
        e_field = 0;
        m_field = (int)(v / ldexp(1.0, -9));
    } else {
        e_field = E + 7;
        m_field = (int)((v / ldexp(1.0, E) - 1.0) * 8.0);
    }
    return (uint8_t)((sign << 7) | (e_field << 3) | m_field);
}

/* fp32 product x * (1/scale) exactly as the format reading fixes it, then encode. */
uint8_t oracle_e4m3_quantize(float x, float scale)
{
    volatile float inv = 1.0f / scale;
    volatile float y = x * inv;
    return oracle_e4m3_encode(y);
}

/* ---------------------------------------------------------------------------------------
 * kv_append [Decode] + [Slot] + [Layout]: for each token t and KV head h with
 * slot = slot_mapping[t] >= 0, write K[t,h,:] and V[t,h,:] into
 * cache[slot / bs][h][slot % bs][:].  bf16 pools copy the 16-bit pattern; FP8 pools store
 * the E4M3 code of x / scale.  Negative slots are padding and are skipped.
 * Returns 0, or 1 if a slot lies beyond the pool (nothing is written for that token).
 * ------------------------------------------------------------------------------------- */
int oracle_kv_append(const uint16_t *k, const uint16_t *v, const int64_t *slot_mapping,
                     int64_t num_tokens, int num_kv_heads, int head_dim, int block_size,
                     int64_t num_blocks, int kv_dtype, float k_scale, float v_scale,
                     void *key_cache, void *value_cache)
{
    int status = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        int64_t blk, off;
        if (slot < 0)
            continue;
        if (slot >= num_blocks * (int64_t)block_size) {
            status = 1;
            continue;
        }
        blk = slot / block_size;
        off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            int64_t src = (t * num_kv_heads + h) * (int64_t)head_dim;
            int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * (int64_t)head_dim;
            for (int d = 0; d < head_dim; ++d) {
                if (kv_dtype == ORC_BF16) {
                    ((uint16_t *)key_cache)[dst + d] = k[src + d];
                    ((uint16_t *)value_cache)[dst + d] = v[src + d];
                } else {
                    ((uint8_t *)key_cache)[dst + d] =
                        oracle_e4m3_quantize(orc_bf16_to_float(k[src + d]), k_scale);
                    ((uint8_t *)value_cache)[dst + d] =
                        oracle_e4m3_quantize(orc_bf16_to_float(v[src + d]), v_scale);
                }
            }
        }
    }
    return status;
}

/* Read one cached element as a double: bf16 exactly, FP8 as value(code) * scale. */
static double orc_cache_elem(const void *cache, int64_t idx, int kv_dtype, float scale)
{
    if (kv_dtype == ORC_BF16)
        return orc_bf16_to_double(((const uint16_t *)cache)[idx]);
    return oracle_e4m3_decode(((const uint8_t *)cache)[idx]) * (double)scale;
}

/* ---------------------------------------------------------------------------------------
 * Paged decode attention [Attn] + [Causal] + [Decode] + [GQA] + [Slot].
 * For every sequence b and query head hq (or for the listed (b, hq) pairs):
 *   h      = hq / (Hq / Hkv)                                   contiguous GQA groups
 *   K_j,V_j = cache[block_table[b][j / bs]][h][j % bs][:],  j = 0 .. seq_len[b]-1
 *   s_j    = scale * sum_d q[b,hq,d] * K_j[d]                  (scale taken as given, fp32)
 *   w_j    = exp(s_j - max_i s_i) / sum_l exp(s_l - max_i s_i)  textbook softmax
 *   out    = sum_j w_j * V_j
 * Positions j >= seq_len[b] are never read: the causal mask of the new (last) query
 * row admits exactly j <= seq_len-1.  out is double [B, Hq, D].
 * Returns 0, or 1 for an invalid argument (seq_len outside [1, MB*bs], bad table id);
 * such (b, hq) rows are filled with NaN.
 * ------------------------------------------------------------------------------------- */
static int orc_decode_pair(const uint16_t *q, const void *key_cache, const void *value_cache,
                           const int32_t *block_tables, const int32_t *seq_lens, int b, int hq,
                           int num_q_heads, int num_kv_heads, int head_dim, int max_blocks,
                           int block_size, int64_t num_blocks, int kv_dtype, float k_scale,
                           float v_scale, float scale, double *out)
{
    int group = num_q_heads / num_kv_heads;
    int h = hq / group;
    int L = seq_lens[b];
    const uint16_t *qrow = q + ((int64_t)b * num_q_heads + hq) * head_dim;
    double *orow = out + ((int64_t)b * num_q_heads + hq) * head_dim;
    double *s, smax, denom;
    if (L < 1 || L > max_blocks * block_size)
        goto bad;
    for (int j = 0; j < L; j += block_size) {
        int32_t phys = block_tables[(int64_t)b * max_blocks + j / block_size];
        if (phys < 0 || phys >= num_blocks)
            goto bad;
    }
    s = (double *)malloc(sizeof(double) * (size_t)L);
    if (!s)
        goto bad;
    for (int j = 0; j < L; ++j) {
        int32_t phys = block_tables[(int64_t)b * max_blocks + j / block_size];
        int off = j % block_size;
        int64_t base = (((int64_t)phys * num_kv_heads + h) * block_size + off) * head_dim;
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d)
            dot += orc_bf16_to_double(qrow[d]) * orc_cache_elem(key_cache, base + d, kv_dtype, k_scale);
        s[j] = (double)scale * dot;
    }
    smax = s[0];
    for (int j = 1; j < L; ++j)
        if (s[j] > smax)
            smax = s[j];
    denom = 0.0;
    for (int j = 0; j < L; ++j)
        denom += exp(s[j] - smax);
    for (int d = 0; d < head_dim; ++d)
        orow[d] = 0.0;
    for (int j = 0; j < L; ++j) {
        int32_t phys = block_tables[(int64_t)b * max_blocks + j / block_size];
        int off = j % block_size;
        int64_t base = (((int64_t)phys * num_kv_heads + h) * block_size + off) * head_dim;
        double w = exp(s[j] - smax) / denom;
        for (int d = 0; d < head_dim; ++d)
            orow[d] += w * orc_cache_elem(value_cache, base + d, kv_dtype, v_scale);
    }
    free(s);
    return 0;
bad:
    for (int d = 0; d < head_dim; ++d)
        orow[d] = NAN;
    return 1;
}

int oracle_paged_decode(const uint16_t *q, const void *key_cache, const void *value_cache,
                        const int32_t *block_tables, const int32_t *seq_lens, int batch,
                        int num_q_heads, int num_kv_heads, int head_dim, int max_blocks,
                        int block_size, int64_t num_blocks, int kv_dtype, float k_scale,
                        float v_scale, float scale, const int32_t *pairs, int num_pairs,
                        int num_threads, double *out)
{
    int status = 0;
    int64_t n;
    if (num_kv_heads < 1 || num_q_heads % num_kv_heads != 0)
        return 1;
    n = pairs ? (int64_t)num_pairs : (int64_t)batch * num_q_heads;
    if (num_threads < 1)
        num_threads = 1;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads) reduction(| : status)
#endif
    for (int64_t i = 0; i < n; ++i) {
        int b = pairs ? pairs[2 * i] : (int)(i / num_q_heads);
        int hq = pairs ? pairs[2 * i + 1] : (int)(i % num_q_heads);
        status |= orc_decode_pair(q, key_cache, value_cache, block_tables, seq_lens, b, hq,
                                  num_q_heads, num_kv_heads, head_dim, max_blocks, block_size,
                                  num_blocks, kv_dtype, k_scale, v_scale, scale, out);
    }
    return status;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
