/*
 * pagedkv_oracle.c -- plain, slow, fp64 CPU oracle for the paged KV-cache
 * decode path.  TEST INFRASTRUCTURE ONLY: it is called by tests/, by the
 * smoke check and by the CPU-baseline leg of bench.py, never by the product
 * path.  It shares no source, header, table or helper with the CUDA library.
 *
 * What it restates (sources are the vLLM web pages this project follows):
 *
 *  - vLLM concept page (compassingai.com), "15 分钟专家深入" item 2 and
 *    "技术原理": the KV cache of a layer is cut into fixed-size blocks
 *    (block_size 16); each sequence owns a page table of physical block ids;
 *    attention gathers the blocks named by the table, concatenates them
 *    into one contiguous K and V, and runs scaled dot-product attention:
 *    scores = Q K^T / sqrt(head_dim), softmax, times V.
 *  - same page, "15 分钟专家深入" item 2: new blocks are filled on demand
 *    as tokens arrive (the slot-mapped write below).
 *  - vLLM v0.17.1 notes (admirer.cn), "修复方案": blocks freshly handed to
 *    attention are zeroed before first use; nothing else is touched.
 *  - same notes, "重点：35219": stale bit patterns in unused positions must
 *    never reach the result (0 x NaN = NaN), so positions past seq_len are
 *    excluded from the softmax rather than multiplied by zero.
 *
 * Readings taken where the pages are silent (each also stated in the design
 * notes of the repository):
 *  - cache layout [num_blocks, block_size, num_kv_heads, head_dim], row-major;
 *  - slot = physical_block * block_size + offset; slot < 0 means "skip";
 *  - GQA: q head h reads kv head h / (Hq / Hkv);
 *  - fp8 is OCP E4M3 (bias 7, max 448, NaN = S.1111.111, no infinities) with
 *    one fp32 scale per cache tensor: stored = rne_satfinite(x / scale),
 *    value = decode(stored) * scale;
 *  - seq_len == 0 gives an all-zero output row.
 *
 * Every floating-point reduction here runs in double; the method is written
 * in the pages' order (gather -> contiguous -> scores -> softmax -> PV) with
 * no blocking, fusion, online softmax or split.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_DTYPE_BF16 0
#define ORACLE_DTYPE_FP8_E4M3 1

/* ------------------------------------------------------------------ */
/* Number formats                                                      */
/* ------------------------------------------------------------------ */

/* bfloat16 -> double: a bf16 is the upper half of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t bits)
{
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* OCP 8-bit floating point, E4M3 variant: 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits.  Exponent field 0 encodes subnormals
 * (m/8 * 2^-6); fields 1..15 encode (1 + m/8) * 2^(e-7), except that
 * exponent 15 with mantissa 7 is NaN.  There is no infinity. */
double oracle_e4m3_to_double(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* Nearest E4M3 value to x, ties to the code with an even mantissa, results
 * beyond the largest finite value (448) clamped to +-448 ("satfinite"),
 * NaN -> 0x7F.  Written as a search over the ordered non-negative codes
 * 0x00..0x7E, whose values increase strictly with the code. */
uint8_t oracle_e4m3_from_float(float x)
{
    double a;
    uint8_t sign;
    int lo = 0, hi = 0x7E;
    if (isnan(x))
        return 0x7F;
    sign = signbit(x) ? 0x80 : 0x00;
    a = fabs((double)x);
    if (a >= oracle_e4m3_to_double(0x7E))
        return (uint8_t)(sign | 0x7E);
    /* largest code whose value is <= a */
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (oracle_e4m3_to_double((uint8_t)mid) <= a)
            lo = mid;
        else
            hi = mid - 1;
    }
    {
        double vlo = oracle_e4m3_to_double((uint8_t)lo);
        double vhi = oracle_e4m3_to_double((uint8_t)(lo + 1));
        double half = 0.5 * (vlo + vhi); /* exact in double */
        int code;
        if (a == vlo)
            code = lo;
        else if (a < half)
            code = lo;
        else if (a > half)
            code = lo + 1;
        else
            code = (lo % 2 == 0) ? lo : lo + 1;
        return (uint8_t)(sign | code);
    }
}

/* Quantise one bf16 value with a per-tensor scale: the stored code is the
 * E4M3 rounding of the IEEE binary32 quotient x / scale. */
uint8_t oracle_quantize_e4m3(uint16_t x_bf16, float scale)
{
    uint32_t w = ((uint32_t)x_bf16) << 16;
    float xf, q;
    memcpy(&xf, &w, sizeof xf);
    q = xf / scale;
    return oracle_e4m3_from_float(q);
}

static double decode_elem(const uint8_t *cache, size_t idx, int dtype,
                          double scale)
{
    if (dtype == ORACLE_DTYPE_BF16) {
        uint16_t b;
        memcpy(&b, cache + 2 * idx, 2);
        return oracle_bf16_to_double(b);
    }
    return oracle_e4m3_to_double(cache[idx]) * scale;
}

static int elem_bytes(int dtype)
{
    return dtype == ORACLE_DTYPE_BF16 ? 2 : 1;
}

/* ------------------------------------------------------------------ */
/* Slot-mapped KV write                                                */
/* ------------------------------------------------------------------ */

/* For every token i with slot s = slot_mapping[i] >= 0, copy k[i] / v[i]
 * (shape [num_kv_heads, head_dim], bf16) into row s % block_size of block
 * s / block_size of each cache.  For fp8 caches each element is quantised
 * with its tensor's scale.  Slots at or past num_blocks * block_size are
 * range errors: they are skipped and counted.  Returns the error count. */
long oracle_kv_write(uint8_t *key_cache, uint8_t *value_cache, int dtype,
                     int num_blocks, int block_size, int num_kv_heads,
                     int head_dim, float k_scale, float v_scale,
                     const uint16_t *k, const uint16_t *v,
                     const int64_t *slot_mapping, long num_tokens)
{
    long i, errors = 0;
    size_t row = (size_t)num_kv_heads * head_dim; /* elements per token */
    int eb = elem_bytes(dtype);
    for (i = 0; i < num_tokens; ++i) {
        int64_t s = slot_mapping[i];
        int64_t blk, off;
        size_t base, e;
        if (s < 0)
            continue;
        if (s >= (int64_t)num_blocks * block_size) {
            ++errors;
            continue;
        }
        blk = s / block_size;
        off = s % block_size;
        base = ((size_t)blk * block_size + (size_t)off) * row;
        for (e = 0; e < row; ++e) {
            uint16_t kb = k[(size_t)i * row + e];
            uint16_t vb = v[(size_t)i * row + e];
            if (dtype == ORACLE_DTYPE_BF16) {
                memcpy(key_cache + (base + e) * eb, &kb, 2);
                memcpy(value_cache + (base + e) * eb, &vb, 2);
            } else {
                key_cache[base + e] = oracle_quantize_e4m3(kb, k_scale);
                value_cache[base + e] = oracle_quantize_e4m3(vb, v_scale);
            }
        }
    }
    return errors;
}

/* ------------------------------------------------------------------ */
/* Zeroing of freshly allocated blocks                                 */
/* ------------------------------------------------------------------ */

/* Every byte of key_cache[id] and value_cache[id] becomes 0 for each id in
 * block_ids; ids outside [0, num_blocks) are skipped and counted. */
long oracle_zero_blocks(uint8_t *key_cache, uint8_t *value_cache,
                        size_t block_bytes, int num_blocks,
                        const int32_t *block_ids, long n)
{
    long i, errors = 0;
    for (i = 0; i < n; ++i) {
        int32_t id = block_ids[i];
        if (id < 0 || id >= num_blocks) {
            ++errors;
            continue;
        }
        memset(key_cache + (size_t)id * block_bytes, 0, block_bytes);
        memset(value_cache + (size_t)id * block_bytes, 0, block_bytes);
    }
    return errors;
}

/* ------------------------------------------------------------------ */
/* Block copy (copy-on-write) and swap to / from host memory           */
/* ------------------------------------------------------------------ */

/* Copy-on-write of shared blocks (vLLM internals, naphjohn.github.io,
 * §1.1: shared prefixes are copied when written): for i = 0 .. n-1 in
 * order, every byte of block dst[i] of both caches becomes the byte of
 * block src[i].  Pairs with an id outside [0, num_blocks) are skipped and
 * counted. */
long oracle_copy_blocks(uint8_t *key_cache, uint8_t *value_cache,
                        size_t block_bytes, int num_blocks,
                        const int32_t *src, const int32_t *dst, long n)
{
    long i, errors = 0;
    for (i = 0; i < n; ++i) {
        if (src[i] < 0 || src[i] >= num_blocks || dst[i] < 0 ||
            dst[i] >= num_blocks) {
            ++errors;
            continue;
        }
        memmove(key_cache + (size_t)dst[i] * block_bytes,
                key_cache + (size_t)src[i] * block_bytes, block_bytes);
        memmove(value_cache + (size_t)dst[i] * block_bytes,
                value_cache + (size_t)src[i] * block_bytes, block_bytes);
    }
    return errors;
}

/* Swap out for preemption (vLLM concept page, compassingai.com,
 * "15 分钟专家深入" item 1: KV blocks of preempted sequences move to CPU
 * memory): out_k[i] / out_v[i] (block_bytes each, packed) receive block
 * ids[i] of each cache.  Out-of-range ids leave their slot untouched. */
long oracle_swap_out(const uint8_t *key_cache, const uint8_t *value_cache,
                     size_t block_bytes, int num_blocks, const int32_t *ids,
                     long n, uint8_t *out_k, uint8_t *out_v)
{
    long i, errors = 0;
    for (i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= num_blocks) {
            ++errors;
            continue;
        }
        memcpy(out_k + (size_t)i * block_bytes,
               key_cache + (size_t)ids[i] * block_bytes, block_bytes);
        memcpy(out_v + (size_t)i * block_bytes,
               value_cache + (size_t)ids[i] * block_bytes, block_bytes);
    }
    return errors;
}

/* Swap in: block ids[i] of each cache receives in_k[i] / in_v[i]. */
long oracle_swap_in(uint8_t *key_cache, uint8_t *value_cache,
                    size_t block_bytes, int num_blocks, const int32_t *ids,
                    long n, const uint8_t *in_k, const uint8_t *in_v)
{
    long i, errors = 0;
    for (i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= num_blocks) {
            ++errors;
            continue;
        }
        memcpy(key_cache + (size_t)ids[i] * block_bytes,
               in_k + (size_t)i * block_bytes, block_bytes);
        memcpy(value_cache + (size_t)ids[i] * block_bytes,
               in_v + (size_t)i * block_bytes, block_bytes);
    }
    return errors;
}

/* ------------------------------------------------------------------ */
/* Step input preparation from a persistent request state table        */
/* ------------------------------------------------------------------ */

/* Model Runner V2 summary (papercache.org), Figure 2 and "GPU原生的输入准备":
 * every active request keeps a stable row of a state table; each step
 * gathers the rows of the scheduled requests, in batch order, into the
 * step's inputs.  For batch entry b with state row r = idx_mapping[b],
 * n = num_scheduled[b] new tokens and c = num_computed[r] tokens already
 * in the cache:
 *   block_tables[b][:]  = state_block_table[r][:]
 *   seq_lens[b]         = c + n
 *   query_start_loc[b]  = n_0 + ... + n_{b-1}   (entry batch = total)
 *   for t = query_start_loc[b] + i, i < n:
 *     positions[t]      = c + i
 *     input_ids[t]      = state_token_ids[r][c + i]
 *     slot_mapping[t]   = state_block_table[r][(c+i)/16]*16 + (c+i)%16
 * Errors are counted and the offending outputs skipped: a negative count
 * schedules nothing; an entry whose tokens do not fit in total_tokens
 * writes nothing (its start offset still advances); an out-of-range row
 * writes slot -1 for its tokens and nothing else; a position past the
 * table or the token buffer writes its position and slot -1.  Returns the
 * error count. */
long oracle_prepare_inputs(const int32_t *idx_mapping,
                           const int32_t *num_scheduled, int batch,
                           const int32_t *state_block_table, int max_blocks,
                           const int32_t *state_num_computed,
                           const int32_t *state_token_ids, int max_model_len,
                           int num_rows, long total_tokens,
                           int32_t *block_tables, int32_t *seq_lens,
                           int32_t *query_start_loc, int32_t *positions,
                           int32_t *input_ids, int64_t *slot_mapping)
{
    long errors = 0, t0 = 0;
    int b, i, j;
    for (b = 0; b < batch; ++b) {
        int r = idx_mapping[b];
        int n = num_scheduled[b];
        if (n < 0) { /* a negative count schedules nothing */
            ++errors;
            n = 0;
        }
        query_start_loc[b] = (int32_t)t0;
        if (t0 + n > total_tokens) { /* no room left in the outputs */
            ++errors;
            t0 += n;
            continue;
        }
        if (r < 0 || r >= num_rows) {
            ++errors;
            for (i = 0; i < n; ++i)
                slot_mapping[t0 + i] = -1;
            t0 += n;
            continue;
        }
        {
            int c = state_num_computed[r];
            for (j = 0; j < max_blocks; ++j)
                block_tables[(size_t)b * max_blocks + j] =
                    state_block_table[(size_t)r * max_blocks + j];
            seq_lens[b] = c + n;
            for (i = 0; i < n; ++i) {
                long t = t0 + i;
                int pos = c + i;
                positions[t] = pos;
                if (pos >= max_blocks * 16 || pos >= max_model_len) {
                    ++errors;
                    slot_mapping[t] = -1;
                    continue;
                }
                input_ids[t] = state_token_ids[(size_t)r * max_model_len + pos];
                slot_mapping[t] =
                    (int64_t)state_block_table[(size_t)r * max_blocks + pos / 16] *
                        16 + pos % 16;
            }
        }
        t0 += n;
    }
    query_start_loc[batch] = (int32_t)t0;
    return errors;
}

/* ------------------------------------------------------------------ */
/* Decode attention                                                    */
/* ------------------------------------------------------------------ */

typedef struct {
    const uint16_t *q;          /* [B, Hq, d] bf16 */
    const uint8_t *key_cache;   /* [NB, bs, Hkv, d] */
    const uint8_t *value_cache; /* [NB, bs, Hkv, d] */
    int dtype;
    double k_scale, v_scale;
    int num_blocks, block_size, num_kv_heads, head_dim;
    const int32_t *block_tables; /* [B, max_blocks] */
    int max_blocks;
    const int32_t *seq_lens; /* [B] */
    int num_heads;
    double scale;
} attn_args;

/* The pages' PagedAttention pseudocode for one query row qrow of q head h
 * against the first L tokens of sequence b.  Returns 0, or 1 on an
 * out-of-range block id / sequence length (the row is then left as
 * zeros). */
static int attend_row(const attn_args *a, const uint16_t *qrow, int b, int h,
                      int L, double *out_row, double *K, double *V, double *p)
{
    const int d = a->head_dim, bs = a->block_size;
    const int group = a->num_heads / a->num_kv_heads;
    const int kvh = h / group;
    const int nblk = (L + bs - 1) / bs;
    double qd[1024];
    int t, j, i;
    double mx, denom;

    for (i = 0; i < d; ++i)
        out_row[i] = 0.0;
    if (L <= 0)
        return L < 0;
    if (nblk > a->max_blocks)
        return 1;

    /* 1. gather: K_all / V_all = concatenation of the blocks named by the
     *    page table, keeping the first L rows (the rest of the last block is
     *    not part of the sequence). */
    for (j = 0; j < nblk; ++j) {
        int32_t blk = a->block_tables[(size_t)b * a->max_blocks + j];
        if (blk < 0 || blk >= a->num_blocks)
            return 1;
        for (t = j * bs; t < (j + 1) * bs && t < L; ++t) {
            size_t base =
                (((size_t)blk * bs + (size_t)(t - j * bs)) * a->num_kv_heads +
                 (size_t)kvh) * d;
            for (i = 0; i < d; ++i) {
                K[(size_t)t * d + i] = decode_elem(a->key_cache, base + i,
                                                   a->dtype, a->k_scale);
                V[(size_t)t * d + i] = decode_elem(a->value_cache, base + i,
                                                   a->dtype, a->v_scale);
            }
        }
    }

    /* 2. scores = scale * q . K[t] */
    for (i = 0; i < d; ++i)
        qd[i] = oracle_bf16_to_double(qrow[i]);
    for (t = 0; t < L; ++t) {
        double s = 0.0;
        for (i = 0; i < d; ++i)
            s += qd[i] * K[(size_t)t * d + i];
        p[t] = a->scale * s;
    }

    /* 3. softmax over the L positions (max subtracted for range). */
    mx = p[0];
    for (t = 1; t < L; ++t)
        if (p[t] > mx)
            mx = p[t];
    denom = 0.0;
    for (t = 0; t < L; ++t) {
        p[t] = exp(p[t] - mx);
        denom += p[t];
    }

    /* 4. output = softmax . V */
    for (t = 0; t < L; ++t) {
        double w = p[t] / denom;
        for (i = 0; i < d; ++i)
            out_row[i] += w * V[(size_t)t * d + i];
    }
    return 0;
}

/* Decode attention for n_pairs (sequence, q head) pairs, or for every pair
 * when pairs == NULL.  out is [B, Hq, d] doubles; only the selected rows are
 * written.  Returns the number of rows that hit a range error.  n_threads
 * <= 0 uses the OpenMP default. */
long oracle_attention_decode(const uint16_t *q, const uint8_t *key_cache,
                             const uint8_t *value_cache, int dtype,
                             double k_scale, double v_scale, int num_blocks,
                             int block_size, int num_kv_heads, int head_dim,
                             const int32_t *block_tables, int max_blocks,
                             const int32_t *seq_lens, int batch, int num_heads,
                             double scale, double *out, const int32_t *pairs,
                             long n_pairs, int n_threads)
{
    attn_args a;
    long total, errors = 0, idx;
    int max_len = 0, b;

    if (head_dim > 1024 || num_kv_heads <= 0 || num_heads % num_kv_heads)
        return -1;
    a.q = q;
    a.key_cache = key_cache;
    a.value_cache = value_cache;
    a.dtype = dtype;
    a.k_scale = dtype == ORACLE_DTYPE_BF16 ? 1.0 : k_scale;
    a.v_scale = dtype == ORACLE_DTYPE_BF16 ? 1.0 : v_scale;
    a.num_blocks = num_blocks;
    a.block_size = block_size;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.block_tables = block_tables;
    a.max_blocks = max_blocks;
    a.seq_lens = seq_lens;
    a.num_heads = num_heads;
    a.scale = scale;
    for (b = 0; b < batch; ++b)
        if (seq_lens[b] > max_len)
            max_len = seq_lens[b];
    if (max_len > max_blocks * block_size)
        max_len = max_blocks * block_size;
    total = pairs ? n_pairs : (long)batch * num_heads;

#ifdef _OPENMP
    if (n_threads > 0)
        omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
#pragma omp parallel reduction(+ : errors)
    {
        size_t n = (size_t)(max_len > 0 ? max_len : 1);
        double *K = (double *)malloc(n * head_dim * sizeof(double));
        double *V = (double *)malloc(n * head_dim * sizeof(double));
        double *p = (double *)malloc(n * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (idx = 0; idx < total; ++idx) {
            int bb, hh;
            if (pairs) {
                bb = pairs[2 * idx];
                hh = pairs[2 * idx + 1];
            } else {
                bb = (int)(idx / num_heads);
                hh = (int)(idx % num_heads);
            }
            if (!K || !V || !p) {
                ++errors;
                continue;
            }
            errors += attend_row(&a, q + ((size_t)bb * num_heads + hh) * head_dim,
                                 bb, hh, seq_lens[bb],
                                 out + ((size_t)bb * num_heads + hh) * head_dim,
                                 K, V, p);
        }
        free(K);
        free(V);
        free(p);
    }
    return errors;
}

/* Prefill / chunked-prefill attention.  vLLM concept page
 * (compassingai.com), "Continuous Batching" with chunked prefill: a long
 * prompt is cut into chunks that share steps with decoding sequences, and
 * every token is inferred incrementally from the tokens before it.  The
 * reading taken here: sequence b brings n_b = query_start_loc[b+1] -
 * query_start_loc[b] query tokens (rows query_start_loc[b] .. +n_b-1 of q,
 * [T, Hq, d]), whose K/V are already in the cache as its last n_b tokens
 * (seq_lens[b] = c_b + n_b, c_b tokens computed in earlier steps).  Query
 * token i sits at position c_b + i and attends to the key positions
 * 0 .. c_b + i, through the pseudocode's gather / scores / softmax / PV; a
 * decode step is the case n_b = 1.
 * out is [T, Hq, d] doubles.  With rows != NULL only those n_rows (token,
 * head) rows are computed.  A sequence with n_b < 0 or c_b < 0 is a range
 * error and its rows stay 0; returns the error count (a bad sequence
 * counts once per computed row). */
long oracle_attention_prefill(const uint16_t *q, const uint8_t *key_cache,
                              const uint8_t *value_cache, int dtype,
                              double k_scale, double v_scale, int num_blocks,
                              int block_size, int num_kv_heads, int head_dim,
                              const int32_t *block_tables, int max_blocks,
                              const int32_t *seq_lens,
                              const int32_t *query_start_loc, int batch,
                              int num_heads, double scale, double *out,
                              const int32_t *rows, long n_rows, int n_threads)
{
    attn_args a;
    long total, errors = 0, idx, T;
    int max_len = 0, b;
    int32_t *seq_of; /* sequence of each query token, -1 when none */

    if (head_dim > 1024 || num_kv_heads <= 0 || num_heads % num_kv_heads ||
        batch < 0)
        return -1;
    T = batch > 0 ? query_start_loc[batch] : 0;
    if (T < 0)
        return -1;
    a.q = q;
    a.key_cache = key_cache;
    a.value_cache = value_cache;
    a.dtype = dtype;
    a.k_scale = dtype == ORACLE_DTYPE_BF16 ? 1.0 : k_scale;
    a.v_scale = dtype == ORACLE_DTYPE_BF16 ? 1.0 : v_scale;
    a.num_blocks = num_blocks;
    a.block_size = block_size;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.block_tables = block_tables;
    a.max_blocks = max_blocks;
    a.seq_lens = seq_lens;
    a.num_heads = num_heads;
    a.scale = scale;
    seq_of = (int32_t *)malloc((size_t)(T > 0 ? T : 1) * sizeof(int32_t));
    if (!seq_of)
        return -1;
    for (idx = 0; idx < T; ++idx)
        seq_of[idx] = -1;
    for (b = 0; b < batch; ++b) {
        long t;
        if (seq_lens[b] > max_len)
            max_len = seq_lens[b];
        for (t = query_start_loc[b]; t < query_start_loc[b + 1]; ++t)
            if (t >= 0 && t < T)
                seq_of[t] = b;
    }
    if (max_len > max_blocks * block_size)
        max_len = max_blocks * block_size;
    total = rows ? n_rows : T * num_heads;

#ifdef _OPENMP
    if (n_threads > 0)
        omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
#pragma omp parallel reduction(+ : errors)
    {
        size_t n = (size_t)(max_len > 0 ? max_len : 1);
        double *K = (double *)malloc(n * head_dim * sizeof(double));
        double *V = (double *)malloc(n * head_dim * sizeof(double));
        double *p = (double *)malloc(n * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (idx = 0; idx < total; ++idx) {
            long t;
            int hh, bb, nq, c, i, k;
            double *orow;
            if (rows) {
                t = rows[2 * idx];
                hh = rows[2 * idx + 1];
            } else {
                t = idx / num_heads;
                hh = (int)(idx % num_heads);
            }
            if (t < 0 || t >= T || hh < 0 || hh >= num_heads || !K || !V || !p) {
                ++errors;
                continue;
            }
            orow = out + ((size_t)t * num_heads + hh) * head_dim;
            for (k = 0; k < head_dim; ++k)
                orow[k] = 0.0;
            bb = seq_of[t];
            if (bb < 0) { /* a token that no sequence owns */
                ++errors;
                continue;
            }
            nq = query_start_loc[bb + 1] - query_start_loc[bb];
            c = seq_lens[bb] - nq; /* tokens before this chunk */
            i = (int)(t - query_start_loc[bb]);
            if (c < 0) {
                ++errors;
                continue;
            }
            errors += attend_row(&a, q + ((size_t)t * num_heads + hh) * head_dim,
                                 bb, hh, c + i + 1, orow, K, V, p);
        }
        free(K);
        free(V);
        free(p);
    }
    free(seq_of);
    return errors;
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int oracle_num_threads(int n_threads)
{
#ifdef _OPENMP
    if (n_threads > 0)
        return n_threads;
    return omp_get_max_threads();
#else
    (void)n_threads;
    return 1;
#endif
}
