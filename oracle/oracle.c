/*
 * oracle.c -- plain, slow, obviously-correct CPU reference for paged decode
 * attention over a block-pooled KV cache.
 *
 * THIS IS TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load it.  It shares no code, header,
 * table or constant with the CUDA library, and it never reads anything the
 * CUDA library produced.
 *
 * Everything is computed in IEEE double precision except where the method
 * itself fixes a narrower type (the FP8/BF16 storage formats and the fp32
 * product x * (1/scale) that feeds the FP8 encoder).
 *
 * Passages followed (page title, section):
 *   - "How does TensorRT-LLM work?", section "The paged KV cache": the KV
 *     cache is one pool of equal fixed-size blocks; a per-request table lists
 *     the request's blocks in order; decode attends over every earlier token.
 *   - "Introduction to TensorRT-LLM", section "2. Paged KV Cache": fixed-size
 *     token blocks, virtual-to-physical block tables.
 *   - "TensorRT-LLM, in depth", section "First principles: where the GPU
 *     memory goes": kv_bytes_per_token = 2 * layers * kv_heads * head_dim *
 *     bytes_per_elem; Llama-3-8B has 8 KV heads (grouped-query attention).
 *   - "TensorRT-LLM, in depth", section "Quantization: fewer bytes per weight
 *     and per cached token": an FP8 KV cache halves cache memory.
 *   - "How does TensorRT-LLM work?", section "Custom attention kernels":
 *     attention is softmax(scale * q K^T) V over the cached tokens (the fused
 *     kernels reach exactly this result, only faster).
 *
 * Readings taken where the pages are silent (each one is listed in the design
 * notes of the repository):
 *   - pool layout [layer][block][kv_head][token_in_block][head_dim], K and V
 *     in separate pools;
 *   - grouped-query mapping: query head hq reads KV head hq / (Hq / Hkv);
 *   - a slot is block_id * block_size + offset; slot -1 means "skip";
 *   - FP8 is OCP E4M3 ("E4M3FN": bias 7, max 448, no infinities, S.1111.111
 *     is NaN); quantisation is e4m3(fp32(x) * fp32(1/scale)) with
 *     round-to-nearest-even and saturation to +-448; dequantisation is
 *     e4m3_value * scale;
 *   - a sequence of length 0 yields a zero output row and lse = -inf.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fPIC -shared oracle.c -lm
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Storage types, numbered for this file only. */
#define OR_F32 0
#define OR_BF16 1
#define OR_E4M3 2

#define OR_OK 0
#define OR_BAD_ARG 1
#define OR_BAD_INDEX 2

static int elem_bytes(int dtype) {
    switch (dtype) {
        case OR_F32: return 4;
        case OR_BF16: return 2;
        case OR_E4M3: return 1;
        default: return 0;
    }
}

/* ---------------------------------------------------------------- formats */

/* bfloat16 is the upper half of an IEEE binary32 word. */
double or_bf16_to_double(uint16_t bits) {
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, 4);
    return (double)f;
}

/* binary32 -> bfloat16, round to nearest, ties to even (by bit arithmetic on
 * the binary32 encoding); NaN maps to the quiet NaN 0x7FC0 with its sign. */
uint16_t or_float_to_bf16(float x) {
    uint32_t w;
    memcpy(&w, &x, 4);
    if ((w & 0x7F800000u) == 0x7F800000u && (w & 0x007FFFFFu) != 0)
        return (uint16_t)(((w >> 16) & 0x8000u) | 0x7FC0u);
    uint32_t lower = w & 0xFFFFu;
    uint32_t upper = w >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

/* OCP E4M3 decode from the bit fields: sign s, exponent e (4 bits, bias 7),
 * mantissa m (3 bits).  e == 0 is subnormal: m/8 * 2^-6.  S.1111.111 is NaN. */
double or_e4m3_to_double(uint8_t code) {
    int s = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* Round-half-to-even of a non-negative double to an integer value. */
static double rne(double a) {
    double f = floor(a);
    double d = a - f;
    if (d > 0.5) return f + 1.0;
    if (d < 0.5) return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* binary32 -> OCP E4M3, round to nearest even on the E4M3 grid, saturating
 * finite (and infinite) magnitudes above 448 to 448; NaN -> S.1111.111. */
uint8_t or_float_to_e4m3(float xf) {
    double x = (double)xf;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    if (isnan(x)) return (uint8_t)(sign | 0x7F);
    double a = fabs(x);
    if (a == 0.0) return sign;
    /* grid spacing: 2^(E-3) inside binade [2^E, 2^(E+1)), E >= -6; the
     * subnormal range shares the spacing of the lowest binade, 2^-9. */
    int E;
    frexp(a, &E); /* a = f * 2^E, f in [0.5, 1) -> binade exponent E-1 */
    E -= 1;
    if (E < -6) E = -6;
    double quantum = ldexp(1.0, E - 3);
    double r = rne(a / quantum) * quantum; /* exact: a is a binary32 value */
    if (r > 448.0) r = 448.0;
    if (r == 0.0) return sign;
    /* encode r exactly */
    int Er;
    frexp(r, &Er);
    Er -= 1;
    if (Er < -6) { /* subnormal: r = m * 2^-9 */
        int m = (int)(r / ldexp(1.0, -9));
        return (uint8_t)(sign | m);
    }
    int e = Er + 7;
    int m = (int)((r / ldexp(1.0, Er) - 1.0) * 8.0);
    return (uint8_t)(sign | (e << 3) | m);
}

/* Value of one stored element, as double. */
static double load_elem(const void* base, int dtype, int64_t idx) {
    switch (dtype) {
        case OR_F32: return (double)((const float*)base)[idx];
        case OR_BF16: return or_bf16_to_double(((const uint16_t*)base)[idx]);
        case OR_E4M3: return or_e4m3_to_double(((const uint8_t*)base)[idx]);
        default: return NAN;
    }
}

/* Value of one input element as binary32 (inputs are f32 or bf16). */
static float load_input_f32(const void* base, int dtype, int64_t idx) {
    if (dtype == OR_F32) return ((const float*)base)[idx];
    uint32_t w = ((uint32_t)((const uint16_t*)base)[idx]) << 16;
    float f;
    memcpy(&f, &w, 4);
    return f;
}

/* ----------------------------------------------------------- closed forms */

/* "TensorRT-LLM, in depth", First principles: K and V, per layer, per KV
 * head, head_dim elements each. */
int64_t or_kv_bytes_per_token(int64_t layers, int64_t kv_heads, int64_t head_dim,
                              int64_t bytes_per_elem) {
    return 2 * layers * kv_heads * head_dim * bytes_per_elem;
}

/* ------------------------------------------------------------ slot mapping */

/* Token at position pos of sequence seq lands in block table[seq][pos / bs]
 * at offset pos % bs; its slot is block * bs + offset.  seq < 0 gives -1. */
int or_slot_mapping(const int32_t* block_tables, int max_blocks_per_seq, int block_size,
                    const int32_t* seq_idx, const int32_t* pos, int num_tokens,
                    int64_t* slots_out) {
    for (int t = 0; t < num_tokens; ++t) {
        if (seq_idx[t] < 0) {
            slots_out[t] = -1;
            continue;
        }
        int32_t p = pos[t];
        if (p < 0 || p / block_size >= max_blocks_per_seq) return OR_BAD_INDEX;
        int32_t blk = block_tables[(int64_t)seq_idx[t] * max_blocks_per_seq + p / block_size];
        if (blk < 0) return OR_BAD_INDEX;
        slots_out[t] = (int64_t)blk * block_size + (p % block_size);
    }
    return OR_OK;
}

/* ---------------------------------------------------------------- append */

/* Write token t's K (or V) row for every KV head into the pool slot named by
 * slots[t].  src is [T][kv_heads][head_dim] in src_dtype (f32 or bf16); the
 * pool is [layers][num_blocks][kv_heads][block_size][head_dim] in pool_dtype.
 * f32->f32 and bf16->bf16 copy bits; f32->bf16 rounds to nearest even;
 * ->E4M3 encodes fp32(x) * fp32(1/scale). */
int or_kv_append(void* pool, int pool_dtype, int num_layers, int num_blocks, int block_size,
                 int kv_heads, int head_dim, int layer, const void* src, int src_dtype,
                 const int64_t* slots, int num_tokens, float scale) {
    if (layer < 0 || layer >= num_layers) return OR_BAD_ARG;
    if (src_dtype != OR_F32 && src_dtype != OR_BF16) return OR_BAD_ARG;
    if (pool_dtype == OR_F32 && src_dtype != OR_F32) return OR_BAD_ARG;
    int eb = elem_bytes(pool_dtype);
    if (eb == 0) return OR_BAD_ARG;
    float inv_scale = 1.0f / scale; /* one IEEE binary32 division */
    int64_t nslots = (int64_t)num_blocks * block_size;
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slots[t];
        if (slot == -1) continue;
        if (slot < 0 || slot >= nslots) return OR_BAD_INDEX;
        int64_t blk = slot / block_size, off = slot % block_size;
        for (int h = 0; h < kv_heads; ++h) {
            int64_t dst_row = ((((int64_t)layer * num_blocks + blk) * kv_heads + h) * block_size + off) * head_dim;
            int64_t src_row = ((int64_t)t * kv_heads + h) * head_dim;
            for (int d = 0; d < head_dim; ++d) {
                int64_t di = dst_row + d, si = src_row + d;
                if (pool_dtype == OR_F32) {
                    ((float*)pool)[di] = ((const float*)src)[si];
                } else if (pool_dtype == OR_BF16) {
                    if (src_dtype == OR_BF16)
                        ((uint16_t*)pool)[di] = ((const uint16_t*)src)[si];
                    else
                        ((uint16_t*)pool)[di] = or_float_to_bf16(((const float*)src)[si]);
                } else {
                    float x = load_input_f32(src, src_dtype, si);
                    float y = x * inv_scale;
                    ((uint8_t*)pool)[di] = or_float_to_e4m3(y);
                }
            }
        }
    }
    return OR_OK;
}

/* -------------------------------------------------------------- attention */

/* Decode attention for every (sequence b, query head hq) over the tokens t
 * with win_begin <= t < min(win_end, seq_lens[b]):
 *     K_t = pool_K[layer][table[b][t / bs]][hq / G][t % bs][:] * k_scale
 *     s_t = scale * sum_d q[b][hq][d] * K_t[d]
 *     w_t = exp(s_t - max s) / sum exp(s - max s)
 *     out[b][hq][:] = sum_t w_t * V_t[:]          lse[b][hq] = ln sum exp(s_t)
 * with V_t gathered like K_t (times v_scale).  Windows let a test split the
 * token range and recombine; the full result is win = [0, INT32_MAX).
 * k_scale / v_scale apply to E4M3 pools only (other pools use 1).
 * q is [B][Hq][D] in q_dtype (f32 or bf16).  out is [B][Hq][D] double;
 * lse is [B][Hq] double (-inf where no token is in the window).
 * num_threads <= 0 uses the OpenMP default.  Returns the number of threads
 * used through *threads_used when it is not NULL. */
int or_paged_attention(const void* q, int q_dtype, const void* k_pool, const void* v_pool,
                       int kv_dtype, int num_layers, int num_blocks, int block_size,
                       int kv_heads, int head_dim, int layer, float k_scale, float v_scale,
                       const int32_t* block_tables, int max_blocks_per_seq,
                       const int32_t* seq_lens, int num_seqs, int num_q_heads, float scale,
                       int win_begin, int win_end, double* out, double* lse, int num_threads,
                       int* threads_used) {
    if (layer < 0 || layer >= num_layers || kv_heads <= 0 || num_q_heads % kv_heads != 0)
        return OR_BAD_ARG;
    if (elem_bytes(kv_dtype) == 0 || (q_dtype != OR_F32 && q_dtype != OR_BF16)) return OR_BAD_ARG;
    const int G = num_q_heads / kv_heads;
    const double ks = (kv_dtype == OR_E4M3) ? (double)k_scale : 1.0;
    const double vs = (kv_dtype == OR_E4M3) ? (double)v_scale : 1.0;
    int status = OR_OK;
    int used = 1;
#ifdef _OPENMP
    if (num_threads <= 0) num_threads = omp_get_max_threads();
#else
    num_threads = 1;
#endif
    const int64_t pairs = (int64_t)num_seqs * num_q_heads;
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads)
    for (int64_t pr = 0; pr < pairs; ++pr) {
#ifdef _OPENMP
        if (pr == 0) used = omp_get_num_threads();
#endif
        const int b = (int)(pr / num_q_heads);
        const int hq = (int)(pr % num_q_heads);
        const int h = hq / G;
        double* o = out + pr * head_dim;
        for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
        lse[pr] = -INFINITY;
        int L = seq_lens[b];
        int t0 = win_begin < 0 ? 0 : win_begin;
        int t1 = win_end < L ? win_end : L;
        if (L < 0 || L > max_blocks_per_seq * block_size) {
#pragma omp atomic write
            status = OR_BAD_INDEX;
            continue;
        }
        if (t1 <= t0) continue;
        const int n = t1 - t0;
        double* s = (double*)malloc(sizeof(double) * (size_t)n);
        int64_t* row = (int64_t*)malloc(sizeof(int64_t) * (size_t)n);
        int bad = 0;
        /* gather: the row of token t lives in block table[b][t / bs] */
        for (int i = 0; i < n; ++i) {
            int t = t0 + i;
            int32_t blk = block_tables[(int64_t)b * max_blocks_per_seq + t / block_size];
            if (blk < 0 || blk >= num_blocks) { bad = 1; break; }
            row[i] = ((((int64_t)layer * num_blocks + blk) * kv_heads + h) * block_size +
                      t % block_size) * head_dim;
        }
        if (bad) {
#pragma omp atomic write
            status = OR_BAD_INDEX;
            free(s);
            free(row);
            continue;
        }
        /* scores */
        const int64_t qrow = pr * head_dim;
        double smax = -INFINITY;
        for (int i = 0; i < n; ++i) {
            double acc = 0.0;
            for (int d = 0; d < head_dim; ++d) {
                double qd = (q_dtype == OR_F32) ? (double)((const float*)q)[qrow + d]
                                                : or_bf16_to_double(((const uint16_t*)q)[qrow + d]);
                acc += qd * (load_elem(k_pool, kv_dtype, row[i] + d) * ks);
            }
            s[i] = (double)scale * acc;
            if (s[i] > smax) smax = s[i];
        }
        /* softmax weights and weighted sum of V */
        double z = 0.0;
        for (int i = 0; i < n; ++i) {
            s[i] = exp(s[i] - smax);
            z += s[i];
        }
        for (int i = 0; i < n; ++i) {
            double w = s[i] / z;
            for (int d = 0; d < head_dim; ++d)
                o[d] += w * (load_elem(v_pool, kv_dtype, row[i] + d) * vs);
        }
        lse[pr] = smax + log(z);
        free(s);
        free(row);
    }
    if (threads_used) *threads_used = used;
    return status;
}

/* Flash-decoding combine of per-window results: given S partial outputs
 * o_s (each already normalised over its window) and their log-sum-exps
 * lse_s, the attention over the union of the windows is
 *     out = sum_s exp(lse_s - M) o_s / sum_s exp(lse_s - M),  M = max_s lse_s.
 * Windows with lse = -inf (no tokens) contribute nothing; if every window is
 * empty the output is zero and lse is -inf.  o_parts is [S][D]. */
void or_lse_combine(const double* o_parts, const double* lse_parts, int num_parts, int head_dim,
                    double* out, double* lse_out) {
    double M = -INFINITY;
    for (int s = 0; s < num_parts; ++s)
        if (lse_parts[s] > M) M = lse_parts[s];
    for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
    if (M == -INFINITY) {
        *lse_out = -INFINITY;
        return;
    }
    double z = 0.0;
    for (int s = 0; s < num_parts; ++s) {
        if (lse_parts[s] == -INFINITY) continue;
        double w = exp(lse_parts[s] - M);
        z += w;
        for (int d = 0; d < head_dim; ++d) out[d] += w * o_parts[(int64_t)s * head_dim + d];
    }
    for (int d = 0; d < head_dim; ++d) out[d] /= z;
    *lse_out = M + log(z);
}

/* ------------------------------------------------ array helpers for tests */

void or_e4m3_encode_array(const float* x, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = or_float_to_e4m3(x[i]);
}

void or_e4m3_decode_array(const uint8_t* c, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = or_e4m3_to_double(c[i]);
}

void or_bf16_encode_array(const float* x, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = or_float_to_bf16(x[i]);
}

void or_bf16_decode_array(const uint16_t* c, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = or_bf16_to_double(c[i]);
}

/* ------------------------------------------------- multi-query attention */

/* Several queries per sequence: the last C tokens of sequence b (positions
 * L_b - C .. L_b - 1) each ask a query, as when a decode step verifies C
 * drafted tokens ("How does TensorRT-LLM work?", "Speculative decoding": the
 * big model checks several guessed tokens in one pass) or a prompt chunk is
 * processed ("TensorRT-LLM, in depth", "In-flight batching and the
 * scheduler": chunked prefill).  Query c sits at position L_b - C + c and
 * attends causally, to tokens 0 .. L_b - C + c:
 *     out[b][c][hq][:] = softmax_t(scale * q[b][c][hq] . K_t) V_t
 * q is [B][C][Hq][D]; out is [B][C][Hq][D] and lse [B][C][Hq] (double).
 * A query with no token (L_b - C + c < 0) gets zeros and lse = -inf. */
int or_paged_attention_mq(const void* q, int q_dtype, const void* k_pool, const void* v_pool,
                          int kv_dtype, int num_layers, int num_blocks, int block_size,
                          int kv_heads, int head_dim, int layer, float k_scale, float v_scale,
                          const int32_t* block_tables, int max_blocks_per_seq,
                          const int32_t* seq_lens, int num_seqs, int num_queries, int num_q_heads,
                          float scale, double* out, double* lse, int num_threads, int* threads_used) {
    if (layer < 0 || layer >= num_layers || kv_heads <= 0 || num_q_heads % kv_heads != 0 ||
        num_queries < 1)
        return OR_BAD_ARG;
    if (elem_bytes(kv_dtype) == 0 || (q_dtype != OR_F32 && q_dtype != OR_BF16)) return OR_BAD_ARG;
    const int G = num_q_heads / kv_heads;
    const int C = num_queries;
    const double ks = (kv_dtype == OR_E4M3) ? (double)k_scale : 1.0;
    const double vs = (kv_dtype == OR_E4M3) ? (double)v_scale : 1.0;
    int status = OR_OK;
#ifdef _OPENMP
    if (num_threads <= 0) num_threads = omp_get_max_threads();
#else
    num_threads = 1;
#endif
    const int64_t rows = (int64_t)num_seqs * C * num_q_heads;
    if (threads_used) *threads_used = num_threads;
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads)
    for (int64_t pr = 0; pr < rows; ++pr) {
        const int b = (int)(pr / ((int64_t)C * num_q_heads));
        const int c = (int)((pr / num_q_heads) % C);
        const int hq = (int)(pr % num_q_heads);
        const int h = hq / G;
        double* o = out + pr * head_dim;
        for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
        lse[pr] = -INFINITY;
        const int L = seq_lens[b];
        if (L < 0 || L > max_blocks_per_seq * block_size) {
#pragma omp atomic write
            status = OR_BAD_INDEX;
            continue;
        }
        const int n = L - C + c + 1; /* tokens 0 .. position of query c */
        if (n <= 0) continue;
        double* s = (double*)malloc(sizeof(double) * (size_t)n);
        int64_t* row = (int64_t*)malloc(sizeof(int64_t) * (size_t)n);
        int bad = 0;
        for (int t = 0; t < n; ++t) {
            int32_t blk = block_tables[(int64_t)b * max_blocks_per_seq + t / block_size];
            if (blk < 0 || blk >= num_blocks) { bad = 1; break; }
            row[t] = ((((int64_t)layer * num_blocks + blk) * kv_heads + h) * block_size +
                      t % block_size) * head_dim;
        }
        if (bad) {
#pragma omp atomic write
            status = OR_BAD_INDEX;
            free(s);
            free(row);
            continue;
        }
        double smax = -INFINITY;
        for (int t = 0; t < n; ++t) {
            double acc = 0.0;
            for (int d = 0; d < head_dim; ++d) {
                double qd = (q_dtype == OR_F32) ? (double)((const float*)q)[pr * head_dim + d]
                                                : or_bf16_to_double(((const uint16_t*)q)[pr * head_dim + d]);
                acc += qd * (load_elem(k_pool, kv_dtype, row[t] + d) * ks);
            }
            s[t] = (double)scale * acc;
            if (s[t] > smax) smax = s[t];
        }
        double z = 0.0;
        for (int t = 0; t < n; ++t) {
            s[t] = exp(s[t] - smax);
            z += s[t];
        }
        for (int t = 0; t < n; ++t) {
            double w = s[t] / z;
            for (int d = 0; d < head_dim; ++d)
                o[d] += w * (load_elem(v_pool, kv_dtype, row[t] + d) * vs);
        }
        lse[pr] = smax + log(z);
        free(s);
        free(row);
    }
    return status;
}
