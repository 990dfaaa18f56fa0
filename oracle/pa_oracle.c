/*
 * pa_oracle.c -- CPU oracle for paged single-token decode attention.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load this library.  It is
 * plain, slow C written to be checked by eye, in double precision, and it
 * shares no source, header or helper with the CUDA library.
 *
 * What it computes follows the pages this project is built from:
 *   - spindle, section "Paging": a pool of fixed-size blocks (block size 16)
 *     shared by all sequences, reached through a per-sequence block table;
 *     refcounted copy-on-write forks share blocks.
 *   - spindle, section "Two bugs worth recording": append takes an explicit
 *     start position and attention (the "gather") takes an explicit length;
 *     nothing here infers a position or advances a length.
 *   - spindle, section "Why write the forward pass": attention reads the
 *     cache sequence by sequence, so nothing may leak across sequences.
 * The attention itself is the plain definition: gather the sequence's keys
 * and values into contiguous buffers, take the dot products with the query,
 * a max-subtracted softmax, and the weighted sum of values.  The oracle does
 * not split the context into partitions; it is the result a split-KV kernel
 * must reproduce within rounding.
 *
 * Pool layout (a choice of this library; the pages fix none):
 *   pool[num_blocks][num_kv_heads][head_dim / X][16][X],  X = 16 / elem_bytes
 * i.e. element (block b, kv head h, slot t, dim d) sits at
 *   ((((b * Hkv + h) * (D / X) + d / X) * 16 + t) * X + d % X)
 * Each (block, head) tile is one contiguous 16*D*elem_bytes chunk.
 *
 * Element types: 0 = fp32, 1 = bf16 (raw 16-bit patterns).  bf16 inputs are
 * widened exactly (bit shift); outputs are rounded once from double.
 *
 * Parity status: the attention values are pinned by closed forms, special
 * cases and a library routine in the test suite, not by printed values (the
 * pages print none for attention).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_BLOCK 16

/* Return codes. */
#define OR_OK 0
#define OR_BAD_ARG 1
#define OR_BAD_BLOCK 2   /* a block-table entry outside [0, num_blocks) */
#define OR_BAD_POS 3     /* a position beyond the block table's capacity */

/* ---- element conversion ------------------------------------------------ */

static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;   /* bf16 is the top half of an fp32 */
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load_elem(const void* base, size_t idx, int dtype) {
    if (dtype == 1) return bf16_bits_to_double(((const uint16_t*)base)[idx]);
    return (double)((const float*)base)[idx];
}

/* Round a double to the nearest bf16, ties to even, in one step.
 * bf16 has 8 exponent bits (like fp32) and 7 stored mantissa bits, so its
 * spacing (ulp) at magnitude m in [2^e, 2^(e+1)) is 2^(e-7), and 2^(-133)
 * below the smallest normal 2^(-126).  x / ulp is exact in double (a power
 * of two scaling), rint() rounds it half-to-even, and the result is a bf16
 * value, which is also an fp32 value, so its top 16 bits are the code. */
uint16_t oracle_double_to_bf16(double x) {
    if (isnan(x)) return 0x7FC0;
    double m = fabs(x);
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isinf(x)) return sign | 0x7F80;
    if (m == 0.0) return sign;
    int e;
    frexp(m, &e);                 /* m = f * 2^e, f in [0.5, 1): m in [2^(e-1), 2^e) */
    int ex = e - 1;               /* m in [2^ex, 2^(ex+1)) */
    if (ex < -126) ex = -126;     /* subnormal range keeps the fixed spacing */
    double ulp = ldexp(1.0, ex - 7);
    double r = rint(m / ulp) * ulp;
    if (r >= ldexp(1.0, 128)) return sign | 0x7F80;   /* overflow to infinity */
    float f = (float)r;           /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

/* Round double -> fp32 (the C conversion rounds to nearest even). */
static float double_to_f32(double x) { return (float)x; }

void oracle_round_out(const double* in, void* out, int64_t n, int dtype) {
    for (int64_t i = 0; i < n; ++i) {
        if (dtype == 1) ((uint16_t*)out)[i] = oracle_double_to_bf16(in[i]);
        else ((float*)out)[i] = double_to_f32(in[i]);
    }
}

double oracle_bf16_to_double(uint16_t b) { return bf16_bits_to_double(b); }

/* ---- layout ------------------------------------------------------------ */

static int elem_bytes_of(int dtype) { return dtype == 1 ? 2 : 4; }

/* Element index of (block, kv head, slot, dim) in a pool. */
static size_t pool_elem(int64_t blk, int h, int slot, int d, int Hkv, int D, int X) {
    return ((((size_t)blk * (size_t)Hkv + (size_t)h) * (size_t)(D / X) + (size_t)(d / X)) * ORACLE_BLOCK
            + (size_t)slot) * (size_t)X + (size_t)(d % X);
}

static int check_dims(int Hkv, int D, int dtype) {
    if (dtype != 0 && dtype != 1) return 0;
    int X = 16 / elem_bytes_of(dtype);
    if (Hkv <= 0 || D <= 0 || D % X != 0) return 0;
    return 1;
}

/* Physical block holding logical position p of sequence s (spindle, "Paging":
 * logical block p / 16 through the table, slot p % 16). */
static int lookup_block(const int32_t* tables, int max_blocks, int s, int p, int num_blocks,
                        int64_t* blk_out) {
    int lb = p / ORACLE_BLOCK;
    if (p < 0 || lb >= max_blocks) return OR_BAD_POS;
    int32_t b = tables[(size_t)s * (size_t)max_blocks + (size_t)lb];
    if (b < 0 || b >= num_blocks) return OR_BAD_BLOCK;
    *blk_out = b;
    return OR_OK;
}

/* ---- append (explicit start position) ---------------------------------- */

/* Write n_s = cu_new[s+1] - cu_new[s] new tokens of sequence s at positions
 * start_pos[s] .. start_pos[s] + n_s - 1.  k_new / v_new rows are
 * [sum n_s][Hkv][D] in plain row-major order.  A pure byte copy. */
int oracle_append_kv(void* k_pool, void* v_pool, const void* k_new, const void* v_new,
                     const int32_t* tables, int max_blocks, const int32_t* start_pos,
                     const int32_t* cu_new, int num_seqs, int num_blocks, int Hkv, int D,
                     int dtype) {
    if (!check_dims(Hkv, D, dtype) || num_seqs < 0) return OR_BAD_ARG;
    int eb = elem_bytes_of(dtype);
    int X = 16 / eb;
    int rc = OR_OK;
    for (int s = 0; s < num_seqs; ++s) {
        int n = cu_new[s + 1] - cu_new[s];
        for (int i = 0; i < n; ++i) {
            int p = start_pos[s] + i;
            int64_t blk;
            int r = lookup_block(tables, max_blocks, s, p, num_blocks, &blk);
            if (r != OR_OK) { rc = r; continue; }
            size_t row = (size_t)(cu_new[s] + i);
            for (int h = 0; h < Hkv; ++h) {
                for (int d = 0; d < D; ++d) {
                    size_t src = (row * (size_t)Hkv + (size_t)h) * (size_t)D + (size_t)d;
                    size_t dst = pool_elem(blk, h, p % ORACLE_BLOCK, d, Hkv, D, X);
                    memcpy((char*)k_pool + dst * eb, (const char*)k_new + src * eb, (size_t)eb);
                    memcpy((char*)v_pool + dst * eb, (const char*)v_new + src * eb, (size_t)eb);
                }
            }
        }
    }
    return rc;
}

/* ---- copy-on-write block copy ------------------------------------------ */

/* For each pair (src, dst), copy every byte of block src to block dst in
 * both pools (all kv heads, all 16 slots).  spindle, "Paging": refcounted
 * copy-on-write forking; the copy is what makes a shared block private. */
int oracle_copy_block(void* k_pool, void* v_pool, const int32_t* pairs, int num_pairs,
                      int num_blocks, int Hkv, int D, int dtype) {
    if (!check_dims(Hkv, D, dtype) || num_pairs < 0) return OR_BAD_ARG;
    size_t block_bytes = (size_t)Hkv * ORACLE_BLOCK * (size_t)D * (size_t)elem_bytes_of(dtype);
    int rc = OR_OK;
    for (int i = 0; i < num_pairs; ++i) {
        int32_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) { rc = OR_BAD_BLOCK; continue; }
        memmove((char*)k_pool + (size_t)dst * block_bytes, (char*)k_pool + (size_t)src * block_bytes, block_bytes);
        memmove((char*)v_pool + (size_t)dst * block_bytes, (char*)v_pool + (size_t)src * block_bytes, block_bytes);
    }
    return rc;
}

/* ---- decode attention --------------------------------------------------- */

/* The plain definition for one query: out = sum_t softmax(scale * <q, K_t>)_t V_t,
 * with the maximum score subtracted before exponentiating.  Kc and Vc are
 * L contiguous rows of D doubles. */
static void attend(double* out_row, const double* qv, const double* Kc, const double* Vc,
                   double* x, int L, int D, double scale) {
    for (int d = 0; d < D; ++d) out_row[d] = 0.0;
    if (L <= 0) return;
    double xmax = -INFINITY;
    for (int t = 0; t < L; ++t) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += qv[d] * Kc[(size_t)t * D + d];
        x[t] = scale * acc;
        if (x[t] > xmax) xmax = x[t];
    }
    double denom = 0.0;
    for (int t = 0; t < L; ++t) { x[t] = exp(x[t] - xmax); denom += x[t]; }
    for (int t = 0; t < L; ++t) {
        double p = x[t] / denom;
        for (int d = 0; d < D; ++d) out_row[d] += p * Vc[(size_t)t * D + d];
    }
}

/* One (sequence, query head): gather the context through the block table
 * into contiguous K and V, then attend in double.  Query head h reads kv head
 * h / (Hq / Hkv) (grouped-query attention).  A zero-length context gives a
 * zero output.  out_row gets D doubles. */
int oracle_decode_one(double* out_row, const void* q, const void* k_pool, const void* v_pool,
                      const int32_t* tables, const int32_t* context_lens, int s, int h,
                      int Hq, int Hkv, int D, int max_blocks, int num_blocks, double scale,
                      int dtype) {
    if (!check_dims(Hkv, D, dtype) || Hq <= 0 || Hq % Hkv != 0) return OR_BAD_ARG;
    int X = 16 / elem_bytes_of(dtype);
    int g = h / (Hq / Hkv);
    int L = context_lens[s];
    for (int d = 0; d < D; ++d) out_row[d] = 0.0;
    if (L <= 0) return L < 0 ? OR_BAD_POS : OR_OK;
    if (L > max_blocks * ORACLE_BLOCK) return OR_BAD_POS;

    double* Kc = (double*)malloc(sizeof(double) * (size_t)L * (size_t)D);
    double* Vc = (double*)malloc(sizeof(double) * (size_t)L * (size_t)D);
    double* x = (double*)malloc(sizeof(double) * (size_t)L);
    double* qv = (double*)malloc(sizeof(double) * (size_t)D);
    int rc = OR_OK;
    if (!Kc || !Vc || !x || !qv) { rc = OR_BAD_ARG; goto done; }

    /* gather to contiguous: logical position t is slot t % 16 of block table[s][t / 16] */
    for (int t = 0; t < L; ++t) {
        int64_t blk;
        rc = lookup_block(tables, max_blocks, s, t, num_blocks, &blk);
        if (rc != OR_OK) goto done;
        for (int d = 0; d < D; ++d) {
            size_t e = pool_elem(blk, g, t % ORACLE_BLOCK, d, Hkv, D, X);
            Kc[(size_t)t * D + d] = load_elem(k_pool, e, dtype);
            Vc[(size_t)t * D + d] = load_elem(v_pool, e, dtype);
        }
    }
    for (int d = 0; d < D; ++d) qv[d] = load_elem(q, ((size_t)s * Hq + h) * (size_t)D + d, dtype);
    attend(out_row, qv, Kc, Vc, x, L, D, scale);
done:
    free(Kc); free(Vc); free(x); free(qv);
    return rc;
}

/* One query against a context already in contiguous rows (no paging at all):
 * q_row is D elements, k_rows / v_rows are [L][Hkv][D] elements, and the query
 * reads kv head g.  This is the "contiguous" side of paged == contiguous. */
int oracle_decode_contig(double* out_row, const void* q_row, const void* k_rows,
                         const void* v_rows, int L, int g, int Hkv, int D, double scale,
                         int dtype) {
    if (dtype != 0 && dtype != 1) return OR_BAD_ARG;
    if (Hkv <= 0 || D <= 0 || g < 0 || g >= Hkv || L < 0) return OR_BAD_ARG;
    double* Kc = (double*)malloc(sizeof(double) * ((size_t)L + 1) * (size_t)D);
    double* Vc = (double*)malloc(sizeof(double) * ((size_t)L + 1) * (size_t)D);
    double* x = (double*)malloc(sizeof(double) * ((size_t)L + 1));
    double* qv = (double*)malloc(sizeof(double) * (size_t)D);
    int rc = OR_OK;
    if (!Kc || !Vc || !x || !qv) { rc = OR_BAD_ARG; goto done; }
    for (int t = 0; t < L; ++t)
        for (int d = 0; d < D; ++d) {
            size_t e = ((size_t)t * Hkv + (size_t)g) * (size_t)D + (size_t)d;
            Kc[(size_t)t * D + d] = load_elem(k_rows, e, dtype);
            Vc[(size_t)t * D + d] = load_elem(v_rows, e, dtype);
        }
    for (int d = 0; d < D; ++d) qv[d] = load_elem(q_row, (size_t)d, dtype);
    attend(out_row, qv, Kc, Vc, x, L, D, scale);
done:
    free(Kc); free(Vc); free(x); free(qv);
    return rc;
}

/* Every (sequence, query head); out is [S][Hq][D] doubles. */
int oracle_decode(double* out, const void* q, const void* k_pool, const void* v_pool,
                  const int32_t* tables, const int32_t* context_lens, int num_seqs, int Hq,
                  int Hkv, int D, int max_blocks, int num_blocks, double scale, int dtype) {
    int rc = OR_OK;
    for (int s = 0; s < num_seqs; ++s)
        for (int h = 0; h < Hq; ++h) {
            int r = oracle_decode_one(out + ((size_t)s * Hq + h) * (size_t)D, q, k_pool, v_pool,
                                      tables, context_lens, s, h, Hq, Hkv, D, max_blocks,
                                      num_blocks, scale, dtype);
            if (r != OR_OK) rc = r;
        }
    return rc;
}

/* A chosen subset of (sequence, query head) pairs: pairs[2i], pairs[2i+1];
 * out is [n][D] doubles.  Used to check full-size runs one output at a time. */
int oracle_decode_pairs(double* out, const int32_t* pairs, int n, const void* q,
                        const void* k_pool, const void* v_pool, const int32_t* tables,
                        const int32_t* context_lens, int Hq, int Hkv, int D, int max_blocks,
                        int num_blocks, double scale, int dtype) {
    int rc = OR_OK;
    for (int i = 0; i < n; ++i) {
        int r = oracle_decode_one(out + (size_t)i * D, q, k_pool, v_pool, tables, context_lens,
                                  pairs[2 * i], pairs[2 * i + 1], Hq, Hkv, D, max_blocks,
                                  num_blocks, scale, dtype);
        if (r != OR_OK) rc = r;
    }
    return rc;
}

/* ---- FP8 (E4M3) KV cache ------------------------------------------------ *
 * Quantised pools hold, per (block, kv head), a record of 16 * D code bytes
 * followed by 16 fp32 scales (one per slot):
 *   K codes: [D / 16][16 slots][16 dims]   (16-byte pieces per slot, as the
 *            bf16 layout with X = 16)
 *   V codes: [D][16 slots]                 (one 16-byte row per dim)
 *   scales : [16] fp32, value = code * scale
 * E4M3: 1 sign, 4 exponent (bias 7) and 3 mantissa bits; no infinities; the
 * code 0x7F / 0xFF is NaN; the largest finite value is 448; below 2^-6 the
 * spacing is fixed at 2^-9 (subnormals).  (The pages name a block-scaled FP4
 * GEMM on the Slipstream page, "Companion work", for the same bandwidth-bound
 * decode; a per-token scale is this library's reading for an 8-bit cache.) */

double oracle_e4m3_to_double(uint8_t c) {
    int sign = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Nearest E4M3 value (ties to even), magnitudes above 448 saturate to 448. */
uint8_t oracle_f32_to_e4m3(float x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double m = fabs((double)x);
    if (m == 0.0) return sign;
    int e;
    frexp(m, &e);
    int ex = e - 1;               /* m in [2^ex, 2^(ex+1)) */
    if (ex < -6) ex = -6;         /* subnormal spacing 2^-9 */
    double ulp = ldexp(1.0, ex - 3);
    double r = rint(m / ulp) * ulp;
    if (r > 448.0) r = 448.0;
    if (r == 0.0) return sign;
    uint8_t code;
    if (r < ldexp(1.0, -6)) {
        code = (uint8_t)(r / ldexp(1.0, -9));           /* subnormal: E = 0 */
    } else {
        int re;
        frexp(r, &re);                                  /* r in [2^(re-1), 2^re) */
        int E = re - 1 + 7;
        int M = (int)(r / ldexp(1.0, re - 1) * 8.0) - 8;
        code = (uint8_t)((E << 3) | M);
    }
    return sign | code;
}

static size_t fp8_record_bytes(int D) { return (size_t)16 * D + 64; }

/* Quantise one row of D values (bf16 bits) with its own scale amax / 448;
 * the arithmetic is fp32, each step correctly rounded. */
static float quantise_row(const uint16_t* row, int D, uint8_t* codes) {
    float amax = 0.0f;
    for (int d = 0; d < D; ++d) {
        uint32_t u = ((uint32_t)row[d]) << 16;
        float f;
        memcpy(&f, &u, sizeof f);
        f = fabsf(f);
        if (f > amax) amax = f;
    }
    float scale = amax / 448.0f;
    for (int d = 0; d < D; ++d) {
        uint32_t u = ((uint32_t)row[d]) << 16;
        float f;
        memcpy(&f, &u, sizeof f);
        codes[d] = scale > 0.0f ? oracle_f32_to_e4m3(f / scale) : 0;
    }
    return scale;
}

/* Append with quantisation: rows of bf16 k_new / v_new ([sum n][Hkv][D]) go
 * to explicit positions like oracle_append_kv, as codes plus per-slot scales. */
int oracle_append_kv_fp8(void* k_pool, void* v_pool, const void* k_new, const void* v_new,
                         const int32_t* tables, int max_blocks, const int32_t* start_pos,
                         const int32_t* cu_new, int num_seqs, int num_blocks, int Hkv, int D) {
    if (Hkv <= 0 || D <= 0 || D % 16 != 0 || num_seqs < 0) return OR_BAD_ARG;
    size_t rec = fp8_record_bytes(D);
    uint8_t* codes = (uint8_t*)malloc((size_t)D);
    if (!codes) return OR_BAD_ARG;
    int rc = OR_OK;
    for (int s = 0; s < num_seqs; ++s) {
        int n = cu_new[s + 1] - cu_new[s];
        for (int i = 0; i < n; ++i) {
            int p = start_pos[s] + i;
            int64_t blk;
            int r = lookup_block(tables, max_blocks, s, p, num_blocks, &blk);
            if (r != OR_OK) { rc = r; continue; }
            int t = p % ORACLE_BLOCK;
            size_t row = (size_t)(cu_new[s] + i);
            for (int h = 0; h < Hkv; ++h) {
                uint8_t* krec = (uint8_t*)k_pool + ((size_t)blk * Hkv + h) * rec;
                uint8_t* vrec = (uint8_t*)v_pool + ((size_t)blk * Hkv + h) * rec;
                const uint16_t* krow = (const uint16_t*)k_new + (row * Hkv + h) * (size_t)D;
                const uint16_t* vrow = (const uint16_t*)v_new + (row * Hkv + h) * (size_t)D;
                float ks = quantise_row(krow, D, codes);
                for (int d = 0; d < D; ++d) krec[((size_t)(d / 16) * 16 + t) * 16 + d % 16] = codes[d];
                memcpy(krec + (size_t)16 * D + 4 * t, &ks, 4);
                float vs = quantise_row(vrow, D, codes);
                for (int d = 0; d < D; ++d) vrec[(size_t)d * 16 + t] = codes[d];
                memcpy(vrec + (size_t)16 * D + 4 * t, &vs, 4);
            }
        }
    }
    free(codes);
    return rc;
}

/* Decode over FP8 pools: gather each position's codes through the table,
 * dequantise (code * scale, exact in double) and attend; q is bf16. */
int oracle_decode_fp8_one(double* out_row, const void* q, const void* k_pool, const void* v_pool,
                          const int32_t* tables, const int32_t* context_lens, int s, int h,
                          int Hq, int Hkv, int D, int max_blocks, int num_blocks, double scale) {
    if (Hkv <= 0 || D <= 0 || D % 16 != 0 || Hq <= 0 || Hq % Hkv != 0) return OR_BAD_ARG;
    int g = h / (Hq / Hkv);
    int L = context_lens[s];
    for (int d = 0; d < D; ++d) out_row[d] = 0.0;
    if (L <= 0) return L < 0 ? OR_BAD_POS : OR_OK;
    if (L > max_blocks * ORACLE_BLOCK) return OR_BAD_POS;
    size_t rec = fp8_record_bytes(D);
    double* Kc = (double*)malloc(sizeof(double) * (size_t)L * (size_t)D);
    double* Vc = (double*)malloc(sizeof(double) * (size_t)L * (size_t)D);
    double* x = (double*)malloc(sizeof(double) * (size_t)L);
    double* qv = (double*)malloc(sizeof(double) * (size_t)D);
    int rc = OR_OK;
    if (!Kc || !Vc || !x || !qv) { rc = OR_BAD_ARG; goto done; }
    for (int t = 0; t < L; ++t) {
        int64_t blk;
        rc = lookup_block(tables, max_blocks, s, t, num_blocks, &blk);
        if (rc != OR_OK) goto done;
        int slot = t % ORACLE_BLOCK;
        const uint8_t* krec = (const uint8_t*)k_pool + ((size_t)blk * Hkv + g) * rec;
        const uint8_t* vrec = (const uint8_t*)v_pool + ((size_t)blk * Hkv + g) * rec;
        float ks, vs;
        memcpy(&ks, krec + (size_t)16 * D + 4 * slot, 4);
        memcpy(&vs, vrec + (size_t)16 * D + 4 * slot, 4);
        for (int d = 0; d < D; ++d) {
            Kc[(size_t)t * D + d] = oracle_e4m3_to_double(krec[((size_t)(d / 16) * 16 + slot) * 16 + d % 16]) * ks;
            Vc[(size_t)t * D + d] = oracle_e4m3_to_double(vrec[(size_t)d * 16 + slot]) * vs;
        }
    }
    for (int d = 0; d < D; ++d) qv[d] = load_elem(q, ((size_t)s * Hq + h) * (size_t)D + d, 1);
    attend(out_row, qv, Kc, Vc, x, L, D, scale);
done:
    free(Kc); free(Vc); free(x); free(qv);
    return rc;
}

int oracle_decode_fp8_pairs(double* out, const int32_t* pairs, int n, const void* q,
                            const void* k_pool, const void* v_pool, const int32_t* tables,
                            const int32_t* context_lens, int Hq, int Hkv, int D, int max_blocks,
                            int num_blocks, double scale) {
    int rc = OR_OK;
    for (int i = 0; i < n; ++i) {
        int r = oracle_decode_fp8_one(out + (size_t)i * D, q, k_pool, v_pool, tables, context_lens,
                                      pairs[2 * i], pairs[2 * i + 1], Hq, Hkv, D, max_blocks,
                                      num_blocks, scale);
        if (r != OR_OK) rc = r;
    }
    return rc;
}

/* ---- block-scaled FP4 (MXFP4) KV cache ------------------------------------ *
 * Slipstream, "Companion work", names a block-scaled FP4 kernel (qgemm-mx) as
 * the next step of the same bandwidth-bound decode.  The reading taken here is
 * the microscaling (MX) format that name refers to: blocks of 32 values along
 * head_dim share one power-of-two scale stored as an E8M0 byte (value
 * 2^(code - 127)); each value is an E2M1 code (1 sign bit, 2 exponent bits
 * with bias 1, 1 mantissa bit: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; no
 * infinity or NaN).  The shared exponent of a block with largest magnitude
 * amax is floor(log2(amax)) - 2 (2 = the exponent of E2M1's largest value,
 * 6 = 1.5 * 2^2), so amax / scale lies in [4, 8) and values above 6 saturate.
 * Each (token, kv head) row gets head_dim / 32 scales.
 *
 * Record of one (block, kv head), 8 * D code bytes then D / 2 scale bytes:
 *   K codes: slot t's row of D / 2 bytes at t * D / 2; the byte at
 *            c * (D / 8) + ks * 2 + half (c < 4, ks < D / 16, half < 2) holds
 *            dims d0 = 16 ks + 8 half + 2 c (low nibble) and d0 + 1 (high).
 *   V codes: the byte at ((r * 4 + c) * (D / 16) + mi) * 4 + dh * 2 + half
 *            (r < 8, c < 4, mi < D / 16, dh < 2, half < 2) holds dim
 *            16 mi + 8 dh + r of slots 2 c + 8 half (low nibble) and that + 1
 *            (high nibble).
 *   scales : at 8 * D, [16 slots][D / 32] E8M0 bytes, K and V alike.
 * (The byte orders are this library's choice: each tensor-core fragment of a
 * decode thread is then a run of adjacent bytes.) */

/* Value of a 4-bit E2M1 code. */
double oracle_e2m1_to_double(uint8_t c) {
    int sign = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -v : v;
}

/* Nearest E2M1 code, ties to the even code (mantissa bit 0); magnitudes above
 * 6 saturate to 6; the sign of a zero result is kept.  Spacing: 0.5 below 2,
 * 1 in [2, 4), 2 in [4, 6]. */
uint8_t oracle_f32_to_e2m1(float x) {
    uint8_t sign = signbit(x) ? 8 : 0;
    double m = fabs((double)x);
    if (isnan(x)) return sign;                     /* outside the format; not drawn */
    double ulp = m < 2.0 ? 0.5 : (m < 4.0 ? 1.0 : 2.0);
    double r = rint(m / ulp) * ulp;                /* half-way cases to the even multiple */
    if (r > 6.0) r = 6.0;
    uint8_t code;
    if (r < 1.0) code = (uint8_t)(r / 0.5);        /* E = 0: 0 or 0.5 */
    else {
        int re;
        frexp(r, &re);                             /* r in [2^(re-1), 2^re) */
        int E = re;                                /* bias 1: r = 2^(E-1) (1 + M / 2) */
        int M = (int)(r / ldexp(1.0, re - 1) * 2.0) - 2;
        code = (uint8_t)((E << 1) | M);
    }
    return sign | code;
}

/* E8M0 code of the shared scale of a block whose largest magnitude is amax:
 * 127 + floor(log2(amax)) - 2, kept in [0, 254]; an all-zero block gets 0. */
uint8_t oracle_mx_scale_code(float amax) {
    if (!(amax > 0.0f)) return 0;
    int e;
    frexp((double)amax, &e);                       /* amax in [2^(e-1), 2^e) */
    int code = 127 + (e - 1) - 2;
    if (code < 0) code = 0;
    if (code > 254) code = 254;
    return (uint8_t)code;
}

static size_t fp4_record_bytes(int D) { return (size_t)8 * D + (size_t)D / 2; }

static size_t fp4_k_byte(int t, int d, int D) {
    int ks = d / 16, half = (d % 16) / 8, c = (d % 8) / 2;
    return (size_t)t * (D / 2) + (size_t)c * (D / 8) + (size_t)ks * 2 + half;
}

static size_t fp4_v_byte(int t, int d, int D) {
    int mi = d / 16, dh = (d % 16) / 8, r = d % 8;
    int half = t / 8, c = (t % 8) / 2;
    return ((size_t)(r * 4 + c) * (D / 16) + mi) * 4 + dh * 2 + half;
}

/* Nibble of a code: the even dim (K) or even slot (V) of a byte is its low nibble. */
static void put_nibble(uint8_t* rec, size_t byte, int high, uint8_t code) {
    if (high) rec[byte] = (uint8_t)((rec[byte] & 0x0F) | (code << 4));
    else rec[byte] = (uint8_t)((rec[byte] & 0xF0) | (code & 0x0F));
}

static uint8_t get_nibble(const uint8_t* rec, size_t byte, int high) {
    return high ? (uint8_t)(rec[byte] >> 4) : (uint8_t)(rec[byte] & 0x0F);
}

/* Quantise one row of D bf16 values: D / 32 scale codes, D E2M1 codes; the
 * division by the power-of-two scale is exact (done in double). */
static void quantise_row_fp4(const uint16_t* row, int D, uint8_t* codes, uint8_t* sc) {
    for (int b = 0; b < D / 32; ++b) {
        float amax = 0.0f;
        for (int d = 32 * b; d < 32 * b + 32; ++d) {
            double v = fabs(bf16_bits_to_double(row[d]));
            if ((float)v > amax) amax = (float)v;
        }
        sc[b] = oracle_mx_scale_code(amax);
        double X = ldexp(1.0, (int)sc[b] - 127);
        for (int d = 32 * b; d < 32 * b + 32; ++d)
            codes[d] = amax > 0.0f ? oracle_f32_to_e2m1((float)(bf16_bits_to_double(row[d]) / X)) : 0;
    }
}

/* Append with MXFP4 quantisation: bf16 rows ([sum n][Hkv][D]) to explicit
 * positions like oracle_append_kv; codes and scales in the record layout above. */
int oracle_append_kv_fp4(void* k_pool, void* v_pool, const void* k_new, const void* v_new,
                         const int32_t* tables, int max_blocks, const int32_t* start_pos,
                         const int32_t* cu_new, int num_seqs, int num_blocks, int Hkv, int D) {
    if (Hkv <= 0 || D <= 0 || D % 32 != 0 || num_seqs < 0) return OR_BAD_ARG;
    size_t rec = fp4_record_bytes(D);
    uint8_t* codes = (uint8_t*)malloc((size_t)D);
    uint8_t* sc = (uint8_t*)malloc((size_t)D / 32);
    if (!codes || !sc) { free(codes); free(sc); return OR_BAD_ARG; }
    int rc = OR_OK;
    for (int s = 0; s < num_seqs; ++s) {
        int n = cu_new[s + 1] - cu_new[s];
        for (int i = 0; i < n; ++i) {
            int p = start_pos[s] + i;
            int64_t blk;
            int r = lookup_block(tables, max_blocks, s, p, num_blocks, &blk);
            if (r != OR_OK) { rc = r; continue; }
            int t = p % ORACLE_BLOCK;
            size_t row = (size_t)(cu_new[s] + i);
            for (int h = 0; h < Hkv; ++h) {
                uint8_t* krec = (uint8_t*)k_pool + ((size_t)blk * Hkv + h) * rec;
                uint8_t* vrec = (uint8_t*)v_pool + ((size_t)blk * Hkv + h) * rec;
                quantise_row_fp4((const uint16_t*)k_new + (row * Hkv + h) * (size_t)D, D, codes, sc);
                for (int d = 0; d < D; ++d) put_nibble(krec, fp4_k_byte(t, d, D), d & 1, codes[d]);
                memcpy(krec + (size_t)8 * D + (size_t)t * (D / 32), sc, (size_t)D / 32);
                quantise_row_fp4((const uint16_t*)v_new + (row * Hkv + h) * (size_t)D, D, codes, sc);
                for (int d = 0; d < D; ++d) put_nibble(vrec, fp4_v_byte(t, d, D), t & 1, codes[d]);
                memcpy(vrec + (size_t)8 * D + (size_t)t * (D / 32), sc, (size_t)D / 32);
            }
        }
    }
    free(codes);
    free(sc);
    return rc;
}

/* Dequantised value of (slot t, dim d) of a record: code * 2^(scale - 127), exact. */
static double fp4_value(const uint8_t* recp, int t, int d, int D, int is_v) {
    uint8_t code = is_v ? get_nibble(recp, fp4_v_byte(t, d, D), t & 1)
                        : get_nibble(recp, fp4_k_byte(t, d, D), d & 1);
    uint8_t sc = recp[(size_t)8 * D + (size_t)t * (D / 32) + d / 32];
    return ldexp(oracle_e2m1_to_double(code), (int)sc - 127);
}

/* Decode over MXFP4 pools: gather each position through the table, dequantise
 * and attend in double; q is bf16. */
int oracle_decode_fp4_one(double* out_row, const void* q, const void* k_pool, const void* v_pool,
                          const int32_t* tables, const int32_t* context_lens, int s, int h,
                          int Hq, int Hkv, int D, int max_blocks, int num_blocks, double scale) {
    if (Hkv <= 0 || D <= 0 || D % 32 != 0 || Hq <= 0 || Hq % Hkv != 0) return OR_BAD_ARG;
    int g = h / (Hq / Hkv);
    int L = context_lens[s];
    for (int d = 0; d < D; ++d) out_row[d] = 0.0;
    if (L <= 0) return L < 0 ? OR_BAD_POS : OR_OK;
    if (L > max_blocks * ORACLE_BLOCK) return OR_BAD_POS;
    size_t rec = fp4_record_bytes(D);
    double* Kc = (double*)malloc(sizeof(double) * (size_t)L * (size_t)D);
    double* Vc = (double*)malloc(sizeof(double) * (size_t)L * (size_t)D);
    double* x = (double*)malloc(sizeof(double) * (size_t)L);
    double* qv = (double*)malloc(sizeof(double) * (size_t)D);
    int rc = OR_OK;
    if (!Kc || !Vc || !x || !qv) { rc = OR_BAD_ARG; goto done; }
    for (int t = 0; t < L; ++t) {
        int64_t blk;
        rc = lookup_block(tables, max_blocks, s, t, num_blocks, &blk);
        if (rc != OR_OK) goto done;
        int t16 = t % ORACLE_BLOCK;
        const uint8_t* krec = (const uint8_t*)k_pool + ((size_t)blk * Hkv + g) * rec;
        const uint8_t* vrec = (const uint8_t*)v_pool + ((size_t)blk * Hkv + g) * rec;
        for (int d = 0; d < D; ++d) {
            Kc[(size_t)t * D + d] = fp4_value(krec, t16, d, D, 0);
            Vc[(size_t)t * D + d] = fp4_value(vrec, t16, d, D, 1);
        }
    }
    for (int d = 0; d < D; ++d) qv[d] = load_elem(q, ((size_t)s * Hq + h) * (size_t)D + d, 1);
    attend(out_row, qv, Kc, Vc, x, L, D, scale);
done:
    free(Kc); free(Vc); free(x); free(qv);
    return rc;
}

int oracle_decode_fp4_pairs(double* out, const int32_t* pairs, int n, const void* q,
                            const void* k_pool, const void* v_pool, const int32_t* tables,
                            const int32_t* context_lens, int Hq, int Hkv, int D, int max_blocks,
                            int num_blocks, double scale) {
    int rc = OR_OK;
    for (int i = 0; i < n; ++i) {
        int r = oracle_decode_fp4_one(out + (size_t)i * D, q, k_pool, v_pool, tables, context_lens,
                                      pairs[2 * i], pairs[2 * i + 1], Hq, Hkv, D, max_blocks,
                                      num_blocks, scale);
        if (r != OR_OK) rc = r;
    }
    return rc;
}

/* Dequantised rows of one (block, kv head) record: k_out, v_out [16][D] doubles
 * (a test view of the stored values). */
int oracle_fp4_record_values(double* k_out, double* v_out, const void* k_rec, const void* v_rec,
                             int D) {
    if (D <= 0 || D % 32 != 0) return OR_BAD_ARG;
    for (int t = 0; t < ORACLE_BLOCK; ++t)
        for (int d = 0; d < D; ++d) {
            k_out[(size_t)t * D + d] = fp4_value((const uint8_t*)k_rec, t, d, D, 0);
            v_out[(size_t)t * D + d] = fp4_value((const uint8_t*)v_rec, t, d, D, 1);
        }
    return OR_OK;
}
