/*
 * us_oracle.c -- plain, slow CPU oracle for bitmap-encoded unstructured-sparse
 * weight matrices and for Y = W.X on them.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may link,
 * load or call this file: only the test-suite, the smoke check and the CPU
 * baseline leg of the benchmark use it.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * Sources (each function below names the passage it restates):
 *  [UnionSparse]  "UnionSparse: An Index-Efficient Sparsity Framework for
 *                 Low-Bit Sparse LLM Inference on Edge", section V-A
 *                 "IE-BME Representation" (Union Bitmaps, Union Value Offsets,
 *                 Compressed Values, Fig. 7) with Q = RA*CA = 1, and Fig. 2
 *                 (INT4 operands, INT32 result, dequantisation to FP16).
 *                 Section V-A with Q = RA*CA areas and section V-B (bitmap-
 *                 aware row reordering, Eq. 3-5, the grouped subset DP).
 *  [SPDP]         "Unified Static-Dynamic Pruning for Efficient LLM
 *                 Inference", section 4.1 "Tiled-CBC" (column tiles, values
 *                 in tile-column order, 4-byte TileOffset) and section 4.2.3
 *                 (16-byte value padding), section 2 (static mask W (.) M,
 *                 dynamic mask W (.) M(x)).
 *
 * Readings taken where the pages leave a step open (all are listed in the
 * design notes of the repository):
 *  - Tiles are TM x TK, numbered t = tm*nTK + tk (row-band major, like the
 *    row-major GTile order of [SPDP] 4.1).
 *  - Scan order inside a tile: ROW  p = i*TK + j  ([UnionSparse] "scanned in
 *    row-major order"), COL  p = j*TM + i  ([SPDP] column-major tiles).
 *  - Bit p%64 of 64-bit word p/64 of the tile; the earlier position is the
 *    less significant bit ([UnionSparse] "leftmost bit ... LSB").
 *  - Presence: a bit is set iff the stored weight is nonzero.  For fp16 both
 *    +0 and -0 count as zero; NaN counts as nonzero.
 *  - Values of tile t start at element tile_off[t], in increasing p; each
 *    tile's run is zero-padded to 16 bytes (8 fp16 or 32 int4 elements);
 *    tile_off[t+1] = tile_off[t] + roundup(P_t, E16) (in elements, uint32).
 *  - int4: element e lives in byte e>>1, even e in the low nibble, two's
 *    complement in [-8, 7].
 *  - W4A4 result: int32 acc = sum_k Wq*Xq; Y = fp16_rn((fp32(acc)*s_w)*s_x),
 *    two fp32 roundings then one round-to-nearest-even to fp16.
 *  - fp16 result: fp16_rn of the fp64 sum over increasing k.
 *  - spMspV: column k takes part iff |x_k| > tau.
 *
 * Built with  gcc -O2 -ffp-contract=off -fopenmp  (scalar loops only; the
 * OpenMP pragmas split independent output rows and never change the order
 * of any sum).
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#include <math.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_OK = 0, OR_BAD_ARG = 1, OR_TOO_LARGE = 3, OR_CAPACITY = 4, OR_CORRUPT = 7 };
enum { OR_F16 = 0, OR_I4 = 1, OR_I2 = 2 };
enum { OR_ROW = 0, OR_COL = 1 };

/* ---------------------------------------------------------------- fp16 ---- */
/* IEEE-754 binary16 <-> binary32/64 through the compiler's _Float16 type
 * (exact widening; narrowing is one round-to-nearest-even). */
float or_half_to_float(uint16_t h) {
    _Float16 v;
    memcpy(&v, &h, 2);
    return (float)v;
}
uint16_t or_float_to_half(float f) {
    _Float16 v = (_Float16)f;
    uint16_t h;
    memcpy(&h, &v, 2);
    return h;
}
uint16_t or_double_to_half(double d) {
    _Float16 v = (_Float16)d;
    uint16_t h;
    memcpy(&h, &v, 2);
    return h;
}

/* ------------------------------------------------------------- format ---- */
static int elem_bits(int elem) { return elem == OR_F16 ? 16 : (elem == OR_I4 ? 4 : 2); }
/* elements per 16-byte padding quantum */
static int elems_per_16B(int elem) { return 128 / elem_bits(elem); }

static int check_shape(int M, int K, int TM, int TK, int elem, int order) {
    if (M <= 0 || K <= 0 || TM <= 0 || TK <= 0) return OR_BAD_ARG;
    if (M % TM || K % TK) return OR_BAD_ARG;
    if (((int64_t)TM * TK) % 64) return OR_BAD_ARG;
    if (elem != OR_F16 && elem != OR_I4 && elem != OR_I2) return OR_BAD_ARG;
    if (order != OR_ROW && order != OR_COL) return OR_BAD_ARG;
    if ((uint64_t)M * (uint64_t)K >= ((uint64_t)1 << 32)) return OR_TOO_LARGE;
    return OR_OK;
}

/* position p inside a TM x TK tile -> (row i, column j) */
static void pos_to_ij(int order, int TM, int TK, int64_t p, int* i, int* j) {
    if (order == OR_ROW) { *i = (int)(p / TK); *j = (int)(p % TK); }
    else                 { *j = (int)(p / TM); *i = (int)(p % TM); }
}

int or_num_tiles(int M, int K, int TM, int TK, int64_t* nT) {
    int rc = check_shape(M, K, TM, TK, OR_F16, OR_ROW);
    if (rc) return rc;
    *nT = (int64_t)(M / TM) * (K / TK);
    return OR_OK;
}

/* read element (r, c) of the dense matrix as "is it nonzero" and as a code */
static int dense_nonzero(const void* W, int64_t ldw, int elem, int r, int c) {
    if (elem == OR_F16) {
        uint16_t h = ((const uint16_t*)W)[(int64_t)r * ldw + c];
        return (h & 0x7FFFu) != 0;           /* +0 and -0 are zero */
    }
    return ((const int8_t*)W)[(int64_t)r * ldw + c] != 0;
}

static void put_value(uint8_t* values, int elem, uint64_t e, const void* W, int64_t ldw, int r, int c) {
    if (elem == OR_F16) {
        uint16_t h = ((const uint16_t*)W)[(int64_t)r * ldw + c];
        values[2 * e] = (uint8_t)(h & 0xFF);
        values[2 * e + 1] = (uint8_t)(h >> 8);
    } else if (elem == OR_I4) {
        int8_t q = ((const int8_t*)W)[(int64_t)r * ldw + c];
        uint8_t nib = (uint8_t)q & 0x0F;
        if (e & 1) values[e >> 1] = (uint8_t)((values[e >> 1] & 0x0F) | (nib << 4));
        else       values[e >> 1] = (uint8_t)((values[e >> 1] & 0xF0) | nib);
    } else {
        /* int2 (W2A4, a reading of UnionSparse Fig. 11): element e in bits
         * 2(e%4) .. 2(e%4)+1 of byte e/4, two's complement in [-2, 1] */
        int8_t q = ((const int8_t*)W)[(int64_t)r * ldw + c];
        const int sh = 2 * (int)(e & 3);
        values[e >> 2] = (uint8_t)((values[e >> 2] & ~(3u << sh)) | (((uint8_t)q & 3u) << sh));
    }
}

/* zero element e of the packed stream (padding) */
static void zero_value(uint8_t* values, int elem, uint64_t e) {
    if (elem == OR_F16) { values[2 * e] = 0; values[2 * e + 1] = 0; }
    else if (elem == OR_I4) values[e >> 1] &= (e & 1) ? 0x0F : 0xF0;
    else values[e >> 2] &= (uint8_t)~(3u << (2 * (e & 3)));
}

/*
 * Encode a dense matrix into bitmap tiles.
 * [UnionSparse] V-A: the mask of tile t is scanned in the tile's scan order
 * and packed into 64-bit words (earlier position = less significant bit);
 * the compact rank of a set position is the number of set positions before
 * it; value with rank rho of tile t sits at CV[o_t + rho]; o_t is the prefix
 * sum of the preceding tiles' payload lengths (Q = 1).  [SPDP] 4.2.3: each
 * tile's payload is padded to 16 bytes.
 * W: fp16 bit patterns (elem F16) or int8 codes in [-8,7] (elem I4),
 * row-major with leading dimension ldw.
 * Outputs: bitmap (nT*TM*TK/64 words), tile_off (nT+1 entries),
 * values (capacity values_cap bytes; used bytes returned).
 */
int or_encode(const void* W, int64_t ldw, int M, int K, int TM, int TK, int elem, int order,
              uint64_t* bitmap, uint32_t* tile_off, uint8_t* values, uint64_t values_cap,
              uint64_t* values_used) {
    int rc = check_shape(M, K, TM, TK, elem, order);
    if (rc) return rc;
    if (ldw < K) return OR_BAD_ARG;
    const int nTM = M / TM, nTK = K / TK;
    const int64_t tile_pos = (int64_t)TM * TK;
    const int64_t words_per_tile = tile_pos / 64;
    const int E = elems_per_16B(elem);
    if (elem != OR_F16) {
        const int lo = elem == OR_I4 ? -8 : -2, hi = elem == OR_I4 ? 7 : 1;
        for (int r = 0; r < M; ++r)
            for (int c = 0; c < K; ++c) {
                int8_t q = ((const int8_t*)W)[(int64_t)r * ldw + c];
                if (q < lo || q > hi) return OR_BAD_ARG;
            }
    }
    uint64_t off = 0;                      /* in elements */
    tile_off[0] = 0;
    for (int tm = 0; tm < nTM; ++tm) {
        for (int tk = 0; tk < nTK; ++tk) {
            const int64_t t = (int64_t)tm * nTK + tk;
            uint64_t* words = bitmap + t * words_per_tile;
            for (int64_t w = 0; w < words_per_tile; ++w) words[w] = 0;
            uint64_t P = 0;                /* active entries of this tile */
            for (int64_t p = 0; p < tile_pos; ++p) {
                int i, j;
                pos_to_ij(order, TM, TK, p, &i, &j);
                const int r = tm * TM + i, c = tk * TK + j;
                if (!dense_nonzero(W, ldw, elem, r, c)) continue;
                words[p / 64] |= (uint64_t)1 << (p % 64);
                const uint64_t e = off + P;               /* o_t + rho */
                if ((e + 1) * elem_bits(elem) > values_cap * 8) return OR_CAPACITY;
                put_value(values, elem, e, W, ldw, r, c);
                ++P;
            }
            /* zero padding up to the next 16-byte boundary */
            uint64_t padded = (P + E - 1) / E * E;
            for (uint64_t e = off + P; e < off + padded; ++e) {
                if ((e + 1) * elem_bits(elem) > values_cap * 8) return OR_CAPACITY;
                zero_value(values, elem, e);
            }
            off += padded;
            if (off >= ((uint64_t)1 << 32)) return OR_TOO_LARGE;
            tile_off[t + 1] = (uint32_t)off;
        }
    }
    *values_used = off * elem_bits(elem) / 8;
    return OR_OK;
}

/* value with element index e of the packed stream, as fp16 bits or int4 code */
static uint16_t get_f16(const uint8_t* values, uint64_t e) {
    return (uint16_t)(values[2 * e] | (values[2 * e + 1] << 8));
}
static int8_t get_i2(const uint8_t* values, uint64_t e) {
    const unsigned c = (values[e >> 2] >> (2 * (e & 3))) & 3u;
    return (int8_t)(c >= 2 ? (int)c - 4 : (int)c);
}
static int8_t get_i4(const uint8_t* values, uint64_t e) {
    uint8_t nib = (e & 1) ? (values[e >> 1] >> 4) : (values[e >> 1] & 0x0F);
    return (int8_t)(nib >= 8 ? (int)nib - 16 : (int)nib);
}

/*
 * Decode (exact inverse of or_encode).  Every set position (i,j) of tile t
 * takes value CV[o_t + rho_t(i,j)], rho = number of set positions scanned
 * before it ([UnionSparse] V-A, "Compressed Values"); clear positions are 0.
 * Checks that each tile's run holds its popcount and lies inside the buffer.
 */
int or_decode(const uint64_t* bitmap, const uint32_t* tile_off, const uint8_t* values,
              uint64_t values_bytes, int M, int K, int TM, int TK, int elem, int order,
              void* W, int64_t ldw) {
    int rc = check_shape(M, K, TM, TK, elem, order);
    if (rc) return rc;
    const int nTM = M / TM, nTK = K / TK;
    const int64_t tile_pos = (int64_t)TM * TK;
    const int64_t words_per_tile = tile_pos / 64;
    if (tile_off[0] != 0) return OR_CORRUPT;
    for (int tm = 0; tm < nTM; ++tm) {
        for (int tk = 0; tk < nTK; ++tk) {
            const int64_t t = (int64_t)tm * nTK + tk;
            const uint64_t o_t = tile_off[t], o_next = tile_off[t + 1];
            if (o_next < o_t) return OR_CORRUPT;
            if (o_next * elem_bits(elem) > values_bytes * 8) return OR_CORRUPT;
            const uint64_t* words = bitmap + t * words_per_tile;
            uint64_t rho = 0;
            for (int64_t p = 0; p < tile_pos; ++p) {
                int i, j;
                pos_to_ij(order, TM, TK, p, &i, &j);
                const int64_t idx = (int64_t)(tm * TM + i) * ldw + (tk * TK + j);
                const int set = (int)((words[p / 64] >> (p % 64)) & 1u);
                if (set) {
                    if (o_t + rho >= o_next) return OR_CORRUPT;
                    if (elem == OR_F16) ((uint16_t*)W)[idx] = get_f16(values, o_t + rho);
                    else if (elem == OR_I4) ((int8_t*)W)[idx] = get_i4(values, o_t + rho);
                    else ((int8_t*)W)[idx] = get_i2(values, o_t + rho);
                    ++rho;
                } else {
                    if (elem == OR_F16) ((uint16_t*)W)[idx] = 0;
                    else ((int8_t*)W)[idx] = 0;
                }
            }
        }
    }
    return OR_OK;
}

/* int4 codes packed two per byte (even index in the low nibble) -> int8 */
void or_unpack_int4(const uint8_t* packed, int64_t n, int8_t* out) {
    for (int64_t e = 0; e < n; ++e) out[e] = get_i4(packed, (uint64_t)e);
}

/* ----------------------------------------------------------- multiply ---- */
/* one W4A4 output: int32 accumulation over increasing k, then dequantise
 * ([UnionSparse] Fig. 2: INT4 x INT4 -> Y INT32 -> Dequant -> FP16). */
static int32_t w4a4_acc(const int8_t* Wd, const int8_t* Xd, int K, int m, int n) {
    int64_t acc = 0;
    for (int k = 0; k < K; ++k)
        acc += (int64_t)Wd[(int64_t)m * K + k] * (int64_t)Xd[(int64_t)n * K + k];
    return (int32_t)acc;   /* |acc| <= 64*K < 2^31 for every supported K */
}
static uint16_t w4a4_dequant(int32_t acc, uint16_t s_w, uint16_t s_x) {
    float a = (float)acc;                  /* exact: |acc| < 2^24 */
    float t = a * or_half_to_float(s_w);   /* fp32 rounding 1 */
    float u = t * or_half_to_float(s_x);   /* fp32 rounding 2 */
    return or_float_to_half(u);            /* fp16 rounding */
}

/* Wd: M x K int8 codes (decoded), Xd: N x K int8 codes (token-major).
 * Yacc: N x M int32, Y: N x M fp16 bits (may be NULL). */
int or_spmm_w4a4(const int8_t* Wd, const int8_t* Xd, const uint16_t* s_w, const uint16_t* s_x,
                 int M, int N, int K, int32_t* Yacc, uint16_t* Y, int nthreads) {
    if (M <= 0 || N <= 0 || K <= 0) return OR_BAD_ARG;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(static)
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n) {
            int32_t acc = w4a4_acc(Wd, Xd, K, m, n);
            Yacc[(int64_t)n * M + m] = acc;
            if (Y) Y[(int64_t)n * M + m] = w4a4_dequant(acc, s_w[m], s_x[n]);
        }
    return OR_OK;
}

/* the same outputs, only at the listed (n, m) pairs */
int or_spmm_w4a4_at(const int8_t* Wd, const int8_t* Xd, const uint16_t* s_w, const uint16_t* s_x,
                    int M, int N, int K, const int32_t* n_idx, const int32_t* m_idx, int64_t count,
                    int32_t* acc_out, uint16_t* y_out) {
    for (int64_t q = 0; q < count; ++q) {
        int n = n_idx[q], m = m_idx[q];
        if (n < 0 || n >= N || m < 0 || m >= M) return OR_BAD_ARG;
        acc_out[q] = w4a4_acc(Wd, Xd, K, m, n);
        y_out[q] = w4a4_dequant(acc_out[q], s_w[m], s_x[n]);
    }
    return OR_OK;
}

/* one fp16 output: fp64 sum over increasing k of exact fp16 products */
static double f16_dot(const uint16_t* Wd, const uint16_t* X, int K, int m, int n, double tau, int skip) {
    double s = 0.0;
    for (int k = 0; k < K; ++k) {
        double x = (double)or_half_to_float(X[(int64_t)n * K + k]);
        if (skip && !(fabs(x) > tau)) continue;     /* dynamic mask M(x) */
        double w = (double)or_half_to_float(Wd[(int64_t)m * K + k]);
        s += w * x;
    }
    return s;
}

/* Wd: M x K fp16 (decoded), X: N x K fp16 token-major, Y: N x M fp16 */
int or_spmm_f16(const uint16_t* Wd, const uint16_t* X, int M, int N, int K, uint16_t* Y, int nthreads) {
    if (M <= 0 || N <= 0 || K <= 0) return OR_BAD_ARG;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(static)
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n)
            Y[(int64_t)n * M + m] = or_double_to_half(f16_dot(Wd, X, K, m, n, 0.0, 0));
    return OR_OK;
}

int or_spmm_f16_at(const uint16_t* Wd, const uint16_t* X, int M, int N, int K,
                   const int32_t* n_idx, const int32_t* m_idx, int64_t count, uint16_t* y_out,
                   double* exact_out) {
    for (int64_t q = 0; q < count; ++q) {
        int n = n_idx[q], m = m_idx[q];
        if (n < 0 || n >= N || m < 0 || m >= M) return OR_BAD_ARG;
        double s = f16_dot(Wd, X, K, m, n, 0.0, 0);
        if (exact_out) exact_out[q] = s;
        y_out[q] = or_double_to_half(s);
    }
    return OR_OK;
}

/* spMspV ([SPDP] section 2 and 4.2): y = (W (.) M) . (x (.) M(x)), where
 * column k is active iff |x_k| > tau; inactive columns are skipped. */
int or_spmspv_f16(const uint16_t* Wd, const uint16_t* x, float tau, int M, int K, uint16_t* y,
                  double* exact_out, int nthreads) {
    if (M <= 0 || K <= 0 || !(tau >= 0.0f)) return OR_BAD_ARG;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(static)
    for (int m = 0; m < M; ++m) {
        double s = f16_dot(Wd, x, K, m, 0, (double)tau, 1);
        if (exact_out) exact_out[m] = s;
        y[m] = or_double_to_half(s);
    }
    return OR_OK;
}

/* ------------------------------------------------ IE-BME with Q areas ---- */
/* [UnionSparse] V-A with Q = RA*CA > 1 (Fig. 7).  A local tile (LT) of TM x TK
 * is split into RA row partitions and CA column partitions; area q = a*CA + c
 * (a-th row partition, c-th column partition; the page leaves the numbering
 * of the areas open, this is the row-partition-major reading) covers rows
 * a*LM .. a*LM+LM-1 and columns c*LK .. c*LK+LK-1, LM = TM/RA, LK = TK/CA.
 * The logical union mask B_t(i,j) = OR_q [W_t^(q)(i,j) != 0] (LM x LK) is
 * scanned row-major and packed like the Q = 1 bitmap.  Every set logical
 * position emits one value per area, zeros included, with the same compact
 * rank rho: CV[o_t + q*P_t + rho] = W_t^(q)(i,j); the run of Q*P_t elements is
 * zero-padded to 16 bytes and o_{t+1} = o_t + roundup(Q*P_t).
 * Row reordering ([UnionSparse] V-B) acts before the areas are cut: perm (TM
 * bytes per tile, tile-major; NULL = identity) names for each row p of the
 * reordered tile the original row perm[t*TM + p] of that tile. */
static int check_ie(int M, int K, int TM, int TK, int RA, int CA, int elem) {
    if (M <= 0 || K <= 0 || TM <= 0 || TK <= 0 || RA <= 0 || CA <= 0) return OR_BAD_ARG;
    if (M % TM || K % TK || TM % RA || TK % CA || TM > 256) return OR_BAD_ARG;
    if (((int64_t)(TM / RA) * (TK / CA)) % 64) return OR_BAD_ARG;
    if (elem != OR_F16 && elem != OR_I4) return OR_BAD_ARG;
    if ((uint64_t)M * (uint64_t)K >= ((uint64_t)1 << 32)) return OR_TOO_LARGE;
    return OR_OK;
}

static int perm_row(const uint8_t* perm, int64_t t, int TM, int p) {
    return perm ? (int)perm[t * TM + p] : p;
}

int or_encode_ie(const void* W, int64_t ldw, int M, int K, int TM, int TK, int RA, int CA, int elem,
                 const uint8_t* perm, uint64_t* bitmap, uint32_t* tile_off, uint8_t* values,
                 uint64_t values_cap, uint64_t* values_used) {
    int rc = check_ie(M, K, TM, TK, RA, CA, elem);
    if (rc) return rc;
    if (ldw < K) return OR_BAD_ARG;
    const int nTM = M / TM, nTK = K / TK, Q = RA * CA, LM = TM / RA, LK = TK / CA;
    const int64_t lpos = (int64_t)LM * LK, words_per_tile = lpos / 64;
    const int E = elems_per_16B(elem);
    if (elem == OR_I4) {
        for (int r = 0; r < M; ++r)
            for (int c = 0; c < K; ++c) {
                int8_t q = ((const int8_t*)W)[(int64_t)r * ldw + c];
                if (q < -8 || q > 7) return OR_BAD_ARG;
            }
    }
    if (perm) {                                  /* each tile's perm must be a permutation */
        for (int64_t t = 0; t < (int64_t)nTM * nTK; ++t) {
            uint8_t seen[256] = {0};
            for (int p = 0; p < TM; ++p) {
                if (perm[t * TM + p] >= TM || seen[perm[t * TM + p]]) return OR_BAD_ARG;
                seen[perm[t * TM + p]] = 1;
            }
        }
    }
    uint64_t off = 0;
    tile_off[0] = 0;
    for (int tm = 0; tm < nTM; ++tm) {
        for (int tk = 0; tk < nTK; ++tk) {
            const int64_t t = (int64_t)tm * nTK + tk;
            uint64_t* words = bitmap + t * words_per_tile;
            for (int64_t w = 0; w < words_per_tile; ++w) words[w] = 0;
            /* the union mask and P_t */
            uint64_t P = 0;
            for (int64_t p = 0; p < lpos; ++p) {
                const int i = (int)(p / LK), j = (int)(p % LK);
                int any = 0;
                for (int a = 0; a < RA; ++a)
                    for (int c = 0; c < CA; ++c) {
                        const int r = tm * TM + perm_row(perm, t, TM, a * LM + i);
                        any |= dense_nonzero(W, ldw, elem, r, tk * TK + c * LK + j);
                    }
                if (any) {
                    words[p / 64] |= (uint64_t)1 << (p % 64);
                    ++P;
                }
            }
            /* the Q aligned streams: CV[o_t + q P_t + rho] */
            uint64_t rho = 0;
            for (int64_t p = 0; p < lpos; ++p) {
                if (!((words[p / 64] >> (p % 64)) & 1u)) continue;
                const int i = (int)(p / LK), j = (int)(p % LK);
                for (int a = 0; a < RA; ++a)
                    for (int c = 0; c < CA; ++c) {
                        const int q = a * CA + c;
                        const uint64_t e = off + (uint64_t)q * P + rho;
                        if ((e + 1) * elem_bits(elem) > values_cap * 8) return OR_CAPACITY;
                        const int r = tm * TM + perm_row(perm, t, TM, a * LM + i);
                        put_value(values, elem, e, W, ldw, r, tk * TK + c * LK + j);
                    }
                ++rho;
            }
            const uint64_t len = (uint64_t)Q * P, padded = (len + E - 1) / E * E;
            for (uint64_t e = off + len; e < off + padded; ++e) {
                if ((e + 1) * elem_bits(elem) > values_cap * 8) return OR_CAPACITY;
                if (elem == OR_F16) { values[2 * e] = 0; values[2 * e + 1] = 0; }
                else if (e & 1) values[e >> 1] &= 0x0F;
                else values[e >> 1] &= 0xF0;
            }
            off += padded;
            if (off >= ((uint64_t)1 << 32)) return OR_TOO_LARGE;
            tile_off[t + 1] = (uint32_t)off;
        }
    }
    *values_used = off * elem_bits(elem) / 8;
    return OR_OK;
}

/* Decode (exact inverse of or_encode_ie): back to the original row order. */
int or_decode_ie(const uint64_t* bitmap, const uint32_t* tile_off, const uint8_t* values, uint64_t values_bytes,
                 int M, int K, int TM, int TK, int RA, int CA, int elem, const uint8_t* perm, void* W,
                 int64_t ldw) {
    int rc = check_ie(M, K, TM, TK, RA, CA, elem);
    if (rc) return rc;
    const int nTM = M / TM, nTK = K / TK, Q = RA * CA, LM = TM / RA, LK = TK / CA;
    const int64_t lpos = (int64_t)LM * LK, words_per_tile = lpos / 64;
    for (int tm = 0; tm < nTM; ++tm) {
        for (int tk = 0; tk < nTK; ++tk) {
            const int64_t t = (int64_t)tm * nTK + tk;
            const uint64_t* words = bitmap + t * words_per_tile;
            uint64_t P = 0;
            for (int64_t w = 0; w < words_per_tile; ++w) P += (uint64_t)__builtin_popcountll(words[w]);
            const uint64_t o0 = tile_off[t], o1 = tile_off[t + 1];
            if (o1 < o0 || (uint64_t)Q * P > o1 - o0 || o1 * elem_bits(elem) > values_bytes * 8) return OR_CORRUPT;
            uint64_t rho = 0;
            for (int64_t p = 0; p < lpos; ++p) {
                const int i = (int)(p / LK), j = (int)(p % LK);
                const int set = (words[p / 64] >> (p % 64)) & 1u;
                for (int a = 0; a < RA; ++a)
                    for (int c = 0; c < CA; ++c) {
                        const int r = tm * TM + perm_row(perm, t, TM, a * LM + i);
                        const int64_t idx = (int64_t)r * ldw + tk * TK + c * LK + j;
                        const uint64_t e = o0 + (uint64_t)(a * CA + c) * P + rho;
                        if (elem == OR_F16) ((uint16_t*)W)[idx] = set ? get_f16(values, e) : 0;
                        else ((int8_t*)W)[idx] = set ? get_i4(values, e) : 0;
                    }
                rho += (uint64_t)set;
            }
        }
    }
    return OR_OK;
}

/* Bitmap-aware row reordering of one local tile ([UnionSparse] V-B, Eq. 3-5,
 * Algorithm 1).  mask: HL x KL bytes (nonzero = nonzero weight).  Rows are
 * partitioned into groups of RA; a group r = (r_0 .. r_{RA-1}) activates, at
 * grouped column j < KL/CA, phi(r;j) = OR_a OR_c mask[r_a][j + c*KL/CA], and
 * costs c(r) = sum_j phi(r;j).  F(S) = min over groups r in S holding the
 * smallest row of S of c(r) + F(S \ r), F(empty) = 0, memoised over row
 * subsets.  The optimal groups are canonicalised (rows ascending inside a
 * group, groups in lexicographic order) and the permutation is built
 * partition-wise: perm[p*(HL/RA) + g] = r_{g,p}.  HL <= 20.  Returns the
 * minimum cost in *cost. */
static int group_cost(const uint8_t* mask, int KL, int RA, int CA, const int* rows) {
    const int LK = KL / CA;
    int cost = 0;
    for (int j = 0; j < LK; ++j) {
        int any = 0;
        for (int a = 0; a < RA; ++a)
            for (int c = 0; c < CA; ++c) any |= mask[rows[a] * KL + c * LK + j] != 0;
        cost += any;
    }
    return cost;
}

typedef struct {
    const uint8_t* mask;
    int HL, KL, RA, CA;
    int32_t* F;                    /* memo, -1 = unknown */
    uint32_t* choice;              /* best group (as a row set) of each state */
} reorder_ctx;

static int32_t dp_solve(reorder_ctx* x, uint32_t S) {
    if (S == 0) return 0;
    if (x->F[S] >= 0) return x->F[S];
    int pivot = 0;
    while (!((S >> pivot) & 1u)) ++pivot;
    /* the other RA-1 rows of the group: every (RA-1)-subset of S without the pivot */
    int others[32], no = 0;
    for (int r = pivot + 1; r < x->HL; ++r)
        if ((S >> r) & 1u) others[no++] = r;
    int32_t best = INT32_MAX;
    uint32_t best_g = 0;
    int idx[4] = {0, 1, 2, 3};
    const int need = x->RA - 1;
    if (need > no) return INT32_MAX;
    for (;;) {
        int rows[4];
        uint32_t g = 1u << pivot;
        rows[0] = pivot;
        for (int k = 0; k < need; ++k) {
            rows[k + 1] = others[idx[k]];
            g |= 1u << others[idx[k]];
        }
        const int32_t rest = dp_solve(x, S & ~g);
        if (rest != INT32_MAX) {
            const int32_t v = group_cost(x->mask, x->KL, x->RA, x->CA, rows) + rest;
            if (v < best) { best = v; best_g = g; }
        }
        /* next combination of `need` indices out of `no` */
        int k = need - 1;
        while (k >= 0 && idx[k] == no - need + k) --k;
        if (k < 0) break;
        ++idx[k];
        for (int m = k + 1; m < need; ++m) idx[m] = idx[m - 1] + 1;
    }
    x->F[S] = best;
    x->choice[S] = best_g;
    return best;
}

int or_reorder_rows(const uint8_t* mask, int HL, int KL, int RA, int CA, uint8_t* perm, int* cost) {
    if (!mask || !perm || HL <= 0 || HL > 20 || KL <= 0 || RA <= 0 || RA > 4 || CA <= 0) return OR_BAD_ARG;
    if (HL % RA || KL % CA) return OR_BAD_ARG;
    reorder_ctx x;
    x.mask = mask; x.HL = HL; x.KL = KL; x.RA = RA; x.CA = CA;
    const size_t ns = (size_t)1 << HL;
    x.F = (int32_t*)malloc(ns * sizeof(int32_t));
    x.choice = (uint32_t*)malloc(ns * sizeof(uint32_t));
    if (!x.F || !x.choice) { free(x.F); free(x.choice); return OR_TOO_LARGE; }
    for (size_t i = 0; i < ns; ++i) x.F[i] = -1;
    const uint32_t all = (uint32_t)(ns - 1);
    const int32_t best = dp_solve(&x, all);
    /* recover the groups, rows ascending inside each (the pivot comes first and
     * the others were enumerated in increasing order) */
    const int G = HL / RA;
    int groups[20][4];
    uint32_t S = all;
    for (int g = 0; g < G; ++g) {
        const uint32_t gs = x.choice[S];
        int k = 0;
        for (int r = 0; r < HL; ++r)
            if ((gs >> r) & 1u) groups[g][k++] = r;
        S &= ~gs;
    }
    /* groups in lexicographic order (insertion sort) */
    for (int a = 1; a < G; ++a)
        for (int b = a; b > 0; --b) {
            int less = 0;
            for (int k = 0; k < RA; ++k)
                if (groups[b][k] != groups[b - 1][k]) { less = groups[b][k] < groups[b - 1][k]; break; }
            if (!less) break;
            for (int k = 0; k < RA; ++k) { int t = groups[b][k]; groups[b][k] = groups[b - 1][k]; groups[b - 1][k] = t; }
        }
    for (int p = 0; p < RA; ++p)
        for (int g = 0; g < G; ++g) perm[p * G + g] = (uint8_t)groups[g][p];
    if (cost) *cost = best;
    free(x.F);
    free(x.choice);
    return OR_OK;
}

/* ColInfo ([SPDP] section 4.1, Tiled-CBC storage structure): for a COL-order
 * matrix, one 32-bit word per column of every tile, tile-major
 * (colinfo[t*TK + j]); the upper 16 bits hold the column's starting offset
 * inside the tile's value run (TileOffset_Col: the nonzeros of the columns
 * before it in the same tile), the lower 16 bits its number of nonzeros
 * (NNZ_Column).  Read off the bitmap one position at a time. */
int or_colinfo(const uint64_t* bitmap, int M, int K, int TM, int TK, uint32_t* colinfo) {
    int64_t nT;
    int rc = or_num_tiles(M, K, TM, TK, &nT);
    if (rc != OR_OK) return rc;
    if (!bitmap || !colinfo) return OR_BAD_ARG;
    const int64_t words = (int64_t)TM * TK / 64;
    for (int64_t t = 0; t < nT; ++t) {
        const uint64_t* bm = bitmap + t * words;
        uint32_t offset = 0;
        for (int j = 0; j < TK; ++j) {
            uint32_t nnz = 0;
            for (int i = 0; i < TM; ++i) {
                const int64_t pos = (int64_t)j * TM + i;          /* COL scan: p = j*TM + i */
                if ((bm[pos / 64] >> (pos % 64)) & 1u) ++nnz;
            }
            colinfo[t * TK + j] = (offset << 16) | nnz;
            offset += nnz;
        }
    }
    return OR_OK;
}

/* ------------------------------------------- activation quantisation ---- */
/* Per-token symmetric int4 quantisation of fp16 activations ([UnionSparse]
 * Fig. 2, the "Quant" step between FP16 X and INT4 X; the page fixes the
 * per-token scale, not its rounding, so the plain reading is used):
 *   amax = max_k |x[n][k]|                       (fp16 values are exact in fp32)
 *   s_x[n] = fp16_rn(amax / 7)                   (fp32 division), 1 if that is 0
 *   code[n][k] = clamp(rint(x[n][k] / s_x[n]), -8, 7)
 *                                                (fp32 division, ties to even)
 * NaN inputs do not take part in amax and give code 0. */
int or_quantize_x(const uint16_t* X, int N, int K, int8_t* codes, uint16_t* s_x) {
    if (N < 0 || K < 0 || (N * (int64_t)K > 0 && (!X || !codes || !s_x))) return OR_BAD_ARG;
    for (int n = 0; n < N; ++n) {
        const uint16_t* x = X + (int64_t)n * K;
        float amax = 0.0f;
        for (int k = 0; k < K; ++k) {
            const float a = fabsf(or_half_to_float(x[k]));
            if (a > amax) amax = a;             /* NaN compares false */
        }
        uint16_t s16 = or_float_to_half(amax / 7.0f);
        if ((s16 & 0x7FFFu) == 0) s16 = 0x3C00u;   /* 1.0 */
        s_x[n] = s16;
        const float s = or_half_to_float(s16);
        for (int k = 0; k < K; ++k) {
            const float v = or_half_to_float(x[k]);
            float q = rintf(v / s);             /* default rounding mode: to nearest even */
            if (!(q == q)) q = 0.0f;
            if (q < -8.0f) q = -8.0f;
            if (q > 7.0f) q = 7.0f;
            codes[(int64_t)n * K + k] = (int8_t)q;
        }
    }
    return OR_OK;
}

int or_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
