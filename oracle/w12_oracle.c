/*
 * W12 oracle — TEST INFRASTRUCTURE ONLY (see w12_oracle.h).
 *
 * Plain scalar restatement of the W12 v1 format.  Every loop visits one weight
 * (or one table slot) at a time, in the order the format definition states:
 *   step 1  split each BF16 pattern into sign, exponent, mantissa;
 *   step 2  per segment (128 rows x 256 columns) build the exponent histogram
 *           and take the 15 most frequent exponents into the table;
 *   step 3  give each weight the code of its exponent, or the escape code 15
 *           with the raw exponent appended to the escape list;
 *   step 4  write the header, the segment headers, the packed chunks and the
 *           escape list at their offsets.
 * Sources: "StargazerX0/SpecPilot" (hotrepo.ai) §What it is (12-bit, decodes
 * bit-exactly inside the GEMM); "SpecPilot" (fasttoolhub.com) §Differentiation
 * (general lossless 12-bit format); "SpecPilot: an agent doubled speculative
 * decoding speed, and the 10.87x needs context" (ai.jakubjirak.com) §The
 * mechanisms it found (~12.01-12.02 bits/weight; a quarter less traffic).
 * The byte layout itself is build-defined; the pages give none.
 */
#include "w12_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- geometry of W12 v1 (restated here; nothing is shared with the library) */
enum {
    O_TILE_ROWS = 128,   /* rows per tile                              */
    O_QUARTER   = 32,    /* rows per quarter (escape ordering unit)    */
    O_CHUNK_K   = 32,    /* columns per packed chunk                   */
    O_SEG_K     = 256,   /* columns per segment (one exponent table)   */
    O_CHUNK_B   = 6144,  /* bytes per packed chunk: 3 slabs x 128 x 16 */
    O_SEGHDR_B  = 32,    /* bytes per segment header                   */
    O_HDR_B     = 256    /* bytes of the blob header                   */
};

typedef struct {
    int64_t N, K, Np, Kp, tiles, chunks, segs;
    int64_t off_seghdr, bytes_seghdr, off_weights, bytes_weights, off_esc;
} o_geom;

static int64_t o_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

static void o_geometry(int64_t N, int64_t K, o_geom *g)
{
    g->N = N;
    g->K = K;
    g->Np = o_up(N, O_TILE_ROWS);
    g->Kp = o_up(K, O_CHUNK_K);
    g->tiles = g->Np / O_TILE_ROWS;
    g->chunks = g->Kp / O_CHUNK_K;
    g->segs = (g->Kp + O_SEG_K - 1) / O_SEG_K;
    g->off_seghdr = O_HDR_B;
    g->bytes_seghdr = (int64_t)O_SEGHDR_B * g->tiles * g->segs;
    g->off_weights = o_up(g->off_seghdr + g->bytes_seghdr, 256);
    g->bytes_weights = (int64_t)O_CHUNK_B * g->tiles * g->chunks;
    g->off_esc = o_up(g->off_weights + g->bytes_weights, 256);
}

static int64_t o_total(const o_geom *g, int64_t n_esc)
{
    return o_up(g->off_esc + o_up(n_esc, 16), 256);
}

/* Weight of the padded matrix: rows >= N and columns >= K are +0.0. */
static uint16_t o_w(const uint16_t *w, const o_geom *g, int64_t n, int64_t k)
{
    if (n >= g->N || k >= g->K)
        return 0;
    return w[n * g->K + k];
}

/* step 1: split a BF16 pattern */
static unsigned o_sign(uint16_t b) { return (unsigned)(b >> 15) & 1u; }
static unsigned o_expo(uint16_t b) { return (unsigned)(b >> 7) & 0xFFu; }
static unsigned o_mant(uint16_t b) { return (unsigned)b & 0x7Fu; }

static int64_t o_seg_k_end(const o_geom *g, int64_t seg)
{
    int64_t e = (seg + 1) * O_SEG_K;
    return e < g->Kp ? e : g->Kp;
}

/*
 * step 2: the exponent table of segment (tile t, segment s).
 *
 * Histogram the exponents of all 128 x (segment width) weights of the padded
 * matrix.  Candidates are the exponents that occur; they are ranked by count,
 * larger first, ties broken by the smaller exponent; the first min(15, #) are
 * selected.  The selected exponents are then placed into code slots 0..14 so
 * that slots j and j+8 (j = 0..6) always hold exponents with the same top bit;
 * slot 7 is paired with the escape slot 15, which always holds 0.  Placement:
 * L = selected exponents < 128 ascending, H = those >= 128 ascending, and the
 * slot visiting order is 7, 0, 8, 1, 9, 2, 10, 3, 11, 4, 12, 5, 13, 6, 14.
 *   |L| odd            : L then H, starting at the first slot of the order;
 *   |L| even, |H| odd  : H then L, starting at the first slot;
 *   both even          : L then H, starting at the second slot (slot 7 unused).
 * A slot left empty copies its pair partner if that one is filled, else 0.
 */
static void o_seg_table(const uint16_t *w, const o_geom *g, int64_t t,
                        int64_t s, uint8_t T[16])
{
    static const int order[15] = {7, 0, 8, 1, 9, 2, 10, 3, 11, 4, 12, 5, 13, 6, 14};
    int64_t hist[256];
    int used[256];
    int nsel = 0;
    int L[15], nL = 0, H[15], nH = 0, seq[15], nseq = 0;
    int filled[16];
    int start, i, e, slot;
    int64_t n, k;

    for (e = 0; e < 256; ++e) {
        hist[e] = 0;
        used[e] = 0;
    }
    for (n = t * O_TILE_ROWS; n < (t + 1) * O_TILE_ROWS; ++n)
        for (k = s * O_SEG_K; k < o_seg_k_end(g, s); ++k)
            hist[o_expo(o_w(w, g, n, k))] += 1;

    /* rank: repeatedly take the unused exponent with the largest count,
     * the smaller exponent winning a tie */
    while (nsel < 15) {
        int best = -1;
        for (e = 0; e < 256; ++e) {
            if (used[e] || hist[e] == 0)
                continue;
            if (best < 0 || hist[e] > hist[best])
                best = e;
        }
        if (best < 0)
            break;
        used[best] = 1;
        nsel += 1;
    }

    /* ascending lists of the selected exponents, split by the top bit */
    for (e = 0; e < 256; ++e) {
        if (!used[e])
            continue;
        if (e < 128)
            L[nL++] = e;
        else
            H[nH++] = e;
    }

    if (nL % 2 == 1) {
        for (i = 0; i < nL; ++i) seq[nseq++] = L[i];
        for (i = 0; i < nH; ++i) seq[nseq++] = H[i];
        start = 0;
    } else if (nH % 2 == 1) {
        for (i = 0; i < nH; ++i) seq[nseq++] = H[i];
        for (i = 0; i < nL; ++i) seq[nseq++] = L[i];
        start = 0;
    } else {
        for (i = 0; i < nL; ++i) seq[nseq++] = L[i];
        for (i = 0; i < nH; ++i) seq[nseq++] = H[i];
        start = 1;
    }

    for (slot = 0; slot < 16; ++slot) {
        T[slot] = 0;
        filled[slot] = 0;
    }
    for (i = 0; i < nseq; ++i) {
        slot = order[start + i];
        T[slot] = (uint8_t)seq[i];
        filled[slot] = 1;
    }
    for (slot = 0; slot < 15; ++slot) {
        int partner;
        if (filled[slot])
            continue;
        if (slot == 7)
            partner = 15;
        else
            partner = slot < 8 ? slot + 8 : slot - 8;
        T[slot] = filled[partner] ? T[partner] : 0;
    }
    T[15] = 0;
}

/* step 3: the code of exponent e is the first slot 0..14 that holds it;
 * an exponent held by no slot gets the escape code 15 */
static int o_code(const uint8_t T[16], unsigned e)
{
    int c;
    for (c = 0; c < 15; ++c)
        if (T[c] == e)
            return c;
    return 15;
}

/* Escapes of one segment, counted per quarter. */
static void o_seg_escapes(const uint16_t *w, const o_geom *g, int64_t t,
                          int64_t s, const uint8_t T[16], int64_t qcount[4])
{
    int q;
    int64_t n, k;
    for (q = 0; q < 4; ++q) {
        qcount[q] = 0;
        for (n = t * O_TILE_ROWS + q * O_QUARTER;
             n < t * O_TILE_ROWS + (q + 1) * O_QUARTER; ++n)
            for (k = s * O_SEG_K; k < o_seg_k_end(g, s); ++k)
                if (o_code(T, o_expo(o_w(w, g, n, k))) == 15)
                    qcount[q] += 1;
    }
}

int64_t oracle_w12_size(const uint16_t *w, int64_t N, int64_t K)
{
    o_geom g;
    int64_t t, s, n_esc = 0;
    uint8_t T[16];
    int64_t qc[4];
    if (w == NULL || N < 1 || K < 1)
        return -1;
    o_geometry(N, K, &g);
    for (t = 0; t < g.tiles; ++t)
        for (s = 0; s < g.segs; ++s) {
            o_seg_table(w, &g, t, s, T);
            o_seg_escapes(w, &g, t, s, T, qc);
            n_esc += qc[0] + qc[1] + qc[2] + qc[3];
        }
    return o_total(&g, n_esc);
}

/* ---- little-endian field access ----------------------------------------- */
static void o_put(uint8_t *p, uint64_t v, int nbytes)
{
    int i;
    for (i = 0; i < nbytes; ++i)
        p[i] = (uint8_t)(v >> (8 * i));
}

static uint64_t o_get(const uint8_t *p, int nbytes)
{
    uint64_t v = 0;
    int i;
    for (i = 0; i < nbytes; ++i)
        v |= (uint64_t)p[i] << (8 * i);
    return v;
}

/*
 * step 4: write the blob.
 *
 * Header (256 bytes): "W12B", version 1, header size, flags 0, N, K, padded
 * N and K, tile rows 128, chunk width 32, segment width 256, quarter rows 32,
 * tile / chunk / segment counts, offset and size of the segment-header plane,
 * of the packed-weight plane and of the escape plane, the escape count, the
 * escape-plane size and the total size.
 *
 * Segment header (32 bytes, tile-major): table T[16]; u32 offset of the
 * segment's first escape byte; u16 escape count of each quarter; u32 mask with
 * bit 8q+j set when quarter q has an escape in the segment's chunk j.
 *
 * Packed chunk (6144 bytes, tile-major, chunks in column order): for row r of
 * the tile, bytes 16r..16r+15 of slab 0 hold columns 0..15, slab 1 (offset
 * 2048) holds columns 16..31; each byte is (mantissa << 1) | sign of the pair
 * partner column (column index xor 1).  Slab 2 (offset 4096), bytes
 * 16r..16r+15, holds the 32 codes, even column in the low nibble.
 *
 * Escape list: one raw exponent byte per escaped weight, ordered by tile,
 * segment, quarter, chunk, row, column.
 */
int64_t oracle_w12_encode(const uint16_t *w, int64_t N, int64_t K,
                          uint8_t *blob, int64_t cap)
{
    o_geom g;
    int64_t total, t, s, esc_cursor = 0, n_esc;
    uint8_t T[16];

    total = oracle_w12_size(w, N, K);
    if (total < 0 || blob == NULL || cap < total)
        return -1;
    o_geometry(N, K, &g);
    memset(blob, 0, (size_t)total);

    for (t = 0; t < g.tiles; ++t) {
        for (s = 0; s < g.segs; ++s) {
            uint8_t *sh = blob + g.off_seghdr + O_SEGHDR_B * (t * g.segs + s);
            int64_t qc[4];
            uint32_t mask = 0;
            int q, c;
            int64_t n, k;

            o_seg_table(w, &g, t, s, T);
            o_seg_escapes(w, &g, t, s, T, qc);
            for (c = 0; c < 16; ++c)
                sh[c] = T[c];
            o_put(sh + 16, (uint64_t)esc_cursor, 4);
            for (q = 0; q < 4; ++q)
                o_put(sh + 20 + 2 * q, (uint64_t)qc[q], 2);

            /* escape list in its order: quarter, chunk, row, column */
            for (q = 0; q < 4; ++q) {
                int64_t j;
                for (j = s * O_SEG_K / O_CHUNK_K; j * O_CHUNK_K < o_seg_k_end(&g, s); ++j)
                    for (n = t * O_TILE_ROWS + q * O_QUARTER;
                         n < t * O_TILE_ROWS + (q + 1) * O_QUARTER; ++n)
                        for (k = j * O_CHUNK_K; k < (j + 1) * O_CHUNK_K; ++k) {
                            unsigned e = o_expo(o_w(w, &g, n, k));
                            if (o_code(T, e) == 15) {
                                blob[g.off_esc + esc_cursor] = (uint8_t)e;
                                esc_cursor += 1;
                                mask |= 1u << (8 * q + (int)(j - s * O_SEG_K / O_CHUNK_K));
                            }
                        }
            }
            o_put(sh + 28, mask, 4);

            /* packed chunks of this segment */
            for (n = t * O_TILE_ROWS; n < (t + 1) * O_TILE_ROWS; ++n) {
                int64_t r = n - t * O_TILE_ROWS;
                for (k = s * O_SEG_K; k < o_seg_k_end(&g, s); ++k) {
                    int64_t j = k / O_CHUNK_K, kk = k % O_CHUNK_K;
                    uint8_t *chunk = blob + g.off_weights + O_CHUNK_B * (t * g.chunks + j);
                    uint16_t b = o_w(w, &g, n, k);
                    uint16_t partner = o_w(w, &g, n, k ^ 1);
                    uint8_t sbyte = (uint8_t)((o_mant(b) << 1) | o_sign(partner));
                    int code = o_code(T, o_expo(b));
                    if (kk < 16)
                        chunk[16 * r + kk] = sbyte;
                    else
                        chunk[2048 + 16 * r + (kk - 16)] = sbyte;
                    chunk[4096 + 16 * r + kk / 2] |= (uint8_t)(code << (4 * (kk % 2)));
                }
            }
        }
    }
    n_esc = esc_cursor;

    /* header */
    memcpy(blob, "W12B", 4);
    o_put(blob + 0x04, 1, 4);
    o_put(blob + 0x08, O_HDR_B, 4);
    o_put(blob + 0x0C, 0, 4);
    o_put(blob + 0x10, (uint64_t)g.N, 8);
    o_put(blob + 0x18, (uint64_t)g.K, 8);
    o_put(blob + 0x20, (uint64_t)g.Np, 8);
    o_put(blob + 0x28, (uint64_t)g.Kp, 8);
    o_put(blob + 0x30, O_TILE_ROWS, 4);
    o_put(blob + 0x34, O_CHUNK_K, 4);
    o_put(blob + 0x38, O_SEG_K, 4);
    o_put(blob + 0x3C, O_QUARTER, 4);
    o_put(blob + 0x40, (uint64_t)g.tiles, 8);
    o_put(blob + 0x48, (uint64_t)g.chunks, 8);
    o_put(blob + 0x50, (uint64_t)g.segs, 8);
    o_put(blob + 0x58, (uint64_t)g.off_seghdr, 8);
    o_put(blob + 0x60, (uint64_t)g.bytes_seghdr, 8);
    o_put(blob + 0x68, (uint64_t)g.off_weights, 8);
    o_put(blob + 0x70, (uint64_t)g.bytes_weights, 8);
    o_put(blob + 0x78, (uint64_t)g.off_esc, 8);
    o_put(blob + 0x80, (uint64_t)n_esc, 8);
    o_put(blob + 0x88, (uint64_t)o_up(n_esc, 16), 8);
    o_put(blob + 0x90, (uint64_t)total, 8);
    return total;
}

/* Header check shared by the readers below: magic, version and that every
 * geometry field equals what N and K imply. */
static int o_read_header(const uint8_t *blob, int64_t len, o_geom *g,
                         int64_t *n_esc)
{
    int64_t N, K;
    if (blob == NULL || len < O_HDR_B || memcmp(blob, "W12B", 4) != 0)
        return -1;
    if (o_get(blob + 0x04, 4) != 1 || o_get(blob + 0x08, 4) != O_HDR_B)
        return -1;
    N = (int64_t)o_get(blob + 0x10, 8);
    K = (int64_t)o_get(blob + 0x18, 8);
    if (N < 1 || K < 1)
        return -1;
    o_geometry(N, K, g);
    *n_esc = (int64_t)o_get(blob + 0x80, 8);
    if ((int64_t)o_get(blob + 0x20, 8) != g->Np || (int64_t)o_get(blob + 0x28, 8) != g->Kp ||
        o_get(blob + 0x30, 4) != O_TILE_ROWS || o_get(blob + 0x34, 4) != O_CHUNK_K ||
        o_get(blob + 0x38, 4) != O_SEG_K || o_get(blob + 0x3C, 4) != O_QUARTER ||
        (int64_t)o_get(blob + 0x40, 8) != g->tiles || (int64_t)o_get(blob + 0x48, 8) != g->chunks ||
        (int64_t)o_get(blob + 0x50, 8) != g->segs ||
        (int64_t)o_get(blob + 0x58, 8) != g->off_seghdr ||
        (int64_t)o_get(blob + 0x60, 8) != g->bytes_seghdr ||
        (int64_t)o_get(blob + 0x68, 8) != g->off_weights ||
        (int64_t)o_get(blob + 0x70, 8) != g->bytes_weights ||
        (int64_t)o_get(blob + 0x78, 8) != g->off_esc ||
        (int64_t)o_get(blob + 0x88, 8) != o_up(*n_esc, 16) ||
        (int64_t)o_get(blob + 0x90, 8) != o_total(g, *n_esc) || len < o_total(g, *n_esc))
        return -1;
    return 0;
}

int oracle_w12_dims(const uint8_t *blob, int64_t len, int64_t *N, int64_t *K)
{
    o_geom g;
    int64_t n_esc;
    if (o_read_header(blob, len, &g, &n_esc) != 0)
        return -1;
    *N = g.N;
    *K = g.K;
    return 0;
}

/* Decode the tiles [t0, t1) of a blob into w_out (original N x K shape).
 * Every weight: sign from the pair partner's S byte, mantissa from its own S
 * byte, exponent from the table or, for code 15, the next byte of its
 * quarter's escape run. */
static int o_decode_tiles(const uint8_t *blob, const o_geom *g, int64_t n_esc,
                          int64_t t0, int64_t t1, uint16_t *w_out)
{
    int64_t t, s;
    for (t = t0; t < t1; ++t) {
        for (s = 0; s < g->segs; ++s) {
            const uint8_t *sh = blob + g->off_seghdr + O_SEGHDR_B * (t * g->segs + s);
            int64_t cursor = (int64_t)o_get(sh + 16, 4);
            int q;
            for (q = 0; q < 4; ++q) {
                int64_t j;
                for (j = s * O_SEG_K / O_CHUNK_K; j * O_CHUNK_K < o_seg_k_end(g, s); ++j) {
                    const uint8_t *chunk = blob + g->off_weights + O_CHUNK_B * (t * g->chunks + j);
                    int64_t n;
                    for (n = t * O_TILE_ROWS + q * O_QUARTER;
                         n < t * O_TILE_ROWS + (q + 1) * O_QUARTER; ++n) {
                        int64_t r = n - t * O_TILE_ROWS, kk;
                        for (kk = 0; kk < O_CHUNK_K; ++kk) {
                            int64_t k = j * O_CHUNK_K + kk, pk = kk ^ 1;
                            unsigned sb = kk < 16 ? chunk[16 * r + kk] : chunk[2048 + 16 * r + kk - 16];
                            unsigned sp = pk < 16 ? chunk[16 * r + pk] : chunk[2048 + 16 * r + pk - 16];
                            unsigned code = (chunk[4096 + 16 * r + kk / 2] >> (4 * (kk % 2))) & 0xFu;
                            unsigned mant = sb >> 1, sign = sp & 1u, e;
                            if (code == 15) {
                                if (cursor >= n_esc)
                                    return -1;
                                e = blob[g->off_esc + cursor];
                                cursor += 1;
                            } else {
                                e = sh[code];
                            }
                            if (n < g->N && k < g->K)
                                w_out[n * g->K + k] = (uint16_t)((sign << 15) | (e << 7) | mant);
                        }
                    }
                }
            }
        }
    }
    return 0;
}

int oracle_w12_decode(const uint8_t *blob, int64_t len, uint16_t *w_out)
{
    o_geom g;
    int64_t n_esc;
    if (w_out == NULL || o_read_header(blob, len, &g, &n_esc) != 0)
        return -1;
    return o_decode_tiles(blob, &g, n_esc, 0, g.tiles, w_out);
}

/* ---- GEMM in fp64 -------------------------------------------------------- */
static double o_bf16_to_double(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

void oracle_gemm_f64(const uint16_t *x, const uint16_t *w, int64_t M,
                     int64_t N, int64_t K, double *y)
{
    int64_t m, n, k;
    for (m = 0; m < M; ++m)
        for (n = 0; n < N; ++n) {
            double acc = 0.0;
            for (k = 0; k < K; ++k)
                acc += o_bf16_to_double(x[m * K + k]) * o_bf16_to_double(w[n * K + k]);
            y[m * N + n] = acc;
        }
}

int oracle_max_threads(int threads)
{
#ifdef _OPENMP
    return threads > 0 ? threads : omp_get_max_threads();
#else
    (void)threads;
    return 1;
#endif
}

int oracle_w12_gemm_f64(const uint16_t *x, const uint8_t *blob, int64_t len,
                        int64_t M, double *y, int threads)
{
    o_geom g;
    int64_t n_esc, t, n;
    uint16_t *w;
    int bad = 0;
    if (x == NULL || y == NULL || M < 1 || o_read_header(blob, len, &g, &n_esc) != 0)
        return -1;
    w = (uint16_t *)malloc((size_t)(g.N * g.K) * sizeof(uint16_t));
    if (w == NULL)
        return -1;
    threads = oracle_max_threads(threads);
    (void)threads;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads) reduction(| : bad)
#endif
    for (t = 0; t < g.tiles; ++t)
        bad |= o_decode_tiles(blob, &g, n_esc, t, t + 1, w) != 0;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(threads)
#endif
    for (n = 0; n < g.N; ++n) {
        int64_t m, k;
        for (m = 0; m < M; ++m) {
            double acc = 0.0;
            for (k = 0; k < g.K; ++k)
                acc += o_bf16_to_double(x[m * g.K + k]) * o_bf16_to_double(w[n * g.K + k]);
            y[m * g.N + n] = acc;
        }
    }
    free(w);
    return bad ? -1 : 0;
}

/* ======================================================================
 * Q8: the 8-bit weight copy used by the first level of a two-level
 * verification ("SpecPilot: an agent doubled speculative decoding speed, and
 * the 10.87x needs context", §The mechanisms it found, names a two-level
 * verification with an 8-bit or INT6/INT8 copy of the weights; the page gives
 * no scheme).  Reading taken: symmetric INT8 per output row.
 *   a[n] = max_k |W[n][k]|, s[n] = a[n] / 127 (fp32), q = rint(W / s) in fp32
 *   (nearest, ties to even), clamped to [-127, 127]; a zero row has s = 0 and
 *   q = 0.  A row holding Inf or NaN cannot be quantized (error).
 *   The product it feeds: y[m][n] = s[n] * sum_k x[m][k] * q[n][k].
 * Layout (Q8 v1): header 256 B | scales fp32[N_pad] (pad rows 0) | q plane,
 * each part 256-byte aligned.  q plane: per 128-row tile, per 32-column
 * chunk, two 2048-byte slabs of 128 rows x 16 bytes (columns 0-15, 16-31);
 * padded entries are 0.  Header: 0x00 "Q8W1", 0x04 u32 1, 0x08 u32 256,
 * 0x0C u32 0, 0x10 N, 0x18 K, 0x20 N_pad, 0x28 K_pad, 0x30 tiles, 0x38 chunks,
 * 0x40/0x48 scales offset/size, 0x50/0x58 q offset/size, 0x60 total.
 * ====================================================================== */

typedef struct {
    int64_t N, K, Npad, Kpad, tiles, chunks;
    int64_t off_s, bytes_s, off_q, bytes_q, total;
} o_q8geom;

static void o_q8_geometry(int64_t N, int64_t K, o_q8geom *g)
{
    g->N = N;
    g->K = K;
    g->Npad = o_up(N, 128);
    g->Kpad = o_up(K, 32);
    g->tiles = g->Npad / 128;
    g->chunks = g->Kpad / 32;
    g->off_s = 256;
    g->bytes_s = 4 * g->Npad;
    g->off_q = o_up(g->off_s + g->bytes_s, 256);
    g->bytes_q = 4096 * g->tiles * g->chunks;
    g->total = o_up(g->off_q + g->bytes_q, 256);
}

static float o_bf16_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

int64_t oracle_q8_size(int64_t N, int64_t K)
{
    o_q8geom g;
    if (N < 1 || K < 1)
        return -1;
    o_q8_geometry(N, K, &g);
    return g.total;
}

int64_t oracle_q8_encode(const uint16_t *w, int64_t N, int64_t K, uint8_t *blob, int64_t cap)
{
    o_q8geom g;
    int64_t n, k;
    if (!w || !blob || N < 1 || K < 1)
        return -1;
    o_q8_geometry(N, K, &g);
    if (cap < g.total)
        return -1;
    memset(blob, 0, (size_t)g.total);
    for (n = 0; n < N; ++n) {
        float a = 0.0f, s;
        for (k = 0; k < K; ++k) {
            float v = o_bf16_to_float(w[n * K + k]);
            if (!(v - v == 0.0f))
                return -1; /* Inf or NaN */
            if (fabsf(v) > a)
                a = fabsf(v);
        }
        s = a / 127.0f;
        memcpy(blob + g.off_s + 4 * n, &s, 4);
        for (k = 0; k < K; ++k) {
            int64_t t = n / 128, r = n % 128, c = k / 32, col = k % 32;
            float q = 0.0f;
            int qi;
            if (a > 0.0f) {
                q = rintf(o_bf16_to_float(w[n * K + k]) / s);
                if (q > 127.0f) q = 127.0f;
                if (q < -127.0f) q = -127.0f;
            }
            qi = (int)q;
            blob[g.off_q + 4096 * (t * g.chunks + c) + 2048 * (col / 16) + 16 * r + col % 16] = (uint8_t)(int8_t)qi;
        }
    }
    o_put(blob + 0x00, 0x31573851u, 4); /* "Q8W1" */
    o_put(blob + 0x04, 1, 4);
    o_put(blob + 0x08, 256, 4);
    o_put(blob + 0x10, (uint64_t)g.N, 8);
    o_put(blob + 0x18, (uint64_t)g.K, 8);
    o_put(blob + 0x20, (uint64_t)g.Npad, 8);
    o_put(blob + 0x28, (uint64_t)g.Kpad, 8);
    o_put(blob + 0x30, (uint64_t)g.tiles, 8);
    o_put(blob + 0x38, (uint64_t)g.chunks, 8);
    o_put(blob + 0x40, (uint64_t)g.off_s, 8);
    o_put(blob + 0x48, (uint64_t)g.bytes_s, 8);
    o_put(blob + 0x50, (uint64_t)g.off_q, 8);
    o_put(blob + 0x58, (uint64_t)g.bytes_q, 8);
    o_put(blob + 0x60, (uint64_t)g.total, 8);
    return g.total;
}

int oracle_q8_decode(const uint8_t *blob, int64_t len, float *scales, int8_t *q)
{
    o_q8geom g;
    int64_t N, K, n, k;
    if (!blob || len < 256 || o_get(blob, 4) != 0x31573851u || o_get(blob + 4, 4) != 1)
        return -1;
    N = (int64_t)o_get(blob + 0x10, 8);
    K = (int64_t)o_get(blob + 0x18, 8);
    if (N < 1 || K < 1)
        return -1;
    o_q8_geometry(N, K, &g);
    if ((int64_t)o_get(blob + 0x60, 8) != g.total || len < g.total ||
        (int64_t)o_get(blob + 0x50, 8) != g.off_q)
        return -1;
    for (n = 0; n < N; ++n) {
        memcpy(&scales[n], blob + g.off_s + 4 * n, 4);
        for (k = 0; k < K; ++k) {
            int64_t t = n / 128, r = n % 128, c = k / 32, col = k % 32;
            q[n * K + k] = (int8_t)blob[g.off_q + 4096 * (t * g.chunks + c) + 2048 * (col / 16) + 16 * r + col % 16];
        }
    }
    return 0;
}
