/*
 * mmq_oracle.c -- plain, slow, obviously correct CPU reference for the prefill
 * quantized matrix multiply (MMQ) of k-quant weight super-blocks (q6_K, q4_K)
 * against per-32 q8 activations.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the CPU
 * baseline leg of bench.py may load or run this library.  It shares no code,
 * header, table or helper with the CUDA path, and never includes anything from
 * it.  Build: gcc -O2 -ffp-contract=off (IEEE single rounding per operation, no
 * fast-math, no FMA contraction).
 *
 * Sources (page title, section):
 *   [r45] "r45 - cp.async for the q6_K A-side staging: mechanism confirmed,
 *          wall-neutral (REVERTED)"
 *   [r56] "r56 - q6_K A-side bundle: A cp.async + W_dsc f32 plane (LANDED)"
 *   [r58] "r58 - q4_K BT spec + cp.async-db2 transplant (REVERTED)"
 *
 * The result the method reaches has a plain closed form,
 *     Y[t,j] = sum_k a[t,k] * w[j,k]
 * with a = d_a * q_a (per 32-element activation chunk) and w the decoded
 * weight; the oracle evaluates it the way the pages state it: an integer dot
 * per sub-block, scaled by the f32 scale products, accumulated in f64.
 *
 * READING marks a point where the pages are silent and the plainest reading
 * was taken (bit mapping inside ql/qh/qs, the scales[12] packing, the
 * activation rounding rule).
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define QK_K 256          /* values per super-block */
#define CHUNK 32          /* activation quantization block, one q8 scale each */
#define Q6K_BYTES 210     /* ql[128] qh[64] scales[16] d(f16)   [r56] §1, §3.2 */
#define Q4K_BYTES 144     /* d dmin (f16) scales[12] qs[128]   [r58] §2.2 */

/* ------------------------------------------------------------------------ */
/* IEEE binary16 -> binary32.  Exact: every half value is a float.           */
/* normal:    (1024 + man) * 2^(exp - 25);  subnormal: man * 2^-24           */
/* ------------------------------------------------------------------------ */
float oracle_f16_to_f32(uint16_t h)
{
    unsigned sign = (h >> 15) & 1u;
    unsigned expo = (h >> 10) & 0x1Fu;
    unsigned man = h & 0x3FFu;
    float mag;
    if (expo == 0)
        mag = ldexpf((float)man, -24);
    else if (expo == 31)
        mag = man ? NAN : INFINITY;
    else
        mag = ldexpf((float)(man | 0x400u), (int)expo - 25);
    return sign ? -mag : mag;
}

void oracle_f16_to_f32_array(const uint16_t* h, float* out, size_t n)
{
    for (size_t i = 0; i < n; ++i)
        out[i] = oracle_f16_to_f32(h[i]);
}

static float load_f16(const uint8_t* p)
{
    return oracle_f16_to_f32((uint16_t)(p[0] | ((unsigned)p[1] << 8)));
}

/* ------------------------------------------------------------------------ */
/* Activation prepass: per (token t, chunk c of 32 along K)                   */
/*   amax = max|x|, d = amax / 127 (f32 divide), q = round(x / d) in         */
/*   [-127, 127] (f32 divide, ties away from zero), ssum = sum q.           */
/* The pages name the planes the prepass writes (qa8 codes and a d/ssum      */
/* scale pair per chunk and row: [r45] §2.3, [r56] §1); the config fixes    */
/* d = amax/127.  READING: x / d is an IEEE f32 division and the rounding    */
/* is half away from zero (C roundf); amax == 0 gives d = 0 and all-zero q. */
/* ------------------------------------------------------------------------ */
void oracle_quantize_act(const float* x, int M, int K, int ldx,
                         int8_t* q, float* d, int32_t* ssum)
{
    const int nchunk = K / CHUNK;
    for (int t = 0; t < M; ++t) {
        for (int c = 0; c < nchunk; ++c) {
            const float* xc = x + (size_t)t * (size_t)ldx + (size_t)c * CHUNK;
            float amax = 0.0f;
            for (int i = 0; i < CHUNK; ++i) {
                float a = fabsf(xc[i]);
                if (a > amax)
                    amax = a;
            }
            const float dd = amax / 127.0f;
            int32_t s = 0;
            for (int i = 0; i < CHUNK; ++i) {
                int v = 0;
                if (dd != 0.0f) {
                    float r = roundf(xc[i] / dd);
                    if (r > 127.0f) r = 127.0f;
                    if (r < -127.0f) r = -127.0f;
                    v = (int)r;
                }
                q[(size_t)t * K + (size_t)c * CHUNK + i] = (int8_t)v;
                s += v;
            }
            d[(size_t)t * nchunk + c] = dd;
            ssum[(size_t)t * nchunk + c] = s;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* q6_K super-block decode.  Byte layout from the pages: ql[128] at 0,      */
/* qh[64] at 128, int8 scales[16] at 192, f16 d at 208 ([r56] §2.2 and the  */
/* expand_q6k_dsc excerpt in §3.2; [r58] §3.2 "ql+qh recomb").  A code is 4  */
/* low bits from ql and 2 high bits from qh, centred by -32; element e uses */
/* scales[e/16], i.e. chunk cc (32 values) uses scales[2cc] for its first   */
/* 16 values and scales[2cc+1] for its last 16 ([r56] §2.2).                */
/* READING (bit positions inside ql/qh): element e takes the nibble         */
/* (ql[e/2] >> 4*(e%2)) & 15 and the pair (qh[e/4] >> 2*(e%4)) & 3.         */
/* ------------------------------------------------------------------------ */
void oracle_decode_q6k(const uint8_t* b, float* d, int8_t sc[16], int8_t q[QK_K])
{
    const uint8_t* ql = b;
    const uint8_t* qh = b + 128;
    for (int i = 0; i < 16; ++i)
        sc[i] = (int8_t)b[192 + i];
    *d = load_f16(b + 208);
    for (int e = 0; e < QK_K; ++e) {
        int lo = (ql[e / 2] >> (4 * (e % 2))) & 15;
        int hi = (qh[e / 4] >> (2 * (e % 4))) & 3;
        q[e] = (int8_t)((lo | (hi << 4)) - 32);
    }
}

/* ------------------------------------------------------------------------ */
/* q4_K super-block decode.  Byte layout: f16 d at 0, f16 dmin at 2, 12     */
/* scale bytes at 4 holding 8 six-bit scales and 8 six-bit mins, 128 bytes  */
/* of nibbles at 16 ([r58] §2.2: the 144-byte block, qs at +16, decoded by  */
/* get_scale_min_k4).  Value = d*sc_c*q - dmin*m_c for chunk c.            */
/* READING (field order): d at 0 and dmin at 2; the 96 scale bits are read  */
/* little-endian as 16 six-bit fields, fields 0..7 = sc_0..7 and fields     */
/* 8..15 = m_0..7; nibble e = (qs[e/2] >> 4*(e%2)) & 15.                    */
/* ------------------------------------------------------------------------ */
void oracle_decode_q4k(const uint8_t* b, float* d, float* dmin,
                       uint8_t sc[8], uint8_t m[8], uint8_t q[QK_K])
{
    *d = load_f16(b + 0);
    *dmin = load_f16(b + 2);
    for (int f = 0; f < 16; ++f) {
        const int bit = 6 * f;
        const int byte = 4 + bit / 8;
        const int sh = bit % 8;
        unsigned v = (unsigned)b[byte] >> sh;
        if (sh > 2)
            v |= (unsigned)b[byte + 1] << (8 - sh);
        v &= 63u;
        if (f < 8)
            sc[f] = (uint8_t)v;
        else
            m[f - 8] = (uint8_t)v;
    }
    for (int e = 0; e < QK_K; ++e)
        q[e] = (uint8_t)((b[16 + e / 2] >> (4 * (e % 2))) & 15);
}

/* ------------------------------------------------------------------------ */
/* Registration-time f32 scale planes.  Each entry is one f32 multiply of   */
/* two exact conversions (f16 -> f32, int -> f32), no FMA contraction       */
/* ([r56] §2.2 "W_dsc" and §2.3 "bit-identical by construction").          */
/* q6_K: dsc[j][c][h] = d * scales[2*(c%8) + h], h = 0, 1.                  */
/* q4_K: dsc[j][c] = d * sc_(c%8), dmn[j][c] = dmin * m_(c%8) (the q4_K     */
/*       plane is the follow-up the r58 page names in §5).                   */
/* Row-major oracle layout: [od][id/32]([2]).                               */
/* ------------------------------------------------------------------------ */
void oracle_scale_planes_q6k(const uint8_t* raw, int od, int id, float* dsc)
{
    const int nsb = id / QK_K, nchunk = id / CHUNK;
    for (int j = 0; j < od; ++j) {
        for (int sb = 0; sb < nsb; ++sb) {
            const uint8_t* b = raw + ((size_t)j * nsb + sb) * Q6K_BYTES;
            const float d = load_f16(b + 208);
            for (int cc = 0; cc < 8; ++cc) {
                const float sc0 = (float)(int8_t)b[192 + 2 * cc];
                const float sc1 = (float)(int8_t)b[192 + 2 * cc + 1];
                const size_t o = ((size_t)j * nchunk + (size_t)sb * 8 + cc) * 2;
                dsc[o + 0] = d * sc0;
                dsc[o + 1] = d * sc1;
            }
        }
    }
}

void oracle_scale_planes_q4k(const uint8_t* raw, int od, int id, float* dsc, float* dmn)
{
    const int nsb = id / QK_K, nchunk = id / CHUNK;
    float d, dmin;
    uint8_t sc[8], m[8], q[QK_K];
    for (int j = 0; j < od; ++j) {
        for (int sb = 0; sb < nsb; ++sb) {
            oracle_decode_q4k(raw + ((size_t)j * nsb + sb) * Q4K_BYTES, &d, &dmin, sc, m, q);
            for (int cc = 0; cc < 8; ++cc) {
                const size_t o = (size_t)j * nchunk + (size_t)sb * 8 + cc;
                dsc[o] = d * (float)sc[cc];
                dmn[o] = dmin * (float)m[cc];
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Per-sub-block integer dots I = sum q_w * q_a (int32, exact).             */
/* q6_K: one dot per 16-value sub-block (each has its own int8 scale).      */
/* q4_K: one dot per 32-value chunk (one six-bit scale/min per chunk).       */
/* dots[(t*od + j)*nsub + s]; q_a row-major [M][id].                         */
/* ------------------------------------------------------------------------ */
void oracle_dots_q6k(const uint8_t* raw, int od, int id, const int8_t* qa, int M, int32_t* dots)
{
    const int nsb = id / QK_K, nsub = id / 16;
    float d;
    int8_t sc[16], q[QK_K];
    for (int j = 0; j < od; ++j) {
        for (int sb = 0; sb < nsb; ++sb) {
            oracle_decode_q6k(raw + ((size_t)j * nsb + sb) * Q6K_BYTES, &d, sc, q);
            for (int t = 0; t < M; ++t) {
                const int8_t* a = qa + (size_t)t * id + (size_t)sb * QK_K;
                for (int s = 0; s < 16; ++s) {
                    int32_t acc = 0;
                    for (int e = 16 * s; e < 16 * s + 16; ++e)
                        acc += (int32_t)q[e] * (int32_t)a[e];
                    dots[((size_t)t * od + j) * nsub + (size_t)sb * 16 + s] = acc;
                }
            }
        }
    }
}

void oracle_dots_q4k(const uint8_t* raw, int od, int id, const int8_t* qa, int M, int32_t* dots)
{
    const int nsb = id / QK_K, nsub = id / CHUNK;
    float d, dmin;
    uint8_t sc[8], m[8], q[QK_K];
    for (int j = 0; j < od; ++j) {
        for (int sb = 0; sb < nsb; ++sb) {
            oracle_decode_q4k(raw + ((size_t)j * nsb + sb) * Q4K_BYTES, &d, &dmin, sc, m, q);
            for (int t = 0; t < M; ++t) {
                const int8_t* a = qa + (size_t)t * id + (size_t)sb * QK_K;
                for (int c = 0; c < 8; ++c) {
                    int32_t acc = 0;
                    for (int e = 32 * c; e < 32 * c + 32; ++e)
                        acc += (int32_t)q[e] * (int32_t)a[e];
                    dots[((size_t)t * od + j) * nsub + (size_t)sb * 8 + c] = acc;
                }
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Y in f64 (spec formula, [r56] §2.2 for the q6_K scale pair):       */
/*   q6_K: Y[t,j] = sum_c sum_h d_a[t,c] * dsc[j,c,h] * I[t,j,c,h]          */
/*   q4_K: Y[t,j] = sum_c d_a[t,c] * (dsc[j,c]*I[t,j,c] - dmn[j,c]*ssum[t,c]) */
/* S[t,j] = sum of |term| (the condition number's numerator; may be NULL).  */
/* Rows j are split over nthreads POSIX threads; each thread runs the same  */
/* scalar code on its own rows.                                             */
/* ------------------------------------------------------------------------ */
typedef struct {
    int type; /* 6 or 4 */
    const uint8_t* raw;
    int od, id;
    const int8_t* qa;
    const float* da;
    const int32_t* ssum;
    int M;
    double* Y;
    double* S;
    int j0, j1;
} gemm_job;

static void gemm_rows_q6k(const gemm_job* g)
{
    const int id = g->id, nsb = id / QK_K, nchunk = id / CHUNK;
    int8_t* qrow = (int8_t*)malloc((size_t)id);
    float* dscrow = (float*)malloc((size_t)nchunk * 2 * sizeof(float));
    float d;
    int8_t sc[16];
    for (int j = g->j0; j < g->j1; ++j) {
        for (int sb = 0; sb < nsb; ++sb) {
            oracle_decode_q6k(g->raw + ((size_t)j * nsb + sb) * Q6K_BYTES, &d, sc,
                              qrow + (size_t)sb * QK_K);
            for (int s = 0; s < 16; ++s)
                dscrow[(size_t)sb * 16 + s] = d * (float)sc[s];
        }
        for (int t = 0; t < g->M; ++t) {
            const int8_t* a = g->qa + (size_t)t * id;
            double y = 0.0, sabs = 0.0;
            for (int c = 0; c < nchunk; ++c) {
                const double dac = (double)g->da[(size_t)t * nchunk + c];
                for (int h = 0; h < 2; ++h) {
                    const int s = 2 * c + h;
                    int32_t I = 0;
                    for (int e = 16 * s; e < 16 * s + 16; ++e)
                        I += (int32_t)qrow[e] * (int32_t)a[e];
                    const double term = dac * (double)dscrow[s] * (double)I;
                    y += term;
                    sabs += fabs(term);
                }
            }
            g->Y[(size_t)t * g->od + j] = y;
            if (g->S)
                g->S[(size_t)t * g->od + j] = sabs;
        }
    }
    free(qrow);
    free(dscrow);
}

static void gemm_rows_q4k(const gemm_job* g)
{
    const int id = g->id, nsb = id / QK_K, nchunk = id / CHUNK;
    uint8_t* qrow = (uint8_t*)malloc((size_t)id);
    float* dscrow = (float*)malloc((size_t)nchunk * sizeof(float));
    float* dmnrow = (float*)malloc((size_t)nchunk * sizeof(float));
    float d, dmin;
    uint8_t sc[8], m[8];
    for (int j = g->j0; j < g->j1; ++j) {
        for (int sb = 0; sb < nsb; ++sb) {
            oracle_decode_q4k(g->raw + ((size_t)j * nsb + sb) * Q4K_BYTES, &d, &dmin, sc, m,
                              qrow + (size_t)sb * QK_K);
            for (int c = 0; c < 8; ++c) {
                dscrow[(size_t)sb * 8 + c] = d * (float)sc[c];
                dmnrow[(size_t)sb * 8 + c] = dmin * (float)m[c];
            }
        }
        for (int t = 0; t < g->M; ++t) {
            const int8_t* a = g->qa + (size_t)t * id;
            double y = 0.0, sabs = 0.0;
            for (int c = 0; c < nchunk; ++c) {
                int32_t I = 0;
                for (int e = 32 * c; e < 32 * c + 32; ++e)
                    I += (int32_t)qrow[e] * (int32_t)a[e];
                const double dac = (double)g->da[(size_t)t * nchunk + c];
                const double main_term = dac * (double)dscrow[c] * (double)I;
                const double min_term = dac * (double)dmnrow[c] * (double)g->ssum[(size_t)t * nchunk + c];
                y += main_term - min_term;
                sabs += fabs(main_term) + fabs(min_term);
            }
            g->Y[(size_t)t * g->od + j] = y;
            if (g->S)
                g->S[(size_t)t * g->od + j] = sabs;
        }
    }
    free(qrow);
    free(dscrow);
    free(dmnrow);
}

static void* gemm_thread(void* p)
{
    const gemm_job* g = (const gemm_job*)p;
    if (g->type == 6)
        gemm_rows_q6k(g);
    else
        gemm_rows_q4k(g);
    return NULL;
}

static void gemm_run(int type, const uint8_t* raw, int od, int id, const int8_t* qa,
                     const float* da, const int32_t* ssum, int M, double* Y, double* S,
                     int nthreads)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > od)
        nthreads = od;
    gemm_job* jobs = (gemm_job*)calloc((size_t)nthreads, sizeof(gemm_job));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    for (int i = 0; i < nthreads; ++i) {
        gemm_job g = {type, raw, od, id, qa, da, ssum, M, Y, S,
                      (int)((long long)od * i / nthreads), (int)((long long)od * (i + 1) / nthreads)};
        jobs[i] = g;
    }
    for (int i = 1; i < nthreads; ++i)
        pthread_create(&th[i], NULL, gemm_thread, &jobs[i]);
    gemm_thread(&jobs[0]);
    for (int i = 1; i < nthreads; ++i)
        pthread_join(th[i], NULL);
    free(jobs);
    free(th);
}

void oracle_gemm_q6k(const uint8_t* raw, int od, int id, const int8_t* qa, const float* da,
                     const int32_t* ssum, int M, double* Y, double* S, int nthreads)
{
    gemm_run(6, raw, od, id, qa, da, ssum, M, Y, S, nthreads);
}

void oracle_gemm_q4k(const uint8_t* raw, int od, int id, const int8_t* qa, const float* da,
                     const int32_t* ssum, int M, double* Y, double* S, int nthreads)
{
    gemm_run(4, raw, od, id, qa, da, ssum, M, Y, S, nthreads);
}

/* ------------------------------------------------------------------------ */
/* Dequantized weights in f64 (for the dense-matmul cross-check):           */
/*   q6_K: w = d * sc[e/16] * q;  q4_K: w = d * sc_c * q - dmin * m_c.      */
/* ------------------------------------------------------------------------ */
void oracle_dequant_q6k(const uint8_t* raw, int od, int id, double* W)
{
    const int nsb = id / QK_K;
    float d;
    int8_t sc[16], q[QK_K];
    for (int j = 0; j < od; ++j)
        for (int sb = 0; sb < nsb; ++sb) {
            oracle_decode_q6k(raw + ((size_t)j * nsb + sb) * Q6K_BYTES, &d, sc, q);
            for (int e = 0; e < QK_K; ++e)
                W[(size_t)j * id + (size_t)sb * QK_K + e] = (double)d * (double)sc[e / 16] * (double)q[e];
        }
}

void oracle_dequant_q4k(const uint8_t* raw, int od, int id, double* W)
{
    const int nsb = id / QK_K;
    float d, dmin;
    uint8_t sc[8], m[8], q[QK_K];
    for (int j = 0; j < od; ++j)
        for (int sb = 0; sb < nsb; ++sb) {
            oracle_decode_q4k(raw + ((size_t)j * nsb + sb) * Q4K_BYTES, &d, &dmin, sc, m, q);
            for (int e = 0; e < QK_K; ++e)
                W[(size_t)j * id + (size_t)sb * QK_K + e] =
                    (double)d * (double)sc[e / 32] * (double)q[e] - (double)dmin * (double)m[e / 32];
        }
}

/* ------------------------------------------------------------------------ */
/* Decoded integer codes of a whole weight matrix, row-major [od][id]       */
/* (q6_K: centred codes in [-32,31]; q4_K: nibbles in [0,15]).              */
/* ------------------------------------------------------------------------ */
void oracle_codes_q6k(const uint8_t* raw, int od, int id, int8_t* codes)
{
    const int nsb = id / QK_K;
    float d;
    int8_t sc[16];
    for (int j = 0; j < od; ++j)
        for (int sb = 0; sb < nsb; ++sb)
            oracle_decode_q6k(raw + ((size_t)j * nsb + sb) * Q6K_BYTES, &d, sc,
                              codes + (size_t)j * id + (size_t)sb * QK_K);
}

void oracle_codes_q4k(const uint8_t* raw, int od, int id, uint8_t* codes)
{
    const int nsb = id / QK_K;
    float d, dmin;
    uint8_t sc[8], m[8];
    for (int j = 0; j < od; ++j)
        for (int sb = 0; sb < nsb; ++sb)
            oracle_decode_q4k(raw + ((size_t)j * nsb + sb) * Q4K_BYTES, &d, &dmin, sc, m,
                              codes + (size_t)j * id + (size_t)sb * QK_K);
}

/* ------------------------------------------------------------------------ */
/* Decoded per-super-block fields of a whole weight matrix, [od][id/256]:   */
/*   q6_K: d, scales[16];  q4_K: d, dmin, sc[8], m[8].                       */
/* ------------------------------------------------------------------------ */
void oracle_fields_q6k(const uint8_t* raw, int od, int id, float* d, int8_t* sc)
{
    const int nsb = id / QK_K;
    int8_t q[QK_K];
    for (int j = 0; j < od; ++j)
        for (int sb = 0; sb < nsb; ++sb) {
            const size_t b = (size_t)j * nsb + sb;
            oracle_decode_q6k(raw + b * Q6K_BYTES, d + b, sc + b * 16, q);
        }
}

void oracle_fields_q4k(const uint8_t* raw, int od, int id, float* d, float* dmin, uint8_t* sc, uint8_t* m)
{
    const int nsb = id / QK_K;
    uint8_t q[QK_K];
    for (int j = 0; j < od; ++j)
        for (int sb = 0; sb < nsb; ++sb) {
            const size_t b = (size_t)j * nsb + sb;
            oracle_decode_q4k(raw + b * Q4K_BYTES, d + b, dmin + b, sc + b * 8, m + b * 8, q);
        }
}

/* ------------------------------------------------------------------------ */
/* GGUF interop: blocks in the public ggml (llama.cpp) q4_K / q6_K layout,
 * rewritten into the reading above (same byte positions of d, dmin, scales and
 * the code arrays; only the order of the codes inside qs / ql / qh and the
 * q4_K scale packing differ).  This part follows the public ggml block format,
 * not the three pages; it is pinned against hand-worked blocks and an
 * independent inverse encoder, not against real GGUF files (parity unpinned
 * against real files).
 *
 * ggml q4_K, value v (0..255), j = v / 64, l = v % 64:
 *   code  = l < 32 ? qs[32 j + l] & 15 : qs[32 j + l - 32] >> 4
 *   sub-block s = v / 32 (0..7) with scale sc_s and min m_s:
 *     s < 4:  sc = S[s] & 63,  m = S[s + 4] & 63
 *     s >= 4: sc = (S[s + 4] & 15) | ((S[s - 4] >> 6) << 4)
 *             m  = (S[s + 4] >> 4) | ((S[s] >> 6) << 4)
 * ggml q6_K, value v, n = v / 128, w = v % 128, p = w / 32, l = w % 32:
 *   low 4 bits  = nibble (p / 2) of ql[64 n + 32 (p % 2) + l]
 *   high 2 bits = (qh[32 n + l] >> (2 p)) & 3
 *   code = (low | high << 4) - 32, scale index 8 n + 2 p + l / 16 = v / 16 (as the
 *   reading: the scales array is copied unchanged). */
static int ggml_q4k_code(const uint8_t* qs, int v)
{
    const int j = v / 64, l = v % 64;
    return l < 32 ? (qs[32 * j + l] & 15) : (qs[32 * j + l - 32] >> 4);
}

static void ggml_q4k_scale_min(const uint8_t* S, int s, int* sc, int* m)
{
    if (s < 4) {
        *sc = S[s] & 63;
        *m = S[s + 4] & 63;
    } else {
        *sc = (S[s + 4] & 15) | ((S[s - 4] >> 6) << 4);
        *m = (S[s + 4] >> 4) | ((S[s] >> 6) << 4);
    }
}

static int ggml_q6k_code_unsigned(const uint8_t* ql, const uint8_t* qh, int v)
{
    const int n = v / 128, w = v % 128, p = w / 32, l = w % 32;
    const int byte = ql[64 * n + 32 * (p % 2) + l];
    const int low = (p / 2) ? (byte >> 4) : (byte & 15);
    const int high = (qh[32 * n + l] >> (2 * p)) & 3;
    return low | (high << 4);
}

/* src and dst may be the same buffer; nblocks blocks of 144 (q4_K) or 210 (q6_K) B. */
void oracle_ggml_to_reading(int type, const uint8_t* src, long long nblocks, uint8_t* dst)
{
    for (long long bi = 0; bi < nblocks; ++bi) {
        if (type == 12) {
            uint8_t in[Q4K_BYTES], out[Q4K_BYTES];
            memcpy(in, src + bi * Q4K_BYTES, Q4K_BYTES);
            memset(out, 0, sizeof out);
            memcpy(out, in, 4);                                  /* d, dmin */
            /* scales: field f (0..15) as 6 bits at bit 6f, little-endian over 12 bytes */
            for (int s = 0; s < 8; ++s) {
                int sc, m;
                ggml_q4k_scale_min(in + 4, s, &sc, &m);
                const int fields[2] = {sc, m};
                for (int t = 0; t < 2; ++t) {
                    const int f = s + 8 * t;
                    for (int b = 0; b < 6; ++b)
                        if ((fields[t] >> b) & 1) {
                            const int bit = 6 * f + b;
                            out[4 + bit / 8] |= (uint8_t)(1u << (bit % 8));
                        }
                }
            }
            /* codes: value e at nibble e % 2 of qs[e / 2] */
            for (int e = 0; e < QK_K; ++e)
                out[16 + e / 2] |= (uint8_t)(ggml_q4k_code(in + 16, e) << (4 * (e % 2)));
            memcpy(dst + bi * Q4K_BYTES, out, Q4K_BYTES);
        } else {
            uint8_t in[Q6K_BYTES], out[Q6K_BYTES];
            memcpy(in, src + bi * Q6K_BYTES, Q6K_BYTES);
            memset(out, 0, sizeof out);
            memcpy(out + 192, in + 192, 18);                     /* scales[16], d */
            for (int e = 0; e < QK_K; ++e) {
                const int u = ggml_q6k_code_unsigned(in, in + 128, e);
                out[e / 2] |= (uint8_t)((u & 15) << (4 * (e % 2)));            /* ql */
                out[128 + e / 4] |= (uint8_t)(((u >> 4) & 3) << (2 * (e % 4))); /* qh */
            }
            memcpy(dst + bi * Q6K_BYTES, out, Q6K_BYTES);
        }
    }
}
