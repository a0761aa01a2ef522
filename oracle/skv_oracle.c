/*
 * skv_oracle.c -- plain, slow CPU oracle of the SKV v1 format.
 *
 * TEST INFRASTRUCTURE. This file is the checker, not the product: only the
 * tests, __graft_entry__.smoke() and bench.py's CPU-baseline leg (and its
 * `--impl reference` arm) may load or call it. It shares no code, header,
 * table or generator with the CUDA library.
 *
 * What it computes follows the method of two pages, cited by title and
 * section:
 *   - "Speculative KV Coding" (aisparkup.com wiki): the pipeline section
 *     (encoder and decoder both hold (mu, sigma); the coder turns KV_full
 *     into bits and back, losslessly) and the mixture section
 *     q(x) = 0.95 N(x; mu, sigma^2) + 0.03 N(x; mu, (3 sigma)^2) + 0.02 p_hat(x).
 *   - "推测性KV编码：用预测模型实现缓存无损压缩4倍" (blog.hotdry.top): the
 *     information-theory section (code length = -log q, Gaussian cost) and the
 *     deployment section (bit-identical CDF on both ends).
 * The discretisation and the bitstream are the SKV v1 format's; each function below
 * names the format section it writes out.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fno-fast-math -fPIC -shared
 *        -pthread (oracle/build.py). No FMA contraction and no flush-to-zero:
 *        the fp32 steps of SKV v1 format §5 must round exactly as written.
 *
 * Parity pins for every function are in tests/test_oracle_*.py.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Status values of the C-ABI (include/skv.h), restated here. */
enum {
    OR_OK = 0,
    OR_ERR_INVALID_ARG = 1,
    OR_ERR_NONFINITE_MU = 3,
    OR_ERR_BAD_SIGMA = 4,
    OR_ERR_EMPTY_MARGINAL = 5,
    OR_ERR_CAPACITY = 6,
    OR_ERR_CORRUPT = 7,
    OR_ERR_NOMEM = 9,
};

enum { DT_BF16 = 0, DT_E4M3 = 1 };

/* SKV v1 format §3: T[j + 2048] = round_half_even(2^24 Phi(j/256)). */
static const uint32_t PHI_T[4097] = {
#include "phi_q24.inc"
};

/* ---------------------------------------------------------------- types */

typedef struct {
    uint32_t dtype;
    uint32_t n_layers, n_kv, n_heads, head_dim;
    uint64_t n_tokens;
    uint32_t tokens_per_chunk, streams_per_chunk;
    uint32_t w_n, w_w, w_h;
    uint32_t sigma_block;  /* 0: one sigma per channel; else tokens per sigma block */
} or_layout;

typedef struct {          /* per-dtype constants, SKV v1 format §1 */
    uint32_t N;           /* number of codes */
    uint32_t m;           /* M = 2^m */
    uint32_t V;           /* scalars per 16-byte vector */
    uint32_t bytes;       /* bytes per code */
} or_dtype;

static or_dtype dtype_info(uint32_t dtype)
{
    or_dtype d;
    if (dtype == DT_BF16) { d.N = 65536; d.m = 24; d.V = 8; d.bytes = 2; }
    else                  { d.N = 256;   d.m = 16; d.V = 16; d.bytes = 1; }
    return d;
}

/* ------------------------------------------------- section 1: code order */

uint32_t oracle_ord(uint32_t dtype, uint32_t b)
{
    uint32_t N = dtype_info(dtype).N;
    uint32_t sign = b & (N / 2);
    return sign ? (b ^ (N - 1)) : (b ^ (N / 2));
}

uint32_t oracle_code(uint32_t dtype, uint32_t o)
{
    uint32_t N = dtype_info(dtype).N;
    return (o < N / 2) ? (o ^ (N - 1)) : (o ^ (N / 2));
}

/* Value of a code as binary32 (exact for both dtypes). */
float oracle_value(uint32_t dtype, uint32_t b)
{
    if (dtype == DT_BF16) {
        uint32_t bits = b << 16;
        float f;
        memcpy(&f, &bits, 4);
        return f;
    }
    /* OCP e4m3: 1 sign, 4 exponent (bias 7), 3 mantissa; S.1111.111 is NaN,
       there is no infinity. */
    uint32_t s = (b >> 7) & 1, e = (b >> 3) & 15, mant = b & 7;
    float v;
    if (e == 15 && mant == 7) v = NAN;
    else if (e == 0) v = ldexpf((float)mant, -9);               /* mant/8 * 2^-6 */
    else v = ldexpf((float)(8 + mant), (int)e - 10);             /* (1+mant/8) 2^(e-7) */
    return s ? -v : v;
}

static int code_is_finite(uint32_t dtype, uint32_t b)
{
    if (dtype == DT_BF16) return ((b >> 7) & 0xFF) != 0xFF;
    return (b & 0x7F) != 0x7F;
}

/* ------------------------------------------------------ section 2: edges */

float oracle_edge(uint32_t dtype, uint32_t o)
{
    uint32_t maxc = (dtype == DT_BF16) ? 0x7F7Fu : 0x7Eu;
    uint32_t sgn = (dtype == DT_BF16) ? 0x8000u : 0x80u;
    uint32_t o_lo = oracle_ord(dtype, maxc | sgn);   /* ord(-max) */
    uint32_t o_hi = oracle_ord(dtype, maxc);         /* ord(+max) */
    if (o <= o_lo) return -INFINITY;
    if (o > o_hi) return INFINITY;
    float a = oracle_value(dtype, oracle_code(dtype, o - 1));
    float b = oracle_value(dtype, oracle_code(dtype, o));
    float ha = 0.5f * a;
    float hb = 0.5f * b;
    return ha + hb;
}

/* ------------------------------------------------ section 3: fixed-point Phi */

void oracle_phi_table(uint32_t *out)
{
    memcpy(out, PHI_T, sizeof PHI_T);
}

uint32_t oracle_phi_q(int32_t zq)
{
    if (zq <= -524288) return 0;
    if (zq >= 524288) return 1u << 24;
    int32_t j = (int32_t)floor((double)zq / 256.0);
    int32_t r = zq - 256 * j;
    uint32_t t0 = PHI_T[j + 2048], t1 = PHI_T[j + 2049];
    return t0 + (uint32_t)(((uint64_t)(t1 - t0) * (uint64_t)r) / 256u);
}

/* --------------------------------------------- section 5: cumulative table */

/* P_hat(o) = floor(2^24 cum(o) / total) for o = 0..N, cum in code order. */
static int phat_table(uint32_t dtype, const uint64_t *counts, uint32_t w_h, uint32_t *P)
{
    uint32_t N = dtype_info(dtype).N;
    if (w_h == 0) {
        for (uint32_t o = 0; o <= N; o++) P[o] = 0;
        return OR_OK;
    }
    unsigned __int128 total = 0;
    for (uint32_t b = 0; b < N; b++) total += counts[b];
    if (total == 0) return OR_ERR_EMPTY_MARGINAL;
    unsigned __int128 cum = 0;
    for (uint32_t o = 0; o <= N; o++) {
        P[o] = (uint32_t)(((cum << 24)) / total);
        if (o < N) cum += counts[oracle_code(dtype, o)];
    }
    return OR_OK;
}

typedef struct {
    uint32_t dtype;
    or_dtype d;
    uint32_t w_n, w_w, w_h;
    const uint32_t *P;       /* P_hat, N + 1 entries */
} or_model;

static int32_t floor_div3(int32_t a)
{
    int32_t q = a / 3;               /* C truncates toward zero */
    if ((a % 3) != 0 && a < 0) q -= 1;
    return q;
}

/* C(o) for one element with predictor value mu and rs = fl32(1/sigma). */
static uint64_t cdf_at(const or_model *md, uint32_t o, float mu, float rs)
{
    float E = oracle_edge(md->dtype, o);
    float d = E - mu;
    float z = d * rs;
    if (z < -24.0f) z = -24.0f;
    if (z > 24.0f) z = 24.0f;
    float zs = z * 65536.0f;
    int32_t zq = (int32_t)floorf(zs);
    int32_t zw = floor_div3(zq);
    uint64_t S = (uint64_t)md->w_n * oracle_phi_q(zq)
               + (uint64_t)md->w_w * oracle_phi_q(zw)
               + (uint64_t)md->w_h * md->P[o];
    uint64_t MN = (1ull << md->d.m) - md->d.N;
    return (uint64_t)o + (S * MN) / (100ull << 24);
}

static int sigma_valid(float s)
{
    return isfinite(s) && s >= 0x1p-126f;
}

/* The model value of a mu code: non-finite mu is reported and replaced by 0
   (SKV v1 format §4). */
static float mu_value(uint32_t dtype, uint32_t code, int *bad)
{
    if (!code_is_finite(dtype, code)) { *bad = 1; return 0.0f; }
    return oracle_value(dtype, code);
}

/* Full cumulative table C[0..N] for one element (tests). */
int oracle_cdf_all(uint32_t dtype, uint32_t mu_code, float sigma,
                   uint32_t w_n, uint32_t w_w, uint32_t w_h,
                   const uint64_t *counts, uint64_t *C)
{
    or_model md;
    md.dtype = dtype; md.d = dtype_info(dtype);
    md.w_n = w_n; md.w_w = w_w; md.w_h = w_h;
    if (w_n + w_w + w_h != 100) return OR_ERR_INVALID_ARG;
    if (!sigma_valid(sigma)) return OR_ERR_BAD_SIGMA;
    uint32_t *P = malloc(sizeof(uint32_t) * (md.d.N + 1));
    if (!P) return OR_ERR_NOMEM;
    int st = phat_table(dtype, counts, w_h, P);
    if (st != OR_OK) { free(P); return st; }
    md.P = P;
    int bad = 0;
    float mu = mu_value(dtype, mu_code, &bad);
    float rs = 1.0f / sigma;
    for (uint32_t o = 0; o <= md.d.N; o++) C[o] = cdf_at(&md, o, mu, rs);
    free(P);
    return bad ? OR_ERR_NONFINITE_MU : OR_OK;
}

/* C(o) for a batch of (mu code, sigma, ord) queries sharing one model. */
int oracle_cdf_eval(uint32_t dtype, uint32_t w_n, uint32_t w_w, uint32_t w_h,
                    const uint64_t *counts, uint64_t n, const uint32_t *mu_code,
                    const float *sigma, const uint32_t *ords, uint64_t *C)
{
    or_model md;
    md.dtype = dtype; md.d = dtype_info(dtype);
    md.w_n = w_n; md.w_w = w_w; md.w_h = w_h;
    if (w_n + w_w + w_h != 100) return OR_ERR_INVALID_ARG;
    uint32_t *P = malloc(sizeof(uint32_t) * (md.d.N + 1));
    if (!P) return OR_ERR_NOMEM;
    int st = phat_table(dtype, counts, w_h, P);
    if (st != OR_OK) { free(P); return st; }
    md.P = P;
    int bad = 0, badsig = 0;
    for (uint64_t i = 0; i < n; i++) {
        float mu = mu_value(dtype, mu_code[i], &bad);
        if (!sigma_valid(sigma[i])) badsig = 1;
        float rs = 1.0f / sigma[i];
        C[i] = cdf_at(&md, ords[i], mu, rs);
    }
    free(P);
    if (badsig) return OR_ERR_BAD_SIGMA;
    return bad ? OR_ERR_NONFINITE_MU : OR_OK;
}

/* Decoder search: the o with C(o) <= s < C(o+1), by bisection on [0, N). */
static uint32_t find_symbol(const or_model *md, uint64_t s, float mu, float rs)
{
    uint32_t lo = 0, hi = md->d.N;     /* C(lo) <= s < C(hi) */
    while (hi - lo > 1) {
        uint32_t mid = lo + (hi - lo) / 2;
        if (cdf_at(md, mid, mu, rs) <= s) lo = mid; else hi = mid;
    }
    return lo;
}

/* Search for a batch of slots (tests of the inversion). */
int oracle_find_symbols(uint32_t dtype, uint32_t mu_code, float sigma,
                        uint32_t w_n, uint32_t w_w, uint32_t w_h,
                        const uint64_t *counts, uint64_t n, const uint64_t *slots,
                        uint32_t *ords)
{
    or_model md;
    md.dtype = dtype; md.d = dtype_info(dtype);
    md.w_n = w_n; md.w_w = w_w; md.w_h = w_h;
    uint32_t *P = malloc(sizeof(uint32_t) * (md.d.N + 1));
    if (!P) return OR_ERR_NOMEM;
    int st = phat_table(dtype, counts, w_h, P);
    if (st != OR_OK) { free(P); return st; }
    md.P = P;
    int bad = 0;
    float mu = mu_value(dtype, mu_code, &bad);
    float rs = 1.0f / sigma;
    for (uint64_t i = 0; i < n; i++) ords[i] = find_symbol(&md, slots[i], mu, rs);
    free(P);
    return OR_OK;
}

/* --------------------------------------------- section 7: chunk geometry */

typedef struct {
    or_layout lay;
    or_dtype d;
    uint64_t HD, P, n_chunks;
    uint64_t n_sblk;       /* sigma rows per (layer, kv) plane */
    uint32_t W, G;
} or_geom;

static int geom_init(const or_layout *lay, or_geom *g)
{
    if (lay->dtype > DT_E4M3) return OR_ERR_INVALID_ARG;
    if (lay->n_layers == 0 || lay->n_kv == 0 || lay->n_heads == 0 || lay->head_dim == 0)
        return OR_ERR_INVALID_ARG;
    if (lay->tokens_per_chunk == 0) return OR_ERR_INVALID_ARG;
    if (lay->sigma_block % lay->tokens_per_chunk != 0) return OR_ERR_INVALID_ARG;
    if (lay->streams_per_chunk == 0 || lay->streams_per_chunk % 32 != 0 ||
        lay->streams_per_chunk > 256) return OR_ERR_INVALID_ARG;
    if (lay->w_n + lay->w_w + lay->w_h != 100) return OR_ERR_INVALID_ARG;
    g->lay = *lay;
    g->d = dtype_info(lay->dtype);
    g->HD = (uint64_t)lay->n_heads * lay->head_dim;
    if ((g->HD * g->d.bytes) % 16 != 0) return OR_ERR_INVALID_ARG;
    g->P = (lay->n_tokens + lay->tokens_per_chunk - 1) / lay->tokens_per_chunk;
    g->n_chunks = (uint64_t)lay->n_layers * lay->n_kv * g->P;
    g->W = lay->streams_per_chunk;
    g->G = g->W / 32;
    g->n_sblk = lay->sigma_block ? (lay->n_tokens + lay->sigma_block - 1) / lay->sigma_block : 1;
    return OR_OK;
}

/* SKV v1 format §4: the sigma entry of global element i. Without sigma
   blocks it is the element's (layer, kv, channel); with blocks of B tokens
   also its token's block t / B. */
static uint64_t sigma_index(const or_geom *g, uint64_t i)
{
    uint64_t T = g->lay.n_tokens;
    uint64_t plane = i / (T * g->HD);
    uint64_t t = (i / g->HD) % T;
    uint64_t c = i % g->HD;
    uint64_t blk = g->lay.sigma_block ? t / g->lay.sigma_block : 0;
    return (plane * g->n_sblk + blk) * g->HD + c;
}

/* Chunk k: first element (global index), its (layer, kv) plane, vector count. */
static void chunk_span(const or_geom *g, uint64_t k, uint64_t *elem0, uint64_t *plane,
                       uint64_t *n_vec)
{
    uint64_t page = k % g->P;
    *plane = k / g->P;
    uint64_t tok0 = page * g->lay.tokens_per_chunk;
    uint64_t ntok = g->lay.n_tokens - tok0;
    if (ntok > g->lay.tokens_per_chunk) ntok = g->lay.tokens_per_chunk;
    *elem0 = (*plane * g->lay.n_tokens + tok0) * g->HD;
    *n_vec = ntok * g->HD / g->d.V;
}

/* Symbols in stream s: V per owned vector q = s, s+W, ... < n_vec. */
static uint64_t stream_len(const or_geom *g, uint64_t n_vec, uint32_t s)
{
    if (n_vec <= s) return 0;
    return ((n_vec - s + g->W - 1) / g->W) * g->d.V;
}

/* Chunk-local element of symbol i of stream s. */
static uint64_t stream_elem(const or_geom *g, uint32_t s, uint64_t i)
{
    uint64_t q = s + (i / g->d.V) * g->W;
    return q * g->d.V + (i % g->d.V);
}

static uint64_t pad16(uint64_t b) { return (b + 15) & ~(uint64_t)15; }

static uint64_t header_bytes(const or_geom *g)
{
    return 8ull * g->W + pad16(4ull * g->G);
}

/* Worst-case group words, SKV v1 format §8. */
static uint64_t group_cap_words(const or_geom *g, uint64_t n_vec, uint32_t grp)
{
    uint64_t nmax = stream_len(g, n_vec, 32 * grp);
    return 32 * ((nmax * (g->d.m + 1) + 31) / 32);
}

static uint64_t chunk_max_bytes(const or_geom *g, uint64_t n_vec)
{
    uint64_t b = header_bytes(g);
    for (uint32_t grp = 0; grp < g->G; grp++) b += pad16(4 * group_cap_words(g, n_vec, grp));
    return b;
}

int oracle_num_chunks(const or_layout *lay, uint64_t *n)
{
    or_geom g;
    int st = geom_init(lay, &g);
    if (st) return st;
    *n = g.n_chunks;
    return OR_OK;
}

int oracle_max_encoded_bytes(const or_layout *lay, uint64_t *bytes)
{
    or_geom g;
    int st = geom_init(lay, &g);
    if (st) return st;
    uint64_t tot = 0;
    for (uint64_t k = 0; k < g.n_chunks; k++) {
        uint64_t e0, pl, nv;
        chunk_span(&g, k, &e0, &pl, &nv);
        tot += chunk_max_bytes(&g, nv);
    }
    *bytes = tot;
    return OR_OK;
}

static uint32_t load_code(const or_geom *g, const void *buf, uint64_t idx)
{
    if (g->d.bytes == 2) return ((const uint16_t *)buf)[idx];
    return ((const uint8_t *)buf)[idx];
}

static void store_code(const or_geom *g, void *buf, uint64_t idx, uint32_t c)
{
    if (g->d.bytes == 2) ((uint16_t *)buf)[idx] = (uint16_t)c;
    else ((uint8_t *)buf)[idx] = (uint8_t)c;
}

static void put_u32(uint8_t *p, uint32_t v)
{
    for (int i = 0; i < 4; i++) p[i] = (uint8_t)(v >> (8 * i));
}
static void put_u64(uint8_t *p, uint64_t v)
{
    for (int i = 0; i < 8; i++) p[i] = (uint8_t)(v >> (8 * i));
}
static uint32_t get_u32(const uint8_t *p)
{
    uint32_t v = 0;
    for (int i = 0; i < 4; i++) v |= (uint32_t)p[i] << (8 * i);
    return v;
}
static uint64_t get_u64(const uint8_t *p)
{
    uint64_t v = 0;
    for (int i = 0; i < 8; i++) v |= (uint64_t)p[i] << (8 * i);
    return v;
}

/* ------------------------------------------------------ section 6: encode */

typedef struct {
    const or_geom *g;
    const or_model *md;
    const void *kv, *mu;
    const float *rs_all;       /* fl32(1/sigma), one per sigma entry */
    int bad_mu;
} or_ctx;

/* Encode chunk k into buf (capacity chunk_max_bytes); returns its size. */
static uint64_t encode_chunk(or_ctx *cx, uint64_t k, uint8_t *buf)
{
    const or_geom *g = cx->g;
    const uint32_t m = g->d.m;
    const uint64_t M = 1ull << m, L = 1ull << (m + 7);
    uint64_t e0, plane, n_vec;
    chunk_span(g, k, &e0, &plane, &n_vec);

    uint64_t hdr = header_bytes(g);
    memset(buf, 0, hdr);
    uint64_t pos = hdr;
    for (uint32_t grp = 0; grp < g->G; grp++) {
        uint64_t nlane[32], nmax = 0;
        uint32_t *word[32];
        uint8_t *has[32];
        for (uint32_t l = 0; l < 32; l++) {
            nlane[l] = stream_len(g, n_vec, 32 * grp + l);
            if (nlane[l] > nmax) nmax = nlane[l];
            word[l] = malloc(sizeof(uint32_t) * (nlane[l] + 1));
            has[l] = calloc(nlane[l] + 1, 1);
        }
        /* Each stream encodes its symbols backwards from x = L. */
        for (uint32_t l = 0; l < 32; l++) {
            uint32_t s = 32 * grp + l;
            uint64_t x = L;
            for (uint64_t i = nlane[l]; i-- > 0;) {
                uint64_t el = stream_elem(g, s, i);
                uint32_t code = load_code(g, cx->kv, e0 + el);
                float mu = mu_value(g->lay.dtype, load_code(g, cx->mu, e0 + el), &cx->bad_mu);
                float r = cx->rs_all[sigma_index(g, e0 + el)];
                uint32_t o = oracle_ord(g->lay.dtype, code);
                uint64_t c = cdf_at(cx->md, o, mu, r);
                uint64_t f = cdf_at(cx->md, o + 1, mu, r) - c;
                if (x >= (f << 39)) {
                    word[l][i] = (uint32_t)(x & 0xFFFFFFFFu);
                    has[l][i] = 1;
                    x >>= 32;
                }
                x = (x / f) * M + (x % f) + c;
            }
            put_u64(buf + 8ull * s, x);
        }
        /* Words in decode order: step i ascending, lane ascending. */
        uint64_t nw = 0;
        for (uint64_t i = 0; i < nmax; i++)
            for (uint32_t l = 0; l < 32; l++)
                if (i < nlane[l] && has[l][i]) {
                    put_u32(buf + pos + 4 * nw, word[l][i]);
                    nw++;
                }
        put_u32(buf + 8ull * g->W + 4ull * grp, (uint32_t)nw);
        uint64_t padded = pad16(4 * nw);
        memset(buf + pos + 4 * nw, 0, padded - 4 * nw);
        pos += padded;
        for (uint32_t l = 0; l < 32; l++) { free(word[l]); free(has[l]); }
    }
    return pos;
}

/* ------------------------------------------------------ section 6: decode */

/* Decode chunk k from its bytes into kv_out (global layout). */
static int decode_chunk(or_ctx *cx, uint64_t k, const uint8_t *buf, uint64_t size,
                        void *kv_out, uint64_t out_elem0)
{
    const or_geom *g = cx->g;
    const uint32_t m = g->d.m;
    const uint64_t M = 1ull << m, L = 1ull << (m + 7);
    uint64_t e0, plane, n_vec;
    chunk_span(g, k, &e0, &plane, &n_vec);

    uint64_t hdr = header_bytes(g);
    if (size < hdr) return OR_ERR_CORRUPT;
    uint64_t nwords[8], start[8], pos = hdr;
    for (uint32_t grp = 0; grp < g->G; grp++) {
        nwords[grp] = get_u32(buf + 8ull * g->W + 4ull * grp);
        start[grp] = pos;
        pos += pad16(4 * nwords[grp]);
        if (pos > size) return OR_ERR_CORRUPT;
    }
    if (pos != size) return OR_ERR_CORRUPT;

    for (uint32_t grp = 0; grp < g->G; grp++) {
        uint64_t x[32], nlane[32], nmax = 0, rp = 0;
        for (uint32_t l = 0; l < 32; l++) {
            x[l] = get_u64(buf + 8ull * (32 * grp + l));
            if (x[l] < L || x[l] >= (1ull << (m + 39))) return OR_ERR_CORRUPT;
            nlane[l] = stream_len(g, n_vec, 32 * grp + l);
            if (nlane[l] > nmax) nmax = nlane[l];
        }
        for (uint64_t i = 0; i < nmax; i++) {
            for (uint32_t l = 0; l < 32; l++) {
                if (i >= nlane[l]) continue;
                uint32_t s = 32 * grp + l;
                uint64_t el = stream_elem(g, s, i);
                float mu = mu_value(g->lay.dtype, load_code(g, cx->mu, e0 + el), &cx->bad_mu);
                float r = cx->rs_all[sigma_index(g, e0 + el)];
                uint64_t slot = x[l] & (M - 1);
                uint32_t o = find_symbol(cx->md, slot, mu, r);
                uint64_t c = cdf_at(cx->md, o, mu, r);
                uint64_t f = cdf_at(cx->md, o + 1, mu, r) - c;
                x[l] = f * (x[l] >> m) + slot - c;
                store_code(g, kv_out, out_elem0 + el, oracle_code(g->lay.dtype, o));
                if (x[l] < L) {
                    if (rp >= nwords[grp]) return OR_ERR_CORRUPT;
                    x[l] = (x[l] << 32) | get_u32(buf + start[grp] + 4 * rp);
                    rp++;
                }
            }
        }
        for (uint32_t l = 0; l < 32; l++)
            if (x[l] != L) return OR_ERR_CORRUPT;
        if (rp != nwords[grp]) return OR_ERR_CORRUPT;
    }
    return OR_OK;
}

/* -------------------------------------------------------- shared set-up */

typedef struct {
    or_geom g;
    or_model md;
    uint32_t *P;
    float *rs;
} or_setup;

static void setup_free(or_setup *su)
{
    free(su->P);
    free(su->rs);
}

static int setup_init(const or_layout *lay, const float *sigma, const uint64_t *counts,
                      or_setup *su)
{
    memset(su, 0, sizeof *su);
    int st = geom_init(lay, &su->g);
    if (st) return st;
    su->P = malloc(sizeof(uint32_t) * (su->g.d.N + 1));
    uint64_t nsig = (uint64_t)lay->n_layers * lay->n_kv * su->g.n_sblk * su->g.HD;
    su->rs = malloc(sizeof(float) * (nsig ? nsig : 1));
    if (!su->P || !su->rs) { setup_free(su); return OR_ERR_NOMEM; }
    for (uint64_t i = 0; i < nsig; i++) {
        if (!sigma_valid(sigma[i])) { setup_free(su); return OR_ERR_BAD_SIGMA; }
        su->rs[i] = 1.0f / sigma[i];
    }
    st = phat_table(lay->dtype, counts, lay->w_h, su->P);
    if (st) { setup_free(su); return st; }
    su->md.dtype = lay->dtype;
    su->md.d = su->g.d;
    su->md.w_n = lay->w_n; su->md.w_w = lay->w_w; su->md.w_h = lay->w_h;
    su->md.P = su->P;
    return OR_OK;
}

/* ------------------------------------------------------ threaded drivers */

typedef struct {
    or_ctx cx;
    const uint64_t *ids;     /* chunk ids to process */
    uint64_t n_ids;
    uint32_t tid, nthreads;
    uint8_t **bufs;          /* encode: per-id buffers */
    uint64_t *sizes;
    const uint8_t *stream;   /* decode: bitstream */
    const uint64_t *offsets;
    uint64_t stream_bytes;
    void *kv_out;
    int pages;               /* decode: write page i at i * page_elems */
    uint64_t page_elems;
    int status;
} or_job;

static void *encode_worker(void *arg)
{
    or_job *jb = arg;
    for (uint64_t i = jb->tid; i < jb->n_ids; i += jb->nthreads) {
        uint64_t k = jb->ids[i];
        uint64_t e0, pl, nv;
        chunk_span(jb->cx.g, k, &e0, &pl, &nv);
        jb->bufs[i] = malloc(chunk_max_bytes(jb->cx.g, nv));
        if (!jb->bufs[i]) { jb->status = OR_ERR_NOMEM; return NULL; }
        jb->sizes[i] = encode_chunk(&jb->cx, k, jb->bufs[i]);
    }
    return NULL;
}

static void *decode_worker(void *arg)
{
    or_job *jb = arg;
    for (uint64_t i = jb->tid; i < jb->n_ids; i += jb->nthreads) {
        uint64_t k = jb->ids[i];
        uint64_t a = jb->offsets[k], b = jb->offsets[k + 1];
        if (b < a || b > jb->stream_bytes) { jb->status = OR_ERR_CORRUPT; continue; }
        uint64_t e0, pl, nv;
        chunk_span(jb->cx.g, k, &e0, &pl, &nv);
        /* a page is written chunk-locally at i * page_elems */
        uint64_t dst0 = jb->pages ? i * jb->page_elems : e0;
        int st = decode_chunk(&jb->cx, k, jb->stream + a, b - a, jb->kv_out, dst0);
        if (st && !jb->status) jb->status = st;
    }
    return NULL;
}

static int run_jobs(or_job *base, uint32_t nthreads, void *(*fn)(void *))
{
    if (nthreads < 1) nthreads = 1;
    or_job *jobs = malloc(sizeof(or_job) * nthreads);
    pthread_t *th = malloc(sizeof(pthread_t) * nthreads);
    if (!jobs || !th) { free(jobs); free(th); return OR_ERR_NOMEM; }
    for (uint32_t t = 0; t < nthreads; t++) {
        jobs[t] = *base;
        jobs[t].tid = t;
        jobs[t].nthreads = nthreads;
        jobs[t].status = 0;
    }
    for (uint32_t t = 1; t < nthreads; t++) pthread_create(&th[t], NULL, fn, &jobs[t]);
    fn(&jobs[0]);
    for (uint32_t t = 1; t < nthreads; t++) pthread_join(th[t], NULL);
    int st = OR_OK, bad = 0;
    for (uint32_t t = 0; t < nthreads; t++) {
        if (jobs[t].status && !st) st = jobs[t].status;
        bad |= jobs[t].cx.bad_mu;
    }
    base->cx.bad_mu = bad;
    free(jobs);
    free(th);
    return st;
}

/*
 * Encode the chunks ids[0..n_ids) (all chunks if ids == NULL) and write them
 * back to back into out; offsets gets n_ids + 1 entries. Returns a status.
 */
int oracle_encode_chunks(const or_layout *lay, const void *kv, const void *mu,
                         const float *sigma, const uint64_t *counts,
                         const uint64_t *ids, uint64_t n_ids,
                         uint8_t *out, uint64_t out_capacity, uint64_t *offsets,
                         uint32_t nthreads)
{
    or_setup su;
    int st = setup_init(lay, sigma, counts, &su);
    if (st) return st;
    uint64_t *all = NULL;
    if (!ids) {
        n_ids = su.g.n_chunks;
        all = malloc(sizeof(uint64_t) * (n_ids ? n_ids : 1));
        for (uint64_t k = 0; k < n_ids; k++) all[k] = k;
        ids = all;
    }
    or_job jb;
    memset(&jb, 0, sizeof jb);
    jb.cx.g = &su.g; jb.cx.md = &su.md; jb.cx.kv = kv; jb.cx.mu = mu; jb.cx.rs_all = su.rs;
    jb.ids = ids; jb.n_ids = n_ids;
    jb.bufs = calloc(n_ids ? n_ids : 1, sizeof(uint8_t *));
    jb.sizes = calloc(n_ids ? n_ids : 1, sizeof(uint64_t));
    st = run_jobs(&jb, nthreads, encode_worker);
    offsets[0] = 0;
    for (uint64_t i = 0; i < n_ids; i++) {
        uint64_t sz = st ? 0 : jb.sizes[i];
        offsets[i + 1] = offsets[i] + sz;
        if (!st && offsets[i + 1] > out_capacity) st = OR_ERR_CAPACITY;
        if (!st) memcpy(out + offsets[i], jb.bufs[i], sz);
    }
    for (uint64_t i = 0; i < n_ids; i++) free(jb.bufs[i]);
    free(jb.bufs);
    free(jb.sizes);
    free(all);
    int bad = jb.cx.bad_mu;
    setup_free(&su);
    if (st) return st;
    return bad ? OR_ERR_NONFINITE_MU : OR_OK;
}

int oracle_encode(const or_layout *lay, const void *kv, const void *mu, const float *sigma,
                  const uint64_t *counts, uint8_t *out, uint64_t out_capacity,
                  uint64_t *offsets, uint32_t nthreads)
{
    return oracle_encode_chunks(lay, kv, mu, sigma, counts, NULL, 0, out, out_capacity,
                                offsets, nthreads);
}

/* Decode a whole bitstream (offsets has n_chunks + 1 entries) into kv_out. */
int oracle_decode(const or_layout *lay, const uint8_t *stream, uint64_t stream_bytes,
                  const uint64_t *offsets, const void *mu, const float *sigma,
                  const uint64_t *counts, void *kv_out, uint32_t nthreads)
{
    or_setup su;
    int st = setup_init(lay, sigma, counts, &su);
    if (st) return st;
    uint64_t n = su.g.n_chunks;
    uint64_t *all = malloc(sizeof(uint64_t) * (n ? n : 1));
    for (uint64_t k = 0; k < n; k++) all[k] = k;
    if (n && offsets[0] != 0) { free(all); setup_free(&su); return OR_ERR_CORRUPT; }
    or_job jb;
    memset(&jb, 0, sizeof jb);
    jb.cx.g = &su.g; jb.cx.md = &su.md; jb.cx.mu = mu; jb.cx.rs_all = su.rs;
    jb.ids = all; jb.n_ids = n;
    jb.stream = stream; jb.offsets = offsets; jb.stream_bytes = stream_bytes;
    jb.kv_out = kv_out;
    st = run_jobs(&jb, nthreads, decode_worker);
    int bad = jb.cx.bad_mu;
    free(all);
    setup_free(&su);
    if (st) return st;
    return bad ? OR_ERR_NONFINITE_MU : OR_OK;
}

/*
 * Decode the chunks ids[0..n_ids) of a full bitstream; chunk ids[i] is written
 * chunk-locally at pages_out + i * tokens_per_chunk * HD codes.
 */
int oracle_decode_pages(const or_layout *lay, const uint8_t *stream, uint64_t stream_bytes,
                        const uint64_t *offsets, const void *mu, const float *sigma,
                        const uint64_t *counts, const uint64_t *ids, uint64_t n_ids,
                        void *pages_out, uint32_t nthreads)
{
    or_setup su;
    int st = setup_init(lay, sigma, counts, &su);
    if (st) return st;
    for (uint64_t i = 0; i < n_ids; i++)
        if (ids[i] >= su.g.n_chunks) { setup_free(&su); return OR_ERR_INVALID_ARG; }
    or_job jb;
    memset(&jb, 0, sizeof jb);
    jb.cx.g = &su.g; jb.cx.md = &su.md; jb.cx.mu = mu; jb.cx.rs_all = su.rs;
    jb.ids = ids; jb.n_ids = n_ids;
    jb.stream = stream; jb.offsets = offsets; jb.stream_bytes = stream_bytes;
    jb.kv_out = pages_out;
    jb.pages = 1;
    jb.page_elems = (uint64_t)lay->tokens_per_chunk * su.g.HD;
    st = run_jobs(&jb, nthreads, decode_worker);
    int bad = jb.cx.bad_mu;
    setup_free(&su);
    if (st) return st;
    return bad ? OR_ERR_NONFINITE_MU : OR_OK;
}

/* ------------------------------------------- ideal cross-entropy (double) */

/* Phi(b) - Phi(a) for a <= b, arranged to avoid cancellation in the tails. */
static double gauss_mass(double a, double b)
{
    const double r2 = 0.70710678118654752440;
    if (a >= 0) return 0.5 * (erfc(a * r2) - erfc(b * r2));
    if (b <= 0) return 0.5 * (erfc(-b * r2) - erfc(-a * r2));
    return 1.0 - 0.5 * erfc(b * r2) - 0.5 * erfc(-a * r2);
}

/*
 * Sum over all elements of -log2 q(x), with q the real-valued mixture
 * (w_n N(mu, sigma^2) + w_w N(mu, 9 sigma^2) + w_h p_hat)/100 integrated over
 * each code's rounding interval: the code length an ideal arithmetic coder
 * would reach under the model (the information-theory section of the
 * 推测性KV编码 blog: bits = cross-entropy). Returns +inf if some element has
 * zero model mass.
 */
double oracle_ideal_bits(const or_layout *lay, const void *kv, const void *mu,
                         const float *sigma, const uint64_t *counts)
{
    or_geom g;
    if (geom_init(lay, &g)) return NAN;
    uint64_t total = 0;
    if (lay->w_h) for (uint32_t b = 0; b < g.d.N; b++) total += counts[b];
    uint64_t n_el = (uint64_t)lay->n_layers * lay->n_kv * lay->n_tokens * g.HD;
    double bits = 0.0;
    for (uint64_t i = 0; i < n_el; i++) {
        double s = sigma[sigma_index(&g, i)];
        uint32_t code = load_code(&g, kv, i);
        uint32_t mc = load_code(&g, mu, i);
        double m = code_is_finite(lay->dtype, mc) ? oracle_value(lay->dtype, mc) : 0.0;
        uint32_t o = oracle_ord(lay->dtype, code);
        double lo = oracle_edge(lay->dtype, o), hi = oracle_edge(lay->dtype, o + 1);
        double q = 0.0;
        if (hi > lo) {
            q += lay->w_n / 100.0 * gauss_mass((lo - m) / s, (hi - m) / s);
            q += lay->w_w / 100.0 * gauss_mass((lo - m) / (3 * s), (hi - m) / (3 * s));
        }
        if (lay->w_h && total) q += lay->w_h / 100.0 * (double)counts[code] / (double)total;
        bits += -log2(q);
    }
    return bits;
}

/* Sum over elements of -log2(f/M): the code length of the integer model. */
double oracle_model_bits(const or_layout *lay, const void *kv, const void *mu,
                         const float *sigma, const uint64_t *counts)
{
    or_setup su;
    if (setup_init(lay, sigma, counts, &su)) return NAN;
    uint64_t n_el = (uint64_t)lay->n_layers * lay->n_kv * lay->n_tokens * su.g.HD;
    double bits = 0.0, M = (double)(1ull << su.g.d.m);
    int bad = 0;
    for (uint64_t i = 0; i < n_el; i++) {
        float r = su.rs[sigma_index(&su.g, i)];
        uint32_t code = load_code(&su.g, kv, i);
        float m = mu_value(lay->dtype, load_code(&su.g, mu, i), &bad);
        uint32_t o = oracle_ord(lay->dtype, code);
        uint64_t c = cdf_at(&su.md, o, m, r);
        uint64_t f = cdf_at(&su.md, o + 1, m, r) - c;
        bits += -log2((double)f / M);
    }
    setup_free(&su);
    return bits;
}

/* ------------------------------------- inputs of the model: p_hat and sigma */

/*
 * counts[b] = number of codes equal to b (every bit pattern, NaN codes too):
 * the empirical marginal p_hat of the wiki's mixture section, before
 * normalisation. Adds to counts when accumulate is nonzero, else starts from 0.
 */
int oracle_histogram(uint32_t dtype, const void *codes, uint64_t n, uint64_t *counts,
                     int accumulate)
{
    if (dtype > DT_E4M3 || !counts || (n && !codes)) return OR_ERR_INVALID_ARG;
    uint32_t N = dtype_info(dtype).N;
    if (!accumulate) memset(counts, 0, sizeof(uint64_t) * N);
    for (uint64_t i = 0; i < n; ++i) {
        uint32_t b = dtype == DT_BF16 ? ((const uint16_t *)codes)[i] : ((const uint8_t *)codes)[i];
        counts[b] += 1;
    }
    return OR_OK;
}

/*
 * Frozen per-(layer, kv, head, channel) sigma from the first t_cal tokens:
 * the calibrate-once scale of the wiki's predictor-choice section and the
 * blog's predictor-engineering section. The blog's information-theory section
 * gives the Gaussian code length's optimum as the mean squared residual about
 * mu, so sigma is the root mean square of r = value(kv) - value(mu) over the
 * counted elements (both codes finite; mask byte nonzero when a mask is
 * given), summed in binary64 in token order and rounded to binary32 at the
 * end, then clamped into the valid range [2^-126, FLT_MAX] (2^-126 when
 * nothing is counted). With sigma blocks of B tokens (the position-aware
 * sigma the blog's limitations section names), each block gets its own sigma
 * from its own first t_cal tokens (t_cal <= B; a short last block uses all).
 */
int oracle_calibrate_sigma(const or_layout *lay, const void *kv, const void *mu,
                           const uint8_t *mask, uint64_t t_cal, float *sigma)
{
    or_geom g;
    int st = geom_init(lay, &g);
    if (st != OR_OK) return st;
    if (t_cal == 0 || t_cal > lay->n_tokens || !kv || !mu || !sigma) return OR_ERR_INVALID_ARG;
    if (lay->sigma_block && t_cal > lay->sigma_block) return OR_ERR_INVALID_ARG;
    uint64_t planes = (uint64_t)lay->n_layers * lay->n_kv;
    uint64_t B = lay->sigma_block ? lay->sigma_block : lay->n_tokens;
    for (uint64_t p = 0; p < planes; ++p) {
        for (uint64_t b = 0; b < g.n_sblk; ++b) {
            uint64_t t0 = b * B;
            uint64_t t1 = t0 + t_cal < lay->n_tokens ? t0 + t_cal : lay->n_tokens;
            for (uint64_t c = 0; c < g.HD; ++c) {
                double S = 0.0;
                uint64_t count = 0;
                for (uint64_t t = t0; t < t1; ++t) {
                    uint64_t el = (p * lay->n_tokens + t) * g.HD + c;
                    if (mask && mask[el] == 0) continue;
                    uint32_t kb = load_code(&g, kv, el), mb = load_code(&g, mu, el);
                    if (!code_is_finite(lay->dtype, kb) || !code_is_finite(lay->dtype, mb)) continue;
                    double r = (double)oracle_value(lay->dtype, kb) - (double)oracle_value(lay->dtype, mb);
                    S += r * r;
                    count += 1;
                }
                float s = 0x1p-126f;
                if (count) {
                    s = (float)sqrt(S / (double)count);
                    if (!(s >= 0x1p-126f)) s = 0x1p-126f;
                    if (s > 0x1.fffffep127f) s = 0x1.fffffep127f;
                }
                sigma[(p * g.n_sblk + b) * g.HD + c] = s;
            }
        }
    }
    return OR_OK;
}

/* ------------------- context page: requantising 2b-bit codes to b bits */

/*
 * The PM-KVQ section of the third page (progressive quantisation of the KV
 * cache, 16 -> 8 -> 4 -> 2 bits) lowers a 2b-bit code to b bits. Its
 * Equivalent Right Shift keeps the zero point and sets the new scale to
 * S_b = (2^b + 1) S_2b, which the page shows equals dequantising and
 * requantising; written here as exactly that: x = z + S_2b q (binary64),
 * q_b = round((x - z) / S_b). The two shift baselines the page's ablation
 * names are written as plain shifts: Direct Right Shift q >> b, and (this
 * build's reading of "rounding-corrected") Modified Right Shift
 * min((q + 2^(b-1)) >> b, 2^b - 1); both imply the scale 2^b S_2b.
 * Codes are packed LSB first (code i in bits [w i, w i + w) of the byte
 * string, w = 2b on input, b on output); one scale (and zero) per `group`
 * consecutive codes. mode: 0 ERS, 1 DRS, 2 MRS.
 */
int oracle_requantize(uint32_t mode, uint32_t b, const uint8_t *in, uint64_t n, uint8_t *out,
                      const float *scale_in, const float *zero_in, float *scale_out, uint64_t group)
{
    if (mode > 2 || !(b == 1 || b == 2 || b == 4 || b == 8) || group == 0) return OR_ERR_INVALID_ARG;
    if ((n * b) % 8 != 0 || (n && (!in || !out || !scale_in || !scale_out))) return OR_ERR_INVALID_ARG;
    const uint32_t w = 2 * b;
    uint64_t n_groups = (n + group - 1) / group;
    if (mode == 0)          /* dequantising needs finite, positive scales */
        for (uint64_t g = 0; g < n_groups; ++g)
            if (!(scale_in[g] > 0.0f && scale_in[g] <= 0x1.fffffep127f)) return OR_ERR_INVALID_ARG;
    memset(out, 0, n * b / 8);
    for (uint64_t i = 0; i < n; ++i) {
        uint64_t bit = i * w;
        uint32_t q = 0;
        for (uint32_t k = 0; k < w; ++k) q |= (uint32_t)((in[(bit + k) / 8] >> ((bit + k) % 8)) & 1u) << k;
        uint64_t g = i / group;
        uint32_t r;
        if (mode == 0) {
            double S2 = scale_in[g], z = zero_in ? zero_in[g] : 0.0;
            double Sb = (double)((1u << b) + 1u) * S2;
            double x = z + S2 * (double)q;
            r = (uint32_t)floor((x - z) / Sb + 0.5);
        } else if (mode == 1) {
            r = q >> b;
        } else {
            r = (q + (1u << (b - 1))) >> b;
            if (r > (1u << b) - 1u) r = (1u << b) - 1u;
        }
        uint64_t ob = i * b;
        for (uint32_t k = 0; k < b; ++k) out[(ob + k) / 8] |= (uint8_t)(((r >> k) & 1u) << ((ob + k) % 8));
    }
    for (uint64_t g = 0; g < n_groups; ++g)
        scale_out[g] = mode == 0 ? (float)((double)((1u << b) + 1u) * (double)scale_in[g])
                                 : (float)((double)(1u << b) * (double)scale_in[g]);
    return OR_OK;
}
