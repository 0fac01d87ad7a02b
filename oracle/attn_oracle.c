/*
 * attn_oracle.c -- CPU oracle for the fused low-precision attention forward pass.
 *
 * TEST INFRASTRUCTURE (see attn_oracle.h): plain, slow, obviously correct C.
 * Compiled with -ffp-contract=off so that every float expression rounds the
 * way it is written. Shares no code with the CUDA library.
 *
 * Readings of the pages where they are silent are stated beside the code that
 * takes them; each is also listed in the repository's design notes.
 */
#define _GNU_SOURCE
#include "attn_oracle.h"

#include <float.h>
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------------- */
/* threads                                                                   */
/* ------------------------------------------------------------------------- */
static int g_threads = 0;

int or_set_threads(int n) { g_threads = n > 0 ? n : 0; return or_threads(); }

int or_threads(void) {
    if (g_threads > 0) return g_threads;
    long c = sysconf(_SC_NPROCESSORS_ONLN);
    return c > 0 ? (int)c : 1;
}

typedef void (*unit_fn)(void* ctx, long unit);
typedef struct { unit_fn fn; void* ctx; long n; long next; } pool_t;

static void* pool_worker(void* arg) {
    pool_t* p = (pool_t*)arg;
    for (;;) {
        long u = __atomic_fetch_add(&p->next, 1, __ATOMIC_RELAXED);
        if (u >= p->n) break;
        p->fn(p->ctx, u);
    }
    return NULL;
}

static void parallel_for(long n, unit_fn fn, void* ctx) {
    int nt = or_threads();
    if (nt > 256) nt = 256;
    if (nt > n) nt = (int)n;
    pool_t p = {fn, ctx, n, 0};
    if (nt <= 1) { pool_worker(&p); return; }
    pthread_t th[256];
    int started = 0;
    for (int i = 0; i < nt - 1; i++)
        if (pthread_create(&th[started], NULL, pool_worker, &p) == 0) started++;
    pool_worker(&p);
    for (int i = 0; i < started; i++) pthread_join(th[i], NULL);
}

/* ------------------------------------------------------------------------- */
/* E4M3 ("Fused attention kernel", 8-bit forward pass: the e4m3 format).     */
/* The pages name the format only; the OCP 8-bit floating point definition   */
/* (E4M3FN) is taken: sign, 4 exponent bits with bias 7, 3 mantissa bits, no */
/* infinities, S.1111.111 is NaN, largest finite 448, subnormals 2^-9 apart. */
/* ------------------------------------------------------------------------- */
double or_e4m3_decode(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    double v = (e == 0) ? ldexp((double)m, -9)            /* m/8 * 2^-6        */
                        : ldexp(8.0 + m, e - 10);         /* (1+m/8) * 2^(e-7) */
    return s ? -v : v;
}

/* round half to even of a non-negative double that is exact */
static double rne_int(double q) {
    double n = floor(q);
    double f = q - n;
    if (f > 0.5 || (f == 0.5 && fmod(n, 2.0) != 0.0)) n += 1.0;
    return n;
}

/* Round to nearest, ties to even; finite values beyond 448 and infinities
 * saturate to +-448 (reading: the "satfinite" conversion); NaN -> 0x7F. */
uint8_t or_e4m3_encode(float x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7E;
    if (a < 0.015625) {                         /* below 2^-6: subnormal grid 2^-9 */
        double n = rne_int(a * 512.0);          /* exact scaling by a power of two */
        return sign | (uint8_t)n;               /* n == 8 is the smallest normal, 0x08 */
    }
    int e;
    double f = frexp(a, &e);                    /* a = f * 2^e, f in [0.5, 1) */
    int E = e - 1;                              /* a = (2f) * 2^E, 2f in [1, 2) */
    double n = rne_int((2.0 * f - 1.0) * 8.0);  /* mantissa in eighths, exact */
    if (n >= 8.0) { E += 1; n = 0.0; }
    int code = ((E + 7) << 3) | (int)n;
    if (code > 0x7E) code = 0x7E;
    return sign | (uint8_t)code;
}

/* E2M1, the element format of NVFP4 (FLAMIA section 2: NVFP4 blocks of 16
 * elements; the OCP 4-bit floating point definition is taken): sign, 2
 * exponent bits with bias 1, 1 mantissa bit; magnitudes 0, 0.5, 1, 1.5, 2,
 * 3, 4, 6; no infinities or NaN. */
double or_e2m1_decode(uint8_t c) {
    int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

/* Nearest magnitude, ties to the even code (mantissa bit 0); beyond 6 and
 * infinities saturate to 6 (satfinite); the sign is kept, zero included;
 * NaN -> 0x7 (the format has none; a quantiser block holding one is reported). */
uint8_t or_e2m1_encode(float x) {
    if (isnan(x)) return 0x7;
    uint8_t sign = signbit(x) ? 0x8 : 0x0;
    double a = fabs((double)x);
    if (a >= 6.0) return sign | 0x7;
    uint8_t best = 0;
    double bd = INFINITY;
    for (uint8_t c = 0; c < 8; c++) {
        double dd = fabs(a - or_e2m1_decode(c));
        if (dd < bd || (dd == bd && (c & 1) == 0)) { bd = dd; best = c; }
    }
    return sign | best;
}

void or_e4m3_encode_range(uint64_t start, uint64_t count, uint8_t* out) {
    for (uint64_t i = 0; i < count; i++) {
        uint32_t bits = (uint32_t)(start + i);
        float x;
        memcpy(&x, &bits, 4);
        out[i] = or_e4m3_encode(x);
    }
}

/* E8M0 shared exponent of a 32-element MX block (FLAMIA, section 2:
 * microscaling formats use 32-element blocks with one shared scale).
 * The pages do not fix the exponent rule. Default reading: the smallest X with
 * amax <= 448 * 2^X, so that no element saturates; with amax = m * 2^E,
 * m in [1, 2): X = E - 8 if m <= 1.75 (448 = 1.75 * 2^8) else E - 7.
 * The OCP MX floor rule X = E - 8 is kept as a switch. amax == 0 -> -127. */
int or_e8m0_exponent(float amax, int rule) {
    if (!(amax > 0.0f)) return -127;
    int e;
    double f = frexp((double)amax, &e);
    int E = e - 1;
    double m = 2.0 * f;
    int X = (rule == OR_MX_RULE_OCP_FLOOR) ? E - 8 : (m <= 1.75 ? E - 8 : E - 7);
    if (X < -127) X = -127;
    if (X > 127) X = 127;
    return X;
}

/* fp32 -> bf16, round to nearest even (the output format: BF16) */
uint16_t or_bf16_rne(float x) {
    uint32_t u;
    memcpy(&u, &x, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------------- */
/* Rotation ("Fused attention kernel", 8-bit forward pass: incoherent        */
/* processing multiplies Q and K by a random sign diagonal and a Hadamard    */
/* matrix; the product cancels in Q K^T).                                    */
/* Readings: the signs are the top bits of a SplitMix64 stream (Steele, Lea, */
/* Flood 2014) started at the seed; the Hadamard matrix is the unnormalised  */
/* Sylvester one (H H^T = d I), applied as a fast Walsh-Hadamard transform   */
/* with stages h = 1, 2, 4, ..., d/2 in that order, each butterfly           */
/* (a, b) -> (a + b, a - b) rounded to fp32. The 1/d is left to the score    */
/* scale. The pages ask for a Hadamard matrix, not for a row order: at       */
/* d = 128 the rotation stores the transform's output channel pi(p) at      */
/* channel p, pi swapping the 3-bit fields at bits 1-3 and 4-6 of the index  */
/* (rows of the Sylvester matrix permuted: still a Hadamard matrix, R R^T =  */
/* d I, so the rotation still cancels in Q K^T); at d = 64 pi is the         */
/* identity.                                                                 */
/* ------------------------------------------------------------------------- */
uint64_t or_splitmix64_next(uint64_t* state) {
    uint64_t z = (*state += 0x9E3779B97F4A7C15ULL);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

void or_signs(uint64_t seed, int d, float* s) {
    uint64_t st = seed;
    for (int j = 0; j < d; j++) s[j] = (or_splitmix64_next(&st) >> 63) ? -1.0f : 1.0f;
}

void or_fwht_f32(float* x, int d) {
    for (int h = 1; h < d; h <<= 1)
        for (int i = 0; i < d; i++)
            if (!(i & h)) {
                float a = x[i], b = x[i + h];
                x[i] = a + b;
                x[i + h] = a - b;
            }
}

int or_rotation_channel(int p, int d) {
    if (d != 128) return p;
    return (p & 1) | (((p >> 4) & 7) << 1) | (((p >> 1) & 7) << 4);
}

/* ------------------------------------------------------------------------- */
/* documents (FLAMIA abstract and section 4.1: packed documents, scales kept */
/* document-local, no repacking). cu_seqlens == NULL means one document.     */
/* ------------------------------------------------------------------------- */
static int doc_of(const int32_t* cu, int nd, int t) {
    int lo = 0, hi = nd - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

long or_num_blocks(const int32_t* cu, int nd, int T, int block) {
    if (!cu) return (T + block - 1) / block;
    long n = 0;
    for (int i = 0; i < nd; i++) n += (cu[i + 1] - cu[i] + block - 1) / block;
    return n;
}

typedef struct { int nd; int32_t* cu; } docs_t;

static docs_t docs_make(const int32_t* cu, int nd, int T) {
    docs_t D;
    if (!cu) { nd = 1; }
    D.nd = nd;
    D.cu = (int32_t*)malloc(sizeof(int32_t) * (nd + 1));
    if (!cu) { D.cu[0] = 0; D.cu[1] = T; }
    else memcpy(D.cu, cu, sizeof(int32_t) * (nd + 1));
    return D;
}

/* block offset of document `doc` for blocks of `block` tokens */
static long block_offset(const docs_t* D, int doc, int block) {
    long n = 0;
    for (int i = 0; i < doc; i++) n += (D->cu[i + 1] - D->cu[i] + block - 1) / block;
    return n;
}

/* ------------------------------------------------------------------------- */
/* O-2 quantiser                                                             */
/* ------------------------------------------------------------------------- */
typedef struct {
    const float* x; int T, H, d; docs_t D;
    int layout, block, rotate, mx_rule;
    float signs[256];
    uint8_t* codes; float* sf; uint8_t* su;
    int err;
} quant_ctx;

static void rotated_row(const quant_ctx* c, int t, int h, float* y) {
    const float* src = c->x + ((long)t * c->H + h) * c->d;
    for (int j = 0; j < c->d; j++) y[j] = c->rotate ? c->signs[j] * src[j] : src[j];
    if (c->rotate) {
        float t[256];
        or_fwht_f32(y, c->d);
        for (int p = 0; p < c->d; p++) t[p] = y[or_rotation_channel(p, c->d)];
        for (int p = 0; p < c->d; p++) y[p] = t[p];
    }
}

/* E4M3 token block (reading: scale = amax / 448 with IEEE division, codes from
 * y * (448 / amax); blocks start at the document start, the last one may be
 * partial; amax == 0 gives scale 0 and zero codes; a non-finite amax is an
 * error). Unit = (document, head). */
static void quant_tokblock_unit(void* vc, long u) {
    quant_ctx* c = (quant_ctx*)vc;
    int doc = (int)(u / c->H), h = (int)(u % c->H);
    int s = c->D.cu[doc], L = c->D.cu[doc + 1] - s, d = c->d, b = c->block;
    long boff = block_offset(&c->D, doc, b);
    long NB = block_offset(&c->D, c->D.nd, b);
    float* y = (float*)malloc(sizeof(float) * (size_t)b * d);
    for (int blk = 0; blk * b < L; blk++) {
        int n = L - blk * b < b ? L - blk * b : b;
        float amax = 0.0f;
        for (int r = 0; r < n; r++) {
            rotated_row(c, s + blk * b + r, h, y + (long)r * d);
            for (int j = 0; j < d; j++) {
                float a = fabsf(y[(long)r * d + j]);
                if (!(a <= amax)) amax = a;        /* NaN propagates */
            }
        }
        float scale, inv;
        if (!isfinite(amax)) { __atomic_store_n(&c->err, OR_ERR_NONFINITE, __ATOMIC_RELAXED); scale = NAN; inv = 0.0f; }
        else if (amax == 0.0f) { scale = 0.0f; inv = 0.0f; }
        else { inv = 448.0f / amax; scale = amax / 448.0f; }
        c->sf[(long)h * NB + boff + blk] = scale;
        for (int r = 0; r < n; r++) {
            uint8_t* dst = c->codes + ((long)(s + blk * b + r) * c->H + h) * d;
            for (int j = 0; j < d; j++) dst[j] = or_e4m3_encode(y[(long)r * d + j] * inv);
        }
    }
    free(y);
}

static float pow2f_exact(int k) { return ldexpf(1.0f, k); }

/* MX row32: one E8M0 exponent per (token, head, 32 consecutive channels);
 * codes = E4M3(y * 2^-X). Unit = token. */
static void quant_mxrow_unit(void* vc, long t) {
    quant_ctx* c = (quant_ctx*)vc;
    int d = c->d;
    float y[256];
    for (int h = 0; h < c->H; h++) {
        rotated_row(c, (int)t, h, y);
        for (int g = 0; g < d / 32; g++) {
            float amax = 0.0f;
            for (int j = 0; j < 32; j++) { float a = fabsf(y[g * 32 + j]); if (!(a <= amax)) amax = a; }
            if (!isfinite(amax)) __atomic_store_n(&c->err, OR_ERR_NONFINITE, __ATOMIC_RELAXED);
            int X = or_e8m0_exponent(amax, c->mx_rule);
            c->su[((long)t * c->H + h) * (d / 32) + g] = (uint8_t)(X + 127);
            float pw = pow2f_exact(-X);
            uint8_t* dst = c->codes + ((long)t * c->H + h) * d + g * 32;
            for (int j = 0; j < 32; j++) dst[j] = or_e4m3_encode(y[g * 32 + j] * pw);
        }
    }
}

/* MX col32 (V): one E8M0 exponent per (32 document-local tokens, head,
 * channel), the blocks running along the sequence, which is the contraction
 * axis of P V. Unit = (document, head). */
static void quant_mxcol_unit(void* vc, long u) {
    quant_ctx* c = (quant_ctx*)vc;
    int doc = (int)(u / c->H), h = (int)(u % c->H);
    int s = c->D.cu[doc], L = c->D.cu[doc + 1] - s, d = c->d;
    long goff = block_offset(&c->D, doc, 32);
    long NG = block_offset(&c->D, c->D.nd, 32);
    float y[32][256];
    for (int g = 0; g * 32 < L; g++) {
        int n = L - g * 32 < 32 ? L - g * 32 : 32;
        for (int r = 0; r < n; r++) rotated_row(c, s + g * 32 + r, h, y[r]);
        for (int j = 0; j < d; j++) {
            float amax = 0.0f;
            for (int r = 0; r < n; r++) { float a = fabsf(y[r][j]); if (!(a <= amax)) amax = a; }
            if (!isfinite(amax)) __atomic_store_n(&c->err, OR_ERR_NONFINITE, __ATOMIC_RELAXED);
            int X = or_e8m0_exponent(amax, c->mx_rule);
            c->su[((long)h * NG + goff + g) * d + j] = (uint8_t)(X + 127);
            float pw = pow2f_exact(-X);
            for (int r = 0; r < n; r++)
                c->codes[((long)(s + g * 32 + r) * c->H + h) * d + j] = or_e4m3_encode(y[r][j] * pw);
        }
    }
}

/* MX token layout (V of the causal-exact MX mode): one E8M0 exponent per
 * (token, head) over all d channels, so that every scale depends on its own
 * token only (FLAMIA sections 1 and 4.5: exact scaling removes within-block
 * dependencies); codes = E4M3(y * 2^-X). Scales [H][T]. Unit = token. */
static void quant_mxtok_unit(void* vc, long t) {
    quant_ctx* c = (quant_ctx*)vc;
    int d = c->d;
    float y[256];
    for (int h = 0; h < c->H; h++) {
        rotated_row(c, (int)t, h, y);
        float amax = 0.0f;
        for (int j = 0; j < d; j++) { float a = fabsf(y[j]); if (!(a <= amax)) amax = a; }
        if (!isfinite(amax)) __atomic_store_n(&c->err, OR_ERR_NONFINITE, __ATOMIC_RELAXED);
        int X = or_e8m0_exponent(amax, c->mx_rule);
        c->su[(long)h * c->T + t] = (uint8_t)(X + 127);
        float pw = pow2f_exact(-X);
        uint8_t* dst = c->codes + ((long)t * c->H + h) * d;
        for (int j = 0; j < d; j++) dst[j] = or_e4m3_encode(y[j] * pw);
    }
}

/* NVFP4 (Q and K of the mixed NVFP4/FP8 path; FLAMIA sections 1 and 2:
 * 16-element blocks with a shared scale plus a tensor-level scale, NVFP4 for
 * Q K^T and 8-bit operands elsewhere). Readings: the tensor-level scale is
 * kept per document-local 128-token block and head (the token-block scaling
 * the pages reuse, document-local like every other scale here), fp32
 * s_t = amax / (448 * 6); each 16-channel group of a row takes the E4M3 scale
 * sf = E4M3(max |z|) with z = fl32(y * fl32(448 / amax)) (the same form as the
 * E4M3 token-block codes), and its codes e = E2M1(fl32(z * fl32(6 / dec(sf)))),
 * zero when sf decodes to 0. Value = e2m1(e) * dec(sf) * s_t. Unit =
 * (document, head). */
static void quant_nvfp4_unit(void* vc, long u) {
    quant_ctx* c = (quant_ctx*)vc;
    int doc = (int)(u / c->H), h = (int)(u % c->H);
    int s = c->D.cu[doc], L = c->D.cu[doc + 1] - s, d = c->d;
    long boff = block_offset(&c->D, doc, 128);
    long NB = block_offset(&c->D, c->D.nd, 128);
    float* y = (float*)malloc(sizeof(float) * 128 * (size_t)d);
    for (int blk = 0; blk * 128 < L; blk++) {
        int n = L - blk * 128 < 128 ? L - blk * 128 : 128;
        float amax = 0.0f;
        for (int r = 0; r < n; r++) {
            rotated_row(c, s + blk * 128 + r, h, y + (long)r * d);
            for (int j = 0; j < d; j++) {
                float a = fabsf(y[(long)r * d + j]);
                if (!(a <= amax)) amax = a;
            }
        }
        float st, inv;
        if (!isfinite(amax)) { __atomic_store_n(&c->err, OR_ERR_NONFINITE, __ATOMIC_RELAXED); st = NAN; inv = 0.0f; }
        else if (amax == 0.0f) { st = 0.0f; inv = 0.0f; }
        else { inv = 448.0f / amax; st = amax / 2688.0f; }
        c->sf[(long)h * NB + boff + blk] = st;
        for (int r = 0; r < n; r++) {
            long t = s + blk * 128 + r;
            uint8_t* dst = c->codes + (t * c->H + h) * (d / 2);
            for (int g = 0; g < d / 16; g++) {
                float z[16], gmax = 0.0f;
                for (int i = 0; i < 16; i++) {
                    z[i] = y[(long)r * d + 16 * g + i] * inv;
                    float a = fabsf(z[i]);
                    if (!(a <= gmax)) gmax = a;
                }
                uint8_t sf = or_e4m3_encode(gmax);
                c->su[(t * c->H + h) * (d / 16) + g] = sf;
                double sv = or_e4m3_decode(sf);
                float rr = sv > 0.0 ? 6.0f / (float)sv : 0.0f;
                for (int i = 0; i < 16; i += 2) {
                    uint8_t lo = sv > 0.0 ? or_e2m1_encode(z[i] * rr) : 0;
                    uint8_t hi = sv > 0.0 ? or_e2m1_encode(z[i + 1] * rr) : 0;
                    dst[8 * g + i / 2] = (uint8_t)(lo | (hi << 4));
                }
            }
        }
    }
    free(y);
}

int or_quantize(const float* x, int T, int H, int d, const int32_t* cu, int nd,
                int layout, int block, int rotate, uint64_t seed, int mx_rule,
                uint8_t* codes, float* scales_f32, uint8_t* scales_u8) {
    if (d < 1 || d > 256 || (d & (d - 1)) || T < 0 || H < 1) return OR_ERR_ARG;
    if (layout == OR_E4M3_TOKBLOCK && (block < 1 || !scales_f32)) return OR_ERR_ARG;
    if ((layout == OR_MX_ROW32 || layout == OR_MX_COL32) && (d % 32 || !scales_u8)) return OR_ERR_ARG;
    if (layout == OR_MX_TOKEN && !scales_u8) return OR_ERR_ARG;
    if (layout == OR_NVFP4 && (d % 16 || block != 128 || !scales_f32 || !scales_u8)) return OR_ERR_ARG;
    quant_ctx c;
    memset(&c, 0, sizeof(c));
    c.x = x; c.T = T; c.H = H; c.d = d; c.D = docs_make(cu, nd, T);
    c.layout = layout; c.block = block; c.rotate = rotate; c.mx_rule = mx_rule;
    c.codes = codes; c.sf = scales_f32; c.su = scales_u8;
    or_signs(seed, d, c.signs);
    if (layout == OR_E4M3_TOKBLOCK) parallel_for((long)c.D.nd * H, quant_tokblock_unit, &c);
    else if (layout == OR_MX_ROW32) parallel_for(T, quant_mxrow_unit, &c);
    else if (layout == OR_MX_COL32) parallel_for((long)c.D.nd * H, quant_mxcol_unit, &c);
    else if (layout == OR_MX_TOKEN) parallel_for(T, quant_mxtok_unit, &c);
    else if (layout == OR_NVFP4) parallel_for((long)c.D.nd * H, quant_nvfp4_unit, &c);
    else { free(c.D.cu); return OR_ERR_ARG; }
    free(c.D.cu);
    return c.err;
}

/* ------------------------------------------------------------------------- */
/* O-1: FP64 softmax attention, the plain definition. Per document and head: */
/* S = scale * Q K^T; causal masks key j > query i (positions local to the   */
/* document, top-left aligned); O = softmax(S) V; lse = max + log(sum).       */
/* ------------------------------------------------------------------------- */
typedef struct {
    const double *q, *k, *v; int T, H, d; docs_t D; int causal; double scale;
    const int32_t* rows; int nrows; double *o, *lse;
} fp64_ctx;

static void fp64_unit(void* vc, long u) {
    fp64_ctx* c = (fp64_ctx*)vc;
    int ri = (int)(u / c->H), h = (int)(u % c->H), d = c->d, H = c->H;
    int t = c->rows ? c->rows[ri] : ri;
    int doc = doc_of(c->D.cu, c->D.nd, t);
    int s0 = c->D.cu[doc], L = c->D.cu[doc + 1] - s0, i = t - s0;
    int nk = c->causal ? i + 1 : L;
    double* sc = (double*)malloc(sizeof(double) * (nk > 0 ? nk : 1));
    const double* qr = c->q + ((long)t * H + h) * d;
    double m = -INFINITY;
    for (int j = 0; j < nk; j++) {
        const double* kr = c->k + ((long)(s0 + j) * H + h) * d;
        double acc = 0.0;
        for (int x = 0; x < d; x++) acc += qr[x] * kr[x];
        sc[j] = c->scale * acc;
        if (sc[j] > m) m = sc[j];
    }
    double l = 0.0;
    double* out = c->o + ((long)ri * H + h) * d;
    for (int x = 0; x < d; x++) out[x] = 0.0;
    for (int j = 0; j < nk; j++) {
        double p = exp(sc[j] - m);
        l += p;
        const double* vr = c->v + ((long)(s0 + j) * H + h) * d;
        for (int x = 0; x < d; x++) out[x] += p * vr[x];
    }
    for (int x = 0; x < d; x++) out[x] = nk > 0 ? out[x] / l : 0.0;
    c->lse[(long)h * c->nrows + ri] = nk > 0 ? m + log(l) : -INFINITY;
    free(sc);
}

void or_attention_fp64(const double* q, const double* k, const double* v, int T, int H, int d,
                       const int32_t* cu, int nd, int causal, double scale,
                       const int32_t* rows, int nrows, double* o, double* lse) {
    fp64_ctx c = {q, k, v, T, H, d, docs_make(cu, nd, T), causal, scale, rows, rows ? nrows : T, o, lse};
    parallel_for((long)c.nrows * H, fp64_unit, &c);
    free(c.D.cu);
}

/* ------------------------------------------------------------------------- */
/* O-1 backward: the gradients of the plain definition above for an upstream */
/* gradient dO (the step after the forward; FLAMIA section 1 lists the       */
/* backward among its kernels). With P = softmax(S) row-wise, S = scale Q K^T */
/* (masked as in the forward) and O = P V:                                   */
/*   dV = P^T dO;  dP = dO V^T;  D_i = sum_j P_ij dP_ij  (= dO_i . O_i);       */
/*   dS = P o (dP - D);  dQ = scale dS K;  dK = scale dS^T Q.                  */
/* One (document, head) per unit, so a thread owns that unit's dK, dV rows.  */
/* With a given output o (the forward's stored output, as a training step    */
/* keeps it), D_i = dO_i . o_i is taken from that o instead; everything else */
/* is unchanged.                                                             */
/* ------------------------------------------------------------------------- */
typedef struct {
    const double *q, *k, *v, *dout; int T, H, d; docs_t D; int causal; double scale;
    double *dq, *dk, *dv;
    const double* o;   /* NULL: D from P and dP */
} bwd_ctx;

static void bwd_unit(void* vc, long u) {
    bwd_ctx* c = (bwd_ctx*)vc;
    int doc = (int)(u / c->H), h = (int)(u % c->H), d = c->d, H = c->H;
    int s0 = c->D.cu[doc], L = c->D.cu[doc + 1] - s0;
    if (L <= 0) return;
    double* p = (double*)malloc(sizeof(double) * L);
    double* dp = (double*)malloc(sizeof(double) * L);
    for (int j = 0; j < L; j++) {
        double* dkr = c->dk + ((long)(s0 + j) * H + h) * d;
        double* dvr = c->dv + ((long)(s0 + j) * H + h) * d;
        for (int x = 0; x < d; x++) dkr[x] = dvr[x] = 0.0;
    }
    for (int i = 0; i < L; i++) {
        int nk = c->causal ? i + 1 : L;
        const double* qr = c->q + ((long)(s0 + i) * H + h) * d;
        const double* gr = c->dout + ((long)(s0 + i) * H + h) * d;
        double m = -INFINITY;
        for (int j = 0; j < nk; j++) {
            const double* kr = c->k + ((long)(s0 + j) * H + h) * d;
            double acc = 0.0;
            for (int x = 0; x < d; x++) acc += qr[x] * kr[x];
            p[j] = c->scale * acc;
            if (p[j] > m) m = p[j];
        }
        double l = 0.0;
        for (int j = 0; j < nk; j++) {
            p[j] = exp(p[j] - m);
            l += p[j];
        }
        double D = 0.0;
        for (int j = 0; j < nk; j++) {
            p[j] /= l;
            const double* vr = c->v + ((long)(s0 + j) * H + h) * d;
            double acc = 0.0;
            for (int x = 0; x < d; x++) acc += gr[x] * vr[x];
            dp[j] = acc;
            D += p[j] * dp[j];
        }
        if (c->o) {
            const double* orow = c->o + ((long)(s0 + i) * H + h) * d;
            D = 0.0;
            for (int x = 0; x < d; x++) D += gr[x] * orow[x];
        }
        double* dqr = c->dq + ((long)(s0 + i) * H + h) * d;
        for (int x = 0; x < d; x++) dqr[x] = 0.0;
        for (int j = 0; j < nk; j++) {
            const double ds = p[j] * (dp[j] - D);
            const double* kr = c->k + ((long)(s0 + j) * H + h) * d;
            double* dkr = c->dk + ((long)(s0 + j) * H + h) * d;
            double* dvr = c->dv + ((long)(s0 + j) * H + h) * d;
            for (int x = 0; x < d; x++) {
                dqr[x] += c->scale * ds * kr[x];
                dkr[x] += c->scale * ds * qr[x];
                dvr[x] += p[j] * gr[x];
            }
        }
    }
    free(p);
    free(dp);
}

void or_attention_fp64_bwd(const double* q, const double* k, const double* v, const double* dout, int T, int H,
                           int d, const int32_t* cu, int nd, int causal, double scale, double* dq, double* dk,
                           double* dv) {
    or_attention_fp64_bwd_o(q, k, v, dout, NULL, T, H, d, cu, nd, causal, scale, dq, dk, dv);
}

void or_attention_fp64_bwd_o(const double* q, const double* k, const double* v, const double* dout,
                             const double* o, int T, int H, int d, const int32_t* cu, int nd, int causal,
                             double scale, double* dq, double* dk, double* dv) {
    bwd_ctx c = {q, k, v, dout, T, H, d, docs_make(cu, nd, T), causal, scale, dq, dk, dv, o};
    parallel_for((long)c.D.nd * H, bwd_unit, &c);
    free(c.D.cu);
}

/* ------------------------------------------------------------------------- */
/* Bit-level exponentials for inference (FLAMIA section 1: two bit-level      */
/* exponential approximations; section 4.3: log-domain probability            */
/* quantisation; section 4.4: Schraudolph's approximation, Mitchell-P).       */
/*                                                                           */
/* A binary floating-point number's bit pattern, read as a fixed-point        */
/* number, is its log2 plus the exponent bias, interpolated linearly between  */
/* powers of two (Mitchell's logarithm). Read backwards, writing 2^23 (u+127) */
/* into an fp32's bits gives 2^floor(u) (1 + frac(u)) ~ 2^u (Schraudolph);    */
/* an E4M3 code (3 mantissa bits, bias 7) of 2^u is round(8 (u + 7)).         */
/* Relative to 2^u that interpolation is (1 + f) 2^-f, f = frac(u), too large */
/* by up to 6.2%; evaluating it at u = x - delta scales it by 2^-delta, and   */
/* delta = log2(1/2 + 3 / (8 ln 2)) minimises the mean square relative error  */
/* over f uniform on [0, 1) (the minimiser of the quadratic in K = 2^-delta   */
/* is K = E[g] / E[g^2], g = (1 + f) 2^-f, E[g] = 1 / (2 ln^2 2),             */
/* E[g^2] = (2 ln 2 + 3/2) / (8 ln^3 2)).                                     */
/* Readings: u resolved to 2^-14 in the fp32 form (its bits carry 23          */
/* fractional bits; the reading keeps the whole fp32 range at 2^-14, well     */
/* below E4M3's 2^-3); ties to even at both roundings; the lower limits keep  */
/* -inf and tiny probabilities at the smallest normal fp32 (E4M3 code 0) and  */
/* at code 0.                                                                 */
/* ------------------------------------------------------------------------- */
float or_exp2_schraudolph(double x) {
    double u = x - OR_SCHRAUDOLPH_DELTA;
    if (!(u > -126.0)) u = -126.0;                        /* also -inf, NaN */
    double n = nearbyint(ldexp(u + 126.0, 14));          /* to nearest even */
    double fl = floor(n / 16384.0);
    double frac = (n - fl * 16384.0) / 16384.0;
    return (float)ldexp(1.0 + frac, (int)fl - 126);
}

uint8_t or_exp2_mitchell_code(double x) {
    double y = 8.0 * (x - OR_SCHRAUDOLPH_DELTA) + 56.0;
    if (!(y > 0.0)) return 0;                             /* also -inf, NaN */
    if (y > 126.0) y = 126.0;
    return (uint8_t)nearbyint(y);
}

/* ------------------------------------------------------------------------- */
/* O-3: the running-softmax loop over quantised operands, the way the kernel */
/* tiles it ("Fused attention kernel", Implementation sketch: running max m, */
/* rescale alpha = exp(m_old - m_new) applied to the old output, every key   */
/* block scored, one normalisation at the end, lse = m + log l).             */
/*                                                                           */
/* Per query row, key tiles of 128 document-local keys in ascending order:   */
/*   S_t   = fl32(sum_c qhat_c khat_c)      (fp64 sum, one rounding: the     */
/*           tensor core's fp32 accumulation, up to its summation order)      */
/*   s'_t  = fl32(S_t * fl32(qs * ks_t * C)), C = softmax_scale*log2(e)/d for  */
/*           rotated Q, K (H H^T = d I) and softmax_scale*log2(e) otherwise;  */
/*           E4M3 layouts multiply the block scales here, MX layouts carry    */
/*           them inside qhat, khat ("folding score scales", FLAMIA 4.3)      */
/*   masked keys (causal t > i, keys past the document end): s' = -inf        */
/*   m'    = max(m, max_t s'_t) if that exceeds fl32(m + tau), else m:        */
/*           the reference maximum moves only by more than tau (log2 units;   */
/*           tau = 0 is the exact running max); alpha = fl32(2^(m - m'))       */
/*   pt_t  = 2^(s'_t - m' + 8)              (probabilities prescaled by 2^8)  */
/*   Phat  = E4M3(fl32(pt_t * r_t))         r_t = fl32(V block scale x        */
/*                                          fl32(1 / reference))              */
/*                                          (E4M3 layouts), 1 (MX layouts)    */
/*   l     = fl32(alpha l + fl32(sum_t pt_t))                                 */
/*   O_c   = fl32(alpha O_c + fl32(sum_t Phat_t vhat_tc))                     */
/* End: O = fl32(O * fl32(ref / l)), lse = ln2 * (m + log2 l - 8), O -> bf16. */
/* Bit-level exponentials (E4M3 tile or MX col32, not exact): with            */
/* x_t = s'_t - m' + 8 + log2 r_t (the V ratio folded into the exponent),     */
/*   Schraudolph: p_t = or_exp2_schraudolph(x_t), Phat = E4M3(p_t),           */
/*                l adds p_t / r_t;                                           */
/*   Mitchell-P:  Phat = the value of or_exp2_mitchell_code(x_t),             */
/*                l adds Phat / r_t.                                          */
/* Their tie band adds 2^-15 to dx (the device rounds u + 126 or 8 u + 56,    */
/* scaled into [0, 1], to fp32 before the final rounding, and forms log2 r    */
/* with an fp32 approximation).                                               */
/* vhat = V code (E4M3 layouts; its scale enters through r_t and ref) or     */
/* code * 2^X (MX col32: the block-scaled MMA applies V's exponents).        */
/* ref = max over the document's V blocks (default), or, in the causal-exact */
/* mode, max of the V token scales at positions <= i, so that no later token */
/* reaches row i (FLAMIA 1 and 4.5: exact options remove within-block        */
/* dependencies).                                                            */
/*                                                                           */
/* Optional second output, amb: where several results are correct. A GPU     */
/* computes S in fp32 in its own summation order and 2^x with an fp32        */
/* approximation, so a probability lying within that rounding of an E4M3     */
/* boundary may take either neighbouring code; both are faithful results.    */
/* For each such key the emulation adds |code_hi - code_lo| * |vhat_tc| to   */
/* amb (rescaled and normalised like O), so that a parity check can accept   */
/* exactly the differences these ties explain. The error model, in log2      */
/* units of the exponent x = s' - m' + 8:                                    */
/*   dx = 2^-20 (|cf| A_t + A_m) + 2^-21 (|s'_t| + |m'| + 8),                */
/*   A_t = sum_c |qhat_c khat_c|; 2^-20 A_t covers an fp32 sum of the d      */
/*   products in any tree of depth <= 16 (each level rounds by 2^-24 A_t),  */
/*   A_m = the largest |cf| A of the keys so far (error of the running max),*/
/*   cf the factor from S to s'; relative band on pt: ln2 dx + 2^-20.        */
/* ------------------------------------------------------------------------- */
typedef struct {
    const or_qtensor *q, *k, *v; int T, H, d; docs_t D; int causal, exact, rotated; double scale;
    int flags; const int32_t* rows; int nrows; float* o; uint16_t* ob; float* lse; float* amb; float* lamb;
    double dec[256];
    float tau;                   /* rescale threshold of the running max, log2 units */
    int expm;                    /* 0: 2^x; OR_EMU_EXP_SCHRAUDOLPH or OR_EMU_EXP_MITCHELL_P */
    const uint8_t* pg;           /* device probability codes [H][T][pstride], or NULL */
    long pstride;
    long counts[4];              /* given codes: same, other tie code, violation, masked non-zero */
    long nbq, nbk, nbv, ngv;     /* block counts of the logical scale arrays */
    int h;                       /* head being evaluated */
    double *kh, *vh;             /* dequantised K and V of head h, [T][d] */
    float* vtok;                 /* MX token layout: V scale 2^X of each token of head h (0 when X = -127) */
} emu_ctx;

/* dequantised element: code value, times 2^X for the MX layouts (the E4M3
 * layouts return the bare code value; their scale is applied per block) */
static double hat(const emu_ctx* c, const or_qtensor* x, int t, int h, int j, long ng) {
    if (x->layout == OR_NVFP4) {   /* e2m1 code times its 16-channel E4M3 scale (s_t enters with cf) */
        uint8_t b = x->codes[((long)t * c->H + h) * (c->d / 2) + j / 2];
        uint8_t e = (j & 1) ? (uint8_t)(b >> 4) : (uint8_t)(b & 15);
        return or_e2m1_decode(e) * c->dec[x->scales_u8[((long)t * c->H + h) * (c->d / 16) + j / 16]];
    }
    uint8_t code = x->codes[((long)t * c->H + h) * c->d + j];
    double v = c->dec[code];
    if (x->layout == OR_MX_ROW32) {
        int X = (int)x->scales_u8[((long)t * c->H + h) * (c->d / 32) + j / 32] - 127;
        v = ldexp(v, X);
    } else if (x->layout == OR_MX_COL32) {
        int doc = doc_of(c->D.cu, c->D.nd, t);
        long g = block_offset(&c->D, doc, 32) + (t - c->D.cu[doc]) / 32;
        int X = (int)x->scales_u8[((long)h * ng + g) * c->d + j] - 127;
        v = ldexp(v, X);
    }
    return v;
}

static void emu_decode_unit(void* vc, long t) {
    emu_ctx* c = (emu_ctx*)vc;
    for (int j = 0; j < c->d; j++) {
        c->kh[t * c->d + j] = hat(c, c->k, (int)t, c->h, j, 0);
        c->vh[t * c->d + j] = hat(c, c->v, (int)t, c->h, j, c->ngv);
    }
    if (c->v->layout == OR_MX_TOKEN) {
        int b = c->v->scales_u8[(long)c->h * c->T + t];
        c->vtok[t] = b ? ldexpf(1.0f, b - 127) : 0.0f;
    }
}

/* One key under a bit-level exponential: x is the exponent with the V ratio
 * r folded in, dx its error band. Sets ph[a] (the probability P V uses, the
 * device's code where given) and tie[a], and adds the key's share to rowsum
 * (and, log-domain P, its tie band to rowtie). */
static void emu_bitexp_key(const emu_ctx* c, int a, double x, double r, double dx, const uint8_t* gcodes,
                           double* ph, double* tie, double* rowsum, double* rowtie, long* n_same, long* n_tie,
                           long* n_bad) {
    const int schr = c->expm == OR_EMU_EXP_SCHRAUDOLPH;
    float pf = 0.0f;
    uint8_t own, lo, hi;
    if (schr) {
        pf = or_exp2_schraudolph(x);
        own = or_e4m3_encode(pf);
        lo = or_e4m3_encode(or_exp2_schraudolph(x - dx));
        hi = or_e4m3_encode(or_exp2_schraudolph(x + dx));
    } else {
        own = or_exp2_mitchell_code(x);
        lo = or_exp2_mitchell_code(x - dx);
        hi = or_exp2_mitchell_code(x + dx);
    }
    uint8_t use = own;
    tie[a] = 0.0;
    if (gcodes) {
        uint8_t gc = gcodes[a];
        if (gc == own) (*n_same)++;
        else if (lo != hi && (gc == lo || gc == hi)) (*n_tie)++;
        else (*n_bad)++;
        use = gc;
    } else if (lo != hi && (c->flags & OR_EMU_QUANTIZE_P)) {
        tie[a] = fabs(c->dec[hi] - c->dec[lo]);
    }
    if (schr) {
        ph[a] = (c->flags & OR_EMU_QUANTIZE_P) ? c->dec[use] : (double)pf;
        *rowsum += (double)pf / r;
    } else {
        ph[a] = c->dec[use];
        *rowsum += c->dec[use] / r;
        *rowtie += tie[a] / r;
    }
}

static void emu_unit(void* vc, long ri) {
    emu_ctx* c = (emu_ctx*)vc;
    int h = c->h, d = c->d;
    int t = c->rows ? c->rows[ri] : (int)ri;
    int doc = doc_of(c->D.cu, c->D.nd, t);
    int s0 = c->D.cu[doc], L = c->D.cu[doc + 1] - s0, i = t - s0;
    const or_qtensor *Q = c->q, *K = c->k, *V = c->v;
    int mx = (Q->layout == OR_MX_ROW32);
    int vmx = (V->layout == OR_MX_COL32);
    double C = c->scale * 1.4426950408889634 / (c->rotated ? (double)d : 1.0);
    float C32 = (float)C;

    double qh[256];
    for (int j = 0; j < d; j++) qh[j] = hat(c, Q, t, h, j, 0);
    float qs = 1.0f;
    const float *ks_row = NULL, *vs_row = NULL;
    int kb = 1, vb = 1;
    if (!mx) {
        qs = Q->scales_f32[(long)h * c->nbq + block_offset(&c->D, doc, Q->block) + i / Q->block];
        ks_row = K->scales_f32 + (long)h * c->nbk + block_offset(&c->D, doc, K->block);
        kb = K->block;
    }
    /* V reference for the E4M3 layouts */
    float ref = 1.0f;
    if (!vmx) {
        /* V's scale per block (E4M3) or per token (MX token layout: 2^X) */
        if (V->layout == OR_MX_TOKEN) {
            vs_row = c->vtok + s0;
            vb = 1;
        } else {
            vs_row = V->scales_f32 + (long)h * c->nbv + block_offset(&c->D, doc, V->block);
            vb = V->block;
        }
        int nblk = (L + vb - 1) / vb;
        int last = c->exact ? i / vb : nblk - 1;
        float mxv = 0.0f;
        for (int b = 0; b <= last; b++) if (vs_row[b] > mxv) mxv = vs_row[b];
        ref = mxv;
    }
    const float inv_ref = ref > 0.0f ? 1.0f / ref : 0.0f;   /* rounded once per row */

    float m = -INFINITY, l = 0.0f;
    double lt = 0.0;             /* tie band of l (log-domain P) */
    float O[256];
    double Am[256];
    for (int x = 0; x < d; x++) O[x] = 0.0f, Am[x] = 0.0;
    int nkeys = c->causal ? i + 1 : L;
    int ntiles = (nkeys + 127) / 128;
    float sp[128];
    double ph[128], at[128], tie[128];
    double amax = 0.0;
    long n_same = 0, n_tie = 0, n_bad = 0, n_mask = 0;
    const uint8_t* prow = c->pg ? c->pg + ((long)h * c->T + t) * c->pstride : NULL;
    for (int jt = 0; jt < ntiles; jt++) {
        int k0 = jt * 128, kn = (nkeys - k0) < 128 ? nkeys - k0 : 128;
        float mt = -INFINITY;
        double cf = 0.0;
        for (int a = 0; a < kn; a++) {
            const double* kr = c->kh + (long)(s0 + k0 + a) * d;
            double acc = 0.0, aa = 0.0;
            for (int j = 0; j < d; j++) {
                acc += qh[j] * kr[j];
                aa += fabs(qh[j] * kr[j]);
            }
            float S = (float)acc;
            float sc;
            if (mx) {
                cf = C32;
                sc = S * C32;
            } else {
                cf = (float)((double)qs * (double)ks_row[(k0 + a) / kb] * C);
                sc = S * (float)cf;
            }
            sp[a] = sc;
            at[a] = fabs(cf) * aa;
            if (at[a] > amax) amax = at[a];
            if (sc > mt) mt = sc;
        }
        /* the reference maximum moves to the new maximum only when that exceeds it
         * by more than tau (log2 units; tau = 0: whenever it grows) */
        float mcand = mt > m ? mt : m;
        float mnew = (m == -INFINITY || mcand > m + c->tau) ? mcand : m;
        float alpha = (m == -INFINITY) ? 0.0f : (float)exp2((double)m - (double)mnew);
        double rowsum = 0.0, rowtie = 0.0;
        for (int a = 0; a < kn; a++) {
            double r = 1.0;
            if (!vmx) {
                float sv = vs_row[(k0 + a) / vb];
                r = (sv > 0.0f && ref > 0.0f) ? (double)(sv * inv_ref) : 1.0;
            }
            if (c->expm) {
                emu_bitexp_key(c, a, (double)sp[a] - (double)mnew + 8.0 + log2(r), r,
                               ldexp(at[a] + amax, -20) +
                                   ldexp(fabs((double)sp[a]) + fabs((double)mnew) + 8.0, -21) + ldexp(1.0, -15),
                               prow ? prow + k0 : NULL, ph, tie, &rowsum, &rowtie, &n_same, &n_tie, &n_bad);
                continue;
            }
            double pt = exp2((double)sp[a] - (double)mnew + 8.0);
            rowsum += pt;
            float pr = (float)(pt * r);
            uint8_t own = or_e4m3_encode(pr);
            ph[a] = (c->flags & OR_EMU_QUANTIZE_P) ? c->dec[own] : (double)pr;
            tie[a] = 0.0;
            if ((c->amb || prow) && (c->flags & OR_EMU_QUANTIZE_P)) {
                uint8_t lo = own, hi = own;
                if (pt > 0.0) {
                    double dx = ldexp(at[a] + amax, -20) +
                                ldexp(fabs((double)sp[a]) + fabs((double)mnew) + 8.0, -21);
                    double band = 0.6931471805599453 * dx + ldexp(1.0, -20);
                    lo = or_e4m3_encode((float)(pr * (1.0 - band)));
                    hi = or_e4m3_encode((float)(pr * (1.0 + band)));
                }
                if (prow) {
                    /* the device's code: the emulation's own, or the other code of a tie */
                    uint8_t gc = prow[k0 + a];
                    if (gc == own) n_same++;
                    else if (lo != hi && (gc == lo || gc == hi)) n_tie++;
                    else n_bad++;
                    ph[a] = c->dec[gc];
                } else if (lo != hi) {
                    tie[a] = fabs(c->dec[hi] - c->dec[lo]);
                }
            }
        }
        l = alpha * l + (float)rowsum;
        lt = (double)alpha * lt + rowtie;
        for (int x = 0; x < d; x++) {
            double acc = 0.0, ta = 0.0;
            for (int a = 0; a < kn; a++) {
                const double vv = c->vh[(long)(s0 + k0 + a) * d + x];
                acc += ph[a] * vv;
                ta += tie[a] * fabs(vv);
            }
            O[x] = alpha * O[x] + (float)acc;
            Am[x] = (double)alpha * Am[x] + ta;
        }
        m = mnew;
    }
    if (prow) {
        /* keys the row does not see (causal future, past the document end) carry code 0 */
        for (long kx = nkeys; kx < c->pstride; kx++)
            if (prow[kx] != 0) n_mask++;
        __atomic_fetch_add(&c->counts[0], n_same, __ATOMIC_RELAXED);
        __atomic_fetch_add(&c->counts[1], n_tie, __ATOMIC_RELAXED);
        __atomic_fetch_add(&c->counts[2], n_bad, __ATOMIC_RELAXED);
        __atomic_fetch_add(&c->counts[3], n_mask, __ATOMIC_RELAXED);
    }
    float fin = (l > 0.0f) ? (float)((double)ref / (double)l) : 0.0f;
    float* out = c->o + ((long)ri * c->H + h) * d;
    for (int x = 0; x < d; x++) {
        out[x] = O[x] * fin;
        if (c->ob) c->ob[((long)ri * c->H + h) * d + x] = or_bf16_rne(out[x]);
        if (c->amb) c->amb[((long)ri * c->H + h) * d + x] = (float)(Am[x] * (double)fin);
    }
    c->lse[(long)h * c->nrows + ri] =
        (l > 0.0f) ? (float)(0.6931471805599453 * ((double)m + log2((double)l) - 8.0)) : -INFINITY;
    if (c->lamb)
        c->lamb[(long)h * c->nrows + ri] =
            (lt <= 0.0 || !(l > 0.0f)) ? 0.0f : (lt < (double)l ? (float)(-log1p(-lt / (double)l)) : INFINITY);
}

static int emulate(const or_qtensor* q, const or_qtensor* k, const or_qtensor* v,
                   int T, int H, int d, const int32_t* cu, int nd,
                   int causal, int exact, int rotated, double scale, float tau, int flags,
                   const int32_t* rows, int nrows, float* o, uint16_t* ob, float* lse, float* amb,
                   float* lamb, const uint8_t* pg, long pstride, long* counts) {
    if (d < 1 || d > 256) return OR_ERR_ARG;
    if (pg && (!(flags & OR_EMU_QUANTIZE_P) || pstride < 1 || amb || lamb)) return OR_ERR_ARG;
    if (!(tau >= 0.0f && tau < 1.0f)) return OR_ERR_ARG;
    int expm = flags & (OR_EMU_EXP_SCHRAUDOLPH | OR_EMU_EXP_MITCHELL_P);
    if (expm == (OR_EMU_EXP_SCHRAUDOLPH | OR_EMU_EXP_MITCHELL_P)) return OR_ERR_ARG;
    /* the bit-level forms: E4M3 with one V scale per key tile, or MX with col32 V; not exact */
    if (expm && (exact || v->layout == OR_MX_TOKEN || (v->layout == OR_E4M3_TOKBLOCK && v->block != 128)))
        return OR_ERR_ARG;
    int mxq = q->layout == OR_MX_ROW32, mxk = k->layout == OR_MX_ROW32;
    if (mxq != mxk) return OR_ERR_ARG;
    /* NVFP4 Q K^T (the mixed path): both NVFP4 with 128-token s_t blocks, an E4M3 V, not exact */
    int nvq = q->layout == OR_NVFP4, nvk = k->layout == OR_NVFP4;
    if (nvq != nvk || v->layout == OR_NVFP4) return OR_ERR_ARG;
    if (nvq && (q->block != 128 || k->block != 128 || v->layout != OR_E4M3_TOKBLOCK || exact || d % 16))
        return OR_ERR_ARG;
    if (q->layout == OR_MX_COL32 || k->layout == OR_MX_COL32 || v->layout == OR_MX_ROW32) return OR_ERR_ARG;
    if (exact && (!causal || !((v->layout == OR_E4M3_TOKBLOCK && v->block == 1) || v->layout == OR_MX_TOKEN)))
        return OR_ERR_ARG;
    if (v->layout == OR_MX_TOKEN && !mxq) return OR_ERR_ARG;
    emu_ctx c;
    memset(&c, 0, sizeof(c));
    c.q = q; c.k = k; c.v = v; c.T = T; c.H = H; c.d = d; c.D = docs_make(cu, nd, T);
    c.causal = causal; c.exact = exact; c.rotated = rotated; c.scale = scale; c.flags = flags;
    c.rows = rows; c.nrows = rows ? nrows : T; c.o = o; c.ob = ob; c.lse = lse; c.amb = amb; c.lamb = lamb;
    c.pg = pg; c.pstride = pstride; c.tau = tau; c.expm = expm;
    for (int i = 0; i < 256; i++) c.dec[i] = or_e4m3_decode((uint8_t)i);
    if (!mxq) { c.nbq = block_offset(&c.D, c.D.nd, q->block); c.nbk = block_offset(&c.D, c.D.nd, k->block); }
    if (v->layout == OR_E4M3_TOKBLOCK) c.nbv = block_offset(&c.D, c.D.nd, v->block);
    else c.ngv = block_offset(&c.D, c.D.nd, 32);
    c.vtok = (float*)malloc(sizeof(float) * (size_t)(T > 0 ? T : 1));
    c.kh = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * d);
    c.vh = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * d);
    if (!c.kh || !c.vh || !c.vtok) { free(c.kh); free(c.vh); free(c.vtok); free(c.D.cu); return OR_ERR_ARG; }
    for (int h = 0; h < H; h++) {
        c.h = h;
        parallel_for(T, emu_decode_unit, &c);
        parallel_for(c.nrows, emu_unit, &c);
    }
    free(c.kh); free(c.vh); free(c.vtok); free(c.D.cu);
    if (counts) for (int i = 0; i < 4; i++) counts[i] = c.counts[i];
    return OR_OK;
}

int or_attention_emulate(const or_qtensor* q, const or_qtensor* k, const or_qtensor* v,
                         int T, int H, int d, const int32_t* cu, int nd,
                         int causal, int exact, int rotated, double scale, float rescale_tau, int flags,
                         const int32_t* rows, int nrows, float* o, uint16_t* ob, float* lse, float* amb,
                         float* lse_amb) {
    return emulate(q, k, v, T, H, d, cu, nd, causal, exact, rotated, scale, rescale_tau, flags, rows, nrows, o, ob,
                   lse, amb, lse_amb, NULL, 0, NULL);
}

/* The same emulation with a device's probability codes in place of its own
 * (where several codes are correct, the device's choice is checked, then
 * used): p_codes[(h * T + t) * p_stride + k] is the code row t of head h gave
 * the document-local key k. Every visible key's device code must be the
 * emulation's own code, or the other code of a tie (the emulation's
 * probability within its rounding band of an E4M3 boundary: both neighbouring
 * codes are faithful results); keys the row does not see must carry code 0.
 * counts: [0] keys with the emulation's code, [1] keys with the other code of
 * a tie, [2] keys with any other code (errors), [3] unseen keys with a
 * non-zero code (errors). O and lse are then computed from the device's
 * codes, so that they can be compared without any tie allowance. */
int or_attention_emulate_given_p(const or_qtensor* q, const or_qtensor* k, const or_qtensor* v,
                                 int T, int H, int d, const int32_t* cu, int nd,
                                 int causal, int exact, int rotated, double scale, float rescale_tau, int flags,
                                 const int32_t* rows, int nrows, float* o, uint16_t* ob, float* lse,
                                 const uint8_t* p_codes, long p_stride, long* counts) {
    if (!p_codes || !counts) return OR_ERR_ARG;
    return emulate(q, k, v, T, H, d, cu, nd, causal, exact, rotated, scale, rescale_tau, flags | OR_EMU_QUANTIZE_P,
                   rows, nrows, o, ob, lse, NULL, NULL, p_codes, p_stride, counts);
}
