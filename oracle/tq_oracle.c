/*
 * tq_oracle.c -- plain, slow, double-precision CPU oracle for rotated-codebook
 * KV-cache compression and attention over the compressed cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this code.  It shares no code, header, table or
 * constant generator with the CUDA library; each side is written from the
 * method's description on its own.
 *
 * Sources (web pages on TurboQuant-style KV compression):
 *   [turbo-attn]   pypi.org/project/turbo-attn/0.24.0, section "How it works"
 *                  (steps 1-3: rotate, normalise with a BF16 norm, quantise
 *                  to a shared codebook; pre-rotated queries; fused decode),
 *                  section "Configuration" (TKV_DECODE_SPLITS: split-K decode).
 *   [0xsero]       gitdiagram.com/0xsero/turboquant, sections "Compression
 *                  Pipeline" (random orthogonal rotation, Lloyd-Max scalar
 *                  codebook, QJL residual-sign projection), "Value
 *                  Compression" (group scale/zero, 4x2-bit / 2x4-bit per byte),
 *                  "Key Storage and Attention Scoring" (paged store + scoring).
 *   [brightcoding] converter.brightcoding.dev blog on TurboQuant-GPU, sections
 *                  "What is TurboQuant-GPU?" (rotation makes coordinates
 *                  ~Gaussian; Lloyd-Max is optimal for Gaussian sources) and
 *                  "Example 4" (normalize -> rotate -> quantize -> pack).
 *   [tiny-tq]      pypi.org/project/tiny-turboquant/0.18.0, section "Measured
 *                  quality" (each value group of 32 gets its own scale/zero).
 *
 * Every step below is the plain definition, in the pages' order:
 *   O1 RNG          SplitMix64 (Steele, Lea & Flood, OOPSLA 2014) streams,
 *                   Box-Muller Gaussians.
 *   O2 rotation     Pi = Q diag(sign(diag R)) from a Householder QR of a
 *                   Gaussian matrix (Haar measure, Mezzadri 2007); y = Pi k.
 *   O3 codebook     Lloyd-Max quantiser for N(0,1), applied to z = sqrt(d) y.
 *   O4 key record   norm (bf16), codes, QJL signs of S r, residual norm (bf16).
 *   O5 value record per-group fp16 (scale, zero), round-half-up codes.
 *   O6 paged layout page records of struct-of-arrays sub-blocks.
 *   O7 dequant      K~ = n Pi^T (c/sqrt d + sqrt(pi/2)/m gamma S^T(2 sigma-1)),
 *                   V~ = code * scale + zero.
 *   O8 decode       dense softmax attention over the dequantised cache, both
 *                   in the original space and in the rotated space.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define OR_PI 3.14159265358979323846

/* ------------------------------------------------------------------------- */
/* O1: SplitMix64 and Gaussian streams                                       */
/* ------------------------------------------------------------------------- */

/* One SplitMix64 step: advance the state by the golden-ratio gamma, then mix. */
static uint64_t or_splitmix64(uint64_t *state)
{
    uint64_t z = (*state += 0x9E3779B97F4A7C15ULL);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Raw SplitMix64 outputs from an initial state (for pinning the generator). */
void tq_or_splitmix64(uint64_t state, int64_t n, uint64_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = or_splitmix64(&state);
}

/* Uniform in (0,1): top 53 bits, centred in their bucket (never 0 or 1). */
static double or_uniform(uint64_t *state)
{
    return ((double)(or_splitmix64(state) >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

/*
 * Gaussian stream `stream` of `seed`: the state starts at
 * seed XOR (0x9E3779B97F4A7C15 * (stream + 1)); each pair of uniforms
 * (u1, u2) gives r cos(2 pi u2) then r sin(2 pi u2), r = sqrt(-2 ln u1).
 */
void tq_or_gaussians(uint64_t seed, int stream, int64_t n, double *out)
{
    uint64_t state = seed ^ (0x9E3779B97F4A7C15ULL * (uint64_t)(stream + 1));
    for (int64_t i = 0; i < n; i += 2) {
        double u1 = or_uniform(&state);
        double u2 = or_uniform(&state);
        double r = sqrt(-2.0 * log(u1));
        out[i] = r * cos(2.0 * OR_PI * u2);
        if (i + 1 < n) out[i + 1] = r * sin(2.0 * OR_PI * u2);
    }
}

/* ------------------------------------------------------------------------- */
/* O2: Haar rotation by Householder QR                                        */
/* ------------------------------------------------------------------------- */

/*
 * Pi (d x d, row-major) = Q diag(sign(R_kk)) where G = Q R, G the d x d
 * Gaussian matrix of stream 0 filled row-major.  Householder reflections
 * H_k = I - 2 v_k v_k^T are applied to G to make it upper triangular; Q is
 * H_0 H_1 ... H_{d-1} accumulated on the identity.
 */
int tq_or_rotation(int d, uint64_t seed, double *Pi)
{
    double *A = malloc(sizeof(double) * d * d);
    double *V = malloc(sizeof(double) * d * d); /* v_k stored in row k, entries k..d-1 */
    double *rdiag = malloc(sizeof(double) * d);
    if (!A || !V || !rdiag) { free(A); free(V); free(rdiag); return -1; }
    tq_or_gaussians(seed, 0, (int64_t)d * d, A);
    memset(V, 0, sizeof(double) * d * d);

    for (int k = 0; k < d; ++k) {
        double nx = 0.0;
        for (int i = k; i < d; ++i) nx += A[i * d + k] * A[i * d + k];
        nx = sqrt(nx);
        double x0 = A[k * d + k];
        double alpha = (x0 >= 0.0) ? -nx : nx; /* reflect x onto alpha e_1 */
        double *v = V + k * d;
        for (int i = k; i < d; ++i) v[i] = A[i * d + k];
        v[k] -= alpha;
        double nv = 0.0;
        for (int i = k; i < d; ++i) nv += v[i] * v[i];
        nv = sqrt(nv);
        if (nv > 0.0)
            for (int i = k; i < d; ++i) v[i] /= nv;
        /* A[k:, k:] -= 2 v (v^T A[k:, k:]) */
        for (int j = k; j < d; ++j) {
            double dot = 0.0;
            for (int i = k; i < d; ++i) dot += v[i] * A[i * d + j];
            for (int i = k; i < d; ++i) A[i * d + j] -= 2.0 * v[i] * dot;
        }
        rdiag[k] = A[k * d + k];
    }
    /* Q = H_0 ... H_{d-1} I: apply reflections right-to-left to the identity. */
    double *Q = A; /* reuse storage */
    for (int i = 0; i < d * d; ++i) Q[i] = 0.0;
    for (int i = 0; i < d; ++i) Q[i * d + i] = 1.0;
    for (int k = d - 1; k >= 0; --k) {
        const double *v = V + k * d;
        for (int j = 0; j < d; ++j) {
            double dot = 0.0;
            for (int i = k; i < d; ++i) dot += v[i] * Q[i * d + j];
            for (int i = k; i < d; ++i) Q[i * d + j] -= 2.0 * v[i] * dot;
        }
    }
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j)
            Pi[i * d + j] = Q[i * d + j] * (rdiag[j] < 0.0 ? -1.0 : 1.0);
    free(A); free(V); free(rdiag);
    return 0;
}

/* QJL matrix S (m x d, m = d rows): Gaussian stream 1, row-major. */
void tq_or_qjl_matrix(int d, uint64_t seed, double *S)
{
    tq_or_gaussians(seed, 1, (int64_t)d * d, S);
}

/* ------------------------------------------------------------------------- */
/* O3: Lloyd-Max codebook for N(0,1)                                          */
/* ------------------------------------------------------------------------- */

static double or_phi(double x) { return isinf(x) ? 0.0 : exp(-0.5 * x * x) / sqrt(2.0 * OR_PI); }

/* P(a < X < b) for X ~ N(0,1), via erfc on the side that avoids cancellation. */
static double or_mass(double a, double b)
{
    const double s = sqrt(0.5);
    if (a >= 0.0) return 0.5 * (erfc(a * s) - erfc(b * s));
    if (b <= 0.0) return 0.5 * (erfc(-b * s) - erfc(-a * s));
    return 1.0 - 0.5 * erfc(b * s) - 0.5 * erfc(-a * s);
}

/*
 * Lloyd-Max fixed point for L = 2^bits levels: thresholds are midpoints of
 * neighbouring centroids; centroids are conditional means of N(0,1) between
 * thresholds, (phi(t_{i-1}) - phi(t_i)) / (Phi(t_i) - Phi(t_{i-1})).
 * Start: uniform spacing on [-3, 3].  Stop: max |delta c| < 1e-15.
 * Returns iterations used, or -1 if it did not converge.
 */
int tq_or_codebook(int bits, double *centroids, double *thresholds)
{
    int L = 1 << bits;
    double c[16], t[17];
    for (int i = 0; i < L; ++i) c[i] = (L == 1) ? 0.0 : -3.0 + 6.0 * i / (L - 1);
    for (int it = 0; it < 1000000; ++it) {
        t[0] = -INFINITY;
        t[L] = INFINITY;
        for (int i = 1; i < L; ++i) t[i] = 0.5 * (c[i - 1] + c[i]);
        double dmax = 0.0;
        for (int i = 0; i < L; ++i) {
            double cn = (or_phi(t[i]) - or_phi(t[i + 1])) / or_mass(t[i], t[i + 1]);
            double dd = fabs(cn - c[i]);
            if (dd > dmax) dmax = dd;
            c[i] = cn;
        }
        if (dmax < 1e-15) {
            for (int i = 0; i < L; ++i) centroids[i] = c[i];
            for (int i = 1; i < L; ++i) thresholds[i - 1] = 0.5 * (c[i - 1] + c[i]);
            return it + 1;
        }
    }
    return -1;
}

/* ------------------------------------------------------------------------- */
/* Rounding helpers (exact definitions of bf16 / fp16 round-to-nearest-even)  */
/* ------------------------------------------------------------------------- */

/* double -> bf16 bits, one rounding: 8 significant bits, min normal 2^-126. */
uint16_t tq_or_bf16_from_double(double x)
{
    if (isnan(x)) return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double ax = fabs(x);
    if (ax == 0.0) return sign;
    if (isinf(ax)) return sign | 0x7F80;
    int e;
    frexp(ax, &e); /* ax = f 2^e, f in [0.5, 1) */
    int qe = e - 8;
    if (qe < -133) qe = -133; /* subnormal quantum */
    double q = ldexp(1.0, qe);
    double r = nearbyint(ax / q) * q; /* default rounding mode: nearest-even */
    if (r > 0x1.FCp127) return sign | 0x7F80;
    float f = (float)r; /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    return sign | (uint16_t)((u >> 16) & 0x7FFF);
}

double tq_or_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* double -> fp16 bits, one rounding: 11 significant bits, min normal 2^-14. */
uint16_t tq_or_f16_from_double(double x)
{
    if (isnan(x)) return 0x7E00;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double ax = fabs(x);
    if (ax == 0.0) return sign;
    if (isinf(ax)) return sign | 0x7C00;
    int e;
    frexp(ax, &e);
    int qe = e - 11;
    if (qe < -24) qe = -24;
    double q = ldexp(1.0, qe);
    double r = nearbyint(ax / q) * q;
    if (r > 65504.0) return sign | 0x7C00;
    if (r < ldexp(1.0, -14)) return sign | (uint16_t)(r / ldexp(1.0, -24)); /* subnormal */
    int ee;
    double f = frexp(r, &ee); /* r = f 2^ee = (2f) 2^(ee-1) */
    uint16_t E = (uint16_t)(ee - 1 + 15);
    uint16_t mant = (uint16_t)((2.0 * f - 1.0) * 1024.0);
    return sign | (uint16_t)(E << 10) | mant;
}

double tq_or_f16_to_double(uint16_t h)
{
    int s = h >> 15, E = (h >> 10) & 31, M = h & 1023;
    double v;
    if (E == 0) v = ldexp((double)M, -24);
    else if (E == 31) v = M ? NAN : INFINITY;
    else v = ldexp(1024.0 + M, E - 25);
    return s ? -v : v;
}

/* ------------------------------------------------------------------------- */
/* Parameters and record geometry                                            */
/* ------------------------------------------------------------------------- */

typedef struct or_ctx {
    int d, kb, vb, g, qjl;
    int vmse;           /* values coded by rotation + Lloyd-Max codebook (else group scale/zero) */
    double vcent[16];   /* 2^vb value centroids (vmse) */
    double vthr[15];
    double *Pi, *S;     /* d x d each, row-major */
    double cent[16];    /* 2^kb centroids, ascending, N(0,1) units */
    double thr[15];     /* 2^kb - 1 thresholds */
    /* per-token-head record field sizes in bytes */
    int kcode, ksign, vcode, vmeta;
} or_ctx;

/*
 * O2': randomized Hadamard rotation ([turbo-attn] "How it works", step 1: a
 * fast Walsh-Hadamard transform).  Pi = H diag(s) / sqrt(d), H the Hadamard
 * matrix of Sylvester's construction (H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]]),
 * s_j = -1 when the top bit of the j-th raw output of SplitMix64 stream 0 is
 * set, else +1 (the pages name no sign source: this stream is the reading).
 * d must be a power of two.
 */
int tq_or_hadamard_rotation(int d, uint64_t seed, double *Pi)
{
    if (d <= 0 || (d & (d - 1))) return -1;
    double *H = malloc(sizeof(double) * d * d);
    if (!H) return -1;
    H[0] = 1.0;
    for (int n = 1; n < d; n *= 2) /* grow H_n (top-left n x n) into H_2n */
        for (int i = 0; i < n; ++i)
            for (int j = 0; j < n; ++j) {
                double h = H[i * d + j];
                H[i * d + (j + n)] = h;
                H[(i + n) * d + j] = h;
                H[(i + n) * d + (j + n)] = -h;
            }
    uint64_t state = seed ^ 0x9E3779B97F4A7C15ULL; /* stream 0 */
    double inv = 1.0 / sqrt((double)d);
    for (int j = 0; j < d; ++j) {
        double sj = (or_splitmix64(&state) >> 63) ? -1.0 : 1.0;
        for (int i = 0; i < d; ++i) Pi[i * d + j] = H[i * d + j] * sj * inv;
    }
    free(H);
    return 0;
}

/* QJL is used iff k_bits <= 3 (one sign bit per coordinate, m = d).
 * Pi comes from seed_rot, S from seed_qjl; the codec uses one seed for both.
 * options: bit 0 -- the randomized Hadamard rotation (O2') instead of the Haar
 * one (O2); bit 1 -- values coded like keys without QJL (O5'). */
or_ctx *tq_or_create3(int d, int kb, int vb, int g, uint64_t seed_rot, uint64_t seed_qjl, int options)
{
    int rotation = options & 1;
    if (d <= 0 || d % 8 || kb < 1 || kb > 4 || vb < 1 || vb > 8 || g <= 0 || d % g) return NULL;
    or_ctx *c = calloc(1, sizeof(or_ctx));
    c->d = d; c->kb = kb; c->vb = vb; c->g = g; c->qjl = kb <= 3;
    c->Pi = malloc(sizeof(double) * d * d);
    c->S = malloc(sizeof(double) * d * d);
    int rc = rotation == 1 ? tq_or_hadamard_rotation(d, seed_rot, c->Pi) : tq_or_rotation(d, seed_rot, c->Pi);
    if (rc != 0 || tq_or_codebook(kb, c->cent, c->thr) < 0) {
        free(c->Pi); free(c->S); free(c);
        return NULL;
    }
    tq_or_qjl_matrix(d, seed_qjl, c->S);
    c->vmse = (options >> 1) & 1;
    if (c->vmse && tq_or_codebook(vb, c->vcent, c->vthr) < 0) {
        free(c->Pi); free(c->S); free(c);
        return NULL;
    }
    c->kcode = d * kb / 8;
    c->ksign = c->qjl ? d / 8 : 0;
    c->vcode = d * vb / 8;
    c->vmeta = c->vmse ? 2 : (d / g) * 4; /* a bf16 norm, or (scale, zero) fp16 per group */
    return c;
}

or_ctx *tq_or_create2(int d, int kb, int vb, int g, uint64_t seed_rot, uint64_t seed_qjl)
{
    return tq_or_create3(d, kb, vb, g, seed_rot, seed_qjl, 0);
}

or_ctx *tq_or_create(int d, int kb, int vb, int g, uint64_t seed)
{
    return tq_or_create3(d, kb, vb, g, seed, seed, 0);
}

void tq_or_destroy(or_ctx *c)
{
    if (!c) return;
    free(c->Pi); free(c->S); free(c);
}

void tq_or_get_params(const or_ctx *c, double *Pi, double *S, double *cent, double *thr)
{
    int d = c->d, L = 1 << c->kb;
    if (Pi) memcpy(Pi, c->Pi, sizeof(double) * d * d);
    if (S) memcpy(S, c->S, sizeof(double) * d * d);
    if (cent) memcpy(cent, c->cent, sizeof(double) * L);
    if (thr) memcpy(thr, c->thr, sizeof(double) * (L - 1));
}

/* sizes[0..3] = key code bytes, key sign bytes, value code bytes, value meta bytes
 * per token-head; sizes[4], sizes[5] = K and V page-record bytes for page size P. */
void tq_or_geometry(const or_ctx *c, int P, int64_t *sizes)
{
    sizes[0] = c->kcode; sizes[1] = c->ksign; sizes[2] = c->vcode; sizes[3] = c->vmeta;
    sizes[4] = (int64_t)P * (c->kcode + c->ksign + 2 + (c->qjl ? 2 : 0));
    sizes[5] = (int64_t)P * (c->vcode + c->vmeta);
}

/* ------------------------------------------------------------------------- */
/* Bit packing: b-bit fields, LSB-first little-endian bitstream              */
/* ------------------------------------------------------------------------- */

void tq_or_pack(const uint8_t *codes, int n, int bits, uint8_t *out)
{
    memset(out, 0, (size_t)(n * bits + 7) / 8);
    for (int j = 0; j < n; ++j)
        for (int b = 0; b < bits; ++b)
            if ((codes[j] >> b) & 1) {
                int pos = j * bits + b;
                out[pos >> 3] |= (uint8_t)(1u << (pos & 7));
            }
}

void tq_or_unpack(const uint8_t *in, int n, int bits, uint8_t *codes)
{
    for (int j = 0; j < n; ++j) {
        int v = 0;
        for (int b = 0; b < bits; ++b) {
            int pos = j * bits + b;
            v |= ((in[pos >> 3] >> (pos & 7)) & 1) << b;
        }
        codes[j] = (uint8_t)v;
    }
}

/* ------------------------------------------------------------------------- */
/* O4 / O5: one token-head                                                    */
/* ------------------------------------------------------------------------- */

typedef struct or_diag {
    double *z;     /* [d] scaled rotated coordinates sqrt(d) Pi k / n   */
    double *pg;    /* [d] QJL projections p_i / gamma                    */
    double *norm;  /* [1] */
    double *gamma; /* [1] */
} or_diag;

/* Key record: kcode bytes of codes, ksign bytes of signs, bf16 norm, bf16 gamma. */
static void or_compress_key(const or_ctx *c, const uint16_t *kin, uint8_t *kcode, uint8_t *ksign,
                            uint16_t *knorm, uint16_t *kgamma, or_diag *dg)
{
    int d = c->d, L = 1 << c->kb;
    double k[256], y[256], r[256];
    uint8_t code[256], sig[256];
    double nsq = 0.0;
    for (int j = 0; j < d; ++j) {
        k[j] = tq_or_bf16_to_double(kin[j]);
        nsq += k[j] * k[j];
    }
    double n = sqrt(nsq);
    *knorm = tq_or_bf16_from_double(n);
    if (dg && dg->norm) *dg->norm = n;
    if (n == 0.0) { /* zero key: all-zero record */
        memset(kcode, 0, c->kcode);
        if (c->qjl) { memset(ksign, 0, c->ksign); *kgamma = 0; }
        if (dg && dg->z) for (int i = 0; i < d; ++i) dg->z[i] = 0.0;
        if (dg && dg->pg) for (int i = 0; i < d; ++i) dg->pg[i] = 0.0;
        if (dg && dg->gamma) *dg->gamma = 0.0;
        return;
    }
    double sd = sqrt((double)d);
    for (int i = 0; i < d; ++i) {
        double acc = 0.0;
        for (int j = 0; j < d; ++j) acc += c->Pi[i * d + j] * k[j];
        y[i] = acc / n;                  /* rotated unit vector */
        double z = sd * y[i];            /* ~ N(0,1) coordinate */
        int cnt = 0;
        for (int t = 0; t < L - 1; ++t) cnt += (c->thr[t] <= z); /* ties -> upper code */
        code[i] = (uint8_t)cnt;
        r[i] = y[i] - c->cent[cnt] / sd; /* residual in the rotated space */
        if (dg && dg->z) dg->z[i] = z;
    }
    tq_or_pack(code, d, c->kb, kcode);
    if (c->qjl) {
        double gsq = 0.0;
        for (int i = 0; i < d; ++i) gsq += r[i] * r[i];
        double gamma = sqrt(gsq);
        *kgamma = tq_or_bf16_from_double(gamma);
        if (dg && dg->gamma) *dg->gamma = gamma;
        for (int i = 0; i < d; ++i) { /* m = d projection rows */
            double p = 0.0;
            for (int j = 0; j < d; ++j) p += c->S[i * d + j] * r[j];
            sig[i] = (p >= 0.0);
            if (dg && dg->pg) dg->pg[i] = (gamma > 0.0) ? p / gamma : 0.0;
        }
        tq_or_pack(sig, d, 1, ksign);
    }
}

/*
 * O5': value record with the MSE codebook ([brightcoding] "What is TurboQuant-GPU?":
 * values get MSE quantization; "Example 4": normalize -> rotate -> Lloyd-Max
 * quantize -> pack): the key steps without QJL, with the v_bits codebook --
 * n = ||v|| stored bf16, z = sqrt(d) Pi v / n, code_j = #{i : t_i <= z_j}.
 * vmeta[0] receives the bf16 norm.  vz (optional) receives z.
 */
static void or_compress_value_mse(const or_ctx *c, const uint16_t *vin, uint8_t *vcode, uint16_t *vmeta, double *vz)
{
    int d = c->d, L = 1 << c->vb;
    double v[256];
    uint8_t code[256];
    double nsq = 0.0;
    for (int j = 0; j < d; ++j) {
        v[j] = tq_or_bf16_to_double(vin[j]);
        nsq += v[j] * v[j];
    }
    double n = sqrt(nsq);
    vmeta[0] = tq_or_bf16_from_double(n);
    double sd = sqrt((double)d);
    for (int i = 0; i < d; ++i) {
        int cnt = 0;
        double z = 0.0;
        if (n > 0.0) {
            double acc = 0.0;
            for (int j = 0; j < d; ++j) acc += c->Pi[i * d + j] * v[j];
            z = sd * acc / n;
            for (int t = 0; t < L - 1; ++t) cnt += (c->vthr[t] <= z);
        }
        code[i] = (uint8_t)cnt; /* a zero value: all-zero codes and norm */
        if (vz) vz[i] = z;
    }
    tq_or_pack(code, d, c->vb, vcode);
}

/* Value record: vcode bytes of codes, (d/g) x (scale, zero) fp16 pairs (O5), or
 * the codes and the bf16 norm (O5'). */
static void or_compress_value(const or_ctx *c, const uint16_t *vin, uint8_t *vcode, uint16_t *vmeta)
{
    if (c->vmse) {
        or_compress_value_mse(c, vin, vcode, vmeta, NULL);
        return;
    }
    int d = c->d, g = c->g, L = (1 << c->vb) - 1;
    uint8_t code[256];
    for (int gi = 0; gi < d / g; ++gi) {
        double mn = INFINITY, mx = -INFINITY;
        for (int j = 0; j < g; ++j) {
            double x = tq_or_bf16_to_double(vin[gi * g + j]);
            if (x < mn) mn = x;
            if (x > mx) mx = x;
        }
        uint16_t s16 = tq_or_f16_from_double((mx - mn) / L);
        uint16_t z16 = tq_or_f16_from_double(mn);
        double s = tq_or_f16_to_double(s16), z = tq_or_f16_to_double(z16);
        for (int j = 0; j < g; ++j) {
            double x = tq_or_bf16_to_double(vin[gi * g + j]);
            int q = 0;
            if (s != 0.0) /* round half up, exactly: count the midpoints at or below x - z */
                for (int m = 0; m < L; ++m) q += (x - z >= (m + 0.5) * s);
            code[gi * g + j] = (uint8_t)q;
        }
        vmeta[2 * gi] = s16;
        vmeta[2 * gi + 1] = z16;
    }
    tq_or_pack(code, d, c->vb, vcode);
}

/*
 * The QJL half of a key record for given codes (O4 steps 4-5): r = y - c/sqrt(d),
 * gamma = ||r||, sigma_i = [(S r)_i >= 0].  Used where two correct encoders may
 * take different codes for a coordinate that sits on a threshold: the signs
 * are then defined by the codes actually stored.
 */
void tq_or_key_qjl_given_codes(const or_ctx *c, const uint16_t *k, const uint8_t *codes, int64_t n,
                               uint8_t *ksign, uint16_t *kgamma, double *pg, double *gamma_out)
{
    int d = c->d;
    double sd = sqrt((double)d);
    for (int64_t row = 0; row < n; ++row) {
        const uint16_t *kin = k + row * d;
        const uint8_t *cd = codes + row * d;
        double kk[256], r[256];
        uint8_t sig[256];
        double nsq = 0.0;
        for (int j = 0; j < d; ++j) {
            kk[j] = tq_or_bf16_to_double(kin[j]);
            nsq += kk[j] * kk[j];
        }
        double nn = sqrt(nsq);
        for (int i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int j = 0; j < d; ++j) acc += c->Pi[i * d + j] * kk[j];
            r[i] = (nn > 0.0 ? acc / nn : 0.0) - c->cent[cd[i]] / sd;
        }
        double gsq = 0.0;
        for (int i = 0; i < d; ++i) gsq += r[i] * r[i];
        double g = sqrt(gsq);
        kgamma[row] = tq_or_bf16_from_double(g);
        if (gamma_out) gamma_out[row] = g;
        for (int i = 0; i < d; ++i) {
            double p = 0.0;
            for (int j = 0; j < d; ++j) p += c->S[i * d + j] * r[j];
            sig[i] = (p >= 0.0);
            if (pg) pg[row * d + i] = g > 0.0 ? p / g : 0.0;
        }
        tq_or_pack(sig, d, 1, ksign + row * (d / 8));
    }
}

/* ------------------------------------------------------------------------- */
/* Threading helper                                                           */
/* ------------------------------------------------------------------------- */

typedef void (*or_job_fn)(void *arg, int64_t lo, int64_t hi);
typedef struct { or_job_fn fn; void *arg; int64_t lo, hi; } or_span;

static void *or_thread_main(void *p)
{
    or_span *s = (or_span *)p;
    s->fn(s->arg, s->lo, s->hi);
    return NULL;
}

/* Runs fn over [0, n) split into contiguous spans, one per thread. */
static void or_parallel(or_job_fn fn, void *arg, int64_t n, int nthreads)
{
    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (n < nthreads) nthreads = n > 0 ? (int)n : 1;
    if (nthreads == 1) { fn(arg, 0, n); return; }
    pthread_t th[256];
    or_span sp[256];
    for (int t = 0; t < nthreads; ++t) {
        sp[t].fn = fn; sp[t].arg = arg;
        sp[t].lo = n * t / nthreads;
        sp[t].hi = n * (t + 1) / nthreads;
        pthread_create(&th[t], NULL, or_thread_main, &sp[t]);
    }
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------------------- */
/* Row-wise compress (records as separate field arrays, plus diagnostics)     */
/* ------------------------------------------------------------------------- */

typedef struct {
    const or_ctx *c;
    const uint16_t *k, *v;
    uint8_t *kcode, *ksign, *vcode;
    uint16_t *knorm, *kgamma, *vmeta;
    double *z, *pg, *norm, *gamma, *vz;
} or_rows_job;

static void or_rows_run(void *p, int64_t lo, int64_t hi)
{
    or_rows_job *J = (or_rows_job *)p;
    const or_ctx *c = J->c;
    int d = c->d;
    for (int64_t i = lo; i < hi; ++i) {
        if (J->k) {
            or_diag dg = {J->z ? J->z + i * d : NULL, J->pg ? J->pg + i * d : NULL,
                          J->norm ? J->norm + i : NULL, J->gamma ? J->gamma + i : NULL};
            uint16_t gdummy;
            uint8_t sdummy[32];
            or_compress_key(c, J->k + i * d, J->kcode + i * c->kcode,
                            c->qjl ? J->ksign + i * c->ksign : sdummy, J->knorm + i,
                            c->qjl ? J->kgamma + i : &gdummy, &dg);
        }
        if (J->v) {
            if (c->vmse)
                or_compress_value_mse(c, J->v + i * d, J->vcode + i * c->vcode, J->vmeta + i * (c->vmeta / 2),
                                      J->vz ? J->vz + i * d : NULL);
            else
                or_compress_value(c, J->v + i * d, J->vcode + i * c->vcode, J->vmeta + i * (c->vmeta / 2));
        }
    }
}

/*
 * Compress n contiguous rows of d bf16 values.  k or v may be NULL to skip
 * that stream.  ksign / kgamma are only written when QJL is on.  Diagnostic
 * arrays (z, pg: [n][d]; norm, gamma: [n]) may be NULL.
 */
void tq_or_compress_rows(const or_ctx *c, const uint16_t *k, const uint16_t *v, int64_t n,
                         uint8_t *kcode, uint8_t *ksign, uint16_t *knorm, uint16_t *kgamma,
                         uint8_t *vcode, uint16_t *vmeta,
                         double *z, double *pg, double *norm, double *gamma, double *vz, int nthreads)
{
    or_rows_job J = {c, k, v, kcode, ksign, vcode, knorm, kgamma, vmeta, z, pg, norm, gamma, vz};
    or_parallel(or_rows_run, &J, n, nthreads);
}

/* ------------------------------------------------------------------------- */
/* O6: paged layout                                                           */
/* ------------------------------------------------------------------------- */
/*
 * Pools: K pool [num_blocks][Hkv] page records of kpage bytes, V pool the same
 * with vpage bytes.  slot -> block = slot / P, offset = slot % P.
 * K record: codes [P][kcode] | signs [P][ksign] (QJL) | norms [P] bf16 | gammas [P] bf16 (QJL)
 * V record: codes [P][vcode] | meta [P][d/g][2] fp16 (scale, zero)
 */

typedef struct {
    const or_ctx *c;
    const uint16_t *k, *v;
    int64_t T;
    int Hkv;
    int64_t ks, vs;
    const int64_t *slots;
    uint8_t *kc, *vc;
    int P;
    int64_t nb;
    int64_t kpage, vpage;
} or_kv_job;

static void or_kv_run(void *p, int64_t lo, int64_t hi)
{
    or_kv_job *J = (or_kv_job *)p;
    const or_ctx *c = J->c;
    int P = J->P;
    for (int64_t i = lo; i < hi; ++i) { /* i = t * Hkv + h */
        int64_t t = i / J->Hkv;
        int h = (int)(i % J->Hkv);
        int64_t slot = J->slots[t];
        if (slot < 0 || slot >= J->nb * P) continue;
        int64_t blk = slot / P;
        int off = (int)(slot % P);
        uint8_t *kr = J->kc + (blk * J->Hkv + h) * J->kpage;
        uint8_t *vr = J->vc + (blk * J->Hkv + h) * J->vpage;
        uint8_t *kcode = kr + (int64_t)off * c->kcode;
        uint8_t *ksign = kr + (int64_t)P * c->kcode + (int64_t)off * c->ksign;
        uint8_t *knorm = kr + (int64_t)P * (c->kcode + c->ksign) + 2 * off;
        uint8_t *kgam = kr + (int64_t)P * (c->kcode + c->ksign + 2) + 2 * off;
        uint16_t nbits, gbits = 0;
        uint8_t sbuf[32];
        or_compress_key(c, J->k + t * J->ks + (int64_t)h * c->d, kcode, c->qjl ? ksign : sbuf, &nbits, &gbits, NULL);
        memcpy(knorm, &nbits, 2); /* little-endian host */
        if (c->qjl) memcpy(kgam, &gbits, 2);
        uint16_t meta[64];
        or_compress_value(c, J->v + t * J->vs + (int64_t)h * c->d, vr + (int64_t)off * c->vcode, meta);
        memcpy(vr + (int64_t)P * c->vcode + (int64_t)off * c->vmeta, meta, c->vmeta);
    }
}

/* Compress K and V ([T][Hkv][d] bf16 with token strides in elements) into the paged pools.
 * Returns the number of skipped tokens (slot -1 or out of range). */
int64_t tq_or_compress_kv(const or_ctx *c, const uint16_t *k, const uint16_t *v, int64_t T, int Hkv,
                          int64_t k_stride_tok, int64_t v_stride_tok, const int64_t *slots,
                          uint8_t *k_cache, uint8_t *v_cache, int P, int64_t num_blocks, int nthreads)
{
    int64_t sz[6];
    tq_or_geometry(c, P, sz);
    or_kv_job J = {c, k, v, T, Hkv, k_stride_tok, v_stride_tok, slots, k_cache, v_cache, P, num_blocks, sz[4], sz[5]};
    or_parallel(or_kv_run, &J, T * Hkv, nthreads);
    int64_t skipped = 0;
    for (int64_t t = 0; t < T; ++t) skipped += (slots[t] < 0 || slots[t] >= num_blocks * P);
    return skipped;
}

/* ------------------------------------------------------------------------- */
/* Reading a token-head back out of the pools                                 */
/* ------------------------------------------------------------------------- */

typedef struct {
    uint8_t code[256];
    uint8_t sig[256];
    double n, gamma;
    double vs[64], vz[64];
    double vn; /* value norm (O5') */
    uint8_t vcode[256];
} or_rec;

static void or_read(const or_ctx *c, const uint8_t *kc, const uint8_t *vc, int P, int Hkv, int64_t slot, int h,
                    or_rec *R)
{
    int64_t sz[6];
    tq_or_geometry(c, P, sz);
    int64_t blk = slot / P;
    int off = (int)(slot % P);
    const uint8_t *kr = kc + (blk * Hkv + h) * sz[4];
    const uint8_t *vr = vc + (blk * Hkv + h) * sz[5];
    tq_or_unpack(kr + (int64_t)off * c->kcode, c->d, c->kb, R->code);
    uint16_t b;
    memcpy(&b, kr + (int64_t)P * (c->kcode + c->ksign) + 2 * off, 2);
    R->n = tq_or_bf16_to_double(b);
    if (c->qjl) {
        tq_or_unpack(kr + (int64_t)P * c->kcode + (int64_t)off * c->ksign, c->d, 1, R->sig);
        memcpy(&b, kr + (int64_t)P * (c->kcode + c->ksign + 2) + 2 * off, 2);
        R->gamma = tq_or_bf16_to_double(b);
    }
    tq_or_unpack(vr + (int64_t)off * c->vcode, c->d, c->vb, R->vcode);
    const uint8_t *meta = vr + (int64_t)P * c->vcode + (int64_t)off * c->vmeta;
    if (c->vmse) {
        memcpy(&b, meta, 2);
        R->vn = tq_or_bf16_to_double(b);
        return;
    }
    for (int gi = 0; gi < c->d / c->g; ++gi) {
        uint16_t s16, z16;
        memcpy(&s16, meta + 4 * gi, 2);
        memcpy(&z16, meta + 4 * gi + 2, 2);
        R->vs[gi] = tq_or_f16_to_double(s16);
        R->vz[gi] = tq_or_f16_to_double(z16);
    }
}

/* O7: K~ in the original space and V~, in double. */
static void or_dequant_rec(const or_ctx *c, const or_rec *R, double *kout, double *vout)
{
    int d = c->d;
    double sd = sqrt((double)d);
    double u[256];
    double qj = c->qjl ? sqrt(OR_PI / 2.0) / d * R->gamma : 0.0;
    for (int j = 0; j < d; ++j) u[j] = c->cent[R->code[j]] / sd; /* rotated-space estimate */
    if (c->qjl)
        for (int j = 0; j < d; ++j) {
            double a = 0.0;
            for (int i = 0; i < d; ++i) a += c->S[i * d + j] * (R->sig[i] ? 1.0 : -1.0);
            u[j] += qj * a;
        }
    for (int j = 0; j < d; ++j) { /* back to the original space: Pi^T u, times the norm */
        double a = 0.0;
        for (int i = 0; i < d; ++i) a += c->Pi[i * d + j] * u[i];
        kout[j] = R->n * a;
    }
    if (c->vmse) { /* O5': V~ = n Pi^T c[code] / sqrt(d) */
        for (int j = 0; j < d; ++j) {
            double a = 0.0;
            for (int i = 0; i < d; ++i) a += c->Pi[i * d + j] * c->vcent[R->vcode[i]];
            vout[j] = R->vn * a / sd;
        }
        return;
    }
    for (int j = 0; j < d; ++j) vout[j] = R->vcode[j] * R->vs[j / c->g] + R->vz[j / c->g];
}

/* Dequantise n_slots slots for all Hkv heads: k_out, v_out are [n_slots][Hkv][d] doubles. */
void tq_or_dequant_slots(const or_ctx *c, const uint8_t *kc, const uint8_t *vc, int P, int Hkv,
                         const int64_t *slots, int64_t n_slots, double *k_out, double *v_out)
{
    or_rec R;
    for (int64_t s = 0; s < n_slots; ++s)
        for (int h = 0; h < Hkv; ++h) {
            or_read(c, kc, vc, P, Hkv, slots[s], h, &R);
            or_dequant_rec(c, &R, k_out + (s * Hkv + h) * c->d, v_out + (s * Hkv + h) * c->d);
        }
}

/* ------------------------------------------------------------------------- */
/* O8: decode attention                                                       */
/* ------------------------------------------------------------------------- */

typedef struct {
    const or_ctx *c;
    const uint16_t *q;
    const uint8_t *kc, *vc;
    const int32_t *bt, *seq;
    int B, Hq, Hkv, P, maxblk;
    double sm_scale;
    int mode;
    const int32_t *jobs; /* pairs (b, kvh) */
    double *out;
} or_dec_job;

static void or_dec_run(void *p, int64_t lo, int64_t hi)
{
    or_dec_job *J = (or_dec_job *)p;
    const or_ctx *c = J->c;
    int d = c->d, G = J->Hq / J->Hkv;
    double sd = sqrt((double)d);
    double qj = sqrt(OR_PI / 2.0) / d;
    double *kt = malloc(sizeof(double) * d), *vt = malloc(sizeof(double) * d);
    double *qrot = malloc(sizeof(double) * G * d), *qs = malloc(sizeof(double) * G * d);
    for (int64_t jb = lo; jb < hi; ++jb) {
        int b = J->jobs[2 * jb], kvh = J->jobs[2 * jb + 1];
        int L = J->seq[b];
        if (L < 0) L = 0;
        double *s = malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * G);
        double *qd = malloc(sizeof(double) * G * d);
        for (int gh = 0; gh < G; ++gh) {
            int h = kvh * G + gh;
            for (int j = 0; j < d; ++j) qd[gh * d + j] = tq_or_bf16_to_double(J->q[((int64_t)b * J->Hq + h) * d + j]);
            if (J->mode == 1) { /* pre-rotate the query: q_rot = Pi q, q_s = S q_rot */
                for (int i = 0; i < d; ++i) {
                    double a = 0.0;
                    for (int j = 0; j < d; ++j) a += c->Pi[i * d + j] * qd[gh * d + j];
                    qrot[gh * d + i] = a;
                }
                for (int i = 0; i < d; ++i) {
                    double a = 0.0;
                    for (int j = 0; j < d; ++j) a += c->S[i * d + j] * qrot[gh * d + j];
                    qs[gh * d + i] = a;
                }
            }
        }
        or_rec R;
        /* pass 1: scores */
        for (int t = 0; t < L; ++t) {
            int64_t slot = (int64_t)J->bt[(int64_t)b * J->maxblk + t / J->P] * J->P + t % J->P;
            or_read(c, J->kc, J->vc, J->P, J->Hkv, slot, kvh, &R);
            if (J->mode == 0) {
                or_dequant_rec(c, &R, kt, vt);
                for (int gh = 0; gh < G; ++gh) {
                    double a = 0.0;
                    for (int j = 0; j < d; ++j) a += qd[gh * d + j] * kt[j];
                    s[(int64_t)t * G + gh] = J->sm_scale * a;
                }
            } else {
                for (int gh = 0; gh < G; ++gh) {
                    double a = 0.0, e = 0.0;
                    for (int j = 0; j < d; ++j) a += qrot[gh * d + j] * c->cent[R.code[j]];
                    a /= sd;
                    if (c->qjl) {
                        for (int i = 0; i < d; ++i) e += qs[gh * d + i] * (R.sig[i] ? 1.0 : -1.0);
                        a += qj * R.gamma * e;
                    }
                    s[(int64_t)t * G + gh] = J->sm_scale * R.n * a;
                }
            }
        }
        /* pass 2: softmax and weighted values */
        for (int gh = 0; gh < G; ++gh) {
            int h = kvh * G + gh;
            double *o = J->out + ((int64_t)b * J->Hq + h) * d;
            for (int j = 0; j < d; ++j) o[j] = 0.0;
            if (L == 0) continue;
            double m = -INFINITY;
            for (int t = 0; t < L; ++t) if (s[(int64_t)t * G + gh] > m) m = s[(int64_t)t * G + gh];
            double den = 0.0;
            for (int t = 0; t < L; ++t) den += exp(s[(int64_t)t * G + gh] - m);
            if (c->vmse) { /* O5' values: sum in the rotated space, then Pi^T once */
                for (int i = 0; i < d; ++i) vt[i] = 0.0;
                for (int t = 0; t < L; ++t) {
                    double w = exp(s[(int64_t)t * G + gh] - m) / den;
                    int64_t slot = (int64_t)J->bt[(int64_t)b * J->maxblk + t / J->P] * J->P + t % J->P;
                    or_read(c, J->kc, J->vc, J->P, J->Hkv, slot, kvh, &R);
                    for (int i = 0; i < d; ++i) vt[i] += w * R.vn * c->vcent[R.vcode[i]] / sd;
                }
                for (int j = 0; j < d; ++j) {
                    double a = 0.0;
                    for (int i = 0; i < d; ++i) a += c->Pi[i * d + j] * vt[i];
                    o[j] = a;
                }
                continue;
            }
            for (int t = 0; t < L; ++t) {
                double w = exp(s[(int64_t)t * G + gh] - m) / den;
                int64_t slot = (int64_t)J->bt[(int64_t)b * J->maxblk + t / J->P] * J->P + t % J->P;
                or_read(c, J->kc, J->vc, J->P, J->Hkv, slot, kvh, &R);
                for (int j = 0; j < d; ++j) o[j] += w * (R.vcode[j] * R.vs[j / c->g] + R.vz[j / c->g]);
            }
        }
        free(s);
        free(qd);
    }
    free(kt); free(vt); free(qrot); free(qs);
}

/*
 * Decode attention for one query token per sequence.  q: [B][Hq][d] bf16;
 * block_table: [B][maxblk]; seq_lens: [B]; out: [B][Hq][d] doubles.
 * Query head h reads KV head h / (Hq / Hkv).  No mask: the token sees its whole
 * context.  mode 0 scores against K~ in the original space, mode 1 scores in
 * the rotated space from the codes.  jobs: n_jobs (b, kvh) pairs to compute
 * (NULL = all); rows not computed are left untouched.
 */
void tq_or_decode(const or_ctx *c, const uint16_t *q, const uint8_t *kc, const uint8_t *vc,
                  const int32_t *block_table, const int32_t *seq_lens, int B, int Hq, int Hkv, int P,
                  int max_blocks, double sm_scale, int mode, const int32_t *jobs, int64_t n_jobs,
                  double *out, int nthreads)
{
    int32_t *all = NULL;
    if (!jobs) {
        n_jobs = (int64_t)B * Hkv;
        all = malloc(sizeof(int32_t) * 2 * n_jobs);
        for (int b = 0; b < B; ++b)
            for (int h = 0; h < Hkv; ++h) { all[2 * (b * Hkv + h)] = b; all[2 * (b * Hkv + h) + 1] = h; }
        jobs = all;
    }
    or_dec_job J = {c, q, kc, vc, block_table, seq_lens, B, Hq, Hkv, P, max_blocks, sm_scale, mode, jobs, out};
    or_parallel(or_dec_run, &J, n_jobs, nthreads);
    free(all);
}

/* ------------------------------------------------------------------------- */
/* Bypass decode over plain bf16 pages                                        */
/* ------------------------------------------------------------------------- */

/*
 * [turbo-attn] "Two independently-usable pieces", item 2: the decode kernel with
 * a bypass loader reads ordinary bf16 pages.  What it computes is plain softmax
 * attention of one query token per sequence over its paged bf16 context:
 * pools [num_blocks][Hkv][P][d]; position t of sequence b is row t % P of block
 * bt[b][t / P]; query head h reads kv head h / (Hq / Hkv); s_t = sm_scale <q, k_t>,
 * p = softmax(s) (max-subtracted), o = sum_t p_t v_t, in double; seq_len 0 gives
 * zeros.  out: [B][Hq][d] doubles.
 */
void tq_or_decode_bf16(const uint16_t *q, const uint16_t *kpool, const uint16_t *vpool, const int32_t *bt,
                       const int32_t *lens, int B, int Hq, int Hkv, int d, int P, int maxblk, double sm_scale,
                       double *out)
{
    int G = Hq / Hkv;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < Hq; ++h) {
            int kvh = h / G;
            int L = lens[b];
            double *o = out + ((int64_t)b * Hq + h) * d;
            for (int j = 0; j < d; ++j) o[j] = 0.0;
            if (L <= 0) continue;
            double *s = malloc(sizeof(double) * L);
            double mx = -INFINITY;
            for (int t = 0; t < L; ++t) {
                int64_t rowi = ((int64_t)bt[(int64_t)b * maxblk + t / P] * Hkv + kvh) * P + t % P;
                double acc = 0.0;
                for (int j = 0; j < d; ++j)
                    acc += tq_or_bf16_to_double(q[((int64_t)b * Hq + h) * d + j]) *
                           tq_or_bf16_to_double(kpool[rowi * d + j]);
                s[t] = sm_scale * acc;
                if (s[t] > mx) mx = s[t];
            }
            double den = 0.0;
            for (int t = 0; t < L; ++t) {
                s[t] = exp(s[t] - mx);
                den += s[t];
            }
            for (int t = 0; t < L; ++t) {
                int64_t rowi = ((int64_t)bt[(int64_t)b * maxblk + t / P] * Hkv + kvh) * P + t % P;
                double w = s[t] / den;
                for (int j = 0; j < d; ++j) o[j] += w * tq_or_bf16_to_double(vpool[rowi * d + j]);
            }
            free(s);
        }
}

