/*
 * ott_oracle.c -- plain CPU oracle for Outlier Tokens Tracing (OTT) KV-cache
 * quantization: the every-G flush and the three-store decode attention.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark load this file. It shares no code, header,
 * table or helper with the CUDA library and is written to be read against
 * the sources, not to be fast. It never calls into the CUDA library.
 *
 * Sources (page title / section):
 *  [blog]  "Accurate KV Cache Quantization with Outlier Tokens Tracing"
 *          (zijie-tian.site): sec. 3.1 (quantize the latest group every G
 *          tokens; rank candidates by the key norm), sec. 3.2 (outlier pool
 *          of capacity P, new tokens compete with pool tokens, a displaced
 *          token is written back to the main cache), sec. 3.3 (decode: the
 *          query meets quantized, residual-window and pool keys; concat,
 *          softmax, times the matching values), the flowchart.
 *  [ss]    "Accurate KV Cache Quantization with Outlier Tokens Tracing"
 *          (sciencestack.ai, arXiv 2505.10938): TL;DR (three KV caches, pool
 *          filled by key magnitude, group quantization every G tokens),
 *          Abstract (keys quantized per channel, values per token),
 *          Fig. 1(c) (keep the tokens whose keys have the smallest
 *          magnitude), Fig. 2 (decoding and quantization stages).
 *  [kivi]  the KIVI reference listed on the mlsanity.com page ("asymmetric
 *          2bit"): min/max asymmetric quantization.
 *
 * Readings taken where the pages are silent (each is restated where used):
 *  R1  The R newest tokens stay fp16; once G+R tokens wait unquantized, the
 *      G oldest of them form the group that is flushed (ring holds < G+R).
 *  R2  A prefill of L tokens is L appends, in token order.
 *  R3  The outlier score is the squared L2 norm of the fp16 key, summed in
 *      fp32 in channel order 0..d-1 (same ranking as the L2 norm).
 *  R4  Candidates at a flush are the pool plus the whole group; the P
 *      smallest (norm, token index) pairs stay, ties go to the lower index.
 *  R5  Evicted pool tokens and the group's non-outliers together form the
 *      new quantized block, stored in ascending token order; a block is
 *      made at every flush, even when it holds no token.
 *  R6  Keys: one (scale, zero) per channel over the block's tokens. Values:
 *      one (scale, zero) per token per 32 consecutive channels. Both fp16.
 *  R7  mn, mx over the valid values (as fp32; -0 orders below +0);
 *      s = fp16_rn((mx - mn) / 3) in fp32 with IEEE division; z = mn;
 *      code = 0 if s == 0, else clamp(rint((x - z) / s), 0, 3) with fp32
 *      subtraction and division and round-half-to-even.
 *  R8  Pool and residual tokens keep their fp16 values ("full precision").
 *  R9  Decode attends over every token seen, with scale 1/sqrt(d); query
 *      head h reads kv head h / (Hq / Hkv).
 *  R10 Batches may be ragged: each sequence keeps its own token count (a
 *      prefill may give every sequence its own length), an append adds one
 *      token to every sequence, and R1 applies to each unit on its own. The
 *      pages state the method for one sequence; this is that method applied
 *      to each sequence of a batch independently.
 *  R11 The cold-pool policy ([blog] sec. 3.2, the alternative to writing a
 *      displaced token back): with cold capacity C, the pool tokens that a
 *      flush displaces do not join the new block; they enter an fp16
 *      first-in-first-out "cold" pool, in ascending token order. When it
 *      holds more than C tokens, the ones that entered first are discarded
 *      and no store holds them any more. The new block is the group's
 *      tokens that did not enter the pool. Decode attends the cold pool like
 *      the outlier pool; discarded tokens are not attended.
 *  R13 A sequence of a batch can be released (it then holds no token) and
 *      refilled with a new prompt; from then on it is a fresh sequence of
 *      its own (R10): its tokens are numbered from 0, and no state of the
 *      released one remains. Appends and decodes need every sequence to
 *      hold at least one token.
 *  R12 Top-K sparse access ([blog] sec. 6, combining OTT with sparse KV
 *      access): a decode call may attend only K of a unit's quantized
 *      blocks, plus every residual, pool and cold token. The K blocks are
 *      the non-empty ones with the largest score bound, ties to the lower
 *      block index. The bound of block j for query head h is the largest
 *      q.k that a key dequantized from the block's per-channel scale s and
 *      zero z can reach: the sum over channels of max(q*z, q*(z + 3*s)),
 *      taken in fp32 (products, 3*s and z + 3*s rounded to nearest, summed
 *      in channel order); the block's bound is the largest over the query
 *      heads that share the kv head. A selected block is attended whole.
 *  R14 The channel-conditioned criterion ([blog] sec. 3.1: a candidate is an
 *      outlier when it lies in an outlier channel and its magnitude is among
 *      the globally smallest p%), a policy beside R4: at a flush, over the
 *      candidates (pool plus group), the outlier channels are the n_oc
 *      channels with the largest max |k| over the candidates (ties to the
 *      lower channel index); each candidate's score is its squared norm over
 *      those channels only (fp32, ascending channel order); the smallest
 *      m = ceil(p * ncand) scores (ties to the lower token index) are the
 *      outliers, p given in units of 1/10000 so that m is exact; the pool
 *      keeps the min(P, m) most outlying of them, and every other candidate
 *      joins the new block (written back). Pool sizes, and so block sizes,
 *      follow from p, P and G alone: the same for every unit.
 *
 * Floating point: decisions that yield integers or stored bits (norms,
 * scales, zeros, codes) are taken in fp32 exactly as the library takes them.
 * The attention output is computed in double. Build with -ffp-contract=off.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16 <-> binary32, written from the format's definition.    */
/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.        */
/* ------------------------------------------------------------------------ */

float orc_h2f(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    float v;
    if (e == 0)
        v = ldexpf((float)m, -24);                   /* zero / subnormal */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexpf((float)(m | 0x400), e - 25);      /* (1024+m) * 2^(e-25) */
    return sign ? -v : v;
}

/* Round |f| to the binary16 grid with ties to even, then encode. */
uint16_t orc_f2h(float f)
{
    uint32_t bits;
    memcpy(&bits, &f, 4);
    uint16_t sign = (uint16_t)((bits >> 16) & 0x8000u);
    if (isnan(f))
        return (uint16_t)(sign | 0x7e00u);
    double a = fabs((double)f);
    if (isinf(f))
        return (uint16_t)(sign | 0x7c00u);
    if (a == 0.0)
        return sign;
    /* grid spacing at a: 2^-24 below 2^-14 (subnormals), else 2^(E-10) */
    int E;
    frexp(a, &E);                 /* a = frac * 2^E, frac in [0.5, 1) */
    E -= 1;                       /* a in [2^E, 2^(E+1)) */
    int qexp = (E < -14) ? -24 : E - 10;
    double y = ldexp(a, -qexp);   /* exact: a has 24 significant bits */
    double r = floor(y);
    double frac = y - r;
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0))
        r += 1.0;
    double rounded = ldexp(r, qexp);
    if (rounded >= 65536.0)
        return (uint16_t)(sign | 0x7c00u);           /* overflow to inf */
    if (rounded < ldexp(1.0, -14))                    /* subnormal (or 0) */
        return (uint16_t)(sign | (uint16_t)(rounded / ldexp(1.0, -24)));
    int E2;
    frexp(rounded, &E2);
    E2 -= 1;
    int mant = (int)(ldexp(rounded, 10 - E2)) - 1024;
    return (uint16_t)(sign | (uint16_t)((E2 + 15) << 10) | (uint16_t)mant);
}

void orc_f2h_array(const float *x, uint16_t *out, long long n)
{
    for (long long i = 0; i < n; ++i)
        out[i] = orc_f2h(x[i]);
}

void orc_h2f_array(const uint16_t *x, float *out, long long n)
{
    for (long long i = 0; i < n; ++i)
        out[i] = orc_h2f(x[i]);
}

/* ------------------------------------------------------------------------ */
/* Outlier score (R3): squared L2 norm of an fp16 key, fp32, channel order. */
/* ------------------------------------------------------------------------ */

float orc_norm(const uint16_t *k, int d)
{
    float s = 0.0f;
    for (int c = 0; c < d; ++c) {
        float kc = orc_h2f(k[c]);
        s = s + kc * kc;
    }
    return s;
}

/* ------------------------------------------------------------------------ */
/* Asymmetric 2-bit quantization of n values x[0], x[stride], ... (R7).     */
/* Writes the fp16 bits of scale and zero, and one code per value.           */
/* ------------------------------------------------------------------------ */

static int below(float a, float b)  /* a < b, with -0 ordered below +0 */
{
    return a < b || (a == b && signbit(a) && !signbit(b));
}

void orc_quant_group(const uint16_t *x, int n, int stride, uint16_t *s_out,
                     uint16_t *z_out, uint8_t *code, int code_stride)
{
    if (n <= 0) {
        *s_out = 0;
        *z_out = 0;
        return;
    }
    float mn = orc_h2f(x[0]), mx = mn;
    for (int i = 1; i < n; ++i) {
        float v = orc_h2f(x[(long)i * stride]);
        if (below(v, mn))
            mn = v;
        if (below(mx, v))
            mx = v;
    }
    uint16_t s16 = orc_f2h((mx - mn) / 3.0f);
    uint16_t z16 = orc_f2h(mn);                       /* exact: mn is fp16 */
    float s = orc_h2f(s16), z = orc_h2f(z16);
    for (int i = 0; i < n; ++i) {
        int q = 0;
        if (s != 0.0f) {
            float v = orc_h2f(x[(long)i * stride]);
            q = (int)rintf((v - z) / s);
            if (q < 0)
                q = 0;
            if (q > 3)
                q = 3;
        }
        code[(long)i * code_stride] = (uint8_t)q;
    }
    *s_out = s16;
    *z_out = z16;
}

/* ------------------------------------------------------------------------ */
/* Cache state, one unit per (sequence b, kv head).                          */
/* ------------------------------------------------------------------------ */

typedef struct {
    int c;              /* valid tokens in the block */
    int32_t *idx;       /* [c] token indices, ascending */
    uint8_t *kcode;     /* [c][d] key codes 0..3 */
    uint16_t *ks, *kz;  /* [d] per-channel key scale/zero (fp16 bits) */
    uint8_t *vcode;     /* [c][d] value codes 0..3 */
    uint16_t *vs, *vz;  /* [c][d/32] per-token value scale/zero (fp16 bits) */
} orc_block;

typedef struct {
    /* unquantized residual tokens, oldest first */
    int tail_n, tail_cap;
    int32_t *tail_idx;
    uint16_t *tail_k, *tail_v;   /* [tail_cap][d] */
    /* outlier pool, kept sorted by (norm, idx) ascending */
    int pool_n;
    int32_t *pool_idx;           /* [P] */
    float *pool_norm;            /* [P] */
    uint16_t *pool_k, *pool_v;   /* [P][d] */
    /* quantized blocks, one per flush */
    int nb, nb_cap;
    orc_block *blk;
    /* cold pool (R11), oldest first */
    int cold_n;
    int32_t *cold_idx;           /* [C] */
    uint16_t *cold_k, *cold_v;   /* [C][d] */
} orc_unit;

typedef struct {
    int B, Hq, Hkv, d, G, R, P;
    long long T;        /* appends plus the longest prefill (0: empty) */
    long long *Tb;      /* [B] tokens seen by each sequence (R10) */
    int C;              /* cold-pool capacity (R11); -1: displaced tokens are written back */
    int pct;            /* R14: p in units of 1/10000; -1: the norm criterion of R4 */
    int n_oc;           /* R14: outlier channels per flush */
    orc_unit *u;        /* [B*Hkv] */
} orc_cache;

typedef struct {
    float norm;
    int32_t idx;
    int from_pool;      /* 1: the candidate was in the pool before this flush */
    const uint16_t *k, *v;
} orc_cand;

static int cand_cmp_norm(const void *a, const void *b)
{
    const orc_cand *x = (const orc_cand *)a, *y = (const orc_cand *)b;
    if (x->norm < y->norm) return -1;
    if (x->norm > y->norm) return 1;
    return (x->idx < y->idx) ? -1 : (x->idx > y->idx);
}

static int cand_cmp_idx(const void *a, const void *b)
{
    const orc_cand *x = (const orc_cand *)a, *y = (const orc_cand *)b;
    return (x->idx < y->idx) ? -1 : (x->idx > y->idx);
}

void orc_destroy(void *hp)
{
    orc_cache *h = (orc_cache *)hp;
    if (!h)
        return;
    for (int i = 0; i < h->B * h->Hkv; ++i) {
        orc_unit *u = &h->u[i];
        free(u->tail_idx); free(u->tail_k); free(u->tail_v);
        free(u->pool_idx); free(u->pool_norm); free(u->pool_k); free(u->pool_v);
        for (int j = 0; j < u->nb; ++j) {
            orc_block *b = &u->blk[j];
            free(b->idx); free(b->kcode); free(b->ks); free(b->kz);
            free(b->vcode); free(b->vs); free(b->vz);
        }
        free(u->blk);
        free(u->cold_idx); free(u->cold_k); free(u->cold_v);
    }
    free(h->u);
    free(h->Tb);
    free(h);
}

/* C < 0: displaced pool tokens are written back (R5); C >= 0: the cold-pool
 * policy with capacity C (R11). */
void *orc_create_policy(int B, int Hq, int Hkv, int d, int G, int R, int P, int C)
{
    if (B < 1 || Hkv < 1 || Hq < Hkv || Hq % Hkv || d < 32 || d % 32 ||
        G < 1 || R < 0 || P < 0)
        return NULL;
    orc_cache *h = (orc_cache *)calloc(1, sizeof(orc_cache));
    h->B = B; h->Hq = Hq; h->Hkv = Hkv; h->d = d; h->G = G; h->R = R; h->P = P;
    h->C = C < 0 ? -1 : C;
    h->pct = -1;
    h->n_oc = 0;
    h->u = (orc_unit *)calloc((size_t)B * Hkv, sizeof(orc_unit));
    h->Tb = (long long *)calloc((size_t)B, sizeof(long long));
    for (int i = 0; i < B * Hkv; ++i) {
        orc_unit *u = &h->u[i];
        u->tail_cap = G + R;
        u->tail_idx = (int32_t *)calloc(u->tail_cap, sizeof(int32_t));
        u->tail_k = (uint16_t *)calloc((size_t)u->tail_cap * d, 2);
        u->tail_v = (uint16_t *)calloc((size_t)u->tail_cap * d, 2);
        u->pool_idx = (int32_t *)calloc(P + 1, sizeof(int32_t));
        u->pool_norm = (float *)calloc(P + 1, sizeof(float));
        u->pool_k = (uint16_t *)calloc((size_t)(P + 1) * d, 2);
        u->pool_v = (uint16_t *)calloc((size_t)(P + 1) * d, 2);
        if (h->C >= 0) {
            u->cold_idx = (int32_t *)calloc(h->C + 1, sizeof(int32_t));
            u->cold_k = (uint16_t *)calloc((size_t)(h->C + 1) * d, 2);
            u->cold_v = (uint16_t *)calloc((size_t)(h->C + 1) * d, 2);
        }
    }
    return h;
}

void *orc_create(int B, int Hq, int Hkv, int d, int G, int R, int P)
{
    return orc_create_policy(B, Hq, Hkv, d, G, R, P, -1);
}

/* R14: the channel-conditioned outlier criterion with p = pct / 10000 and
 * n_oc outlier channels; displaced pool tokens are written back. */
void *orc_create_pct(int B, int Hq, int Hkv, int d, int G, int R, int P, int pct, int n_oc)
{
    if (pct < 0 || pct > 10000 || n_oc < 1 || n_oc > d)
        return NULL;
    orc_cache *h = (orc_cache *)orc_create_policy(B, Hq, Hkv, d, G, R, P, -1);
    if (h) {
        h->pct = pct;
        h->n_oc = n_oc;
    }
    return h;
}

/* R14, step 1: the n_oc channels with the largest max |k| over the
 * candidates, ties to the lower channel index; out[0..n_oc) ascending. */
static void outlier_channels(const orc_cand *cand, int ncand, int d, int n_oc, int *out)
{
    float *amax = (float *)calloc(d, sizeof(float));
    char *taken = (char *)calloc(d, 1);
    for (int c = 0; c < d; ++c)
        for (int t = 0; t < ncand; ++t) {
            float a = fabsf(orc_h2f(cand[t].k[c]));
            if (a > amax[c])
                amax[c] = a;
        }
    for (int n = 0; n < n_oc; ++n) {     /* pick the largest remaining, lower index first */
        int best = -1;
        for (int c = 0; c < d; ++c)
            if (!taken[c] && (best < 0 || amax[c] > amax[best]))
                best = c;
        taken[best] = 1;
    }
    int n = 0;
    for (int c = 0; c < d; ++c)
        if (taken[c])
            out[n++] = c;
    free(amax);
    free(taken);
}

/* R14, step 2: squared norm over the chosen channels (fp32, ascending). */
static float outlier_channel_norm(const uint16_t *k, const int *oc, int n_oc)
{
    float s = 0.0f;
    for (int n = 0; n < n_oc; ++n) {
        float kc = orc_h2f(k[oc[n]]);
        s = s + kc * kc;
    }
    return s;
}

/* R11: the displaced pool tokens ev[0..n) (ascending token order) enter the
 * cold pool one by one; while it is full, the token that entered first
 * leaves. */
static void cold_push(orc_cache *h, orc_unit *u, const orc_cand *ev, int n)
{
    const int d = h->d;
    if (h->C == 0)
        return;
    for (int e = 0; e < n; ++e) {
        if (u->cold_n == h->C) {
            memmove(u->cold_idx, u->cold_idx + 1, sizeof(int32_t) * (h->C - 1));
            memmove(u->cold_k, u->cold_k + d, (size_t)(h->C - 1) * d * 2);
            memmove(u->cold_v, u->cold_v + d, (size_t)(h->C - 1) * d * 2);
            u->cold_n -= 1;
        }
        u->cold_idx[u->cold_n] = ev[e].idx;
        memcpy(u->cold_k + (size_t)u->cold_n * d, ev[e].k, (size_t)d * 2);
        memcpy(u->cold_v + (size_t)u->cold_n * d, ev[e].v, (size_t)d * 2);
        u->cold_n += 1;
    }
}

/* The flush (R1, R3-R7): the oldest G residual tokens meet the pool. */
static void flush_unit(orc_cache *h, orc_unit *u)
{
    const int d = h->d, G = h->G, P = h->P, ng = d / 32;
    const int ncand = u->pool_n + G;
    orc_cand *cand = (orc_cand *)malloc(sizeof(orc_cand) * ncand);
    for (int i = 0; i < u->pool_n; ++i) {
        cand[i].norm = u->pool_norm[i];
        cand[i].idx = u->pool_idx[i];
        cand[i].from_pool = 1;
        cand[i].k = u->pool_k + (size_t)i * d;
        cand[i].v = u->pool_v + (size_t)i * d;
    }
    for (int i = 0; i < G; ++i) {
        orc_cand *c = &cand[u->pool_n + i];
        c->k = u->tail_k + (size_t)i * d;
        c->v = u->tail_v + (size_t)i * d;
        c->idx = u->tail_idx[i];
        c->from_pool = 0;
        c->norm = orc_norm(c->k, d);
    }
    int keep = ncand < P ? ncand : P;
    if (h->pct >= 0) {
        /* R14: scores over the outlier channels for every candidate (the
         * channels depend on this flush's candidates, so old pool tokens are
         * scored again); the smallest ceil(p * ncand) are the outliers. */
        int *oc = (int *)malloc(sizeof(int) * h->n_oc);
        outlier_channels(cand, ncand, d, h->n_oc, oc);
        for (int t = 0; t < ncand; ++t)
            cand[t].norm = outlier_channel_norm(cand[t].k, oc, h->n_oc);
        free(oc);
        const int m = (int)(((long long)h->pct * ncand + 9999) / 10000);
        if (m < keep)
            keep = m;
    }
    /* R4: order by (norm, index); the first `keep` stay in the pool. */
    qsort(cand, ncand, sizeof(orc_cand), cand_cmp_norm);
    int c = ncand - keep;
    /* R5: the rest, in token order, become the new block. */
    qsort(cand + keep, c, sizeof(orc_cand), cand_cmp_idx);
    /* R11: under the cold-pool policy the displaced pool tokens leave the
     * block for the cold pool; the group's tokens keep their order. */
    orc_cand *ev = NULL;
    int nev = 0;
    if (h->C >= 0) {
        ev = (orc_cand *)malloc(sizeof(orc_cand) * (c + 1));
        int nblk = 0;
        for (int t = 0; t < c; ++t) {
            const orc_cand x = cand[keep + t];
            if (x.from_pool)
                ev[nev++] = x;
            else
                cand[keep + nblk++] = x;
        }
        c = nblk;
    }

    if (u->nb == u->nb_cap) {
        u->nb_cap = u->nb_cap ? 2 * u->nb_cap : 16;
        u->blk = (orc_block *)realloc(u->blk, sizeof(orc_block) * u->nb_cap);
    }
    orc_block *b = &u->blk[u->nb++];
    b->c = c;
    b->idx = (int32_t *)malloc(sizeof(int32_t) * (c + 1));
    b->kcode = (uint8_t *)calloc((size_t)c * d + 1, 1);
    b->vcode = (uint8_t *)calloc((size_t)c * d + 1, 1);
    b->ks = (uint16_t *)calloc(d, 2);
    b->kz = (uint16_t *)calloc(d, 2);
    b->vs = (uint16_t *)calloc((size_t)c * ng + 1, 2);
    b->vz = (uint16_t *)calloc((size_t)c * ng + 1, 2);
    uint16_t *bk = (uint16_t *)malloc((size_t)(c + 1) * d * 2);
    uint16_t *bv = (uint16_t *)malloc((size_t)(c + 1) * d * 2);
    for (int t = 0; t < c; ++t) {
        b->idx[t] = cand[keep + t].idx;
        memcpy(bk + (size_t)t * d, cand[keep + t].k, (size_t)d * 2);
        memcpy(bv + (size_t)t * d, cand[keep + t].v, (size_t)d * 2);
    }
    /* R6/R7: keys per channel over the block's tokens ... */
    for (int ch = 0; ch < d; ++ch)
        orc_quant_group(bk + ch, c, d, &b->ks[ch], &b->kz[ch], b->kcode + ch, d);
    /* ... values per token per 32 channels. */
    for (int t = 0; t < c; ++t)
        for (int g = 0; g < ng; ++g)
            orc_quant_group(bv + (size_t)t * d + 32 * g, 32, 1,
                            &b->vs[(size_t)t * ng + g], &b->vz[(size_t)t * ng + g],
                            b->vcode + (size_t)t * d + 32 * g, 1);

    /* new pool: the first `keep` candidates (copy out before overwriting) */
    uint16_t *nk = (uint16_t *)malloc((size_t)(keep + 1) * d * 2);
    uint16_t *nv = (uint16_t *)malloc((size_t)(keep + 1) * d * 2);
    int32_t *ni = (int32_t *)malloc(sizeof(int32_t) * (keep + 1));
    float *nn = (float *)malloc(sizeof(float) * (keep + 1));
    for (int i = 0; i < keep; ++i) {
        memcpy(nk + (size_t)i * d, cand[i].k, (size_t)d * 2);
        memcpy(nv + (size_t)i * d, cand[i].v, (size_t)d * 2);
        ni[i] = cand[i].idx;
        nn[i] = cand[i].norm;
    }
    /* the displaced tokens' rows still live in the old pool arrays */
    if (ev)
        cold_push(h, u, ev, nev);
    memcpy(u->pool_k, nk, (size_t)keep * d * 2);
    memcpy(u->pool_v, nv, (size_t)keep * d * 2);
    memcpy(u->pool_idx, ni, sizeof(int32_t) * keep);
    memcpy(u->pool_norm, nn, sizeof(float) * keep);
    u->pool_n = keep;

    /* drop the group from the residual list */
    u->tail_n -= G;
    memmove(u->tail_idx, u->tail_idx + G, sizeof(int32_t) * u->tail_n);
    memmove(u->tail_k, u->tail_k + (size_t)G * d, (size_t)u->tail_n * d * 2);
    memmove(u->tail_v, u->tail_v + (size_t)G * d, (size_t)u->tail_n * d * 2);

    free(nk); free(nv); free(ni); free(nn);
    free(bk); free(bv);
    free(ev);
    free(cand);
}

/* Append one token to unit u (R1): store it fp16, flush when G+R wait. */
static void append_unit(orc_cache *h, orc_unit *u, long long t,
                        const uint16_t *k, const uint16_t *v)
{
    const int d = h->d;
    u->tail_idx[u->tail_n] = (int32_t)t;
    memcpy(u->tail_k + (size_t)u->tail_n * d, k, (size_t)d * 2);
    memcpy(u->tail_v + (size_t)u->tail_n * d, v, (size_t)d * 2);
    u->tail_n += 1;
    if (u->tail_n >= h->G + h->R)
        flush_unit(h, u);
}

/* k, v: fp16 bits [B][Hkv][d]. */
int orc_append(void *hp, const uint16_t *k, const uint16_t *v)
{
    orc_cache *h = (orc_cache *)hp;
    const int U = h->B * h->Hkv;
    for (int b = 0; b < h->B; ++b)     /* R13: every sequence holds a token */
        if (h->T > 0 && h->Tb[b] == 0)
            return -2;
    for (int i = 0; i < U; ++i)
        append_unit(h, &h->u[i], h->Tb[i / h->Hkv], k + (size_t)i * h->d, v + (size_t)i * h->d);
    for (int b = 0; b < h->B; ++b)
        h->Tb[b] += 1;
    h->T += 1;
    return 0;
}

/* R2. K, V: fp16 bits [B][Hkv][L][d]; only on an empty cache. */
int orc_prefill(void *hp, const uint16_t *K, const uint16_t *V, int L)
{
    orc_cache *h = (orc_cache *)hp;
    if (h->T != 0 || L < 0)
        return -2;
    const int U = h->B * h->Hkv, d = h->d;
    for (int i = 0; i < U; ++i)
        for (int t = 0; t < L; ++t)
            append_unit(h, &h->u[i], t, K + ((size_t)i * L + t) * d,
                        V + ((size_t)i * L + t) * d);
    h->T = L;
    for (int b = 0; b < h->B; ++b)
        h->Tb[b] = L;
    return 0;
}

/* R10. K, V: fp16 bits [B][Hkv][Lmax][d]; sequence b takes its first
 * lens[b] tokens (0 <= lens[b] <= Lmax); only on an empty cache. */
int orc_prefill_lens(void *hp, const uint16_t *K, const uint16_t *V, const int32_t *lens, int Lmax)
{
    orc_cache *h = (orc_cache *)hp;
    if (h->T != 0 || Lmax < 0)
        return -2;
    for (int b = 0; b < h->B; ++b)
        if (lens[b] < 0 || lens[b] > Lmax)
            return -1;
    const int U = h->B * h->Hkv, d = h->d;
    long long longest = 0;
    for (int i = 0; i < U; ++i) {
        const int L = lens[i / h->Hkv];
        for (int t = 0; t < L; ++t)
            append_unit(h, &h->u[i], t, K + ((size_t)i * Lmax + t) * d,
                        V + ((size_t)i * Lmax + t) * d);
    }
    for (int b = 0; b < h->B; ++b) {
        h->Tb[b] = lens[b];
        longest = lens[b] > longest ? lens[b] : longest;
    }
    h->T = longest;
    return 0;
}

/* R13: release sequence b: its units drop every token and block. */
static void clear_unit(orc_unit *u)
{
    for (int j = 0; j < u->nb; ++j) {
        orc_block *b = &u->blk[j];
        free(b->idx); free(b->kcode); free(b->ks); free(b->kz);
        free(b->vcode); free(b->vs); free(b->vz);
    }
    u->nb = 0;
    u->tail_n = 0;
    u->pool_n = 0;
    u->cold_n = 0;
}

int orc_release_seq(void *hp, int b)
{
    orc_cache *h = (orc_cache *)hp;
    if (b < 0 || b >= h->B)
        return -1;
    for (int x = 0; x < h->Hkv; ++x)
        clear_unit(&h->u[b * h->Hkv + x]);
    h->Tb[b] = 0;
    return 0;
}

/* R13: fill the empty sequence b with a prompt of L tokens.
 * K, V: fp16 bits [Hkv][L][d]. */
int orc_prefill_seq(void *hp, int b, const uint16_t *K, const uint16_t *V, int L)
{
    orc_cache *h = (orc_cache *)hp;
    if (b < 0 || b >= h->B || L < 1)
        return -1;
    if (h->Tb[b] != 0)
        return -2;
    const int d = h->d;
    for (int x = 0; x < h->Hkv; ++x)
        for (int t = 0; t < L; ++t)
            append_unit(h, &h->u[b * h->Hkv + x], t, K + ((size_t)x * L + t) * d, V + ((size_t)x * L + t) * d);
    h->Tb[b] = L;
    if (L > h->T)
        h->T = L;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Decode attention for one query head (R8, R9), in double:                  */
/* scores against every quantized, residual and pool key; one softmax over   */
/* the concatenation; the weights times the matching (dequantized) values.   */
/* ------------------------------------------------------------------------ */

/* use_block: NULL attends every block; else block j is attended iff use_block[j]. */
static int decode_head_blocks(orc_cache *h, int b, int hq, const uint16_t *qv, const char *use_block,
                              double *out)
{
    if (b < 0 || b >= h->B || hq < 0 || hq >= h->Hq || h->Tb[b] < 1)
        return -2;
    const int d = h->d, ng = d / 32;
    const orc_unit *u = &h->u[b * h->Hkv + hq / (h->Hq / h->Hkv)];
    const double sigma = 1.0 / sqrt((double)d);
    const long long n = h->Tb[b];
    double *score = (double *)malloc(sizeof(double) * n);
    double *q = (double *)malloc(sizeof(double) * d);
    for (int c = 0; c < d; ++c)
        q[c] = orc_h2f(qv[c]);

    /* scores, segment by segment: quantized blocks, residual, pool */
    long long m = 0;
    for (int j = 0; j < u->nb; ++j) {
        const orc_block *bl = &u->blk[j];
        if (use_block && !use_block[j])
            continue;
        for (int t = 0; t < bl->c; ++t) {
            double acc = 0.0;
            for (int c = 0; c < d; ++c) {
                double kh = bl->kcode[(size_t)t * d + c] * (double)orc_h2f(bl->ks[c]) +
                            (double)orc_h2f(bl->kz[c]);
                acc += q[c] * kh;
            }
            score[m++] = sigma * acc;
        }
    }
    for (int t = 0; t < u->tail_n; ++t) {
        double acc = 0.0;
        for (int c = 0; c < d; ++c)
            acc += q[c] * orc_h2f(u->tail_k[(size_t)t * d + c]);
        score[m++] = sigma * acc;
    }
    for (int t = 0; t < u->pool_n; ++t) {
        double acc = 0.0;
        for (int c = 0; c < d; ++c)
            acc += q[c] * orc_h2f(u->pool_k[(size_t)t * d + c]);
        score[m++] = sigma * acc;
    }
    for (int t = 0; t < u->cold_n; ++t) {       /* R11 */
        double acc = 0.0;
        for (int c = 0; c < d; ++c)
            acc += q[c] * orc_h2f(u->cold_k[(size_t)t * d + c]);
        score[m++] = sigma * acc;
    }

    /* softmax over the concatenated scores */
    double mx = -INFINITY;
    for (long long i = 0; i < m; ++i)
        if (score[i] > mx)
            mx = score[i];
    double sum = 0.0;
    for (long long i = 0; i < m; ++i) {
        score[i] = exp(score[i] - mx);
        sum += score[i];
    }

    /* weights times values, same segment order */
    for (int c = 0; c < d; ++c)
        out[c] = 0.0;
    m = 0;
    for (int j = 0; j < u->nb; ++j) {
        const orc_block *bl = &u->blk[j];
        if (use_block && !use_block[j])
            continue;
        for (int t = 0; t < bl->c; ++t) {
            double p = score[m++];
            for (int c = 0; c < d; ++c) {
                size_t sg = (size_t)t * ng + c / 32;
                double vh = bl->vcode[(size_t)t * d + c] * (double)orc_h2f(bl->vs[sg]) +
                            (double)orc_h2f(bl->vz[sg]);
                out[c] += p * vh;
            }
        }
    }
    for (int t = 0; t < u->tail_n; ++t) {
        double p = score[m++];
        for (int c = 0; c < d; ++c)
            out[c] += p * orc_h2f(u->tail_v[(size_t)t * d + c]);
    }
    for (int t = 0; t < u->pool_n; ++t) {
        double p = score[m++];
        for (int c = 0; c < d; ++c)
            out[c] += p * orc_h2f(u->pool_v[(size_t)t * d + c]);
    }
    for (int t = 0; t < u->cold_n; ++t) {
        double p = score[m++];
        for (int c = 0; c < d; ++c)
            out[c] += p * orc_h2f(u->cold_v[(size_t)t * d + c]);
    }
    for (int c = 0; c < d; ++c)
        out[c] /= sum;
    free(score);
    free(q);
    return 0;
}

int orc_decode_head(void *hp, int b, int hq, const uint16_t *qv, double *out)
{
    return decode_head_blocks((orc_cache *)hp, b, hq, qv, NULL, out);
}

/* R12: the score bound of block bl for the fp16 query qv [d], in fp32. */
static float block_bound(const orc_block *bl, const uint16_t *qv, int d)
{
    float beta = 0.0f;
    for (int c = 0; c < d; ++c) {
        const float q = orc_h2f(qv[c]);
        const float s = orc_h2f(bl->ks[c]);
        const float z = orc_h2f(bl->kz[c]);
        const float three_s = 3.0f * s;
        const float top = z + three_s;       /* the largest dequantized value */
        const float lo = q * z, hi = q * top;
        beta = beta + (hi > lo ? hi : lo);
    }
    return beta;
}

typedef struct {
    float bound;
    int j;
} orc_rank;

static int rank_cmp(const void *a, const void *b)
{
    const orc_rank *x = (const orc_rank *)a, *y = (const orc_rank *)b;
    if (x->bound > y->bound) return -1;
    if (x->bound < y->bound) return 1;
    return (x->j > y->j) - (x->j < y->j);
}

static int cmp_int(const void *a, const void *b)
{
    const int x = *(const int *)a, y = *(const int *)b;
    return (x > y) - (x < y);
}

/* R12: the blocks that a top-K decode of sequence b attends for kv head hk.
 * qb: fp16 bits [Hq][d] (sequence b's queries). Writes the selected block
 * indices in ascending order to sel and returns how many there are
 * (min(K, non-empty blocks)). bounds, if not NULL, receives [nb] block
 * bounds (-inf for an empty block). */
int orc_topk_select(void *hp, int b, int hk, const uint16_t *qb, int K, int32_t *sel, float *bounds)
{
    orc_cache *h = (orc_cache *)hp;
    const int g = h->Hq / h->Hkv, d = h->d;
    const orc_unit *u = &h->u[b * h->Hkv + hk];
    orc_rank *r = (orc_rank *)malloc(sizeof(orc_rank) * (u->nb + 1));
    int n = 0;
    for (int j = 0; j < u->nb; ++j) {
        const orc_block *bl = &u->blk[j];
        float best = -INFINITY;
        if (bl->c > 0)
            for (int x = 0; x < g; ++x) {
                const float bx = block_bound(bl, qb + (size_t)(hk * g + x) * d, d);
                if (bx > best)
                    best = bx;
            }
        if (bounds)
            bounds[j] = best;
        if (bl->c > 0) {
            r[n].bound = best;
            r[n].j = j;
            ++n;
        }
    }
    qsort(r, n, sizeof(orc_rank), rank_cmp);
    const int m = K < n ? (K < 0 ? 0 : K) : n;
    int *js = (int *)malloc(sizeof(int) * (m + 1));
    for (int i = 0; i < m; ++i)
        js[i] = r[i].j;
    qsort(js, m, sizeof(int), cmp_int);
    for (int i = 0; i < m; ++i)
        sel[i] = js[i];
    free(js);
    free(r);
    return m;
}

/* R12. q: fp16 bits [B][Hq][d]; out: double [B][Hq][d]. */
int orc_decode_topk(void *hp, const uint16_t *q, int K, double *out)
{
    orc_cache *h = (orc_cache *)hp;
    const int g = h->Hq / h->Hkv, d = h->d;
    for (int b = 0; b < h->B; ++b)
        if (h->Tb[b] < 1)
            return -2;
    for (int b = 0; b < h->B; ++b)
        for (int hk = 0; hk < h->Hkv; ++hk) {
            const orc_unit *u = &h->u[b * h->Hkv + hk];
            int32_t *sel = (int32_t *)malloc(sizeof(int32_t) * (u->nb + 1));
            char *use = (char *)calloc(u->nb + 1, 1);
            const int m = orc_topk_select(h, b, hk, q + (size_t)b * h->Hq * d, K, sel, NULL);
            for (int i = 0; i < m; ++i)
                use[sel[i]] = 1;
            for (int x = 0; x < g; ++x) {
                const int hq = hk * g + x;
                const size_t o = ((size_t)b * h->Hq + hq) * d;
                decode_head_blocks(h, b, hq, q + o, use, out + o);
            }
            free(use);
            free(sel);
        }
    return 0;
}

/* q: fp16 bits [B][Hq][d]; out: double [B][Hq][d]. */
int orc_decode(void *hp, const uint16_t *q, double *out)
{
    orc_cache *h = (orc_cache *)hp;
    for (int b = 0; b < h->B; ++b)
        if (h->Tb[b] < 1)
            return -2;
    for (int b = 0; b < h->B; ++b)
        for (int hq = 0; hq < h->Hq; ++hq) {
            size_t o = ((size_t)b * h->Hq + hq) * h->d;
            orc_decode_head(h, b, hq, q + o, out + o);
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Introspection and canonical export.                                       */
/* ------------------------------------------------------------------------ */

void orc_counts(void *hp, int u, long long *T, int *nf, int *tail, int *npool)
{
    orc_cache *h = (orc_cache *)hp;
    *T = h->Tb[u / h->Hkv];
    *nf = h->u[u].nb;
    *tail = h->u[u].tail_n;
    *npool = h->u[u].pool_n;
}

int orc_block_count(void *hp, int u, int j)
{
    orc_cache *h = (orc_cache *)hp;
    return (j >= 0 && j < h->u[u].nb) ? h->u[u].blk[j].c : -1;
}

/*
 * Canonical export of unit u. Any pointer may be NULL (skipped). Shapes, with
 * nf blocks, residual length nt and d channels:
 *   bcount [nf] int32             block token counts
 *   bidx   [nf][G] int32          token indices ascending, -1 padded
 *   kcode  [nf][G][d/4] uint8     packed: code of channel c at bits 2(c%4)
 *   ks, kz [nf][d] uint16         of byte c/4; padding rows are zero
 *   vcode  [nf][G][d/4] uint8     same packing
 *   vs, vz [nf][G][d/32] uint16   zero padded
 *   tidx   [nt] int32, tk, tv [nt][d] uint16   residual tokens, oldest first
 *   pidx   [P] int32 ascending (-1 pad), pnorm [P] fp32 bits,
 *   pk, pv [P][d] uint16          pool tokens in ascending index order
 */
int orc_export_unit(void *hp, int ui, int32_t *bcount, int32_t *bidx, uint8_t *kcode,
                    uint16_t *ks, uint16_t *kz, uint8_t *vcode, uint16_t *vs, uint16_t *vz,
                    int32_t *tidx, uint16_t *tk, uint16_t *tv, int32_t *pidx,
                    uint32_t *pnorm, uint16_t *pk, uint16_t *pv)
{
    orc_cache *h = (orc_cache *)hp;
    const orc_unit *u = &h->u[ui];
    const int d = h->d, G = h->G, P = h->P, ng = d / 32, rb = d / 4;
    for (int j = 0; j < u->nb; ++j) {
        const orc_block *bl = &u->blk[j];
        if (bcount) bcount[j] = bl->c;
        for (int t = 0; t < G; ++t) {
            int valid = t < bl->c;
            if (bidx) bidx[(size_t)j * G + t] = valid ? bl->idx[t] : -1;
            for (int by = 0; by < rb; ++by) {
                uint8_t kb = 0, vb = 0;
                if (valid)
                    for (int e = 0; e < 4; ++e) {
                        kb |= (uint8_t)(bl->kcode[(size_t)t * d + 4 * by + e] << (2 * e));
                        vb |= (uint8_t)(bl->vcode[(size_t)t * d + 4 * by + e] << (2 * e));
                    }
                if (kcode) kcode[((size_t)j * G + t) * rb + by] = kb;
                if (vcode) vcode[((size_t)j * G + t) * rb + by] = vb;
            }
            for (int g = 0; g < ng; ++g) {
                size_t o = ((size_t)j * G + t) * ng + g;
                if (vs) vs[o] = valid ? bl->vs[(size_t)t * ng + g] : 0;
                if (vz) vz[o] = valid ? bl->vz[(size_t)t * ng + g] : 0;
            }
        }
        for (int c = 0; c < d; ++c) {
            if (ks) ks[(size_t)j * d + c] = bl->ks[c];
            if (kz) kz[(size_t)j * d + c] = bl->kz[c];
        }
    }
    for (int t = 0; t < u->tail_n; ++t) {
        if (tidx) tidx[t] = u->tail_idx[t];
        if (tk) memcpy(tk + (size_t)t * d, u->tail_k + (size_t)t * d, (size_t)d * 2);
        if (tv) memcpy(tv + (size_t)t * d, u->tail_v + (size_t)t * d, (size_t)d * 2);
    }
    /* pool in ascending token order */
    int *ord = (int *)malloc(sizeof(int) * (P + 1));
    for (int i = 0; i < u->pool_n; ++i)
        ord[i] = i;
    for (int i = 1; i < u->pool_n; ++i)          /* insertion sort by index */
        for (int j = i; j > 0 && u->pool_idx[ord[j - 1]] > u->pool_idx[ord[j]]; --j) {
            int tmp = ord[j]; ord[j] = ord[j - 1]; ord[j - 1] = tmp;
        }
    for (int i = 0; i < P; ++i) {
        int valid = i < u->pool_n;
        int s = valid ? ord[i] : 0;
        if (pidx) pidx[i] = valid ? u->pool_idx[s] : -1;
        if (pnorm) {
            uint32_t nb = 0;
            if (valid) memcpy(&nb, &u->pool_norm[s], 4);
            pnorm[i] = nb;
        }
        if (pk) {
            if (valid) memcpy(pk + (size_t)i * d, u->pool_k + (size_t)s * d, (size_t)d * 2);
            else memset(pk + (size_t)i * d, 0, (size_t)d * 2);
        }
        if (pv) {
            if (valid) memcpy(pv + (size_t)i * d, u->pool_v + (size_t)s * d, (size_t)d * 2);
            else memset(pv + (size_t)i * d, 0, (size_t)d * 2);
        }
    }
    free(ord);
    return 0;
}

/* R11: the cold pool of unit u, oldest first. Any pointer may be NULL.
 * cidx [C] int32 (-1 padded), ck, cv [C][d] fp16 bits (zero padded).
 * Returns the number of cold tokens, or -1 without the cold-pool policy. */
int orc_export_cold(void *hp, int ui, int32_t *cidx, uint16_t *ck, uint16_t *cv)
{
    orc_cache *h = (orc_cache *)hp;
    if (h->C < 0)
        return -1;
    const orc_unit *u = &h->u[ui];
    const int d = h->d;
    for (int i = 0; i < h->C; ++i) {
        const int valid = i < u->cold_n;
        if (cidx) cidx[i] = valid ? u->cold_idx[i] : -1;
        if (ck) {
            if (valid) memcpy(ck + (size_t)i * d, u->cold_k + (size_t)i * d, (size_t)d * 2);
            else memset(ck + (size_t)i * d, 0, (size_t)d * 2);
        }
        if (cv) {
            if (valid) memcpy(cv + (size_t)i * d, u->cold_v + (size_t)i * d, (size_t)d * 2);
            else memset(cv + (size_t)i * d, 0, (size_t)d * 2);
        }
    }
    return u->cold_n;
}
