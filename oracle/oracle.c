/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the compressed-KV decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file: only the tests, the package's smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA library; where both sides need the same definition (the binary16
 * format, the Philox4x32-10 generator, the packed KIVI block layout) each side
 * restates it from its published definition or from the layout specification.
 *
 * Every input arrives as the exact binary16 bit pattern the GPU sees and is
 * widened exactly to fp64; every step below is the plain definition, with no
 * blocking, splitting or reordering beyond what the definition states.
 *
 * Sources (web pages; cited by title and section):
 *   [RKV]  "Rethinking KV Cache Compression: 从显存节省回到真实 serving 端到端收益"
 *          (guide to the paper), §2 "4 种 baseline 的成本结构" (KIVI G=32, R=128;
 *          StreamingLLM / H2O 64 + 448 = 512), §16 "4 种方法逐步执行" (KIVI
 *          per-channel K / per-token V with an fp16 residual; StreamingLLM sink
 *          + recent; H2O accumulated attention score and keep-set update) and
 *          §16 "局限与最终结论" (residual flush when full; H2O needs the
 *          attention probabilities that FlashAttention does not expose).
 *   [EVP]  "KV Cache 驱逐实战：什么时候该放弃打分器，直接随机扔", section
 *          "参考实现" (per-head uniform random eviction with the prompt locked:
 *          n_keep = max(1, int(n_cand * keep_ratio)), per-head gather to
 *          [n_heads, prompt_len + n_keep, head_dim], never a union over heads).
 *   [PHX]  Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
 *          1, 2, 3", SC'11 -- the Philox4x32-10 counter-based generator.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   softmax scale 1/sqrt(D); KIVI zero = group minimum, scale = binary16
 *   round-to-nearest-even of (max - min) / (2^bits - 1), code = exact
 *   round-half-even of (x - zero) / scale clamped to [0, 2^bits - 1], a
 *   degenerate group (scale 0) gets code 0; the quantised prefix length is
 *   n_q = G * floor(max(0, T - R) / G); H2O's recent window is by absolute
 *   position and heavy hitters are ranked by (score desc, position asc);
 *   random eviction keys are 64-bit Philox outputs with counter
 *   (position, kv_head, batch, epoch), smallest keys kept, ties by position.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16 <-> binary64, written from the format definition:      */
/* 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; subnormals have */
/* exponent field 0 and value fraction * 2^-24.                             */
/* ------------------------------------------------------------------------ */

ORC_API double orc_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return sign ? -v : v;
}

/* Round-to-nearest, ties-to-even conversion of a double to binary16. */
ORC_API uint16_t orc_double_to_half(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(x))
        return 0x7e00;
    if (a == 0.0)
        return sign;
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: quantum 2^-24; rounding up to 1024 lands exactly on
           the smallest normal, whose encoding is fraction 0, exponent 1. */
        double m = nearbyint(a * ldexp(1.0, 24));
        return (uint16_t)(sign | (uint16_t)m);
    }
    int E;
    frexp(a, &E);               /* a = f * 2^E, f in [0.5, 1) */
    int e = E - 1;              /* a in [2^e, 2^(e+1)) */
    double m = nearbyint(ldexp(a, 10 - e));   /* in [1024, 2048] */
    if (m == 2048.0) {
        m = 1024.0;
        e += 1;
    }
    int biased = e + 15;
    if (biased >= 31)
        return (uint16_t)(sign | 0x7c00);
    return (uint16_t)(sign | (uint16_t)(biased << 10) | (uint16_t)((int)m - 1024));
}

ORC_API void orc_half_to_double_array(long n, const uint16_t *in, double *out)
{
    for (long i = 0; i < n; ++i)
        out[i] = orc_half_to_double(in[i]);
}

ORC_API void orc_double_to_half_array(long n, const double *in, uint16_t *out)
{
    for (long i = 0; i < n; ++i)
        out[i] = orc_double_to_half(in[i]);
}

/* ------------------------------------------------------------------------ */
/* A tiny parallel-for over independent units (batch x kv-head).  The units */
/* do not interact, so threading changes no arithmetic.                     */
/* ------------------------------------------------------------------------ */

typedef void (*unit_fn)(void *ctx, long unit);

typedef struct {
    unit_fn fn;
    void *ctx;
    long n_units;
    int n_threads;
    int tid;
} par_job;

static void *par_worker(void *arg)
{
    par_job *j = (par_job *)arg;
    for (long u = j->tid; u < j->n_units; u += j->n_threads)
        j->fn(j->ctx, u);
    return NULL;
}

static void parallel_for(long n_units, int n_threads, unit_fn fn, void *ctx)
{
    if (n_threads <= 1 || n_units <= 1) {
        for (long u = 0; u < n_units; ++u)
            fn(ctx, u);
        return;
    }
    if (n_threads > n_units)
        n_threads = (int)n_units;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    par_job *jobs = (par_job *)malloc(sizeof(par_job) * (size_t)n_threads);
    for (int t = 0; t < n_threads; ++t) {
        jobs[t].fn = fn;
        jobs[t].ctx = ctx;
        jobs[t].n_units = n_units;
        jobs[t].n_threads = n_threads;
        jobs[t].tid = t;
        pthread_create(&th[t], NULL, par_worker, &jobs[t]);
    }
    for (int t = 0; t < n_threads; ++t)
        pthread_join(th[t], NULL);
    free(th);
    free(jobs);
}

/* ------------------------------------------------------------------------ */
/* Scaled dot-product attention of one query over n keys (fp64).            */
/*   logit_j = scale * sum_d q_d k_{j,d}                                    */
/*   p_j     = exp(logit_j - lse),  lse = log sum_j exp(logit_j)            */
/*   out_d   = sum_j p_j v_{j,d}                                            */
/* The maximum is subtracted before exponentiation (exact identity).        */
/* n == 0 gives out = 0 and lse = -inf (an empty softmax has no mass).      */
/* ------------------------------------------------------------------------ */

static double attend_one(const double *q, const double *K, const double *V, int n, int D,
                         double scale, double *out, double *logits_out)
{
    for (int d = 0; d < D; ++d)
        out[d] = 0.0;
    if (n <= 0)
        return -INFINITY;
    double *lg = (double *)malloc(sizeof(double) * (size_t)n);
    double mx = -INFINITY;
    for (int j = 0; j < n; ++j) {
        double s = 0.0;
        for (int d = 0; d < D; ++d)
            s += q[d] * K[(size_t)j * D + d];
        lg[j] = s * scale;
        if (lg[j] > mx)
            mx = lg[j];
    }
    double l = 0.0;
    for (int j = 0; j < n; ++j)
        l += exp(lg[j] - mx);
    double lse = mx + log(l);
    for (int j = 0; j < n; ++j) {
        double p = exp(lg[j] - lse);
        for (int d = 0; d < D; ++d)
            out[d] += p * V[(size_t)j * D + d];
    }
    if (logits_out)
        memcpy(logits_out, lg, sizeof(double) * (size_t)n);
    free(lg);
    return lse;
}

/* ------------------------------------------------------------------------ */
/* Decode attention over a slot cache with GQA head mapping.                */
/*   q [B,Hq,D] f16;  K,V [B,Hkv,C,D] f16;  n [B,Hkv] valid slots           */
/*   query head h reads kv head h / (Hq/Hkv) (contiguous grouping)          */
/*   out [B,Hq,D] f64; lse [B,Hq] f64; logits [B,Hq,C] f64 or NULL          */
/* ------------------------------------------------------------------------ */

typedef struct {
    int B, Hq, Hkv, D, C;
    const uint16_t *q, *K, *V;
    const int32_t *n;
    double scale;
    double *out, *lse, *logits;
} attend_ctx;

static void attend_unit(void *vctx, long u)
{
    attend_ctx *c = (attend_ctx *)vctx;
    int b = (int)(u / c->Hkv), hk = (int)(u % c->Hkv);
    int g = c->Hq / c->Hkv, D = c->D;
    int n = c->n[u];
    if (n > c->C)
        n = c->C;
    size_t base = (size_t)u * c->C * D;
    double *K = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * D);
    double *V = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * D);
    double *q = (double *)malloc(sizeof(double) * (size_t)D);
    for (size_t i = 0; i < (size_t)n * D; ++i) {
        K[i] = orc_half_to_double(c->K[base + i]);
        V[i] = orc_half_to_double(c->V[base + i]);
    }
    for (int j = 0; j < g; ++j) {
        int h = hk * g + j;
        size_t qo = ((size_t)b * c->Hq + h) * D;
        for (int d = 0; d < D; ++d)
            q[d] = orc_half_to_double(c->q[qo + d]);
        double *lg = c->logits ? c->logits + ((size_t)b * c->Hq + h) * c->C : NULL;
        c->lse[(size_t)b * c->Hq + h] = attend_one(q, K, V, n, D, c->scale, c->out + qo, lg);
    }
    free(K);
    free(V);
    free(q);
}

ORC_API void orc_decode_attend(int B, int Hq, int Hkv, int D, int C, const uint16_t *q,
                               const uint16_t *K, const uint16_t *V, const int32_t *n,
                               double scale, double *out, double *lse, double *logits,
                               int n_threads)
{
    attend_ctx c = {B, Hq, Hkv, D, C, q, K, V, n, scale, out, lse, logits};
    parallel_for((long)B * Hkv, n_threads, attend_unit, &c);
}

/* ------------------------------------------------------------------------ */
/* KIVI asymmetric group quantisation ([RKV] §2, §16).                      */
/*   zero  = min of the group (a binary16 value; -0 is written as +0)       */
/*   scale = RN16((max - min) / (2^bits - 1))                               */
/*   code  = clamp(round_half_even((x - zero) / scale), 0, 2^bits - 1)      */
/*   dequantised value = zero + code * scale (exact in fp64)                */
/* x - zero is exact in fp64 (both are binary16 values: at most 41          */
/* significant bits); the code is found from exact comparisons against      */
/* (c + 1/2) * scale, which are exact as well.                              */
/* ------------------------------------------------------------------------ */

static uint8_t kivi_code(double x, double zero, double scale, int bits)
{
    int cmax = (1 << bits) - 1;
    if (scale == 0.0)
        return 0;
    double diff = x - zero; /* exact, >= 0 */
    double c = floor(diff / scale);
    /* make c the exact floor of diff / scale */
    while ((c + 1.0) * scale <= diff)
        c += 1.0;
    while (c > 0.0 && c * scale > diff)
        c -= 1.0;
    double rem = diff - c * scale; /* exact: 0 <= rem < scale */
    double twice = 2.0 * rem;
    if (twice > scale)
        c += 1.0;
    else if (twice == scale && fmod(c, 2.0) != 0.0)
        c += 1.0;
    if (c > cmax)
        c = cmax;
    if (c < 0)
        c = 0;
    return (uint8_t)c;
}

/* Quantise cnt values x[0], x[stride], ... as one group. */
static void kivi_group(const uint16_t *x, long stride, int cnt, int bits, uint16_t *scale_bits,
                       uint16_t *zero_bits, uint8_t *codes, long code_stride)
{
    double mn = INFINITY, mx = -INFINITY;
    for (int i = 0; i < cnt; ++i) {
        double v = orc_half_to_double(x[i * stride]);
        if (v < mn)
            mn = v;
        if (v > mx)
            mx = v;
    }
    uint16_t zb = orc_double_to_half(mn);
    if (zb == 0x8000)
        zb = 0x0000;
    double range = mx - mn; /* exact in fp64 */
    uint16_t sb = orc_double_to_half(range / (double)((1 << bits) - 1));
    *zero_bits = zb;
    *scale_bits = sb;
    double zero = orc_half_to_double(zb), scale = orc_half_to_double(sb);
    for (int i = 0; i < cnt; ++i)
        codes[i * code_stride] = kivi_code(orc_half_to_double(x[i * stride]), zero, scale, bits);
}

/* Number of tokens held in the quantised store for a sequence of T tokens
   (the residual keeps the newest tokens in fp16 and flushes whole groups of G
   once it would exceed R + G - 1 tokens). */
ORC_API long orc_kivi_nq(long T, int G, int R)
{
    long over = T - R;
    if (over < 0)
        over = 0;
    return (long)G * (over / G);
}

/*
 * Quantise one (batch, kv-head) unit's first n_q tokens.
 *   K, V: [T, D] f16 of this unit (tokens in position order).
 *   Outputs, per group g < n_q / G (G = 32):
 *     k_scale, k_zero [n_q/G, D] bits;  k_codes [n_q, D] (one code per byte)
 *     v_scale, v_zero [n_q, D/G] bits;  v_codes [n_q, D]
 */
ORC_API void orc_kivi_quantize_unit(int D, int G, int bits, long n_q, const uint16_t *K,
                                    const uint16_t *V, uint16_t *k_scale, uint16_t *k_zero,
                                    uint8_t *k_codes, uint16_t *v_scale, uint16_t *v_zero,
                                    uint8_t *v_codes)
{
    long n_groups = n_q / G;
    for (long g = 0; g < n_groups; ++g) {
        /* K: per channel d, over the G tokens of the group */
        for (int d = 0; d < D; ++d)
            kivi_group(K + (g * G) * D + d, D, G, bits, &k_scale[g * D + d],
                       &k_zero[g * D + d], &k_codes[(g * G) * D + d], D);
    }
    int ng = D / G;
    for (long t = 0; t < n_q; ++t) {
        /* V: per token, over channel groups of G */
        for (int j = 0; j < ng; ++j)
            kivi_group(V + t * D + j * G, 1, G, bits, &v_scale[t * ng + j], &v_zero[t * ng + j],
                       &v_codes[t * D + j * G], 1);
    }
}

/*
 * Pack one group of codes into the documented block layout (restated here
 * from the layout specification; the GPU library restates it separately).
 *
 * K block (bytes): [G tokens x WK u32 words][D f16 scales][D f16 zeros],
 *   WK = D*bits/32; in token t's word w, field i (bits [bits*i, bits*(i+1)))
 *   holds channel d = (32/bits)*w + i.
 * V block (bytes): [G/2 token pairs x 2*WK u32 words][G tokens x (D/G scales,
 *   D/G zeros) f16].  Pair i holds tokens 2i (low 16 bits of every word) and
 *   2i+1 (high 16 bits).  Word index ((r + 2i) mod 8)*W + k (r in [0,8),
 *   k in [0,W), W = D*bits/128); field j (bits [bits*j, bits*(j+1)) of each
 *   16-bit half) holds channel d = 16*(k*(8/bits) + j/2) + 8*(j%2) + r.  Then the V scales
 *   as D/G rows of G values (row j: channel group j of tokens 0..G-1), then the
 *   V zeros in the same order.
 */
ORC_API void orc_kivi_pack_group(int D, int G, int bits, const uint8_t *k_codes,
                                 const uint16_t *k_scale, const uint16_t *k_zero,
                                 const uint8_t *v_codes, const uint16_t *v_scale,
                                 const uint16_t *v_zero, uint8_t *k_block, uint8_t *v_block)
{
    int WK = D * bits / 32;
    int per_word = 32 / bits;
    uint32_t *kw = (uint32_t *)k_block;
    for (int t = 0; t < G; ++t)
        for (int w = 0; w < WK; ++w) {
            uint32_t word = 0;
            for (int i = 0; i < per_word; ++i)
                word |= (uint32_t)k_codes[t * D + per_word * w + i] << (bits * i);
            kw[t * WK + w] = word;
        }
    uint16_t *ks = (uint16_t *)(k_block + (size_t)G * WK * 4);
    memcpy(ks, k_scale, sizeof(uint16_t) * (size_t)D);
    memcpy(ks + D, k_zero, sizeof(uint16_t) * (size_t)D);

    int W = D * bits / 128;
    int per_half = 16 / bits;
    int mt_per_word = 8 / bits;
    uint32_t *vw = (uint32_t *)v_block;
    for (int i = 0; i < G / 2; ++i)
        for (int r = 0; r < 8; ++r)
            for (int k = 0; k < W; ++k) {
                uint32_t word = 0;
                for (int j = 0; j < per_half; ++j) {
                    int d = 16 * (k * mt_per_word + j / 2) + 8 * (j % 2) + r;
                    word |= (uint32_t)v_codes[(2 * i) * D + d] << (bits * j);
                    word |= (uint32_t)v_codes[(2 * i + 1) * D + d] << (16 + bits * j);
                }
                vw[(size_t)i * (2 * WK) + ((r + 2 * i) % 8) * W + k] = word;
            }
    uint16_t *vs = (uint16_t *)(v_block + (size_t)(G / 2) * (2 * WK) * 4);
    int ng = D / G;
    for (int j = 0; j < ng; ++j)
        for (int t = 0; t < G; ++t) {
            vs[j * G + t] = v_scale[t * ng + j];
            vs[ng * G + j * G + t] = v_zero[t * ng + j];
        }
}

/*
 * KIVI decode attention for one unit: full attention of each of the g query
 * heads over the dequantised quantised tokens [0, n_q) followed by the fp16
 * residual tokens [n_q, T).  Dequantisation is exact in fp64.
 *   q [g, D] f16;  K, V [T, D] f16 (the unit's raw tokens, used only for the
 *   residual);  quantised parts as produced by orc_kivi_quantize_unit.
 */
ORC_API void orc_kivi_attend_unit(int g, int D, int G, long T, long n_q, const uint16_t *q,
                                  const uint16_t *K, const uint16_t *V,
                                  const uint16_t *k_scale, const uint16_t *k_zero,
                                  const uint8_t *k_codes, const uint16_t *v_scale,
                                  const uint16_t *v_zero, const uint8_t *v_codes, double scale,
                                  double *out, double *lse)
{
    double *Kd = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * D);
    double *Vd = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * D);
    int ng = D / G;
    for (long t = 0; t < T; ++t)
        for (int d = 0; d < D; ++d) {
            size_t i = (size_t)t * D + d;
            if (t < n_q) {
                long grp = t / G;
                Kd[i] = orc_half_to_double(k_zero[grp * D + d]) +
                        (double)k_codes[i] * orc_half_to_double(k_scale[grp * D + d]);
                Vd[i] = orc_half_to_double(v_zero[t * ng + d / G]) +
                        (double)v_codes[i] * orc_half_to_double(v_scale[t * ng + d / G]);
            } else {
                Kd[i] = orc_half_to_double(K[i]);
                Vd[i] = orc_half_to_double(V[i]);
            }
        }
    double *qd = (double *)malloc(sizeof(double) * (size_t)D);
    for (int j = 0; j < g; ++j) {
        for (int d = 0; d < D; ++d)
            qd[d] = orc_half_to_double(q[(size_t)j * D + d]);
        lse[j] = attend_one(qd, Kd, Vd, (int)T, D, scale, out + (size_t)j * D, NULL);
    }
    free(qd);
    free(Kd);
    free(Vd);
}

/* ------------------------------------------------------------------------ */
/* H2O heavy-hitter scores ([RKV] §2, §16).                                 */
/* ------------------------------------------------------------------------ */

/*
 * Prefill scores over a causal prompt of L tokens, one (batch, kv-head)
 * unit:  score[j] = sum over the g query heads of the unit, and over rows
 * i >= j, of softmax_i(scale * q_i . k_.)_j.
 *   Qp [g, L, D] f16 (this unit's query heads);  Kp [L, D] f16.
 */
typedef struct {
    int Hq, Hkv, D, L;
    long kp_cap, score_cap;
    const uint16_t *Qp, *Kp;
    double scale;
    double *scores;
} prefill_ctx;

static void prefill_unit(void *vctx, long u)
{
    prefill_ctx *c = (prefill_ctx *)vctx;
    int b = (int)(u / c->Hkv), hk = (int)(u % c->Hkv);
    int g = c->Hq / c->Hkv, D = c->D, L = c->L;
    double *K = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * D);
    const uint16_t *kp = c->Kp + (size_t)u * c->kp_cap * D;
    for (size_t i = 0; i < (size_t)L * D; ++i)
        K[i] = orc_half_to_double(kp[i]);
    double *score = c->scores + (size_t)u * c->score_cap;
    for (int j = 0; j < L; ++j)
        score[j] = 0.0;
    double *q = (double *)malloc(sizeof(double) * (size_t)D);
    double *lg = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    for (int hh = 0; hh < g; ++hh) {
        int h = hk * g + hh;
        const uint16_t *qp = c->Qp + ((size_t)b * c->Hq + h) * (size_t)L * D;
        for (int i = 0; i < L; ++i) {
            for (int d = 0; d < D; ++d)
                q[d] = orc_half_to_double(qp[(size_t)i * D + d]);
            double mx = -INFINITY;
            for (int j = 0; j <= i; ++j) {
                double s = 0.0;
                for (int d = 0; d < D; ++d)
                    s += q[d] * K[(size_t)j * D + d];
                lg[j] = s * c->scale;
                if (lg[j] > mx)
                    mx = lg[j];
            }
            double l = 0.0;
            for (int j = 0; j <= i; ++j)
                l += exp(lg[j] - mx);
            double lse = mx + log(l);
            for (int j = 0; j <= i; ++j)
                score[j] += exp(lg[j] - lse);
        }
    }
    free(K);
    free(q);
    free(lg);
}

/* Qp [B,Hq,L,D]; Kp [B,Hkv,kp_cap,D] (prompt in rows [0,L)); scores
   [B,Hkv,score_cap] f64 (entries [0,L) written).  Units may be restricted to
   a list (unit_list, n_list) so large shapes can be sampled. */
ORC_API void orc_h2o_prefill_scores(int B, int Hq, int Hkv, int D, int L, long kp_cap,
                                    long score_cap, const uint16_t *Qp, const uint16_t *Kp,
                                    double scale, double *scores, int n_threads)
{
    prefill_ctx c = {Hq, Hkv, D, L, kp_cap, score_cap, Qp, Kp, scale, scores};
    parallel_for((long)B * Hkv, n_threads, prefill_unit, &c);
}

/*
 * Decode accumulation: for every valid slot j of unit (b, hk), with
 *   p[j] = sum over the unit's query heads h of exp(logit[h][j] - lse[h]),
 * decay == 0 (plain H2O, "Rethinking KV Cache Compression" §16):
 *   score[j] += p[j];
 * 0 < decay < 1 (the incremental activity score A_i <- lambda A_i +
 * (1 - lambda) attn_i of "Practical Online KV Cache Compaction for LLM
 * Agents", §4.1, with attn_i summed over the KV head's query group):
 *   score[j] = decay * score[j] + (1 - decay) * p[j].
 * logits [B,Hq,C] f64 and lse [B,Hq] are the oracle's own attention outputs.
 */
ORC_API void orc_h2o_accumulate(int B, int Hq, int Hkv, int C, const int32_t *n,
                                const double *logits, const double *lse, double decay,
                                double *scores)
{
    int g = Hq / Hkv;
    for (int b = 0; b < B; ++b)
        for (int hk = 0; hk < Hkv; ++hk) {
            int nn = n[b * Hkv + hk];
            double *sc = scores + ((size_t)b * Hkv + hk) * C;
            for (int j = 0; j < nn; ++j) {
                double p = 0.0;
                for (int hh = 0; hh < g; ++hh) {
                    int h = hk * g + hh;
                    p += exp(logits[((size_t)b * Hq + h) * C + j] - lse[(size_t)b * Hq + h]);
                }
                if (decay == 0.0)
                    sc[j] += p;
                else
                    sc[j] = decay * sc[j] + (1.0 - decay) * p;
            }
        }
}

/*
 * H2O keep-set of one unit: recent = slots with pos >= T - n_recent; among
 * the other slots keep the n_heavy largest by (score desc, pos asc).
 *   keep[j] = 1 for kept slots.  Returns the number kept.  *margin receives
 *   the relative gap between the last kept and first dropped heavy candidate
 *   ((a - b) / max(|a|, |b|), +inf when nothing is dropped).
 */
ORC_API int orc_h2o_keep(int n, const int32_t *pos, const double *score, long T, int n_heavy,
                         int n_recent, uint8_t *keep, double *margin)
{
    int *cand = (int *)malloc(sizeof(int) * (size_t)(n > 0 ? n : 1));
    int nc = 0, kept = 0;
    for (int j = 0; j < n; ++j) {
        if ((long)pos[j] >= T - n_recent) {
            keep[j] = 1;
            ++kept;
        } else {
            keep[j] = 0;
            cand[nc++] = j;
        }
    }
    /* selection by repeated maximum: plain O(n * n_heavy), obviously correct */
    int take = nc < n_heavy ? nc : n_heavy;
    double last = INFINITY;
    for (int t = 0; t < take; ++t) {
        int best = -1;
        for (int i = 0; i < nc; ++i) {
            int j = cand[i];
            if (keep[j])
                continue;
            if (best < 0 || score[j] > score[best] ||
                (score[j] == score[best] && pos[j] < pos[best]))
                best = j;
        }
        keep[best] = 1;
        last = score[best];
        ++kept;
    }
    double first_dropped = -INFINITY;
    int any_dropped = 0;
    for (int i = 0; i < nc; ++i) {
        int j = cand[i];
        if (!keep[j]) {
            if (!any_dropped || score[j] > first_dropped)
                first_dropped = score[j];
            any_dropped = 1;
        }
    }
    if (margin) {
        if (!any_dropped || take == 0)
            *margin = INFINITY;
        else {
            double den = fmax(fabs(last), fabs(first_dropped));
            *margin = den > 0 ? (last - first_dropped) / den : 0.0;
        }
    }
    free(cand);
    return kept;
}

/* ------------------------------------------------------------------------ */
/* StreamingLLM ([RKV] §2, §16): keep the first n_sink positions and the    */
/* newest n_recent; everything between is dropped.  Closed form.            */
/* ------------------------------------------------------------------------ */

ORC_API int orc_stream_keep(int n, const int32_t *pos, long T, int n_sink, int n_recent,
                            uint8_t *keep)
{
    int kept = 0;
    for (int j = 0; j < n; ++j) {
        keep[j] = ((long)pos[j] < n_sink || (long)pos[j] >= T - n_recent) ? 1 : 0;
        kept += keep[j];
    }
    return kept;
}

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 ([PHX]): 10 rounds of the S-box                            */
/*   (c0,c1,c2,c3) -> (hi(M1*c2)^c1^k0, lo(M1*c2), hi(M0*c0)^c3^k1,         */
/*                     lo(M0*c0))                                           */
/* with M0 = 0xD2511F53, M1 = 0xCD9E8D57, the key bumped by the Weyl        */
/* constants (0x9E3779B9, 0xBB67AE85) between rounds.                       */
/* ------------------------------------------------------------------------ */

ORC_API void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2],
                               uint32_t out[4])
{
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)p0;
        c0 = n0;
        c1 = n1;
        c2 = n2;
        c3 = n3;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

/* 64-bit eviction key of the token at absolute position pos. */
ORC_API uint64_t orc_random_key(uint64_t seed, int32_t pos, int kv_head, int batch,
                                uint32_t epoch)
{
    uint32_t ctr[4] = {(uint32_t)pos, (uint32_t)kv_head, (uint32_t)batch, epoch};
    uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
    uint32_t o[4];
    orc_philox4x32_10(ctr, key, o);
    return ((uint64_t)o[0] << 32) | o[1];
}

/*
 * Per-head uniform random eviction of one unit ([EVP] 参考实现): slots whose
 * position is < prompt_len are locked; of the n_cand others keep
 * n_keep = max(1, int(n_cand * keep_ratio)) chosen uniformly at random (the
 * n_keep smallest Philox keys, ties by position).  n_cand == 0 is a no-op.
 * keep[j] = 1 for kept slots; returns the count kept.
 */
ORC_API int orc_random_keep(int n, const int32_t *pos, int prompt_len, double keep_ratio,
                            uint64_t seed, uint32_t epoch, int batch, int kv_head, uint8_t *keep)
{
    int n_cand = 0, kept = 0;
    for (int j = 0; j < n; ++j) {
        if (pos[j] < prompt_len) {
            keep[j] = 1;
            ++kept;
        } else {
            keep[j] = 0;
            ++n_cand;
        }
    }
    if (n_cand == 0)
        return kept;
    int n_keep = (int)((double)n_cand * keep_ratio);
    if (n_keep < 1)
        n_keep = 1;
    if (n_keep > n_cand)
        n_keep = n_cand;
    for (int t = 0; t < n_keep; ++t) {
        int best = -1;
        uint64_t bk = 0;
        for (int j = 0; j < n; ++j) {
            if (keep[j] || pos[j] < prompt_len)
                continue;
            uint64_t k = orc_random_key(seed, pos[j], kv_head, batch, epoch);
            if (best < 0 || k < bk || (k == bk && pos[j] < pos[best])) {
                best = j;
                bk = k;
            }
        }
        keep[best] = 1;
        ++kept;
    }
    return kept;
}
