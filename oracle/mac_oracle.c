/*
 * fp64 CPU oracle of the MAC-Attention decode step (Match, Amend, Complete).
 *
 * TEST INFRASTRUCTURE ONLY.  This library is loaded by the test suite, by the
 * package's smoke check and by the benchmark's CPU-baseline / reference leg,
 * and by nothing else.  The CUDA library that implements the method never
 * links, loads or calls it, and the two share no source, header, table or
 * helper.  It is plain C, fp64 throughout, with no blocking, fusion or
 * reordering beyond what the definitions below state.
 *
 * Source: "MAC-Attention" (arXiv 2604.00235), as extracted on the
 * thelatestinai.com paper page:
 *   - Figure 2 caption: the three stages; the attention summary AS; the
 *     log-domain merge (+) and log-domain removal (-); the ring insert of
 *     <pre-RoPE query, AS_{1:m-r}>.
 *   - Abstract: pre-RoPE L2 matching over a short local window; a band near
 *     the match boundary is recomputed; fresh attention on the KV tail is
 *     fused through a numerically stable merge.
 *   - Figure 3 caption: per-request rings; per-head band+tail spans.
 *
 * Conventions.  A token's 0-based index j is the paper's 1-based position
 * P = j + 1.  Ranges [lo, hi) are half-open over 0-based indices, so the
 * paper's band+tail [p-r+1, m] is [p-r, m), its reused prefix AS_{1:p-r} is
 * [0, p-r) and the amend band [m-r+1, m] is [m-r, m).  KV is stored per
 * request as [t_max][Hkv][d] bf16 bit patterns; queries as [B][H][d].
 *
 * Readings where the pages are silent or garbled (each is restated at the
 * function it governs):
 *   R1  Figure 2(c) prints the rectification term and the stored summary
 *       with damaged subscripts; they are read as AS_{m-r+1:m} (the last r
 *       tokens, with the current query) and AS_{1:m-r}, the only reading
 *       under which a later hit at p can reuse the entry as AS_{1:p-r}.
 *   R2  The threshold is relative: hit iff ||q~_m - q~_e|| < tau * ||q~_m||,
 *       compared in squared form, strict.
 *   R3  Nearest entry: smallest squared distance; ties go to the entry with
 *       the larger position (the most recent one).
 *   R4  Amend subtracts from the step's own merged output AS_{1:m} (on a hit
 *       that output already contains the reused prefix).
 *   R5  Every decode step inserts into the ring (hit or miss), at slot
 *       (step mod L), overwriting the oldest entry.  The ring is empty after
 *       a reset; prefill tokens do not enter it.
 *   R6  If m <= r the stored summary AS_{1:m-r} is the empty summary
 *       (0, -inf).  If p - r < 1 the reused prefix is empty and the span
 *       starts at the first token.
 *   R7  The removal is evaluated in fp64 as defined; only when 1 - e^delta
 *       falls below 2^-20 (fp64 would then lose more than 20 of its 53 bits)
 *       is AS_{1:m-r} formed directly as the merge of its parts, which is the
 *       same quantity by definition.  Such steps are counted.
 *   R8  Attention scale: the caller passes it (1/sqrt(d) by default).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* bf16 bit pattern -> double (exact: a bf16 value is an fp32 value).        */
/* ------------------------------------------------------------------------ */
double orc_bf16_to_double(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads for the following parallel loops (timing runs on fewer cores).   */
void orc_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------------ */
/* Attention summary AS_S(q) over S = [lo, hi) of one (request, kv-head).    */
/*   z_j = scale * <q, k_j>,  lse = log sum_j exp(z_j),                      */
/*   o   = sum_j exp(z_j - lse) v_j   (the normalised output).               */
/* The empty set gives (0, -inf).  K, V point at token 0 of the head; token  */
/* j starts tok_stride elements after token j-1.                             */
/* (Figure 2 caption: "attention summary AS" = (normalised output, LSE).)    */
/* ------------------------------------------------------------------------ */
void orc_attention_summary(const double *q, const uint16_t *K, const uint16_t *V,
                           long tok_stride, long lo, long hi, int d, double scale,
                           double *o, double *lse)
{
    for (int i = 0; i < d; i++) o[i] = 0.0;
    if (hi <= lo) { *lse = -INFINITY; return; }
    long n = hi - lo;
    double *z = (double *)malloc((size_t)n * sizeof(double));
    double zmax = -INFINITY;
    for (long j = lo; j < hi; j++) {
        const uint16_t *k = K + j * tok_stride;
        double dot = 0.0;
        for (int i = 0; i < d; i++) dot += q[i] * orc_bf16_to_double(k[i]);
        z[j - lo] = scale * dot;
        if (z[j - lo] > zmax) zmax = z[j - lo];
    }
    double sum = 0.0;
    for (long j = 0; j < n; j++) sum += exp(z[j] - zmax);
    double l = zmax + log(sum);
    for (long j = lo; j < hi; j++) {
        const uint16_t *v = V + j * tok_stride;
        double w = exp(z[j - lo] - l);
        for (int i = 0; i < d; i++) o[i] += w * orc_bf16_to_double(v[i]);
    }
    *lse = l;
    free(z);
}

/* ------------------------------------------------------------------------ */
/* Log-domain merge (Figure 2 caption, the (+) operator; abstract,          */
/* "numerically stable merge"): summaries of two disjoint segments A, B      */
/*   lse = max + log(e^{lA - max} + e^{lB - max}),                           */
/*   o   = e^{lA - lse} oA + e^{lB - lse} oB.                                */
/* The empty summary (0, -inf) is the identity.  o may alias oa or ob.       */
/* ------------------------------------------------------------------------ */
void orc_merge(const double *oa, double la, const double *ob, double lb, int d,
               double *o, double *l)
{
    if (la == -INFINITY && lb == -INFINITY) {
        for (int i = 0; i < d; i++) o[i] = 0.0;
        *l = -INFINITY;
        return;
    }
    double mx = la > lb ? la : lb;
    double lse = mx + log(exp(la - mx) + exp(lb - mx));
    double wa = exp(la - lse), wb = exp(lb - lse);
    for (int i = 0; i < d; i++) o[i] = wa * oa[i] + wb * ob[i];
    *l = lse;
}

/* log(1 - e^x) for x <= 0, by the two-branch rule of Maechler (2012),
 * "Accurately computing log(1 - exp(-|a|))": log(-expm1(x)) above -ln 2,
 * log1p(-exp(x)) below.  x = 0 gives -inf. */
double orc_log1mexp(double x)
{
    if (x > -0.6931471805599453) return log(-expm1(x));
    return log1p(-exp(x));
}

/* ------------------------------------------------------------------------ */
/* Log-domain removal (Figure 2 caption, the (-) operator; "update the cache */
/* via online subtraction"): given the summary of A u B and of B, recover A. */
/*   delta = lB - lAuB (<= 0),  lA = lAuB + log(1 - e^delta),                */
/*   oA = (oAuB - e^delta oB) / (1 - e^delta).                               */
/* Returns the conditioning 1 - e^delta so the caller can test it (R7).      */
/* ------------------------------------------------------------------------ */
double orc_remove(const double *oab, double lab, const double *ob, double lb, int d,
                  double *o, double *l)
{
    if (lb == -INFINITY) {               /* removing the empty set */
        for (int i = 0; i < d; i++) o[i] = oab[i];
        *l = lab;
        return 1.0;
    }
    double delta = lb - lab;
    double one_minus_w = -expm1(delta);  /* 1 - e^delta */
    double w = exp(delta);
    *l = lab + orc_log1mexp(delta);
    for (int i = 0; i < d; i++) o[i] = (oab[i] - w * ob[i]) / one_minus_w;
    return one_minus_w;
}

/* ------------------------------------------------------------------------ */
/* Match (Figure 2(a); abstract, "pre-RoPE L2 matching over a short local    */
/* window").  Over the valid ring entries e (ring_pos[e] > 0):               */
/*   D_e = sum_i (q~_m[i] - q~_e[i])^2,  e* = argmin D_e (R3),               */
/*   hit iff D_{e*} < tau^2 * ||q~_m||^2 (R2).                               */
/* Returns e* (or -1 when no entry is valid).  *D2 is the runner-up distance */
/* (+inf if none), reported so a caller can recognise near-ties.             */
/* ------------------------------------------------------------------------ */
int orc_match(const uint16_t *q_pre, const uint16_t *ring_q, const int64_t *ring_pos,
              int L, int d, double tau, double *D, double *D2, double *qn2, int *hit)
{
    double n2 = 0.0;
    for (int i = 0; i < d; i++) {
        double a = orc_bf16_to_double(q_pre[i]);
        n2 += a * a;
    }
    int best = -1;
    double bestD = INFINITY, secondD = INFINITY;
    int64_t bestPos = -1;
    for (int e = 0; e < L; e++) {
        if (ring_pos[e] <= 0) continue;
        double De = 0.0;
        for (int i = 0; i < d; i++) {
            double diff = orc_bf16_to_double(q_pre[i]) - orc_bf16_to_double(ring_q[(long)e * d + i]);
            De += diff * diff;
        }
        if (best < 0 || De < bestD || (De == bestD && ring_pos[e] > bestPos)) {
            if (best >= 0) secondD = bestD < secondD ? bestD : secondD;
            best = e;
            bestD = De;
            bestPos = ring_pos[e];
        } else if (De < secondD) {
            secondD = De;
        }
    }
    *qn2 = n2;
    *D = bestD;
    *D2 = secondD;
    *hit = (best >= 0) && (bestD < tau * tau * n2);
    return best;
}

/* ------------------------------------------------------------------------ */
/* Per-request, per-head rings and the MAC decode step.                      */
/* ------------------------------------------------------------------------ */
typedef struct orc_mac {
    int B, H, Hkv, d, L, r;
    double tau, scale;
    long t_max;
    uint16_t *K, *V;      /* caller-owned: [B][t_max][Hkv][d] bf16 bits     */
    int64_t *kv_len;      /* [B] tokens stored                              */
    int64_t *step;        /* [B] decode steps since reset                   */
    int64_t *ring_pos;    /* [B][L] 1-based position of the entry, 0 empty  */
    uint16_t *ring_q;     /* [B][H][L][d] pre-RoPE query, bf16 bits         */
    double *ring_o;       /* [B][H][L][d] AS_{1:pos-r}: normalised output   */
    double *ring_lse;     /* [B][H][L]    AS_{1:pos-r}: log-sum-exp         */
    int64_t n_direct;     /* removals formed directly (R7)                  */
} orc_mac;

orc_mac *orc_mac_create(int B, int H, int Hkv, int d, int L, int r, double tau,
                        double scale, long t_max, uint16_t *K, uint16_t *V)
{
    if (B < 1 || H < 1 || Hkv < 1 || H % Hkv || d < 1 || L < 1 || r < 1 || tau < 0 || t_max < 1)
        return NULL;
    orc_mac *s = (orc_mac *)calloc(1, sizeof *s);
    s->B = B; s->H = H; s->Hkv = Hkv; s->d = d; s->L = L; s->r = r;
    s->tau = tau; s->scale = scale; s->t_max = t_max; s->K = K; s->V = V;
    s->kv_len = (int64_t *)calloc((size_t)B, sizeof(int64_t));
    s->step = (int64_t *)calloc((size_t)B, sizeof(int64_t));
    s->ring_pos = (int64_t *)calloc((size_t)B * L, sizeof(int64_t));
    s->ring_q = (uint16_t *)calloc((size_t)B * H * L * d, sizeof(uint16_t));
    s->ring_o = (double *)calloc((size_t)B * H * L * d, sizeof(double));
    s->ring_lse = (double *)malloc((size_t)B * H * L * sizeof(double));
    for (long i = 0; i < (long)B * H * L; i++) s->ring_lse[i] = -INFINITY;
    return s;
}

void orc_mac_destroy(orc_mac *s)
{
    if (!s) return;
    free(s->kv_len); free(s->step); free(s->ring_pos);
    free(s->ring_q); free(s->ring_o); free(s->ring_lse);
    free(s);
}

/* Declare that request b holds len tokens (the caller wrote them into K/V)
 * and empty its rings. */
int orc_mac_reset(orc_mac *s, int b, long len)
{
    if (b < 0 || b >= s->B || len < 0 || len > s->t_max) return -1;
    s->kv_len[b] = len;
    s->step[b] = 0;
    for (int e = 0; e < s->L; e++) s->ring_pos[(long)b * s->L + e] = 0;
    for (int h = 0; h < s->H; h++)
        for (int e = 0; e < s->L; e++) {
            long slot = ((long)b * s->H + h) * s->L + e;
            s->ring_lse[slot] = -INFINITY;
            memset(s->ring_o + slot * s->d, 0, (size_t)s->d * sizeof(double));
            memset(s->ring_q + slot * s->d, 0, (size_t)s->d * sizeof(uint16_t));
        }
    return 0;
}

int64_t orc_mac_direct_count(const orc_mac *s) { return s->n_direct; }

void orc_mac_read_ring(const orc_mac *s, int64_t *pos, uint16_t *q, double *o, double *lse,
                       int64_t *kv_len, int64_t *step)
{
    long BL = (long)s->B * s->L, BHL = (long)s->B * s->H * s->L;
    if (pos) memcpy(pos, s->ring_pos, (size_t)BL * sizeof(int64_t));
    if (q) memcpy(q, s->ring_q, (size_t)BHL * s->d * sizeof(uint16_t));
    if (o) memcpy(o, s->ring_o, (size_t)BHL * s->d * sizeof(double));
    if (lse) memcpy(lse, s->ring_lse, (size_t)BHL * sizeof(double));
    if (kv_len) memcpy(kv_len, s->kv_len, (size_t)s->B * sizeof(int64_t));
    if (step) memcpy(step, s->step, (size_t)s->B * sizeof(int64_t));
}

/* Seed request b's rings with n entries <q~, AS_{1:pos-r}> at 1-based
 * positions pos[i] (strictly increasing, each <= kv_len[b]), inserted in
 * order exactly as decode steps insert them: slot (step mod L), step + 1.
 * q_pre [n][H][d] bf16 bits; o [n][H][d]; lse [n][H].  The pages do not say
 * how prefill queries enter the rings; the caller supplies the entries (its
 * prefill attention yields the summaries). */
int orc_mac_seed(orc_mac *s, int b, int n, const uint16_t *q_pre, const double *o, const double *lse,
                 const int64_t *pos)
{
    if (b < 0 || b >= s->B || n < 0) return -1;
    for (int i = 0; i < n; i++)
        if (pos[i] < 1 || pos[i] > s->kv_len[b] || (i > 0 && pos[i] <= pos[i - 1])) return -1;
    const int H = s->H, d = s->d, L = s->L;
    for (int i = 0; i < n; i++) {
        const long slot = (long)(s->step[b] % L);
        s->ring_pos[(long)b * L + slot] = pos[i];
        for (int h = 0; h < H; h++) {
            const long e = ((long)b * H + h) * L + slot;
            memcpy(s->ring_q + e * d, q_pre + ((long)i * H + h) * d, (size_t)d * sizeof(uint16_t));
            memcpy(s->ring_o + e * d, o + ((long)i * H + h) * d, (size_t)d * sizeof(double));
            s->ring_lse[e] = lse[(long)i * H + h];
        }
        s->step[b] += 1;
    }
    return 0;
}

/* Append the new token's K and V at index kv_len[b] of each request. */
static int append_new_token(orc_mac *s, int batch, const uint16_t *k_new, const uint16_t *v_new)
{
    for (int b = 0; b < batch; b++)
        if (s->kv_len[b] + 1 > s->t_max) return -2;
    long row = (long)s->Hkv * s->d;
    for (int b = 0; b < batch; b++) {
        long at = ((long)b * s->t_max + s->kv_len[b]) * row;
        memcpy(s->K + at, k_new + (long)b * row, (size_t)row * sizeof(uint16_t));
        memcpy(s->V + at, v_new + (long)b * row, (size_t)row * sizeof(uint16_t));
    }
    return 0;
}

/*
 * One MAC decode step for requests 0..batch-1 (Figure 2 (a) -> (b) -> (c)).
 * Inputs: q_pre, q_post [batch][H][d] (pre- and post-RoPE query, bf16 bits),
 * k_new, v_new [batch][Hkv][d].  Outputs: out_o [batch][H][d], out_lse
 * [batch][H] (the merged AS_{1:m}), and the decision per (request, head):
 * ring slot (-1 none), D, runner-up D2, ||q~||^2, hit, reuse position p.
 * Returns 0, or a negative code on bad arguments / a full KV store.
 * orc_mac_step_heads evaluates only query heads [h_lo, h_hi) (a timing
 * sample); the others' outputs, decisions and ring entries are left as they
 * were, while lengths, positions and step counters advance as usual.
 */
int orc_mac_step_heads(orc_mac *s, int batch, int h_lo, int h_hi, const uint16_t *q_pre,
                       const uint16_t *q_post, const uint16_t *k_new, const uint16_t *v_new,
                       double *out_o, double *out_lse, int32_t *dec_slot, double *dec_D,
                       double *dec_D2, double *dec_qn2, int32_t *dec_hit, int64_t *dec_p)
{
    if (batch < 1 || batch > s->B || h_lo < 0 || h_hi > s->H || h_lo >= h_hi) return -1;
    int rc = append_new_token(s, batch, k_new, v_new);
    if (rc) return rc;
    const int H = s->H, d = s->d, L = s->L, G = s->H / s->Hkv;
    const long r = s->r;
    const long row = (long)s->Hkv * d;
    int64_t n_direct = 0;

#pragma omp parallel for schedule(dynamic, 1) reduction(+ : n_direct)
    for (long bh = 0; bh < (long)batch * H; bh++) {
        const int b = (int)(bh / H), h = (int)(bh % H), g = h / G;
        if (h < h_lo || h >= h_hi) continue;             /* heads outside the sample */
        const long m = s->kv_len[b] + 1;                 /* 1-based position of the new token */
        const long slot_new = (long)(s->step[b] % L);    /* R5 */
        const uint16_t *Kh = s->K + (long)b * s->t_max * row + (long)g * d;
        const uint16_t *Vh = s->V + (long)b * s->t_max * row + (long)g * d;
        const uint16_t *qp = q_pre + bh * d;
        double *q = (double *)malloc((size_t)d * sizeof(double));
        double *o = (double *)malloc((size_t)d * sizeof(double));
        double *ot = (double *)malloc((size_t)d * sizeof(double));
        double *ob = (double *)malloc((size_t)d * sizeof(double));
        double *oe = (double *)malloc((size_t)d * sizeof(double));
        for (int i = 0; i < d; i++) q[i] = orc_bf16_to_double(q_post[bh * d + i]);

        /* (a) Match against this head's ring. */
        const long ring_base = ((long)b * H + h) * L;
        double D, D2, qn2;
        int hit;
        int e = orc_match(qp, s->ring_q + ring_base * d, s->ring_pos + (long)b * L, L, d,
                          s->tau, &D, &D2, &qn2, &hit);
        long p = (e >= 0) ? (long)s->ring_pos[(long)b * L + e] : 0;

        /* (b) Complete: attention over the band+tail [p-r+1, m] merged with the
         * reused AS_{1:p-r}; on a miss, attention over [1, m]. */
        double l, lt;
        long lo = 0;
        if (hit) {
            lo = p - r > 0 ? p - r : 0;                  /* R6 */
            orc_attention_summary(q, Kh, Vh, row, lo, m, d, s->scale, ot, &lt);
            orc_merge(s->ring_o + (ring_base + e) * d, s->ring_lse[ring_base + e], ot, lt, d, o, &l);
        } else {
            orc_attention_summary(q, Kh, Vh, row, 0, m, d, s->scale, o, &l);
        }

        /* (c) Amend: AS_{1:m-r} = AS_{1:m} (-) AS_{m-r+1:m}  (R1, R4, R6, R7). */
        double le;
        if (m <= r) {
            for (int i = 0; i < d; i++) oe[i] = 0.0;
            le = -INFINITY;
        } else {
            double lb;
            orc_attention_summary(q, Kh, Vh, row, m - r, m, d, s->scale, ob, &lb);
            double cond = orc_remove(o, l, ob, lb, d, oe, &le);
            if (cond < 0x1p-20) {
                n_direct += 1;
                if (hit) {
                    orc_attention_summary(q, Kh, Vh, row, lo, m - r, d, s->scale, ot, &lt);
                    orc_merge(s->ring_o + (ring_base + e) * d, s->ring_lse[ring_base + e], ot, lt, d, oe, &le);
                } else {
                    orc_attention_summary(q, Kh, Vh, row, 0, m - r, d, s->scale, oe, &le);
                }
            }
        }

        /* Outputs and the decision. */
        memcpy(out_o + bh * d, o, (size_t)d * sizeof(double));
        out_lse[bh] = l;
        if (dec_slot) dec_slot[bh] = e;
        if (dec_D) dec_D[bh] = D;
        if (dec_D2) dec_D2[bh] = D2;
        if (dec_qn2) dec_qn2[bh] = qn2;
        if (dec_hit) dec_hit[bh] = hit;
        if (dec_p) dec_p[bh] = hit ? p : 0;

        /* Insert <q~_m, AS_{1:m-r}> into this head's ring (Figure 2(c)). */
        memcpy(s->ring_q + (ring_base + slot_new) * d, qp, (size_t)d * sizeof(uint16_t));
        memcpy(s->ring_o + (ring_base + slot_new) * d, oe, (size_t)d * sizeof(double));
        s->ring_lse[ring_base + slot_new] = le;
        free(q); free(o); free(ot); free(ob); free(oe);
    }
    for (int b = 0; b < batch; b++) {
        s->ring_pos[(long)b * L + (s->step[b] % L)] = s->kv_len[b] + 1;
        s->kv_len[b] += 1;
        s->step[b] += 1;
    }
    s->n_direct += n_direct;
    return 0;
}

int orc_mac_step(orc_mac *s, int batch, const uint16_t *q_pre, const uint16_t *q_post,
                 const uint16_t *k_new, const uint16_t *v_new, double *out_o, double *out_lse,
                 int32_t *dec_slot, double *dec_D, double *dec_D2, double *dec_qn2,
                 int32_t *dec_hit, int64_t *dec_p)
{
    return orc_mac_step_heads(s, batch, 0, s->H, q_pre, q_post, k_new, v_new, out_o, out_lse,
                              dec_slot, dec_D, dec_D2, dec_qn2, dec_hit, dec_p);
}

/* Full attention decode step (the miss path for every head, no ring): append
 * the new token, then AS_{1:m} for every (request, head). */
int orc_full_step(orc_mac *s, int batch, const uint16_t *q_post, const uint16_t *k_new,
                  const uint16_t *v_new, double *out_o, double *out_lse)
{
    if (batch < 1 || batch > s->B) return -1;
    int rc = append_new_token(s, batch, k_new, v_new);
    if (rc) return rc;
    const int H = s->H, d = s->d, G = s->H / s->Hkv;
    const long row = (long)s->Hkv * d;
#pragma omp parallel for schedule(dynamic, 1)
    for (long bh = 0; bh < (long)batch * H; bh++) {
        const int b = (int)(bh / H), h = (int)(bh % H), g = h / G;
        const long m = s->kv_len[b] + 1;
        double *q = (double *)malloc((size_t)d * sizeof(double));
        for (int i = 0; i < d; i++) q[i] = orc_bf16_to_double(q_post[bh * d + i]);
        orc_attention_summary(q, s->K + (long)b * s->t_max * row + (long)g * d,
                              s->V + (long)b * s->t_max * row + (long)g * d, row, 0, m, d,
                              s->scale, out_o + bh * d, out_lse + bh);
        free(q);
    }
    for (int b = 0; b < batch; b++) s->kv_len[b] += 1;
    return 0;
}
