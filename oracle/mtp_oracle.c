/*
 * mtp_oracle.c -- plain, slow CPU oracle for the MTP draft block and the
 * verify-accept step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file: only the test suite, the package's smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA library; the two meet only through the seeded inputs of the `synth`
 * module.
 *
 * Arithmetic is fp64 throughout.  bf16 inputs are widened exactly (bits << 16).
 * Loops run in the order the definitions are written; the only parallelism is
 * an OpenMP split of independent output rows / sequences, which does not
 * change any row's summation order.
 *
 * Sources (page title, section):
 *  [G4]  "Gemma 4 MTP -- Multi-Token Prediction speculative decoding",
 *        sec. 3 (pre/post projection shapes; the centroid / ordered-embeddings
 *        LM head), sec. 4 "Per-step MTP graph"
 *        (embedding scale, concat + pre-projection, block order, final norm,
 *        post-projection, LM head, softcap, in-graph argmax), sec. 5 "KV
 *        sharing" (mask admits every position <= attn_pos; one mask for all
 *        steps; draft positions are > attn_pos).
 *  [NX]  "MTP decoding (--mtp)", "Requirements" (NextN enorm / hnorm / eh_proj:
 *        separate norms of the token embedding and of the hidden state before
 *        the projection; the NextN block's own attention and feed-forward and
 *        the shared head with its norm), "How it is wired" (accept the longest
 *        prefix whose argmax matches, the next token comes from the first
 *        unverified row; the draft context catches up on the accepted rows)
 *        and "The catch-up runs on the accepted prefix" (the catch-up rows are
 *        [confirmed token, accepted drafts]; no rollback of the draft KV).
 *  [SP]  "opus-mtp-turbo: Track 1 report", item 4 "temp > 0 verification"
 *        (sample_dist: top-k, penalties over history + input[0..i], temp,
 *        min-p, top-p; accept with p(x)/q(x); on reject sample
 *        norm(max(p - q, 0)); a fully accepted window samples its last row).
 *  [FN]  "Fused NextN draft graph", delta 6 (the fused steps cross-attend the
 *        frozen prefix read-only; the recurrence is carried by the hidden
 *        state chain alone).
 *        Item 3 "Q4_0 / Q5_0 draft weights": the Q8_0 weight format of its
 *        quantisation-error table (ggml's rule, see orc_quantize_q8_0).
 *        "The two MTP lanes": the NextN drafter runs its own block with its own
 *        (unified) KV, unlike the assistant that reads the target's.
 *  [PH]  Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
 *        1, 2, 3" (SC'11): the Philox-4x32-10 counter-based generator.
 *
 * Readings taken where the pages are silent (each is also listed in the
 * design notes): RMSNorm y = x / sqrt(mean(x^2) + eps) * g with the gain g
 * stored directly; RoPE rotates Q only, NeoX half-split pairs (i, i + hd/2),
 * angle pos * theta^(-2i/hd), pos = kv_len + step; GQA maps q head h to kv
 * head h / (Hq / Hkv); GELU is the tanh form; argmax ties go to the lowest
 * index and NaN never wins; the sliding window reads the last W positions
 * [kv_len - W, kv_len) at every step; KV views are ring buffers (position t in
 * slot t % cap).  The NextN drafter (the pages name its tensors, not its
 * arithmetic): one pre-norm block at the backbone width, x += w_o attn and
 * x += w_down(silu(w_gate n) * w_up n) with n = ffn_norm(x); a fused query /
 * key / value projection; per-head q and k norms; NeoX RoPE of queries and
 * keys at the row's position (the row index in its own KV); causal attention
 * over rows [0, pos]; keys and values stored rounded to the weights' type;
 * embedding scale 1; the next step's hidden state is the block output before
 * head_norm.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* types (the oracle's own; the CUDA library declares its own elsewhere)     */
/* ------------------------------------------------------------------------ */

typedef struct {
    int32_t d_t, d_a, n_blocks, n_q_heads, head_dim, n_kv_heads, d_ff, vocab;
    int32_t wbf16;        /* 1: weight matrices and KV are bf16 bit patterns; 0: fp32 */
    int32_t n_centroids;  /* 0: dense tied LM head; > 0: centroid-routed head */
    int32_t centroid_top_k;
    int32_t kv_bf16;      /* NextN: 1 when the drafter's own KV is stored as bf16 (its weights may be widened) */
    double rms_eps, attn_scale, emb_scale, logit_softcap;
} orc_model;

typedef struct {
    const void *k, *v;
    int64_t stride_b, stride_h, stride_t;   /* elements; head_dim is contiguous */
    int32_t cap, window;                    /* slots; 0 = full attention */
    int32_t sink, pad_;                     /* attention-sink positions read with a window */
    double rope_theta;
} orc_view;

typedef struct {
    double temp, top_p, min_p, rep_penalty, presence_penalty;
    int32_t top_k, pad_;
} orc_sample_params;

/* tensor table: globals first, then B_COUNT entries per block */
enum { T_TOK_EMBD, T_NORM_E, T_NORM_H, T_W_PRE, T_FINAL_NORM, T_W_POST, T_CENTROIDS, T_ORDERING,
       T_GLOBAL_COUNT };
enum { B_ATTN_NORM, B_W_Q, B_Q_NORM, B_W_O, B_POST_ATTN_NORM, B_PRE_FFN_NORM,
       B_W_GATE, B_W_UP, B_W_DOWN, B_POST_FFN_NORM, B_COUNT };

/* ------------------------------------------------------------------------ */
/* element access                                                            */
/* ------------------------------------------------------------------------ */

static double bf16_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double elem(const void *p, int64_t i, int bf16) {
    if (bf16) return bf16_to_double(((const uint16_t *)p)[i]);
    return (double)((const float *)p)[i];
}

/* ------------------------------------------------------------------------ */
/* building blocks                                                           */
/* ------------------------------------------------------------------------ */

/* RMSNorm (reading: y = x / sqrt(mean(x^2) + eps) * g; g == NULL means unit gains) */
void orc_rmsnorm(const double *x, int n, const float *g, double eps, double *y) {
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double r = 1.0 / sqrt(ss / (double)n + eps);
    for (int i = 0; i < n; ++i) y[i] = x[i] * r * (g ? (double)g[i] : 1.0);
}

/* y[r] = sum_c W[r, c] * x[c], W row-major [rows, cols]; plain dot per row */
void orc_matvec(const void *W, int rows, int cols, int bf16, const double *x, double *y) {
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r) {
        double acc = 0.0;
        const int64_t base = (int64_t)r * cols;
        for (int c = 0; c < cols; ++c) acc += elem(W, base + c, bf16) * x[c];
        y[r] = acc;
    }
}

/* GELU, tanh form: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))) */
double orc_gelu_tanh(double x) {
    const double k = sqrt(2.0 / M_PI);
    return 0.5 * x * (1.0 + tanh(k * (x + 0.044715 * x * x * x)));
}

/* RoPE on one head vector, NeoX half-split pairs (i, i + hd/2) */
void orc_rope_neox(double *q, int hd, int64_t pos, double theta) {
    const int half = hd / 2;
    for (int i = 0; i < half; ++i) {
        double ang = (double)pos * pow(theta, -2.0 * (double)i / (double)hd);
        double c = cos(ang), s = sin(ang);
        double a = q[i], b = q[i + half];
        q[i] = a * c - b * s;
        q[i + half] = a * s + b * c;
    }
}

/* first index of the largest value; NaN never wins; all-NaN -> 0 */
int64_t orc_argmax_f64(const double *z, int64_t n) {
    int64_t best = -1;
    double bv = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double v = z[i];
        if (isnan(v)) continue;
        if (best < 0 || v > bv) { best = i; bv = v; }
    }
    return best < 0 ? 0 : best;
}

static int64_t argmax_stored(const void *z, int64_t n, int bf16) {
    int64_t best = -1;
    double bv = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double v = elem(z, i, bf16);
        if (isnan(v)) continue;
        if (best < 0 || v > bv) { best = i; bv = v; }
    }
    return best < 0 ? 0 : best;
}

/* The slot of position t in a view: t below the sink, then a ring over the
 * remaining cap - sink slots ("opus-mtp-turbo: Track 1 report", item 2 keeps
 * the first `sink` cells beside the window). */
static int64_t view_slot(const orc_view *vw, int64_t t) {
    const int64_t sk = vw->window > 0 ? vw->sink : 0;
    return t < sk ? t : sk + (t - sk) % (vw->cap - sk);
}

/* Cross-attention of one query head into one KV view ([G4] sec. 4-5, [FN] delta 6).
 * Keys: positions t in [lo, kv_len), lo = max(0, kv_len - window) for a sliding
 * view, 0 for a full one, and for a sliding view the sink positions
 * [0, min(sink, lo)) (the sink + window read of "opus-mtp-turbo", item 2).  V is
 * used as stored. */
void orc_attend_head(const double *q, const orc_view *vw, int b, int g, int hd, int kv_len,
                     double scale, int bf16, double *out) {
    const int lo = (vw->window > 0 && kv_len > vw->window) ? kv_len - vw->window : 0;
    const int s0 = vw->window > 0 ? (vw->sink < lo ? vw->sink : lo) : 0;   /* sink keys */
    const int n = s0 + kv_len - lo;
    double *s = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) {
        const int64_t pos = j < s0 ? j : lo + (j - s0);
        int64_t slot = view_slot(vw, pos);
        int64_t base = (int64_t)b * vw->stride_b + (int64_t)g * vw->stride_h + slot * vw->stride_t;
        double acc = 0.0;
        for (int d = 0; d < hd; ++d) acc += q[d] * elem(vw->k, base + d, bf16);
        s[j] = scale * acc;
        if (s[j] > m) m = s[j];
    }
    double den = 0.0;
    for (int d = 0; d < hd; ++d) out[d] = 0.0;
    for (int j = 0; j < n; ++j) {
        double w = exp(s[j] - m);
        den += w;
        const int64_t pos = j < s0 ? j : lo + (j - s0);
        int64_t slot = view_slot(vw, pos);
        int64_t base = (int64_t)b * vw->stride_b + (int64_t)g * vw->stride_h + slot * vw->stride_t;
        for (int d = 0; d < hd; ++d) out[d] += w * elem(vw->v, base + d, bf16);
    }
    for (int d = 0; d < hd; ++d) out[d] /= den;
    free(s);
}

/* ------------------------------------------------------------------------ */
/* Philox-4x32-10 [PH]                                                       */
/* ------------------------------------------------------------------------ */

static void mulhilo32(uint32_t a, uint32_t b, uint32_t *hi, uint32_t *lo) {
    uint64_t p = (uint64_t)a * (uint64_t)b;
    *hi = (uint32_t)(p >> 32);
    *lo = (uint32_t)p;
}

void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int r = 0; r < 10; ++r) {
        uint32_t hi0, lo0, hi1, lo1;
        mulhilo32(0xD2511F53u, c0, &hi0, &lo0);
        mulhilo32(0xCD9E8D57u, c2, &hi1, &lo1);
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* uniform in [0, 1) for (sequence b, row i, purpose): counter (b, 4 i + purpose,
 * offset lo, offset hi), key (seed lo, seed hi); u = (word0 >> 8) * 2^-24 */
double orc_uniform(uint64_t seed, uint64_t offset, uint32_t b, uint32_t i, uint32_t purpose) {
    uint32_t ctr[4] = { b, i * 4u + purpose, (uint32_t)offset, (uint32_t)(offset >> 32) };
    uint32_t key[2] = { (uint32_t)seed, (uint32_t)(seed >> 32) };
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    return (double)(out[0] >> 8) * (1.0 / 16777216.0);
}

/* ------------------------------------------------------------------------ */
/* sample_dist [SP item 4]                                                   */
/*                                                                          */
/* The sampler's arithmetic decides integers (kept sets, orders, picks), so */
/* it is carried out in IEEE fp32 with every rounding step written out:     */
/* penalties, temperature, the difference l - lmax, and every sum taken     */
/* sequentially in the documented order.  A weight is exp(l - lmax) rounded */
/* once to fp32: libm's exp in fp64, then one conversion.  Any other        */
/* implementation whose weights are the correctly rounded exp takes the     */
/* same decisions; one whose exp is off by an ulp may differ only where a   */
/* decision lies within about 1e-6 of its threshold, which *margin reports. */
/* ------------------------------------------------------------------------ */

typedef struct { int id; float w; float l; } cand;

static int cand_cmp(const void *a, const void *b) {   /* weight desc, id asc */
    const cand *x = (const cand *)a, *y = (const cand *)b;
    if (x->w > y->w) return -1;
    if (x->w < y->w) return 1;
    return (x->id < y->id) ? -1 : (x->id > y->id);
}

static float rel_gap(float a, float b, float scale) {
    float d = fabsf(a - b) / (scale > 0.0f ? scale : 1.0f);
    return d;
}

/* Builds sample_dist(z) for one row.
 *   z     raw logits, V entries (values exactly representable in fp32)
 *   pen   penalty token list (history + this window's inputs); duplicates and
 *         out-of-range ids are ignored; each distinct token is penalised once
 *   order top-k (off when top_k <= 0) -> repetition penalty (z > 0: z / r,
 *         else z * r) then presence penalty (- pres) -> temperature (/ temp)
 *         -> weights w = exp(l - lmax) -> min-p (keep w >= min_p, i.e.
 *         p >= min_p * p_max) -> sort by (w desc, id asc) -> top-p (keep the
 *         shortest prefix whose running sum / total reaches top_p, the
 *         crossing token included) -> the kept weights, renormalised by their
 *         sequential sum.
 * Output: n kept candidates, ids[] / w[] in order; *wsum the kept sum.
 * *margin (optional): the smallest nonzero relative distance of any keep/cut
 * decision or ordering to its threshold (diagnostic). */
int orc_sample_dist_f32(const double *z, int V, const int32_t *pen, int n_pen, const orc_sample_params *sp,
                        int32_t *ids, float *w, float *wsum, double *margin) {
    const float rep = (float)sp->rep_penalty, pres = (float)sp->presence_penalty;
    const float temp = (float)sp->temp, min_p = (float)sp->min_p, top_p = (float)sp->top_p;
    float *l = (float *)malloc(sizeof(float) * (size_t)V);
    unsigned char *alive = (unsigned char *)malloc((size_t)V);
    for (int x = 0; x < V; ++x) { l[x] = (float)z[x]; alive[x] = !isnan(l[x]); }
    double mg = INFINITY;

    if (sp->top_k > 0 && sp->top_k < V) {
        cand *all = (cand *)malloc(sizeof(cand) * (size_t)V);
        int na = 0;
        for (int x = 0; x < V; ++x) if (alive[x]) { all[na].id = x; all[na].w = l[x]; ++na; }
        qsort(all, (size_t)na, sizeof(cand), cand_cmp);
        memset(alive, 0, (size_t)V);
        for (int j = 0; j < na && j < sp->top_k; ++j) alive[all[j].id] = 1;
        free(all);
    }

    unsigned char *seen = (unsigned char *)calloc((size_t)V, 1);
    for (int j = 0; j < n_pen; ++j) {
        int x = pen[j];
        if (x < 0 || x >= V || seen[x]) continue;
        seen[x] = 1;
        float y = l[x] > 0.0f ? l[x] / rep : l[x] * rep;
        l[x] = y - pres;
    }
    free(seen);
    for (int x = 0; x < V; ++x) l[x] = l[x] / temp;

    float lmax = -INFINITY;
    for (int x = 0; x < V; ++x) if (alive[x] && l[x] > lmax) lmax = l[x];

    cand *c = (cand *)malloc(sizeof(cand) * (size_t)V);
    int n = 0;
    for (int x = 0; x < V; ++x) {
        if (!alive[x]) continue;
        const float d = l[x] - lmax;
        const float wx = (float)exp((double)d);
        if (min_p > 0.0f) {
            double dd = rel_gap(wx, min_p, min_p);
            if (dd < mg) mg = dd;
        }
        if (wx >= min_p) { c[n].id = x; c[n].w = wx; c[n].l = l[x]; ++n; }
    }
    qsort(c, (size_t)n, sizeof(cand), cand_cmp);
    /* order margins: equal weights of equal scaled logits are ordered by id
     * on any implementation; equal weights of different logits, or nearly
     * equal weights, could swap under another exp */
    for (int j = 1; j < n; ++j) {
        if (c[j - 1].l == c[j].l) continue;
        double d = rel_gap(c[j - 1].w, c[j].w, c[j - 1].w);
        if (d < mg) mg = d;
    }
    if (top_p < 1.0f && n > 0) {
        float tot = 0.0f;
        for (int j = 0; j < n; ++j) tot += c[j].w;
        float cum = 0.0f;
        int keep = n;
        for (int j = 0; j < n; ++j) {
            cum += c[j].w;
            const float share = cum / tot;
            double d = fabs((double)share - (double)top_p);
            if (d < mg) mg = d;
            if (share >= top_p) { keep = j + 1; break; }
        }
        n = keep;
    }
    float ssum = 0.0f;
    for (int j = 0; j < n; ++j) { ids[j] = c[j].id; w[j] = c[j].w; ssum += c[j].w; }
    *wsum = ssum;
    if (margin) *margin = mg;
    free(c); free(alive); free(l);
    return n;
}

/* double-typed wrapper for callers outside this file (weights are fp32 values) */
int orc_sample_dist(const double *z, int V, const int32_t *pen, int n_pen, const orc_sample_params *sp,
                    int32_t *ids, double *w, double *wsum, double *margin) {
    float *wf = (float *)malloc(sizeof(float) * (size_t)(V > 0 ? V : 1));
    float ws;
    int n = orc_sample_dist_f32(z, V, pen, n_pen, sp, ids, wf, &ws, margin);
    for (int j = 0; j < n; ++j) w[j] = (double)wf[j];
    *wsum = (double)ws;
    free(wf);
    return n;
}

/* Inverse-CDF pick over candidates in their stored order: the first j with
 * u * wsum < w[0] + ... + w[j] (fp32, running sum in order).  *margin: the
 * distance of u * wsum to the nearer edge of the chosen interval, relative to
 * wsum (diagnostic). */
int32_t orc_pick_f32(const int32_t *ids, const float *w, int n, float wsum, float u, double *margin) {
    const float target = u * wsum;
    float acc = 0.0f, prev = 0.0f;
    for (int j = 0; j < n; ++j) {
        prev = acc;
        acc += w[j];
        if (target < acc) {
            double a = (double)target - (double)prev, b = (double)acc - (double)target;
            if (margin) *margin = (a < b ? a : b) / (wsum > 0.0f ? (double)wsum : 1.0);
            return ids[j];
        }
    }
    if (margin) *margin = 0.0;
    return n > 0 ? ids[n - 1] : 0;
}

int32_t orc_pick(const int32_t *ids, const double *w, int n, double wsum, double u, double *margin) {
    float *wf = (float *)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1));
    for (int j = 0; j < n; ++j) wf[j] = (float)w[j];
    int32_t r = orc_pick_f32(ids, wf, n, (float)wsum, (float)u, margin);
    free(wf);
    return r;
}

/* ------------------------------------------------------------------------ */
/* Q8_0 drafter weights ([SP] item 3)                                        */
/* ------------------------------------------------------------------------ */

/* IEEE binary16 from a float, round to nearest even (subnormals kept,
 * overflow to infinity), and back. */
static uint16_t f32_to_f16(float xf) {
    double x = xf;
    uint16_t sign = 0;
    if (signbit(x)) { sign = 0x8000; x = -x; }
    if (isnan(x)) return 0x7e00;
    if (x >= 65520.0) return sign | 0x7c00;                 /* rounds past the largest finite */
    if (x < ldexp(1.0, -14)) {                              /* subnormal: steps of 2^-24 */
        const double r = nearbyint(x / ldexp(1.0, -24));    /* 1024 is the smallest normal */
        return sign | (uint16_t)r;
    }
    int e;
    frexp(x, &e);
    e -= 1;                                                 /* x in [2^e, 2^(e+1)) */
    double m = nearbyint(x / ldexp(1.0, e - 10));           /* 11 significant bits */
    if (m == 2048.0) { m = 1024.0; e += 1; }
    if (e > 15) return sign | 0x7c00;
    return sign | (uint16_t)((e + 15) << 10) | (uint16_t)((int)m - 1024);
}
static double f16_to_double(uint16_t h) {
    const int e = (h >> 10) & 31, m = h & 1023;
    const double v = e == 0 ? ldexp((double)m, -24) : e == 31 ? (m ? NAN : INFINITY) : ldexp(1024.0 + m, e - 25);
    return (h & 0x8000) ? -v : v;
}

/* Q8_0 quantisation of a row-major [rows, cols] fp32 matrix, cols a multiple
 * of 32 (the Q8_0 format the report's error table measures, ggml's rule):
 * per block of 32 consecutive weights of a row, d = max |w| / 127 in fp32,
 * stored as binary16; codes q = round(w * (1 / d)) in fp32, halves away from
 * zero, all 0 when d = 0.  Codes go to q[rows, cols] (int8), block scales to
 * d16[rows, cols / 32] (binary16 bits).  The weight a code stands for is
 * f16(d) * q (f16_to_double). */
void orc_quantize_q8_0(const float *w, int64_t rows, int64_t cols, int8_t *q, uint16_t *d16) {
    const int64_t nb = cols / 32;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < nb; ++j) {
            const float *x = w + r * cols + j * 32;
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) amax = fabsf(x[i]) > amax ? fabsf(x[i]) : amax;
            const float d = amax / 127.0f;
            const float id = d != 0.0f ? 1.0f / d : 0.0f;
            for (int i = 0; i < 32; ++i) {
                const float v = x[i] * id;
                q[r * cols + j * 32 + i] = (int8_t)roundf(v);
            }
            d16[r * nb + j] = f32_to_f16(d);
        }
}

/* The weights the codes stand for, fp32 (exact: an 11-bit scale times an
 * 8-bit code). */
void orc_dequantize_q8_0(const int8_t *q, const uint16_t *d16, int64_t rows, int64_t cols, float *w) {
    const int64_t nb = cols / 32;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            w[r * cols + c] = (float)(f16_to_double(d16[r * nb + c / 32]) * (double)q[r * cols + c]);
}

/* Q4_0 quantisation of a row-major [rows, cols] fp32 matrix, cols a multiple
 * of 32 (the Q4_0 format of the report's Q4_0 column, with ggml's rule for
 * the scale -- the report's own quantiser picks it by Lloyd iterations, which
 * the page does not spell out): per block of 32 consecutive weights of a row,
 * m = the weight of largest magnitude (the first on ties), d = m / -8 in fp32,
 * stored as binary16; codes q = min(15, trunc(w * (1 / d) + 8.5)) in fp32
 * (all 8 when d = 0), so m itself gets code 0.  The weight a code stands for
 * is f16(d) * (q - 8).  Storage: 16 bytes per block, byte j holding the code
 * of weight j in its low four bits and that of weight j + 16 in its high
 * four: codes go to q[rows, cols / 2] (uint8), block scales to
 * d16[rows, cols / 32] (binary16 bits). */
void orc_quantize_q4_0(const float *w, int64_t rows, int64_t cols, uint8_t *q, uint16_t *d16) {
    const int64_t nb = cols / 32;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < nb; ++j) {
            const float *x = w + r * cols + j * 32;
            float amax = 0.0f, m = 0.0f;
            for (int i = 0; i < 32; ++i)
                if (fabsf(x[i]) > amax) { amax = fabsf(x[i]); m = x[i]; }
            const float d = m / -8.0f;
            const float id = d != 0.0f ? 1.0f / d : 0.0f;
            int code[32];
            for (int i = 0; i < 32; ++i) {
                const int t = (int)(x[i] * id + 8.5f);   /* truncation toward zero; the value lies in [0.5, 16.5] */
                code[i] = t < 15 ? t : 15;
            }
            uint8_t *qb = q + r * (cols / 2) + j * 16;
            for (int i = 0; i < 16; ++i) qb[i] = (uint8_t)(code[i] | (code[i + 16] << 4));
            d16[r * nb + j] = f32_to_f16(d);
        }
}

/* The weights Q4_0 codes stand for, fp32 (exact: an 11-bit scale times a
 * small integer). */
void orc_dequantize_q4_0(const uint8_t *q, const uint16_t *d16, int64_t rows, int64_t cols, float *w) {
    const int64_t nb = cols / 32;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            const int64_t j = c / 32, i = c % 32;
            const uint8_t byte = q[r * (cols / 2) + j * 16 + (i % 16)];
            const int code = i < 16 ? (byte & 15) : (byte >> 4);
            w[r * cols + c] = (float)(f16_to_double(d16[r * nb + j]) * (double)(code - 8));
        }
}

/* ------------------------------------------------------------------------ */
/* centroid-routed LM head ([G4] sec. 3, "Centroid / ordered-embeddings LM  */
/* head", steps 1-5)                                                         */
/* ------------------------------------------------------------------------ */

/* The full-vocabulary logit row of the centroid-routed head for one hidden
 * state h [d_t]:
 *   1. centroid logits c_j = centroids[j] . h, j < n_c (centroids [n_c, d_t]);
 *   2. the top_k centroids by c_j (reading: ties go to the lower centroid id;
 *      the chosen set is all that matters, not its order);
 *   3. token_ordering [V] int32 read as n_c consecutive lists of
 *      vsc = V / n_c token ids, list j belonging to centroid j (reading of
 *      the [vsc, n_c] view: vsc is the contiguous dimension, get_rows takes
 *      one list per chosen centroid); the chosen lists are the candidates;
 *   4. each candidate t gets the dense head's logit tok_embd[t] . h, with the
 *      same final softcap (reading: the cap applies to the candidates'
 *      logits, before the scatter);
 *   5. every other entry of the row holds -1e30.
 * cgap (optional): the chosen set's margin, the top_k-th largest centroid
 * logit minus the next one, over the population standard deviation of the
 * centroid logits (+inf when top_k = n_c or that deviation is 0).
 * cl (optional): the centroid logits [n_c].
 * Returns 0, or -1 for invalid sizes or an ordering entry outside [0, V). */
int orc_centroid_head(const orc_model *m, const void *centroids, const int32_t *ordering,
                      const void *tok_embd, const double *h, double *z, double *cgap, double *cl_out) {
    const int nc = m->n_centroids, kc = m->centroid_top_k, V = m->vocab, d_t = m->d_t, bf = m->wbf16;
    if (nc <= 0 || kc <= 0 || kc > nc || V % nc != 0) return -1;
    const int vsc = V / nc;
    double *cl = malloc(sizeof(double) * (size_t)nc);
    char *taken = calloc((size_t)nc, 1);
    orc_matvec(centroids, nc, d_t, bf, h, cl);
    for (int v = 0; v < V; ++v) z[v] = -1e30;
    int rc = 0;
    double last = INFINITY;
    for (int r = 0; r < kc && rc == 0; ++r) {
        /* the next centroid: largest remaining logit, lowest id on ties, NaN last */
        int best = -1;
        for (int j = 0; j < nc; ++j) {
            if (taken[j]) continue;
            if (best < 0 || (isnan(cl[best]) && !isnan(cl[j])) || cl[j] > cl[best]) best = j;
        }
        taken[best] = 1;
        last = cl[best];
        for (int i = 0; i < vsc; ++i) {
            const int32_t tk = ordering[(size_t)best * vsc + i];
            if (tk < 0 || tk >= V) { rc = -1; break; }
            double acc = 0.0;
            for (int c = 0; c < d_t; ++c) acc += elem(tok_embd, (int64_t)tk * d_t + c, bf) * h[c];
            if (m->logit_softcap > 0.0) acc = m->logit_softcap * tanh(acc / m->logit_softcap);
            z[tk] = acc;
        }
    }
    if (cgap) {
        double next = -INFINITY, mean = 0.0, var = 0.0;
        int cnt = 0;
        for (int j = 0; j < nc; ++j) {
            if (!taken[j] && cl[j] > next) next = cl[j];
            if (!isnan(cl[j])) { mean += cl[j]; ++cnt; }
        }
        mean = cnt ? mean / cnt : 0.0;
        for (int j = 0; j < nc; ++j) if (!isnan(cl[j])) var += (cl[j] - mean) * (cl[j] - mean);
        const double sd = cnt ? sqrt(var / cnt) : 0.0;
        *cgap = kc < nc && sd > 0.0 ? (last - next) / sd : INFINITY;
    }
    if (cl_out) memcpy(cl_out, cl, sizeof(double) * (size_t)nc);
    free(cl);
    free(taken);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* the draft step ([G4] sec. 4, [NX] Requirements)                           */
/* ------------------------------------------------------------------------ */

#define TT(i) (t[(i)])
#define BT(blk, i) (t[T_GLOBAL_COUNT + (blk) * B_COUNT + (i)])

/* One draft step for B independent sequences.
 *   tok[b]      token consumed at this step (the last token for step 0, the
 *               previous step's draft afterwards)
 *   h_prev[b]   hidden state carried from the target (step 0) or from the
 *               previous step's post-projection, [B, d_t]
 *   step        k: RoPE position of the query is kv_len[b] + k
 * Outputs h_next [B, d_t] (the next step's h_prev), logits [B, V] and, for a
 * centroid-routed head, cgap [B] (optional; see orc_centroid_head). */
int orc_draft_step(const orc_model *m, const void *const *t, const int32_t *block_view,
                   const orc_view *views, int n_views, int B, const int32_t *kv_len, int step,
                   const int32_t *tok, const double *h_prev, double *h_next, double *logits, double *cgap) {
    const int d_t = m->d_t, d_a = m->d_a, hd = m->head_dim, Hq = m->n_q_heads, Hkv = m->n_kv_heads;
    const int qw = Hq * hd, F = m->d_ff, V = m->vocab, bf = m->wbf16;
    const int grp = Hq / Hkv;
    double *e = malloc(sizeof(double) * d_t), *u = malloc(sizeof(double) * 2 * d_t);
    double *x = malloc(sizeof(double) * d_a), *a = malloc(sizeof(double) * d_a);
    double *q = malloc(sizeof(double) * qw), *o = malloc(sizeof(double) * qw);
    double *y = malloc(sizeof(double) * (d_a > d_t ? d_a : d_t));
    double *yn = malloc(sizeof(double) * d_a);
    double *gt = malloc(sizeof(double) * F), *up = malloc(sizeof(double) * F);
    for (int b = 0; b < B; ++b) {
        int32_t tk = tok[b];
        if (tk < 0 || tk >= V) { free(e); free(u); free(x); free(a); free(q); free(o); free(y); free(yn); free(gt); free(up); return -1; }
        /* token embedding from the tied table, scaled ([G4] sec. 4 item 2) */
        for (int c = 0; c < d_t; ++c) e[c] = elem(TT(T_TOK_EMBD), (int64_t)tk * d_t + c, bf) * m->emb_scale;
        /* separate norms of the embedding and of h_prev, then concat ([NX] Requirements) */
        orc_rmsnorm(e, d_t, (const float *)TT(T_NORM_E), m->rms_eps, u);
        orc_rmsnorm(h_prev + (size_t)b * d_t, d_t, (const float *)TT(T_NORM_H), m->rms_eps, u + d_t);
        /* pre-projection 2 d_t -> d_a ([G4] sec. 4 item 3) */
        orc_matvec(TT(T_W_PRE), d_a, 2 * d_t, bf, u, x);
        for (int l = 0; l < m->n_blocks; ++l) {
            const orc_view *vw = &views[block_view[l]];
            /* RMSNorm -> Q proj -> Q-norm -> RoPE ([G4] sec. 4 item 4) */
            orc_rmsnorm(x, d_a, (const float *)BT(l, B_ATTN_NORM), m->rms_eps, a);
            orc_matvec(BT(l, B_W_Q), qw, d_a, bf, a, q);
            for (int h = 0; h < Hq; ++h) {
                double tmp[1024];
                double *qh = q + (size_t)h * hd;
                orc_rmsnorm(qh, hd, (const float *)BT(l, B_Q_NORM), m->rms_eps, tmp);
                memcpy(qh, tmp, sizeof(double) * hd);
                orc_rope_neox(qh, hd, (int64_t)kv_len[b] + step, vw->rope_theta);
            }
            /* cross-attention into the target KV, no draft KV ([G4] sec. 5, [FN] delta 6) */
            for (int h = 0; h < Hq; ++h)
                orc_attend_head(q + (size_t)h * hd, vw, b, h / grp, hd, kv_len[b], m->attn_scale, bf,
                                o + (size_t)h * hd);
            /* o-projection, post-attention norm, residual ([G4] sec. 4 item 4) */
            orc_matvec(BT(l, B_W_O), d_a, qw, bf, o, y);
            orc_rmsnorm(y, d_a, (const float *)BT(l, B_POST_ATTN_NORM), m->rms_eps, yn);
            for (int c = 0; c < d_a; ++c) x[c] += yn[c];
            /* pre-FFN norm, GeGLU, post-FFN norm, residual */
            orc_rmsnorm(x, d_a, (const float *)BT(l, B_PRE_FFN_NORM), m->rms_eps, a);
            orc_matvec(BT(l, B_W_GATE), F, d_a, bf, a, gt);
            orc_matvec(BT(l, B_W_UP), F, d_a, bf, a, up);
            for (int f = 0; f < F; ++f) gt[f] = orc_gelu_tanh(gt[f]) * up[f];
            orc_matvec(BT(l, B_W_DOWN), d_a, F, bf, gt, y);
            orc_rmsnorm(y, d_a, (const float *)BT(l, B_POST_FFN_NORM), m->rms_eps, yn);
            for (int c = 0; c < d_a; ++c) x[c] += yn[c];
        }
        /* final norm -> post-projection = next h_prev ([G4] sec. 4 item 5) */
        orc_rmsnorm(x, d_a, (const float *)TT(T_FINAL_NORM), m->rms_eps, a);
        double *hn = h_next + (size_t)b * d_t;
        orc_matvec(TT(T_W_POST), d_t, d_a, bf, a, hn);
        double *z = logits + (size_t)b * V;
        if (m->n_centroids > 0) {
            /* centroid-routed head ([G4] sec. 3) */
            if (orc_centroid_head(m, TT(T_CENTROIDS), (const int32_t *)TT(T_ORDERING), TT(T_TOK_EMBD), hn, z,
                                  cgap ? cgap + b : NULL, NULL)) {
                free(e); free(u); free(x); free(a); free(q); free(o); free(y); free(yn); free(gt); free(up);
                return -1;
            }
        } else {
            /* tied dense LM head, optional final-logit softcap ([G4] sec. 4 items 6-7) */
            orc_matvec(TT(T_TOK_EMBD), V, d_t, bf, hn, z);
            if (m->logit_softcap > 0.0)
                for (int v = 0; v < V; ++v) z[v] = m->logit_softcap * tanh(z[v] / m->logit_softcap);
        }
    }
    (void)n_views;
    free(e); free(u); free(x); free(a); free(q); free(o); free(y); free(yn); free(gt); free(up);
    return 0;
}

/* Confidence of a draft step ("MTP decoding (--mtp)", "Stopping early when the
 * head is unsure": the draft loop's confidence in the token it proposes, the
 * probability of the top candidate): the softmax probability of the largest
 * logit, 1 / sum_v exp(z_v - z_max), over the step's logits z (after the
 * softcap), NaN entries left out. */
double orc_top1_prob(const double *z, int64_t n) {
    double zm = -INFINITY;
    for (int64_t i = 0; i < n; ++i) if (!isnan(z[i]) && z[i] > zm) zm = z[i];
    if (!(zm > -INFINITY)) return 0.0;
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i) if (!isnan(z[i])) s += exp(z[i] - zm);
    return 1.0 / s;
}

/* N chained draft steps with the token chosen on "device" each step ([G4]
 * sec. 4 item 8; [FN] the fused chain: argmax -> embed -> h chain).
 *   sp == NULL or sp->temp <= 0: greedy (argmax).  Otherwise the token of
 *   step k is drawn from sample_dist(z_k) with penalty set hist[b] u
 *   drafts[b][0..k-1] and the uniform of (seq0 + b, k, purpose 0): seq0 is
 *   the batch index of row 0 when the rows are a slice of a larger batch.
 * Outputs drafts [B, N], h_last [B, d_t] (optional), logits [B, N, V]
 * (optional), margin [B, N] (optional: top1 - top2 logit gap of each greedy
 * step, or the sampling decision's relative margin), conf [B, N] (optional:
 * the step's confidence, see orc_top1_prob), cgap [B, N] (optional: the
 * centroid-routed head's set margin, see orc_centroid_head). */
int orc_draft_block(const orc_model *m, const void *const *t, const int32_t *block_view,
                    const orc_view *views, int n_views, int B, int N, const int32_t *kv_len,
                    const int32_t *last_tok, const float *h_prev, const orc_sample_params *sp,
                    uint64_t seed, uint64_t offset, int seq0, const int32_t *hist, int H,
                    const int32_t *force_tok, int32_t *drafts, double *h_last, double *logits,
                    double *margin, double *conf, double *cgap) {
    const int d_t = m->d_t, V = m->vocab;
    double *h = malloc(sizeof(double) * (size_t)B * d_t), *hn = malloc(sizeof(double) * (size_t)B * d_t);
    double *z = malloc(sizeof(double) * (size_t)B * V);
    int32_t *tok = malloc(sizeof(int32_t) * (size_t)B);
    int32_t *ids = malloc(sizeof(int32_t) * (size_t)V);
    float *wf = malloc(sizeof(float) * (size_t)V);
    int32_t *pen = malloc(sizeof(int32_t) * (size_t)(H + N + 1));
    double *cg = malloc(sizeof(double) * (size_t)B);
    int rc = 0;
    for (size_t i = 0; i < (size_t)B * d_t; ++i) h[i] = (double)h_prev[i];
    for (int b = 0; b < B; ++b) tok[b] = last_tok[b];
    const int sampling = sp && sp->temp > 0.0;
    for (int k = 0; k < N && rc == 0; ++k) {
        rc = orc_draft_step(m, t, block_view, views, n_views, B, kv_len, k, tok, h, hn, z, cg);
        if (rc) break;
        for (int b = 0; b < B; ++b) {
            const double *zb = z + (size_t)b * V;
            int32_t pick;
            double mg;
            if (!sampling) {
                pick = (int32_t)orc_argmax_f64(zb, V);
                double second = -INFINITY;
                for (int v = 0; v < V; ++v) if (v != pick && zb[v] > second) second = zb[v];
                mg = zb[pick] - second;
            } else {
                int np = 0;
                for (int j = 0; j < H; ++j) pen[np++] = hist[(size_t)b * H + j];
                for (int j = 0; j < k; ++j) pen[np++] = drafts[(size_t)b * N + j];
                float ws;
                double m1, m2;
                int n = orc_sample_dist_f32(zb, V, pen, np, sp, ids, wf, &ws, &m1);
                float u = (float)orc_uniform(seed, offset, (uint32_t)(seq0 + b), (uint32_t)k, 0u);
                pick = orc_pick_f32(ids, wf, n, ws, u, &m2);
                mg = m1 < m2 ? m1 : m2;
            }
            if (margin) margin[(size_t)b * N + k] = mg;
            if (conf) conf[(size_t)b * N + k] = orc_top1_prob(zb, V);
            if (cgap) cgap[(size_t)b * N + k] = m->n_centroids > 0 ? cg[b] : INFINITY;
            if (logits) memcpy(logits + ((size_t)b * N + k) * V, zb, sizeof(double) * (size_t)V);
            drafts[(size_t)b * N + k] = pick;
            tok[b] = force_tok ? force_tok[(size_t)b * N + k] : pick;
        }
        double *sw = h; h = hn; hn = sw;
    }
    if (h_last && rc == 0) memcpy(h_last, h, sizeof(double) * (size_t)B * d_t);
    free(h); free(hn); free(z); free(tok); free(ids); free(wf); free(pen); free(cg);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* the dense NextN drafter ([NX] "Requirements", "How it is wired", "The     */
/* catch-up runs on the accepted prefix"; [FN] "The two MTP lanes")          */
/* ------------------------------------------------------------------------ */

/* NextN tensor table: its own order (the assistant's table above is not
 * used).  One block at the backbone width d = d_t:
 *   tok_embd [V, d]   the table, also the (shared) LM head
 *   enorm, hnorm [d]  norms of the token embedding and of the hidden state
 *   eh_proj [d, 2d]   projection of [enorm(e); hnorm(h)]
 *   head_norm [d]     the shared head's norm
 *   attn_norm [d], w_qkv [(Hq + 2 Hkv) hd, d] (query rows, then key rows,
 *   then value rows), q_norm [hd], k_norm [hd], w_o [d, Hq hd],
 *   ffn_norm [d], w_gate, w_up [F, d], w_down [d, F] */
enum { NX_TOK_EMBD, NX_ENORM, NX_HNORM, NX_EH_PROJ, NX_HEAD_NORM, NX_ATTN_NORM, NX_W_QKV, NX_Q_NORM, NX_K_NORM,
       NX_W_O, NX_FFN_NORM, NX_W_GATE, NX_W_UP, NX_W_DOWN, NX_COUNT };

/* SiLU, the gate of the NextN block's feed-forward (SwiGLU) */
double orc_silu(double x) { return x / (1.0 + exp(-x)); }

/* A real number rounded once to bf16, nearest with ties to even; returns the
 * bit pattern.  The drafter stores its own keys and values in the weights'
 * type, so the oracle writes them rounded the same way. */
uint16_t orc_to_bf16(double x) {
    if (isnan(x)) return 0x7FC0;
    if (x == 0.0) return signbit(x) ? 0x8000 : 0x0000;
    int e;
    frexp(x, &e);                      /* |x| in [2^(e-1), 2^e) */
    int eu = e - 8;                    /* 8 significant bits: ulp 2^(e-8) */
    if (eu < -133) eu = -133;          /* below the normal range: bf16's subnormal spacing */
    const double r = rint(ldexp(x, -eu));   /* the default rounding mode: nearest, ties to even */
    const float y = (float)ldexp(r, eu);    /* exact in fp32 (or infinite past the range) */
    uint32_t u;
    memcpy(&u, &y, sizeof u);
    return (uint16_t)(u >> 16);
}

static void store_elem(const void *p, int64_t i, int bf16, double x) {
    if (bf16) ((uint16_t *)(uintptr_t)p)[i] = orc_to_bf16(x);
    else ((float *)(uintptr_t)p)[i] = (float)x;
}

#define NT(i) (t[(i)])

/* One position of the NextN block for sequence b of the drafter's KV `dkv`
 * (K and V [B][Hkv][cap][hd], position p in slot p).
 *   tk, hin  the token at position pos and the hidden state paired with it:
 *            the target's at the previous position (catch-up rows and the
 *            first draft step), the block's own output after that
 *   full 0   a catch-up row: its key and value are written at slot pos and
 *            nothing else is computed (nothing downstream reads the rest)
 *   full 1   a draft step: also the causal attention over positions
 *            [0, pos], the feed-forward and the head; hout [d] receives the
 *            block output (the next step's hidden state) and z [V] the logits
 * The block follows the NextN layout of [NX] "Requirements" (enorm, hnorm,
 * eh_proj, one attention + feed-forward block, the shared head with its
 * norm); the pre-norm residual structure, per-head q/k norms, NeoX RoPE at
 * the row's position and SwiGLU are the readings listed in the design notes. */
static int nextn_row(const orc_model *m, const void *const *t, const orc_view *dkv, int b, int32_t tk,
                     const double *hin, int64_t pos, int full, double *hout, double *z) {
    const int d = m->d_t, hd = m->head_dim, Hq = m->n_q_heads, Hkv = m->n_kv_heads, F = m->d_ff, V = m->vocab;
    const int bf = m->wbf16, kvb = m->kv_bf16, grp = Hq / Hkv, qkv = (Hq + 2 * Hkv) * hd;
    if (tk < 0 || tk >= V || pos < 0 || pos >= dkv->cap) return -1;
    double *e = malloc(sizeof(double) * d), *u = malloc(sizeof(double) * 2 * d);
    double *x = malloc(sizeof(double) * d), *a = malloc(sizeof(double) * d), *y = malloc(sizeof(double) * d);
    double *q = malloc(sizeof(double) * qkv), *o = malloc(sizeof(double) * Hq * hd);
    double *gt = malloc(sizeof(double) * F), *up = malloc(sizeof(double) * F), *tmp = malloc(sizeof(double) * hd);
    /* [enorm(e); hnorm(h)] -> eh_proj ([NX] Requirements) */
    for (int c = 0; c < d; ++c) e[c] = elem(NT(NX_TOK_EMBD), (int64_t)tk * d + c, bf) * m->emb_scale;
    orc_rmsnorm(e, d, (const float *)NT(NX_ENORM), m->rms_eps, u);
    orc_rmsnorm(hin, d, (const float *)NT(NX_HNORM), m->rms_eps, u + d);
    orc_matvec(NT(NX_EH_PROJ), d, 2 * d, bf, u, x);
    /* attention input norm, the fused query / key / value projection */
    orc_rmsnorm(x, d, (const float *)NT(NX_ATTN_NORM), m->rms_eps, a);
    orc_matvec(NT(NX_W_QKV), qkv, d, bf, a, q);
    /* keys: per-head norm, RoPE at pos; key and value stored at slot pos */
    for (int g = 0; g < Hkv; ++g) {
        double *kh = q + (size_t)(Hq + g) * hd, *vh = q + (size_t)(Hq + Hkv + g) * hd;
        orc_rmsnorm(kh, hd, (const float *)NT(NX_K_NORM), m->rms_eps, tmp);
        orc_rope_neox(tmp, hd, pos, dkv->rope_theta);
        const int64_t base = (int64_t)b * dkv->stride_b + (int64_t)g * dkv->stride_h + pos * dkv->stride_t;
        for (int c = 0; c < hd; ++c) {
            store_elem(dkv->k, base + c, kvb, tmp[c]);
            store_elem(dkv->v, base + c, kvb, vh[c]);
        }
    }
    if (full) {
        /* queries: per-head norm, RoPE at pos; attention over [0, pos] as stored */
        for (int h = 0; h < Hq; ++h) {
            double *qh = q + (size_t)h * hd;
            orc_rmsnorm(qh, hd, (const float *)NT(NX_Q_NORM), m->rms_eps, tmp);
            orc_rope_neox(tmp, hd, pos, dkv->rope_theta);
            orc_attend_head(tmp, dkv, b, h / grp, hd, (int)(pos + 1), m->attn_scale, kvb, o + (size_t)h * hd);
        }
        orc_matvec(NT(NX_W_O), d, Hq * hd, bf, o, y);
        for (int c = 0; c < d; ++c) x[c] += y[c];
        /* feed-forward: norm, SwiGLU, residual */
        orc_rmsnorm(x, d, (const float *)NT(NX_FFN_NORM), m->rms_eps, a);
        orc_matvec(NT(NX_W_GATE), F, d, bf, a, gt);
        orc_matvec(NT(NX_W_UP), F, d, bf, a, up);
        for (int f = 0; f < F; ++f) gt[f] = orc_silu(gt[f]) * up[f];
        orc_matvec(NT(NX_W_DOWN), d, F, bf, gt, y);
        for (int c = 0; c < d; ++c) x[c] += y[c];
        memcpy(hout, x, sizeof(double) * d);
        /* the shared head: its norm, then the tied table (optional softcap) */
        orc_rmsnorm(x, d, (const float *)NT(NX_HEAD_NORM), m->rms_eps, a);
        orc_matvec(NT(NX_TOK_EMBD), V, d, bf, a, z);
        if (m->logit_softcap > 0.0)
            for (int v = 0; v < V; ++v) z[v] = m->logit_softcap * tanh(z[v] / m->logit_softcap);
    }
    free(e); free(u); free(x); free(a); free(y); free(q); free(o); free(gt); free(up); free(tmp);
    return 0;
}

/* One drafting call of the NextN drafter for B sequences ([NX] "How it is
 * wired": draft from the head, and "The catch-up runs on the accepted
 * prefix": the draft context re-runs the block on the accepted rows only).
 * The drafter's KV holds kv_len[b] rows (positions 0..kv_len[b]-1).
 *   catch-up: rows j < n_cu[b] (0 <= n_cu[b] <= M) consume cu_tok[b, j] with
 *             the target's hidden state cu_h[b, j] and write their key and
 *             value at position kv_len[b] + j;
 *   drafts:   step k consumes tok_k (last_tok[b] for k = 0, then the previous
 *             draft, or force_tok[b, k-1] when given) with h_k (h_prev[b], the
 *             target's, for k = 0; the previous step's block output after) at
 *             position kv_len[b] + n_cu[b] + k, writes its key and value there
 *             and drafts argmax z (lowest index on ties).
 * Outputs: drafts [B, N]; optional h_last [B, d] (the last step's block
 * output), logits [B, N, V], margin [B, N] (top-1 minus top-2 logit), conf
 * [B, N] (orc_top1_prob).  The rows written beyond the accepted ones (steps
 * k >= 1) are the drafter's own guesses; the next call's catch-up overwrites
 * the ones that get accepted. */
int orc_nextn_draft(const orc_model *m, const void *const *t, const orc_view *dkv, int B, int N,
                    const int32_t *kv_len, int M, const int32_t *n_cu, const int32_t *cu_tok, const float *cu_h,
                    const int32_t *last_tok, const float *h_prev, const int32_t *force_tok, int32_t *drafts,
                    double *h_last, double *logits, double *margin, double *conf) {
    const int d = m->d_t, V = m->vocab;
    double *h = malloc(sizeof(double) * d), *hn = malloc(sizeof(double) * d), *z = malloc(sizeof(double) * V);
    int rc = 0;
    for (int b = 0; b < B && rc == 0; ++b) {
        const int nc = n_cu ? n_cu[b] : 0;
        if (nc < 0 || nc > M || kv_len[b] < 0 || (int64_t)kv_len[b] + nc + N > dkv->cap) { rc = -1; break; }
        for (int j = 0; j < nc && rc == 0; ++j) {
            for (int c = 0; c < d; ++c) h[c] = (double)cu_h[((size_t)b * M + j) * d + c];
            rc = nextn_row(m, t, dkv, b, cu_tok[(size_t)b * M + j], h, (int64_t)kv_len[b] + j, 0, NULL, NULL);
        }
        for (int c = 0; c < d; ++c) h[c] = (double)h_prev[(size_t)b * d + c];
        int32_t tok = last_tok[b];
        for (int k = 0; k < N && rc == 0; ++k) {
            rc = nextn_row(m, t, dkv, b, tok, h, (int64_t)kv_len[b] + nc + k, 1, hn, z);
            if (rc) break;
            const int32_t pick = (int32_t)orc_argmax_f64(z, V);
            double second = -INFINITY;
            for (int v = 0; v < V; ++v) if (v != pick && z[v] > second) second = z[v];
            if (margin) margin[(size_t)b * N + k] = z[pick] - second;
            if (conf) conf[(size_t)b * N + k] = orc_top1_prob(z, V);
            if (logits) memcpy(logits + ((size_t)b * N + k) * V, z, sizeof(double) * (size_t)V);
            drafts[(size_t)b * N + k] = pick;
            tok = force_tok ? force_tok[(size_t)b * N + k] : pick;
            double *sw = h; h = hn; hn = sw;
        }
        if (h_last && rc == 0) memcpy(h_last + (size_t)b * d, h, sizeof(double) * d);
    }
    free(h); free(hn); free(z);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* verify-accept                                                             */
/* ------------------------------------------------------------------------ */

/* Greedy verify ([NX] How it is wired): t_i = argmax of target row i (rows
 * 0..N); n_accept = the largest k with drafts[j] == t_j for all j < k; the
 * emitted tokens are drafts[0..k-1] followed by the bonus t_k, padded with -1.
 * logits [B, 1+N, V] (bf16 bits or fp32). */
void orc_verify_greedy(const void *logits, int bf16, int B, int N, int V, const int32_t *drafts,
                       int32_t *out_tokens, int32_t *out_n_accept) {
#pragma omp parallel for schedule(static)
    for (int b = 0; b < B; ++b) {
        int k = 0;
        int32_t *ot = out_tokens + (size_t)b * (N + 1);
        for (int i = 0; i <= N; ++i) ot[i] = -1;
        for (;;) {
            const int64_t row = ((int64_t)b * (N + 1) + k) * V;
            int32_t tk = (int32_t)argmax_stored((const char *)logits + row * (bf16 ? 2 : 4), V, bf16);
            if (k < N && drafts[(size_t)b * N + k] == tk) { ot[k] = tk; ++k; continue; }
            ot[k] = tk;
            break;
        }
        out_n_accept[b] = k;
    }
}

/* Exact speculative sampling at temp > 0 ([SP] item 4).
 * Row i (0..N-1): p_i = sample_dist(target row i), q_i = sample_dist(draft row
 * i), both with penalty set hist[b] u drafts[b][0..i-1].  With x = d_i,
 * p_i(x) = w_x / W_p and q_i(x) = w'_x / W_q (0 when x is not kept); x is
 * accepted iff u < p_i(x) / q_i(x) (fp32; q = 0 gives +inf, or NaN -> reject,
 * when p = 0 too), u of (b, i, purpose 1).  On the first rejection the emitted
 * token is drawn from r_j = max(p_j - q(id_j), 0) over p's kept candidates in
 * p's order (from p itself when sum r = 0) with the uniform of (b, i, purpose
 * 2) and the window ends.  If every draft is accepted, the bonus token is
 * drawn from p_N (penalty set hist u d_0..d_{N-1}) with the uniform of
 * (b, N, purpose 3).  Sampler arithmetic is fp32 as in orc_sample_dist_f32.
 * margin[b] (optional): smallest relative distance of any decision taken for
 * sequence b to its threshold (diagnostic). */
void orc_verify_sample(const void *tgt, const void *dft, int bf16, int B, int N, int V,
                       const int32_t *drafts, const int32_t *hist, int H,
                       const orc_sample_params *sp, uint64_t seed, uint64_t offset,
                       int32_t *out_tokens, int32_t *out_n_accept, double *margin) {
#pragma omp parallel
    {
        double *z = malloc(sizeof(double) * (size_t)V);
        int32_t *pid = malloc(sizeof(int32_t) * (size_t)V), *qid = malloc(sizeof(int32_t) * (size_t)V);
        float *pw = malloc(sizeof(float) * (size_t)V), *qw = malloc(sizeof(float) * (size_t)V);
        float *r = malloc(sizeof(float) * (size_t)V);
        int32_t *pen = malloc(sizeof(int32_t) * (size_t)(H + N + 1));
#pragma omp for schedule(dynamic, 64)
        for (int b = 0; b < B; ++b) {
            int32_t *ot = out_tokens + (size_t)b * (N + 1);
            for (int i = 0; i <= N; ++i) ot[i] = -1;
            double mg = INFINITY, m1;
            int np = 0;
            for (int j = 0; j < H; ++j) pen[np++] = hist[(size_t)b * H + j];
            int i;
            for (i = 0; i < N; ++i) {
                const int64_t trow = ((int64_t)b * (N + 1) + i) * V;
                const int64_t drow = ((int64_t)b * N + i) * V;
                for (int v = 0; v < V; ++v) z[v] = elem(tgt, trow + v, bf16);
                float ps, qs;
                int np_ = orc_sample_dist_f32(z, V, pen, np, sp, pid, pw, &ps, &m1);
                if (m1 < mg) mg = m1;
                for (int v = 0; v < V; ++v) z[v] = elem(dft, drow + v, bf16);
                int nq = orc_sample_dist_f32(z, V, pen, np, sp, qid, qw, &qs, &m1);
                if (m1 < mg) mg = m1;
                const int32_t x = drafts[(size_t)b * N + i];
                float px = 0.0f, qx = 0.0f;
                for (int j = 0; j < np_; ++j) if (pid[j] == x) { px = pw[j] / ps; break; }
                for (int j = 0; j < nq; ++j) if (qid[j] == x) { qx = qw[j] / qs; break; }
                const float u = (float)orc_uniform(seed, offset, (uint32_t)b, (uint32_t)i, 1u);
                const float ratio = px / qx;
                if (!isnan(ratio) && isfinite(ratio)) {
                    double d = fabs((double)u - (double)ratio);
                    if (d > 0.0 && d < mg) mg = d;
                }
                if (u < ratio) { ot[i] = x; pen[np++] = x; continue; }
                float R = 0.0f;
                for (int j = 0; j < np_; ++j) {
                    const float pj = pw[j] / ps;
                    float qj = 0.0f;
                    for (int jj = 0; jj < nq; ++jj) if (qid[jj] == pid[j]) { qj = qw[jj] / qs; break; }
                    r[j] = pj > qj ? pj - qj : 0.0f;
                    R += r[j];
                }
                const float u2 = (float)orc_uniform(seed, offset, (uint32_t)b, (uint32_t)i, 2u);
                if (R > 0.0f) ot[i] = orc_pick_f32(pid, r, np_, R, u2, &m1);
                else ot[i] = orc_pick_f32(pid, pw, np_, ps, u2, &m1);
                if (m1 < mg) mg = m1;
                break;
            }
            if (i == N) {
                const int64_t trow = ((int64_t)b * (N + 1) + N) * V;
                for (int v = 0; v < V; ++v) z[v] = elem(tgt, trow + v, bf16);
                float ps;
                int np_ = orc_sample_dist_f32(z, V, pen, np, sp, pid, pw, &ps, &m1);
                if (m1 < mg) mg = m1;
                const float u3 = (float)orc_uniform(seed, offset, (uint32_t)b, (uint32_t)N, 3u);
                ot[N] = orc_pick_f32(pid, pw, np_, ps, u3, &m1);
                if (m1 < mg) mg = m1;
            }
            out_n_accept[b] = i;
            if (margin) margin[b] = mg;
        }
        free(z); free(pid); free(qid); free(pw); free(qw); free(r); free(pen);
    }
}

/* Draws of a sampling drafter ([SP] item 4: the drafted token of row i is a
 * draw from q_i = sample_dist(draft row i)).  For sequence b and row i in
 * order: q_i = sample_dist(dft row (b, i)) with penalty set hist[b] u
 * drafts[b][0..i-1], and drafts[b][i] = the inverse-CDF pick of q_i with the
 * uniform of (b, i, purpose 0).  dft [B, N, V] (bf16 bits or fp32); hist
 * [B, H]; drafts [B, N] out; margin[b] (optional) the smallest relative
 * distance of any of the sequence's decisions to its threshold. */
void orc_sample_drafts(const void *dft, int bf16, int B, int N, int V, const int32_t *hist, int H,
                       const orc_sample_params *sp, uint64_t seed, uint64_t offset, int32_t *drafts,
                       double *margin) {
#pragma omp parallel
    {
        double *z = malloc(sizeof(double) * (size_t)V);
        int32_t *ids = malloc(sizeof(int32_t) * (size_t)V);
        float *w = malloc(sizeof(float) * (size_t)V);
        int32_t *pen = malloc(sizeof(int32_t) * (size_t)(H + N + 1));
#pragma omp for schedule(dynamic, 1)
        for (int b = 0; b < B; ++b) {
            double mg = INFINITY, m1, m2;
            int np = 0;
            for (int j = 0; j < H; ++j) pen[np++] = hist[(size_t)b * H + j];
            for (int i = 0; i < N; ++i) {
                const int64_t row = ((int64_t)b * N + i) * V;
                for (int v = 0; v < V; ++v) z[v] = elem(dft, row + v, bf16);
                float ws;
                const int n = orc_sample_dist_f32(z, V, pen, np, sp, ids, w, &ws, &m1);
                const float u = (float)orc_uniform(seed, offset, (uint32_t)b, (uint32_t)i, 0u);
                const int32_t d = orc_pick_f32(ids, w, n, ws, u, &m2);
                if (m1 < mg) mg = m1;
                if (m2 < mg) mg = m2;
                drafts[(size_t)b * N + i] = d;
                pen[np++] = d;
            }
            if (margin) margin[b] = mg;
        }
        free(z); free(ids); free(w); free(pen);
    }
}

void orc_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
