/*
 * smoe_oracle.c -- CPU oracle for the routed Mixture-of-Experts layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library; it defines its own layer struct and its own bf16 and Q4
 * decoding from the written definitions below.
 *
 * What it computes is the plain definition of one routed-MoE layer, per
 * token, in fp64 (every dot product and every intermediate is a double):
 *
 *   0. optional RMSNorm of the residual r: xn = bf16(r / sqrt(mean(r^2) + eps) * gain)
 *      ("Optimizations" page, "The Dense Ceiling -- GPU-Resident Epilogue":
 *      residual-add, RMSNorm and router gate run between layers)
 *   1. exact router gate on the true hidden state: l_e = sum_d Wr[e][d] * xn[d]
 *      ("Optimizations", "Routing Is Exact -- Prompt and Generation Alike";
 *      "System Overview", "What Happens at Each Generated Token Step")
 *   2. top-k experts by logit, descending; ties go to the lower expert id.
 *      The decision is taken on the logits rounded to fp32, the precision of
 *      the pages' own gate (fp32 FMA lanes, "Optimizations", "The NEON
 *      Dense Path").
 *   3. mixing weights: p = softmax(l) over all experts; with norm_topk_prob
 *      w_i = p[idx_i] / sum_j p[idx_j], otherwise w_i = p[idx_i]  (Qwen3's
 *      definition, named by "Routing Is Exact").
 *   4. SMOE-Q4 expert FFN, gate and up in one pass, SiLU(gate)*up, then down
 *      ("Optimizations", "Coalesced GPU Kernels -- Expert FFN and Dense
 *      Matvec"; "System Overview", the Metal Kernel row of the per-token
 *      table).  Weights are the stored quantised values, taken as exact:
 *      w = scale * q + bias, q a 4-bit unsigned code, one bf16 scale and one
 *      bf16 bias per group of 64 along the input dimension.
 *   5. weighted sum into the residual, in rank order: y = r + sum_i w_i * o_i
 *      (the same table row: "weighted-summed into the residual").
 *
 * The prefill chunk path ("Optimizations", "Prefill Reads Each Expert Once,
 * Not Once Per Token": chunks of up to 64 tokens, each layer's routed experts
 * deduplicated into a union read once per chunk) builds the union and the
 * per-expert token buckets by brute force, evaluates each expert for the
 * tokens of its bucket and sums each token's outputs in rank order, so that
 * it is bit-identical to the per-token path.
 *
 * Q4 storage (fixed by this project, since the pages leave it open):
 *   codes: row-major [rows][cols/2] bytes; element 2j is the low nibble of
 *          byte j, element 2j+1 the high nibble;
 *   (SMOE-Q2, the pages' 2-bit vault -- "Optimizations", "Q2 Vaults -- the
 *   Next 2x, Twice Over"; "System Overview", the "SMOE-Q2/Q4 fused dequant"
 *   kernel: the same groups, scales and biases with 2-bit codes,
 *   [rows][cols/4] bytes, element 4j+k in bits 2k..2k+1 of byte j; a layer
 *   says which with code_bits, 4 or 2;)
 *   scale, bias: bf16 [rows][cols/64];
 *   per layer the experts are contiguous: gate and up [E][F][D], down [E][D][F]
 *   (rows x input columns); router bf16 [E][D].
 *
 * Built with -ffp-contract=off so that no multiply-add is fused and the
 * results are the same on every host.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct orc_layer {
    int d_model;
    int n_experts;
    int top_k;
    int ffn_dim;
    int group_size;
    int norm_topk_prob;
    double rms_eps;
    const uint16_t *rms_gain; /* [D] bf16, NULL = no RMSNorm */
    const uint16_t *router_w; /* [E][D] bf16 */
    const uint8_t *gate_q;    /* [E][F][D/2] */
    const uint16_t *gate_s;   /* [E][F][D/G] bf16 */
    const uint16_t *gate_b;
    const uint8_t *up_q;
    const uint16_t *up_s;
    const uint16_t *up_b;
    const uint8_t *down_q;    /* [E][D][F/2] */
    const uint16_t *down_s;   /* [E][D][F/G] */
    const uint16_t *down_b;
    int code_bits;            /* 4 (SMOE-Q4) or 2 (SMOE-Q2); 0 reads as 4 */
} orc_layer;

/* ---- bf16 <-> double --------------------------------------------------- */

/* A bf16 value is the upper half of an IEEE binary32. */
double orc_bf16_to_f64(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 (8 significant bits, binary32 exponent
 * range), ties to even, in one rounding step. */
uint16_t orc_f64_to_bf16(double v)
{
    if (isnan(v))
        return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    double q;
    if (a < 0x1p-126) {
        /* subnormal range: multiples of 2^-133 */
        q = nearbyint(a * 0x1p133) * 0x1p-133;
    } else {
        int e;
        double m = frexp(a, &e);          /* a = m * 2^e, m in [0.5, 1) */
        q = ldexp(nearbyint(ldexp(m, 8)), e - 8);
    }
    if (q > 0x1.FEp127) /* largest finite bf16 */
        return sign | 0x7F80;
    float f = (float)q; /* exact: q has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)((u >> 16) & 0x7FFF);
}

/* ---- Q4 dequantisation -------------------------------------------------- */

/* Weight (row, col) of a Q4 matrix with `cols` input columns. */
static double q4_weight(const uint8_t *q, const uint16_t *s, const uint16_t *b,
                        long row, long cols, long group, long col)
{
    uint8_t byte = q[row * (cols / 2) + col / 2];
    int code = (col & 1) ? (byte >> 4) : (byte & 0x0F);
    long gi = row * (cols / group) + col / group;
    return orc_bf16_to_f64(s[gi]) * (double)code + orc_bf16_to_f64(b[gi]);
}

double orc_q4_weight(const uint8_t *q, const uint16_t *s, const uint16_t *b,
                     long row, long cols, long group, long col)
{
    return q4_weight(q, s, b, row, cols, group, col);
}

/* Weight (row, col) of a Q2 matrix: code = bits 2k..2k+1 of byte col/4, k = col % 4. */
static double q2_weight(const uint8_t *q, const uint16_t *s, const uint16_t *b,
                        long row, long cols, long group, long col)
{
    uint8_t byte = q[row * (cols / 4) + col / 4];
    int code = (byte >> (2 * (col & 3))) & 0x03;
    long gi = row * (cols / group) + col / group;
    return orc_bf16_to_f64(s[gi]) * (double)code + orc_bf16_to_f64(b[gi]);
}

double orc_q2_weight(const uint8_t *q, const uint16_t *s, const uint16_t *b,
                     long row, long cols, long group, long col)
{
    return q2_weight(q, s, b, row, cols, group, col);
}

static double code_weight(int bits, const uint8_t *q, const uint16_t *s, const uint16_t *b,
                          long row, long cols, long group, long col)
{
    return bits == 2 ? q2_weight(q, s, b, row, cols, group, col)
                     : q4_weight(q, s, b, row, cols, group, col);
}

/* ---- step 0: RMSNorm ----------------------------------------------------- */

void orc_rmsnorm(const orc_layer *L, const uint16_t *r, uint16_t *xn)
{
    int D = L->d_model;
    if (!L->rms_gain) {
        memcpy(xn, r, sizeof(uint16_t) * (size_t)D);
        return;
    }
    double ss = 0.0;
    for (int d = 0; d < D; ++d) {
        double v = orc_bf16_to_f64(r[d]);
        ss += v * v;
    }
    double inv = 1.0 / sqrt(ss / (double)D + L->rms_eps);
    for (int d = 0; d < D; ++d)
        xn[d] = orc_f64_to_bf16(orc_bf16_to_f64(r[d]) * inv * orc_bf16_to_f64(L->rms_gain[d]));
}

/* ---- step 1: router gate ------------------------------------------------- */

void orc_router_logits(const orc_layer *L, const uint16_t *xn, double *logits)
{
    int D = L->d_model, E = L->n_experts;
    for (int e = 0; e < E; ++e) {
        double acc = 0.0;
        const uint16_t *w = L->router_w + (size_t)e * D;
        for (int d = 0; d < D; ++d)
            acc += orc_bf16_to_f64(w[d]) * orc_bf16_to_f64(xn[d]);
        logits[e] = acc;
    }
}

/* ---- step 2: top-k -------------------------------------------------------- */

/* Selection by (fp32 logit descending, expert id ascending), i.e. the first
 * k entries of a full sort on that key. */
void orc_topk(const double *logits, int E, int k, int32_t *idx)
{
    char *taken = (char *)calloc((size_t)E, 1);
    for (int i = 0; i < k; ++i) {
        int best = -1;
        float bv = 0.0f;
        for (int e = 0; e < E; ++e) {
            if (taken[e])
                continue;
            float v = (float)logits[e];
            if (best < 0 || v > bv) { /* strict: equal keeps the lower id */
                best = e;
                bv = v;
            }
        }
        taken[best] = 1;
        idx[i] = best;
    }
    free(taken);
}

/* ---- step 3: mixing weights ---------------------------------------------- */

void orc_mix_weights(const double *logits, int E, const int32_t *idx, int k,
                     int norm_topk_prob, double *w)
{
    double m = logits[0];
    for (int e = 1; e < E; ++e)
        if (logits[e] > m)
            m = logits[e];
    double *p = (double *)malloc(sizeof(double) * (size_t)E);
    double z = 0.0;
    for (int e = 0; e < E; ++e) {
        p[e] = exp(logits[e] - m);
        z += p[e];
    }
    for (int e = 0; e < E; ++e)
        p[e] /= z; /* softmax over all experts */
    double sel = 0.0;
    for (int i = 0; i < k; ++i)
        sel += p[idx[i]];
    for (int i = 0; i < k; ++i)
        w[i] = norm_topk_prob ? p[idx[i]] / sel : p[idx[i]];
    free(p);
}

/* ---- step 4: one expert's FFN --------------------------------------------- */

/* o = Wdown * (SiLU(Wgate x) * (Wup x)) for expert e; h (optional) gets the
 * F-vector between the two projections. */
void orc_expert_ffn(const orc_layer *L, int e, const uint16_t *xn, double *o, double *h_out)
{
    long D = L->d_model, F = L->ffn_dim, G = L->group_size;
    const int bits = L->code_bits == 2 ? 2 : 4;
    double *x = (double *)malloc(sizeof(double) * (size_t)D);
    double *h = (double *)malloc(sizeof(double) * (size_t)F);
    for (long d = 0; d < D; ++d)
        x[d] = orc_bf16_to_f64(xn[d]);
    for (long j = 0; j < F; ++j) {
        long row = (long)e * F + j;
        double g = 0.0, u = 0.0;
        for (long d = 0; d < D; ++d) {
            g += code_weight(bits, L->gate_q, L->gate_s, L->gate_b, row, D, G, d) * x[d];
            u += code_weight(bits, L->up_q, L->up_s, L->up_b, row, D, G, d) * x[d];
        }
        h[j] = g / (1.0 + exp(-g)) * u; /* SiLU(g) * u */
    }
    for (long d = 0; d < D; ++d) {
        long row = (long)e * D + d;
        double acc = 0.0;
        for (long f = 0; f < F; ++f)
            acc += code_weight(bits, L->down_q, L->down_s, L->down_b, row, F, G, f) * h[f];
        o[d] = acc;
    }
    if (h_out)
        memcpy(h_out, h, sizeof(double) * (size_t)F);
    free(h);
    free(x);
}

/* ---- one token through the layer ----------------------------------------- */

/* Route one token (steps 0-3).  Any output pointer may be NULL except idx, w. */
static void route_token(const orc_layer *L, const uint16_t *r, uint16_t *xn,
                        double *logits, int32_t *idx, double *w)
{
    orc_rmsnorm(L, r, xn);
    orc_router_logits(L, xn, logits);
    orc_topk(logits, L->n_experts, L->top_k, idx);
    orc_mix_weights(logits, L->n_experts, idx, L->top_k, L->norm_topk_prob, w);
}

/* step 5: y = r + sum_i w_i o_i, rank order */
static void combine(int D, int K, const uint16_t *r, const double *w, const double *o,
                    double *y, uint16_t *y_bf16)
{
    for (int d = 0; d < D; ++d) {
        double acc = orc_bf16_to_f64(r[d]);
        for (int i = 0; i < K; ++i)
            acc += w[i] * o[(size_t)i * D + d];
        y[d] = acc;
        if (y_bf16)
            y_bf16[d] = orc_f64_to_bf16(acc);
    }
}

/* Full layer for one token.  expert_out ([K][D], optional) receives o_i. */
void orc_moe_token(const orc_layer *L, const uint16_t *r, double *y, uint16_t *y_bf16,
                   int32_t *idx, double *w, double *logits_opt, uint16_t *xn_opt,
                   double *expert_out_opt)
{
    int D = L->d_model, E = L->n_experts, K = L->top_k;
    uint16_t *xn = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)D);
    double *logits = (double *)malloc(sizeof(double) * (size_t)E);
    double *o = (double *)malloc(sizeof(double) * (size_t)K * D);
    route_token(L, r, xn, logits, idx, w);
    for (int i = 0; i < K; ++i)
        orc_expert_ffn(L, idx[i], xn, o + (size_t)i * D, NULL);
    combine(D, K, r, w, o, y, y_bf16);
    if (logits_opt)
        memcpy(logits_opt, logits, sizeof(double) * (size_t)E);
    if (xn_opt)
        memcpy(xn_opt, xn, sizeof(uint16_t) * (size_t)D);
    if (expert_out_opt)
        memcpy(expert_out_opt, o, sizeof(double) * (size_t)K * D);
    free(o);
    free(logits);
    free(xn);
}

/* T independent tokens (a batch of decode steps).  Tokens are independent,
 * so they may run on several host threads; each token's arithmetic is the
 * single-token path above, unchanged. */
void orc_moe_tokens(const orc_layer *L, const uint16_t *r, int T, double *y, uint16_t *y_bf16,
                    int32_t *idx, double *w)
{
    int D = L->d_model, K = L->top_k;
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < T; ++t)
        orc_moe_token(L, r + (size_t)t * D, y + (size_t)t * D,
                      y_bf16 ? y_bf16 + (size_t)t * D : NULL,
                      idx + (size_t)t * K, w + (size_t)t * K, NULL, NULL, NULL);
}

/* The same, also returning every token's unweighted expert outputs
 * expert_out [T][K][D] (rank order): the per-token path above, unchanged. */
void orc_moe_tokens_experts(const orc_layer *L, const uint16_t *r, int T, double *y,
                            uint16_t *y_bf16, int32_t *idx, double *w, double *expert_out)
{
    int D = L->d_model, K = L->top_k;
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < T; ++t)
        orc_moe_token(L, r + (size_t)t * D, y + (size_t)t * D,
                      y_bf16 ? y_bf16 + (size_t)t * D : NULL,
                      idx + (size_t)t * K, w + (size_t)t * K, NULL, NULL,
                      expert_out + (size_t)t * K * D);
}

/* ---- per-chunk expert union and token buckets ----------------------------- */

/* union_ids: the distinct expert ids of idx[T][k], ascending, then -1 up to E.
 * offsets[u] .. offsets[u+1]: bucket of union entry u; entries past n_union
 * hold the total.  A bucket lists its tokens ascending with the rank at which
 * each token chose the expert.  Returns the number of idx entries outside
 * [0, E), which are skipped. */
int orc_expert_union(const int32_t *idx, int T, int k, int E, int32_t *union_ids,
                     int32_t *n_union, int32_t *offsets, int32_t *bucket_tok,
                     int32_t *bucket_rank)
{
    int n = 0, pos = 0, bad = 0;
    for (int t = 0; t < T; ++t)
        for (int i = 0; i < k; ++i)
            if (idx[t * k + i] < 0 || idx[t * k + i] >= E)
                ++bad;
    for (int e = 0; e < E; ++e) {
        int start = pos;
        for (int t = 0; t < T; ++t)
            for (int i = 0; i < k; ++i)
                if (idx[t * k + i] == e) {
                    bucket_tok[pos] = t;
                    bucket_rank[pos] = i;
                    ++pos;
                }
        if (pos > start) {
            union_ids[n] = e;
            offsets[n] = start;
            ++n;
        }
    }
    for (int u = n; u < E; ++u)
        union_ids[u] = -1;
    for (int u = n; u <= E; ++u)
        offsets[u] = pos;
    *n_union = n;
    return bad;
}

/* ---- one prefill chunk ------------------------------------------------------ */

/* T tokens (T <= 64 in the pages' prefill) through the layer: route every
 * token, build the union, read each union expert once and apply it to every
 * token of its bucket, then combine per token in rank order. */
void orc_moe_prefill_chunk(const orc_layer *L, const uint16_t *r, int T, double *y,
                           uint16_t *y_bf16, int32_t *idx, double *w, int32_t *union_ids,
                           int32_t *n_union, int32_t *offsets, int32_t *bucket_tok,
                           int32_t *bucket_rank)
{
    int D = L->d_model, E = L->n_experts, K = L->top_k;
    uint16_t *xn = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)T * D);
    double *logits = (double *)malloc(sizeof(double) * (size_t)E);
    double *o = (double *)malloc(sizeof(double) * (size_t)T * K * D);
    for (int t = 0; t < T; ++t)
        route_token(L, r + (size_t)t * D, xn + (size_t)t * D, logits,
                    idx + (size_t)t * K, w + (size_t)t * K);
    orc_expert_union(idx, T, K, E, union_ids, n_union, offsets, bucket_tok, bucket_rank);
    for (int u = 0; u < *n_union; ++u)
        for (int p = offsets[u]; p < offsets[u + 1]; ++p) {
            int t = bucket_tok[p], i = bucket_rank[p];
            orc_expert_ffn(L, union_ids[u], xn + (size_t)t * D,
                           o + ((size_t)t * K + i) * D, NULL);
        }
    for (int t = 0; t < T; ++t)
        combine(D, K, r + (size_t)t * D, w + (size_t)t * K, o + (size_t)t * K * D,
                y + (size_t)t * D, y_bf16 ? y_bf16 + (size_t)t * D : NULL);
    free(o);
    free(logits);
    free(xn);
}

/* ---- dense bf16 matrix-vector product ------------------------------------
 * "Optimizations" page, "Coalesced GPU Kernels -- Expert FFN and Dense
 * Matvec": the bf16 dense matvec twin of the expert kernels, which carries
 * decode's QKV/O projections and the LM head.  Its plain definition:
 *   y[r] = sum_c W[r][c] * x[c],   W bf16 [rows][cols] row-major, x bf16 [cols],
 * every product and every partial sum in fp64 (rows are independent, so the
 * OpenMP split over rows does not change any result). */
void orc_dense_matvec(const uint16_t *w, const uint16_t *x, long rows, long cols, double *y)
{
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r) {
        double acc = 0.0;
        for (long c = 0; c < cols; ++c)
            acc += orc_bf16_to_f64(w[r * cols + c]) * orc_bf16_to_f64(x[c]);
        y[r] = acc;
    }
}

/* ---- SMOE-Q4 quantiser ----------------------------------------------------
 * The offline step before the path: "System Overview", "The Four-Component
 * Architecture" and "What Happens at Each Generated Token Step" (the
 * Sculptor turns a model's routed experts into the vault's "aggressively
 * quantised" blocks).  The pages give no formula; this project reads it as
 * min/max affine quantisation per group of 64 consecutive weights of a row,
 * into the Q4 storage above:
 *   mn, mx = the least and the greatest weight of the group (bf16, exact)
 *   scale  = bf16 nearest-even of the binary32 value ((mx - mn) + 0) / 15
 *   bias   = bf16 of mn + 0  (exact; the "+ 0" turns a -0 into +0)
 *   q      = the code of the level scale*q + bias nearest to w: the integer
 *            nearest to the EXACT quotient (w - mn) / scale, halves to even;
 *            0 wherever scale is 0.  (w - mn) / scale <= 15 * (1 + 2^-8), so
 *            q never leaves [0, 15].
 * Decoding is w' = scale * q + bias, the layout's own definition.
 *
 * How q is evaluated, exactly.  The integer nearest to t = d / s (d = w - mn
 * >= 0, s > 0), halves to even, is the number of midpoints k + 1/2
 * (k = 0 .. levels-1) that lie strictly below t, plus one for a midpoint
 * that t hits exactly when k is odd (k + 1 is then the even neighbour).
 * Since s > 0, "k + 1/2 < t" is "s (k + 1/2) < d".  Both sides are exact here:
 *   - c = s (k + 1/2): 8 significant bits times at most 6, a binary64 value;
 *   - d = w - mn is held as dh + dl, the binary64 sum and its exact rounding
 *     error (Knuth's TwoSum; no overflow or underflow is possible for bf16
 *     inputs in binary64).  Because rounding is monotonic, dh > c implies
 *     d > c and dh < c implies d < c; when dh == c, d - c = dl.
 * No reciprocal, division or other rounding enters the decision. */
static float bf16_to_f32_orc(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Sign of (dh + dl) - c, exactly, for dh = RN(d), dl = d - dh, c a binary64. */
static int cmp_exact(double dh, double dl, double c)
{
    if (dh != c)
        return dh > c ? 1 : -1;
    return dl > 0.0 ? 1 : (dl < 0.0 ? -1 : 0);
}

/* The integer nearest to (w - mn) / s, halves to even, for s > 0, w >= mn. */
static int nearest_level(double w, double mn, double s, int levels)
{
    const double dh = w - mn;            /* Knuth's TwoSum: w - mn = dh + dl exactly */
    const double bb = dh - w;
    const double dl = (w - (dh - bb)) + (-mn - bb);
    int q = 0;
    for (int k = 0; k < levels; ++k) {
        const int c = cmp_exact(dh, dl, s * ((double)k + 0.5));
        if (c > 0 || (c == 0 && (k & 1)))
            ++q;
    }
    return q;
}

/* The same reading for SMOE-Q2 (bits = 2): levels = 2^bits - 1 = 3 replaces 15
 * (scale = bf16 of ((mx - mn) + 0) / 3, codes in [0, 3]), codes stored as in
 * the Q2 layout above. */
static void quantize_codes(const uint16_t *w, long rows, long cols, int bits, uint8_t *codes,
                           uint16_t *scale, uint16_t *bias)
{
    const long G = 64, ng = cols / G;
    const int levels = (1 << bits) - 1, per_byte = 8 / bits;
    const float flev = (float)levels;
    for (long r = 0; r < rows; ++r) {
        for (long g = 0; g < ng; ++g) {
            const uint16_t *p = w + r * cols + g * G;
            float mn = bf16_to_f32_orc(p[0]), mx = mn;
            for (long i = 1; i < G; ++i) {
                const float v = bf16_to_f32_orc(p[i]);
                if (v < mn) mn = v;
                if (v > mx) mx = v;
            }
            const float range = (mx - mn) + 0.0f;
            const float quot = range / flev;
            const uint16_t sb = orc_f64_to_bf16((double)quot);
            const double s = orc_bf16_to_f64(sb);
            scale[r * ng + g] = sb;
            bias[r * ng + g] = orc_f64_to_bf16((double)(mn + 0.0f));
            uint8_t *cq = codes + r * (cols / per_byte) + g * (G / per_byte);
            memset(cq, 0, (size_t)(G / per_byte));
            for (long i = 0; i < G; ++i) {
                const int q = s != 0.0 ? nearest_level(orc_bf16_to_f64(p[i]), (double)mn, s, levels) : 0;
                cq[i / per_byte] = (uint8_t)(cq[i / per_byte] | (q << (bits * (i % per_byte))));
            }
        }
    }
}

void orc_quantize_q4(const uint16_t *w, long rows, long cols, uint8_t *codes, uint16_t *scale,
                     uint16_t *bias)
{
    quantize_codes(w, rows, cols, 4, codes, scale, bias);
}

void orc_quantize_q2(const uint16_t *w, long rows, long cols, uint8_t *codes, uint16_t *scale,
                     uint16_t *bias)
{
    quantize_codes(w, rows, cols, 2, codes, scale, bias);
}
