/*
 * flint_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct CPU evaluation of one Flint
 * mixture-of-experts FFN layer in IEEE double precision.  It exists to check
 * the CUDA library; nothing in the product links, loads or calls it.  It
 * shares no code, header, table or constant with the CUDA sources: only the
 * seeded input generators (the `synth` module) feed both sides.
 *
 * What it computes (Flint vLLM recipe page, "Overview": 256 routed experts,
 * the top 6 chosen by sigmoid score, and one shared expert; the expert activation, hidden and
 * intermediate sizes, the renormalisation of the routing weights and the
 * unweighted shared expert are not printed on the pages and follow the
 * readings written next to each function):
 *
 *   l[t,e]  = sum_h x[t,h] * Wr[e,h] + b[e]                      (router)
 *   S_t     = the k experts with the largest l[t,e]; equal logits
 *             go to the lower expert index                        (top-k)
 *   s       = 1 / (1 + exp(-l))                                   (sigmoid)
 *   w[t,j]  = s[t,S_tj] / sum_{j'} s[t,S_tj']                     (renorm)
 *   g = Wg x, u = Wu x, a = g / (1 + exp(-g)) * u, o = Wd a       (SwiGLU)
 *   y[t]    = sum_j w[t,j] * o_{S_tj}(x_t) + o_shared(x_t)        (combine)
 *
 * Every bf16 input is widened exactly to double; an NVFP4 weight is decoded
 * exactly (E2M1 code x E4M3 block scale x fp32 tensor scale is exact in
 * double).  Nothing is rounded between the widening and the final double
 * result.  Ranking by logit equals ranking by sigmoid score (the sigmoid is
 * strictly increasing) and avoids the saturation of the score.
 *
 * Layouts (row-major, the nn.Linear [out][in] convention):
 *   x      [T][H]      bf16 bits (uint16)
 *   Wr     [E][H]      bf16 bits
 *   b      [E]         fp32 or NULL
 *   gate_up[2I][H]     rows 0..I-1 are the gate, rows I..2I-1 the up projection
 *   down   [H][I]
 *   NVFP4 matrix [R][K]: packed[R][K/2] (low nibble = even column),
 *                        scales[R][K/16] E4M3 codes, one fp32 tensor scale.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* number formats                                                           */
/* ------------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32: widen by placing the 16 bits
 * on top of 16 zero bits.  Exact. */
double oracle_bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* FP4 E2M1 (OCP Microscaling Formats v1.0, "FP4 E2M1"): bit 3 sign, bits
 * 2..1 exponent with bias 1, bit 0 mantissa; exponent 0 is subnormal with
 * value m * 2^(1-1) * 0.5.  No infinities or NaN. */
double oracle_e2m1_decode(uint8_t code)
{
    int sign = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double v;
    if (e == 0)
        v = 0.5 * m;
    else
        v = ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -v : v;
}

/* FP8 E4M3 (OCP 8-bit floating point, "E4M3"): bit 7 sign, bits 6..3
 * exponent with bias 7, bits 2..0 mantissa; exponent 0 is subnormal
 * (m/8 * 2^-6); S.1111.111 is NaN; there are no infinities. */
double oracle_e4m3_decode(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 15;
    int m = code & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* A weight matrix as the oracle sees it: either bf16 rows or NVFP4 rows. */
typedef struct {
    int32_t kind;            /* 0 = bf16, 1 = NVFP4 */
    int32_t rows, cols;
    const uint16_t* bf16;    /* kind 0: [rows][cols] */
    const uint8_t* packed;   /* kind 1: [rows][cols/2] */
    const uint8_t* scales;   /* kind 1: [rows][cols/16] */
    float tensor_scale;      /* kind 1 */
    int32_t pad_;
} oracle_mat;

/* Widen / decode row r of m into out[cols] (exact in double). */
static void mat_row(const oracle_mat* m, int r, double* out)
{
    int K = m->cols;
    if (m->kind == 0) {
        const uint16_t* p = m->bf16 + (size_t)r * K;
        for (int c = 0; c < K; ++c)
            out[c] = oracle_bf16_to_double(p[c]);
    } else {
        const uint8_t* q = m->packed + (size_t)r * (K / 2);
        const uint8_t* s = m->scales + (size_t)r * (K / 16);
        double ts = (double)m->tensor_scale;
        for (int c = 0; c < K; ++c) {
            uint8_t byte = q[c / 2];
            uint8_t nib = (c % 2 == 0) ? (byte & 0xF) : (byte >> 4);
            out[c] = oracle_e2m1_decode(nib) * oracle_e4m3_decode(s[c / 16]) * ts;
        }
    }
}

/* Decode a whole NVFP4 matrix to double (used by tests to build the
 * dequantised reference weights). */
void oracle_nvfp4_dequant(int rows, int cols, const uint8_t* packed,
                          const uint8_t* scales, float tensor_scale, double* out)
{
    oracle_mat m = {1, rows, cols, NULL, packed, scales, tensor_scale, 0};
    for (int r = 0; r < rows; ++r)
        mat_row(&m, r, out + (size_t)r * cols);
}

/* ------------------------------------------------------------------------ */
/* router                                                                   */
/* ------------------------------------------------------------------------ */

/* l[t][e] = sum_h x[t][h] Wr[e][h] (+ b[e]).  The pages name "sigmoid
 * routing" but no bias; a per-expert bias, when given, is added to the logit
 * before both the selection and the sigmoid (the plainest reading). */
void oracle_router_logits(int T, int E, int H, const uint16_t* x,
                          const uint16_t* Wr, const float* bias, double* logits)
{
    double* xr = (double*)malloc(sizeof(double) * H);
    double* wr = (double*)malloc(sizeof(double) * H);
    for (int t = 0; t < T; ++t) {
        for (int h = 0; h < H; ++h)
            xr[h] = oracle_bf16_to_double(x[(size_t)t * H + h]);
        for (int e = 0; e < E; ++e) {
            for (int h = 0; h < H; ++h)
                wr[h] = oracle_bf16_to_double(Wr[(size_t)e * H + h]);
            double acc = 0.0;
            for (int h = 0; h < H; ++h)
                acc += xr[h] * wr[h];
            if (bias)
                acc += (double)bias[e];
            logits[(size_t)t * E + e] = acc;
        }
    }
    free(xr);
    free(wr);
}

double oracle_sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* Top-k by logit, then sigmoid and renormalisation.  Selection is k passes
 * of "largest logit not yet taken"; a strictly-greater comparison scanning
 * from expert 0 upward keeps the lower index on equal logits.  The weights
 * are the selected sigmoid scores divided by their sum, so they sum to one
 * (the renormalisation is a reading: the pages give no formula).  Output
 * order: decreasing logit (ties: increasing index). */
void oracle_select(int T, int E, int k, const double* logits, int32_t* idx, double* w)
{
    char* taken = (char*)malloc((size_t)E);
    for (int t = 0; t < T; ++t) {
        const double* l = logits + (size_t)t * E;
        memset(taken, 0, (size_t)E);
        double ssum = 0.0;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e])
                    continue;
                if (best < 0 || l[e] > l[best])
                    best = e;
            }
            taken[best] = 1;
            idx[(size_t)t * k + j] = best;
            w[(size_t)t * k + j] = oracle_sigmoid(l[best]);
            ssum += w[(size_t)t * k + j];
        }
        for (int j = 0; j < k; ++j)
            w[(size_t)t * k + j] /= ssum;
    }
    free(taken);
}

/* ------------------------------------------------------------------------ */
/* experts                                                                  */
/* ------------------------------------------------------------------------ */

/* SwiGLU: silu(z) = z * sigmoid(z) = z / (1 + exp(-z)). */
double oracle_silu(double z) { return z / (1.0 + exp(-z)); }

/* One expert on one token: o[h] = sum_i Wd[h][i] * silu(g_i) * u_i with
 * g_i = sum_c Wg[i][c] x[c] and u_i = sum_c Wu[i][c] x[c].
 * gate_up is [2I][H] (gate rows first), down is [H][I].  scratch holds at
 * least 2I + max(H, I) doubles. */
static void expert_apply(int H, int I, const oracle_mat* gate_up, const oracle_mat* down,
                         const double* x, double* o, double* scratch)
{
    double* a = scratch;             /* [I]              */
    double* row = scratch + I;       /* [max(H, I)]      */
    double* g = scratch + I + (H > I ? H : I); /* [I]    */
    for (int i = 0; i < I; ++i) {
        mat_row(gate_up, i, row);
        double acc = 0.0;
        for (int c = 0; c < H; ++c)
            acc += row[c] * x[c];
        g[i] = acc;
    }
    for (int i = 0; i < I; ++i) {
        mat_row(gate_up, I + i, row);
        double u = 0.0;
        for (int c = 0; c < H; ++c)
            u += row[c] * x[c];
        a[i] = oracle_silu(g[i]) * u;
    }
    for (int h = 0; h < H; ++h) {
        mat_row(down, h, row);
        double acc = 0.0;
        for (int i = 0; i < I; ++i)
            acc += row[i] * a[i];
        o[h] = acc;
    }
}

/* Exposed for tests: one expert, one token, x given in double. */
void oracle_expert(int H, int I, const oracle_mat* gate_up, const oracle_mat* down,
                   const double* x, double* o)
{
    double* scratch = (double*)malloc(sizeof(double) * (2 * (size_t)I + (H > I ? H : I)));
    expert_apply(H, I, gate_up, down, x, o, scratch);
    free(scratch);
}

/* ------------------------------------------------------------------------ */
/* output layer                                                             */
/* ------------------------------------------------------------------------ */

/* The 4-bit output layer (lm_head) as a plain matrix-vector product: the
 * pages report that the output head was quantised to 4 bits too (the
 * mrchatgpt.org article, section 4, the quantisation item; the
 * qantcore.space review, section 04, the quantised variants).  The
 * vocabulary size is not on the pages.  logits[t][j] = sum_h x[t][h] * W[rows[j]][h]
 * for the nrows requested rows of W ([V][H], bf16 or NVFP4, decoded
 * exactly), all of them in order when rows is NULL (nrows = V). */
void oracle_lm_head(int T, int H, const uint16_t* x, const oracle_mat* W,
                    int nrows, const int32_t* rows, double* out)
{
    double* w = (double*)malloc(sizeof(double) * (size_t)H);
    double* xd = (double*)malloc(sizeof(double) * (size_t)T * H);
    for (size_t i = 0; i < (size_t)T * H; ++i)
        xd[i] = oracle_bf16_to_double(x[i]);
    for (int j = 0; j < nrows; ++j) {
        mat_row(W, rows ? rows[j] : j, w);
        for (int t = 0; t < T; ++t) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h)
                acc += xd[(size_t)t * H + h] * w[h];
            out[(size_t)t * nrows + j] = acc;
        }
    }
    free(xd);
    free(w);
}

/* ------------------------------------------------------------------------ */
/* the layer                                                                */
/* ------------------------------------------------------------------------ */

typedef struct {
    int T, E, H, I, k;
    const uint16_t* x;
    const oracle_mat* gate_up;   /* [E] routed experts; entry kind<0 = absent */
    const oracle_mat* down;      /* [E] */
    const oracle_mat* sh_gate_up;/* shared expert (may be NULL = no shared) */
    const oracle_mat* sh_down;
    const int32_t* idx;          /* [T][k] selection */
    const double* w;             /* [T][k] weights   */
    double* y;                   /* [T][H] out       */
    int next;                    /* work counter     */
    int bad;                     /* set if a selected expert is absent */
    pthread_mutex_t mu;
} layer_job;

static void* layer_worker(void* arg)
{
    layer_job* J = (layer_job*)arg;
    int H = J->H, I = J->I, k = J->k;
    double* xr = (double*)malloc(sizeof(double) * H);
    double* o = (double*)malloc(sizeof(double) * H);
    double* scratch = (double*)malloc(sizeof(double) * (2 * (size_t)I + (H > I ? H : I)));
    for (;;) {
        pthread_mutex_lock(&J->mu);
        int t = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (t >= J->T)
            break;
        for (int h = 0; h < H; ++h)
            xr[h] = oracle_bf16_to_double(J->x[(size_t)t * H + h]);
        double* yt = J->y + (size_t)t * H;
        for (int h = 0; h < H; ++h)
            yt[h] = 0.0;
        for (int j = 0; j < k; ++j) {
            int e = J->idx[(size_t)t * k + j];
            if (e < 0 || e >= J->E || J->gate_up[e].kind < 0 || J->down[e].kind < 0) {
                pthread_mutex_lock(&J->mu);
                J->bad = 1;
                pthread_mutex_unlock(&J->mu);
                continue;
            }
            expert_apply(H, I, &J->gate_up[e], &J->down[e], xr, o, scratch);
            double wj = J->w[(size_t)t * k + j];
            for (int h = 0; h < H; ++h)
                yt[h] += wj * o[h];
        }
        if (J->sh_gate_up && J->sh_down) {
            /* the shared expert is always active and added with weight one */
            expert_apply(H, I, J->sh_gate_up, J->sh_down, xr, o, scratch);
            for (int h = 0; h < H; ++h)
                yt[h] += o[h];
        }
    }
    free(xr);
    free(o);
    free(scratch);
    return NULL;
}

/* Full layer.  If idx_in is non-NULL it fixes the selection S_t (k distinct
 * expert ids per token, e.g. the runner-up set of a near tie computed from
 * this oracle's own logits); the weights are then the renormalised sigmoid
 * scores of that set.  Outputs: y[T][H] (double), and optionally the logits
 * [T][E], the selection [T][k] and the weights [T][k] actually used.
 * Returns 0, or -1 if a selected expert has no weights supplied. */
int oracle_moe_forward(int T, int E, int H, int I, int k,
                       const uint16_t* x, const uint16_t* Wr, const float* bias,
                       const oracle_mat* gate_up, const oracle_mat* down,
                       const oracle_mat* sh_gate_up, const oracle_mat* sh_down,
                       const int32_t* idx_in, double* y,
                       double* logits_out, int32_t* idx_out, double* w_out, int nthreads)
{
    double* logits = (double*)malloc(sizeof(double) * (size_t)T * E);
    int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)T * k);
    double* w = (double*)malloc(sizeof(double) * (size_t)T * k);
    oracle_router_logits(T, E, H, x, Wr, bias, logits);
    if (idx_in) {
        for (int t = 0; t < T; ++t) {
            double ssum = 0.0;
            for (int j = 0; j < k; ++j) {
                int e = idx_in[(size_t)t * k + j];
                idx[(size_t)t * k + j] = e;
                w[(size_t)t * k + j] = oracle_sigmoid(logits[(size_t)t * E + e]);
                ssum += w[(size_t)t * k + j];
            }
            for (int j = 0; j < k; ++j)
                w[(size_t)t * k + j] /= ssum;
        }
    } else {
        oracle_select(T, E, k, logits, idx, w);
    }

    layer_job J;
    J.T = T; J.E = E; J.H = H; J.I = I; J.k = k;
    J.x = x; J.gate_up = gate_up; J.down = down;
    J.sh_gate_up = sh_gate_up; J.sh_down = sh_down;
    J.idx = idx; J.w = w; J.y = y; J.next = 0; J.bad = 0;
    pthread_mutex_init(&J.mu, NULL);
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > T)
        nthreads = T > 0 ? T : 1;
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * nthreads);
    for (int i = 1; i < nthreads; ++i)
        pthread_create(&th[i], NULL, layer_worker, &J);
    layer_worker(&J);
    for (int i = 1; i < nthreads; ++i)
        pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.mu);

    if (logits_out)
        memcpy(logits_out, logits, sizeof(double) * (size_t)T * E);
    if (idx_out)
        memcpy(idx_out, idx, sizeof(int32_t) * (size_t)T * k);
    if (w_out)
        memcpy(w_out, w, sizeof(double) * (size_t)T * k);
    free(logits);
    free(idx);
    free(w);
    return J.bad ? -1 : 0;
}

/* The token -> expert permutation the routing implies, as a plain counting
 * sort: count[e] = number of (token, slot) pairs choosing e, offsets = its
 * exclusive prefix sum (offsets[E] = T*k), and gather[offsets[e] + r] = the
 * pair id t*k + j of the r-th pair choosing e in increasing pair-id order. */
void oracle_permutation(int T, int E, int k, const int32_t* idx,
                        int32_t* offsets, int32_t* gather)
{
    int32_t* fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    for (int e = 0; e <= E; ++e)
        offsets[e] = 0;
    for (int p = 0; p < T * k; ++p)
        offsets[idx[p] + 1] += 1;
    for (int e = 0; e < E; ++e)
        offsets[e + 1] += offsets[e];
    for (int p = 0; p < T * k; ++p) {
        int e = idx[p];
        gather[offsets[e] + fill[e]] = p;
        fill[e] += 1;
    }
    free(fill);
}
