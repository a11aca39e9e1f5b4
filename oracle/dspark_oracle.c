/*
 * dspark_oracle.c -- plain, slow, fp64 CPU reference of one DSpark round.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library. The product path never calls it,
 * and it shares no code, header or constant generator with the CUDA library.
 *
 * Sources (web pages about DSpark; cited by title and section/equation):
 *   [V4.1 blog]  "DeepSeek-V4.1 模型结构（6）：解码，DSpark" (blog.javazero.top)
 *   [spec_dspark] zdszero.github.io "spec_dspark", section "在 SGLang 里"
 *   [ailearn]    "DSpark：不让大模型更聪明，而让它「吐字更快」", sections 02 and 05
 *   [csdn]       deepseek.csdn.net close reading of the DSpark paper, sections 2.1-8
 *
 * What each function computes, in the pages' notation:
 *   draft   -- eq. (4)/(5): p_k = softmax(U_k + W1[x_{k-1}] W2), x_0 = anchor,
 *              sampled left to right (the sequential Markov loop of [V4.1 blog],
 *              section "Markov head"), plus eq. (7) c_k = sigma(w^T[h_k; W1[x_{k-1}]] / T_k)
 *              with the STS temperature of [spec_dspark] (sigmoid(raw / T)).
 *   plan    -- survival a_j = prod_{i<=j} c_i, B = sum(1 + l_r),
 *              tau = sum(1 + sum_{j<=l_r} a_{r,j}), Theta = tau * SPS(B), and
 *              Algorithm 1: admit candidates in decreasing a while Theta rises
 *              ([V4.1 blog] "目标函数", "贪心就能解"; [csdn] 5.3). The
 *              asynchronous variant takes the capacity K = argmax Theta from
 *              lagged confidences and the top-K current candidates ([csdn] 8).
 *   loss    -- the draft head's training objective, teacher-forced, eqs.
 *              (9)-(12) ([V4.1 blog] "训练"; [csdn] 6; [ailearn] 07).
 *   sts     -- sequential temperature scaling of c_k: per position, left to
 *              right, the grid temperature that minimises the ECE of the
 *              cumulative product against cumulative soft labels
 *              ([spec_dspark] "STS 校准"; [ailearn] 05; [csdn] 5.2).
 *   verify  -- accept x with probability min(1, p_t(x)/p_d(x)); at the first
 *              rejection resample from norm(max(0, p_t - p_d)); if every
 *              verified draft is accepted draw the bonus token from the
 *              target ([V4.1 blog] "投机解码"; [ailearn] 02; [csdn] 2.1).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   * sampler: the pages only write sample(logits). Every sample here (the
 *     draft, the bonus and the residual draw) is an exact two-level draw over
 *     vocabulary blocks of 64 tokens: a block is drawn with probability
 *     (block mass / total mass) by a Gumbel-max, argmax_s (log mass_s + G_s),
 *     then a token inside it with probability (weight / block mass) by a
 *     second Gumbel-max, argmax_v (log weight_v + G_v) over the block's
 *     tokens. Each level is an exact categorical draw, so the pair is an
 *     exact draw from the softmax, and each level's decision has a key gap
 *     as its margin. Temperature is 1.
 *   * teacher forcing (for parity checks only): the draft may be handed a
 *     token to adopt at a position whose draw was too close to call; the
 *     position's logits, margin and probability are still computed, and the
 *     chain continues from the adopted token.
 *   * random stream: Philox4x32-10 (Salmon et al., SC'11), key = seed,
 *     counter = (v >> 2, b, j, purpose << 24 | round mod 2^24), word v & 3,
 *     u = (2 * (word >> 9) + 1) * 2^-24, G = -log(-log u).
 *   * accept test written as u * p_d < p_t (no division).
 *   * a residual with no positive mass falls back to sampling p_t.
 *
 * Margins: each decision also reports how far it was from flipping, in the
 * units the parity rule uses (key gap for samples, |u - p_t/p_d| for accept
 * tests, relative Theta gap for the planner); see the header of each entry.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_BLOCK 64

enum {
    ORC_P_DRAFT_BLOCK = 1,
    ORC_P_DRAFT_TOKEN = 2,
    ORC_P_ACCEPT = 3,
    ORC_P_BONUS_BLOCK = 4,
    ORC_P_BONUS_TOKEN = 5,
    ORC_P_RESID_BLOCK = 6,
    ORC_P_RESID_TOKEN = 7,
    ORC_P_TREE_ACCEPT = 8,
    ORC_P_TREE_BLOCK = 9,
    ORC_P_TREE_TOKEN = 10
};

/* ------------------------------------------------------------------ */
/* Philox4x32-10, from the round function and key schedule of Salmon,  */
/* Moraes, Dror and Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3" */
/* ------------------------------------------------------------------ */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;   /* golden ratio */
            k1 += 0xBB67AE85u;   /* sqrt(3) - 1 */
        }
        uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)x0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)x2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t y0 = hi1 ^ x1 ^ k0;
        uint32_t y1 = lo1;
        uint32_t y2 = hi0 ^ x3 ^ k1;
        uint32_t y3 = lo0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

uint32_t orc_word(uint64_t seed, uint64_t round, uint32_t purpose,
                  uint32_t b, uint32_t j, uint32_t v)
{
    uint32_t ctr[4] = { v >> 2, b, j, (purpose << 24) | (uint32_t)(round & 0xFFFFFFu) };
    uint32_t key[2] = { (uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32) };
    uint32_t o[4];
    orc_philox4x32_10(ctr, key, o);
    return o[v & 3u];
}

/* Uniform on the odd grid {(2m+1) 2^-24}: never 0 or 1, exact in fp32 and fp64. */
double orc_uniform(uint64_t seed, uint64_t round, uint32_t purpose,
                   uint32_t b, uint32_t j, uint32_t v)
{
    uint32_t x = orc_word(seed, round, purpose, b, j, v);
    return (double)(2u * (x >> 9) + 1u) * 0x1p-24;
}

double orc_gumbel(uint64_t seed, uint64_t round, uint32_t purpose,
                  uint32_t b, uint32_t j, uint32_t v)
{
    double u = orc_uniform(seed, round, purpose, b, j, v);
    return -log(-log(u));
}

/* ------------------------------------------------------------------ */
/* small fp64 helpers                                                  */
/* ------------------------------------------------------------------ */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* element (i, c) of a row-major [rows, cols] weight stored as fp32 or bf16 */
static double wget(const void* W, int bf16, long i, long cols, long c)
{
    if (bf16) return bf16_to_double(((const uint16_t*)W)[i * cols + c]);
    return (double)((const float*)W)[i * cols + c];
}

/* log sum_v exp(x_v), max-subtracted; -inf entries contribute nothing */
double orc_logsumexp(const double* x, long n)
{
    double m = -INFINITY;
    for (long i = 0; i < n; ++i) if (x[i] > m) m = x[i];
    if (m == -INFINITY) return -INFINITY;
    double s = 0.0;
    for (long i = 0; i < n; ++i) s += exp(x[i] - m);
    return m + log(s);
}

/* ------------------------------------------------------------------ */
/* Two-level draws of v with probability exp(logw_v)/sum.             */
/* tol[v] (optional) widens the margin of token keys whose fp32        */
/* evaluation is known to be loose (the residual), and tol_mass[v] the */
/* block keys: a block's tolerance is sum(tol_mass) / block mass.      */
/* margin = top-2 key gap minus the two tolerances, minimised over     */
/* both levels.                                                        */
/* Returns -1 if no token has positive weight.                         */
/* ------------------------------------------------------------------ */
/* The block level: argmax_s (log mass_s + G_s) over the blocks with positive
 * mass. Returns the block (-1 if none) and its key gap to the runner-up,
 * less both blocks' mass tolerances, in *m1. */
static long pick_block(const double* logw, const double* tol_mass, long V, uint64_t seed,
                       uint64_t round, uint32_t pblk, uint32_t b, uint32_t j, double* m1)
{
    long nblk = (V + ORC_BLOCK - 1) / ORC_BLOCK;
    double best = -INFINITY, second = -INFINITY, tb = 0.0, ts = 0.0;
    long bs = -1;
    for (long s = 0; s < nblk; ++s) {
        long lo = s * ORC_BLOCK, hi = lo + ORC_BLOCK < V ? lo + ORC_BLOCK : V;
        double mass_log = orc_logsumexp(logw + lo, hi - lo);
        if (mass_log == -INFINITY) continue;
        double t = 0.0;
        if (tol_mass) {
            /* block tolerance: absolute error bound of the block mass over the mass */
            double num = 0.0;
            for (long v = lo; v < hi; ++v) num += tol_mass[v];
            t = num / exp(mass_log);
        }
        double key = mass_log + orc_gumbel(seed, round, pblk, b, j, (uint32_t)s);
        if (key > best) { second = best; ts = tb; best = key; tb = t; bs = s; }
        else if (key > second) { second = key; ts = t; }
    }
    *m1 = (bs < 0 || second == -INFINITY) ? INFINITY : (best - second) - (tb + ts);
    return bs;
}

/* Two-level draw, token level by Gumbel-max (every draw). The margin is the
 * smaller of the block and token key gaps; tol/tol_mass (may be NULL) are
 * per-token absolute error bounds of exp(logw) that widen the gaps.
 * Returns -1 if no token has positive weight. */
static int sample_two_level(const double* logw, const double* tol, const double* tol_mass, long V,
                            uint64_t seed, uint64_t round, uint32_t pblk, uint32_t ptok,
                            uint32_t b, uint32_t j, double* margin)
{
    double m1;
    long bs = pick_block(logw, tol_mass, V, seed, round, pblk, b, j, &m1);
    if (bs < 0) { *margin = INFINITY; return -1; }
    long lo = bs * ORC_BLOCK, hi = lo + ORC_BLOCK < V ? lo + ORC_BLOCK : V;
    double kb = -INFINITY, k2 = -INFINITY, t1 = 0.0, t2 = 0.0;
    long vb = -1;
    for (long v = lo; v < hi; ++v) {
        if (logw[v] == -INFINITY) continue;
        double key = logw[v] + orc_gumbel(seed, round, ptok, b, j, (uint32_t)v);
        double t = tol ? tol[v] : 0.0;
        if (key > kb) { k2 = kb; t2 = t1; kb = key; t1 = t; vb = v; }
        else if (key > k2) { k2 = key; t2 = t; }
    }
    double m2 = (k2 == -INFINITY) ? INFINITY : (kb - k2) - (t1 + t2);
    *margin = m1 < m2 ? m1 : m2;
    return (int)vb;
}

/* ------------------------------------------------------------------ */
/* Draft: eq. (4), (5) and (7).                                        */
/* ------------------------------------------------------------------ */
typedef struct {
    int B, gamma, V, r, H;
    int w_bf16;   /* W1/W2 stored as bf16 bit patterns (else fp32) */
} orc_dims;

/* z_v = U_k(v) + sum_i W1[x, i] W2[i, v] for one draft position, fp64 */
static void markov_logits(const orc_dims* d, const float* Urow, const void* W1,
                          const void* W2, int x_prev, double* z)
{
    long V = d->V, r = d->r;
    for (long v = 0; v < V; ++v) z[v] = 0.0;
    for (long i = 0; i < r; ++i) {
        double e = wget(W1, d->w_bf16, x_prev, r, i);   /* W1[x_{k-1}] row */
        for (long v = 0; v < V; ++v) z[v] += e * wget(W2, d->w_bf16, i, V, v);
    }
    for (long v = 0; v < V; ++v) z[v] += (double)Urow[v];
}

/* z_v = U_k(v) + sum_i o_i W2[i, v]: the draft logits of a head whose bias is
 * an r-vector o times W2 (the RNN head's o_k, eq. (6)), fp64 */
static void head_logits(const orc_dims* d, const float* Urow, const void* W2, const double* o, double* z)
{
    long V = d->V, r = d->r;
    for (long v = 0; v < V; ++v) z[v] = 0.0;
    for (long i = 0; i < r; ++i)
        for (long v = 0; v < V; ++v) z[v] += o[i] * wget(W2, d->w_bf16, i, V, v);
    for (long v = 0; v < V; ++v) z[v] += (double)Urow[v];
}

/*
 * For each request b in reqs[0..n_req): draft x_1..x_gamma.
 * Outputs (indexed [b][k-1], full-size arrays, only listed rows written):
 *   tokens, pd_tok = p_k(x_k), lse = log sum exp(z_k), conf = c_k,
 *   margin = the draw's margin (see sample_two_level).
 * force (may be NULL): force[b][k-1] >= 0 replaces the drawn x_k by that token
 * (teacher forcing at a flagged position); the margin is still the draw's.
 */
void orc_draft(const orc_dims* d, const float* U, const void* W1, const void* W2,
               const int32_t* anchor, const float* h, const float* w, const float* T,
               uint64_t seed, uint64_t round, const int32_t* reqs, int n_req, const int32_t* force,
               int32_t* tokens, double* pd_tok, double* lse, double* conf, double* margin)
{
    const long V = d->V, g = d->gamma, r = d->r, H = d->H;
#pragma omp parallel for schedule(dynamic, 1)
    for (int q = 0; q < n_req; ++q) {
        const long b = reqs[q];
        double* z = (double*)malloc(sizeof(double) * (size_t)V);
        int x_prev = anchor[b];                 /* x_0 = anchor */
        for (long k = 1; k <= g; ++k) {
            const long o = b * g + (k - 1);
            /* eq. (7): c_k = sigma(w^T [h_k; W1[x_{k-1}]] / T_k) */
            double s = 0.0;
            for (long i = 0; i < H; ++i) s += (double)w[i] * (double)h[o * H + i];
            for (long i = 0; i < r; ++i) s += (double)w[H + i] * wget(W1, d->w_bf16, x_prev, r, i);
            conf[o] = 1.0 / (1.0 + exp(-s / (double)T[k - 1]));
            /* eq. (4)/(5) */
            markov_logits(d, U + o * V, W1, W2, x_prev, z);
            double L = orc_logsumexp(z, V);
            double m = 0.0;
            int x = sample_two_level(z, NULL, NULL, V, seed, round, ORC_P_DRAFT_BLOCK,
                                     ORC_P_DRAFT_TOKEN, (uint32_t)b, (uint32_t)k, &m);
            if (force && force[o] >= 0) x = force[o];
            tokens[o] = x;
            pd_tok[o] = exp(z[x] - L);
            lse[o] = L;
            margin[o] = m;
            x_prev = x;
        }
        free(z);
    }
}

/* ------------------------------------------------------------------ */
/* RNN head ([V4.1 blog] section on the Markov head (the RNN variant    */
/* the paper also tried); [ailearn] "RNN 头（可选）"; [csdn] §4.2,       */
/* eq. (6)). A gated recurrent state s_k in R^r summarises the block's  */
/* prefix: with z_k = [s_{k-1}; W1[x_{k-1}]; h_k] (length 2r + H),       */
/*   g_k = sigma(W_g z_k),                                              */
/*   s_k = g_k * s_{k-1} + (1 - g_k) * tanh(W_c z_k),                   */
/*   o_k = tanh(W_o z_k),   z = U_k + o_k W2  (the bias B_k = W2^T o_k), */
/* s_0 = 0, x_0 = the anchor; W_g, W_c, W_o are [r][2r + H] (no bias,   */
/* as the equation shows none), stored one after the other in Wr in the */
/* weights' dtype. Sampling and the confidence head (eq. (7), with      */
/* W1[x_{k-1}]) are the Markov draft's. ovec [B][gamma][r] receives o_k. */
/* ------------------------------------------------------------------ */
void orc_rnn_draft(const orc_dims* d, const float* U, const void* W1, const void* W2, const void* Wr,
                   const int32_t* anchor, const float* h, const float* w, const float* T,
                   uint64_t seed, uint64_t round, const int32_t* reqs, int n_req, const int32_t* force,
                   int32_t* tokens, double* pd_tok, double* lse, double* conf, double* margin,
                   double* ovec)
{
    const long V = d->V, g = d->gamma, r = d->r, H = d->H, Z = 2 * r + H;
#pragma omp parallel for schedule(dynamic, 1)
    for (int q = 0; q < n_req; ++q) {
        const long b = reqs[q];
        double* z = (double*)malloc(sizeof(double) * (size_t)V);
        double* zin = (double*)malloc(sizeof(double) * (size_t)Z);
        double* st = (double*)calloc((size_t)r, sizeof(double));     /* s_0 = 0 */
        double* ov = (double*)malloc(sizeof(double) * (size_t)r);
        int x_prev = anchor[b];
        for (long k = 1; k <= g; ++k) {
            const long o = b * g + (k - 1);
            /* z_k = [s_{k-1}; W1[x_{k-1}]; h_k] */
            for (long i = 0; i < r; ++i) zin[i] = st[i];
            for (long i = 0; i < r; ++i) zin[r + i] = wget(W1, d->w_bf16, x_prev, r, i);
            for (long i = 0; i < H; ++i) zin[2 * r + i] = (double)h[o * H + i];
            /* gate, candidate and output of every state entry (all from z_k) */
            for (long j = 0; j < r; ++j) {
                double ag = 0.0, ac = 0.0, ao = 0.0;
                for (long i = 0; i < Z; ++i) {
                    ag += wget(Wr, d->w_bf16, j, Z, i) * zin[i];
                    ac += wget(Wr, d->w_bf16, r + j, Z, i) * zin[i];
                    ao += wget(Wr, d->w_bf16, 2 * r + j, Z, i) * zin[i];
                }
                const double gk = 1.0 / (1.0 + exp(-ag));
                st[j] = gk * zin[j] + (1.0 - gk) * tanh(ac);
                ov[j] = tanh(ao);
                ovec[o * r + j] = ov[j];
            }
            /* eq. (7) as for the Markov head */
            double s = 0.0;
            for (long i = 0; i < H; ++i) s += (double)w[i] * (double)h[o * H + i];
            for (long i = 0; i < r; ++i) s += (double)w[H + i] * zin[r + i];
            conf[o] = 1.0 / (1.0 + exp(-s / (double)T[k - 1]));
            /* z = U_k + o_k W2 */
            head_logits(d, U + o * V, W2, ov, z);
            const double L = orc_logsumexp(z, V);
            double m = 0.0;
            int x = sample_two_level(z, NULL, NULL, V, seed, round, ORC_P_DRAFT_BLOCK,
                                     ORC_P_DRAFT_TOKEN, (uint32_t)b, (uint32_t)k, &m);
            if (force && force[o] >= 0) x = force[o];
            tokens[o] = x;
            pd_tok[o] = exp(z[x] - L);
            lse[o] = L;
            margin[o] = m;
            x_prev = x;
        }
        free(z); free(zin); free(st); free(ov);
    }
}

/* ------------------------------------------------------------------ */
/* Planner                                                             */
/* ------------------------------------------------------------------ */
typedef struct { double a; int j; int b; } orc_cand;

/* order: a descending, then position j ascending, then request b ascending */
static int cand_cmp(const void* pa, const void* pb)
{
    const orc_cand* x = (const orc_cand*)pa;
    const orc_cand* y = (const orc_cand*)pb;
    if (x->a > y->a) return -1;
    if (x->a < y->a) return 1;
    if (x->j != y->j) return x->j < y->j ? -1 : 1;
    if (x->b != y->b) return x->b < y->b ? -1 : 1;
    return 0;
}

/* a_{b,j} = prod_{i<=j} c_{b,i} (left-to-right fp64 products), sorted */
static orc_cand* sorted_candidates(int B, int g, const float* conf)
{
    orc_cand* c = (orc_cand*)malloc(sizeof(orc_cand) * (size_t)B * (size_t)g);
    for (int b = 0; b < B; ++b) {
        double a = 1.0;
        for (int j = 1; j <= g; ++j) {
            a = a * (double)conf[(long)b * g + (j - 1)];
            orc_cand* e = &c[(long)b * g + (j - 1)];
            e->a = a; e->j = j; e->b = b;
        }
    }
    qsort(c, (size_t)B * (size_t)g, sizeof(orc_cand), cand_cmp);
    return c;
}

static double rel_gap(double x, double y)
{
    double m = fabs(x) > fabs(y) ? fabs(x) : fabs(y);
    return m > 0.0 ? fabs(x - y) / m : INFINITY;
}

/* survival probabilities of each request in candidate order (for tests) */
void orc_survival(int B, int g, const float* conf, double* a_out)
{
    for (int b = 0; b < B; ++b) {
        double a = 1.0;
        for (int j = 1; j <= g; ++j) {
            a = a * (double)conf[(long)b * g + (j - 1)];
            a_out[(long)b * g + (j - 1)] = a;
        }
    }
}

/*
 * Algorithm 1 with early stop. sps[n] = SPS(n) for n = 1 .. B*(g+1).
 * lengths[b] = 1 + number of admitted drafts of b (the anchor is always verified).
 * The admission test "Theta rises", (tau + a) SPS(n+1) > tau SPS(n), is taken
 * in the blog's threshold form a SPS(n+1) > tau (SPS(n) - SPS(n+1))
 * ("阈值随负载变化"): the same inequality, without absorbing a tiny a into tau
 * (so that a flat table admits every a > 0: full verify, as "spec_dspark"
 * states for the SGLang planner without an SPS table).
 * Returns the number of admitted candidates m*. margin[0] = smallest relative
 * difference between the two sides over the decisions taken (how far a
 * comparison was from flipping); margin[1] = relative gap between the
 * survival values on the two sides of the cut (how far two candidates were
 * from swapping across it).
 */
int orc_plan_sync(int B, int g, const float* conf, const double* sps,
                  int32_t* lengths, double* margin)
{
    orc_cand* c = sorted_candidates(B, g, conf);
    const int M = B * g;
    double tau = (double)B;           /* every request yields at least one token */
    long n = B;                        /* verify batch: one anchor per request */
    double mg = INFINITY;
    int m = 0;
    for (; m < M; ++m) {
        double gain = c[m].a * sps[n + 1];            /* expected tokens won, at the new rate */
        double cost = tau * (sps[n] - sps[n + 1]);    /* rate lost on the tokens already expected */
        double gap = rel_gap(gain, cost);
        if (gap < mg) mg = gap;
        if (!(gain > cost)) break;    /* stop as soon as Theta no longer rises */
        tau += c[m].a;
        n += 1;
    }
    for (int b = 0; b < B; ++b) lengths[b] = 1;
    for (int i = 0; i < m; ++i) lengths[c[i].b] += 1;
    margin[0] = mg;
    margin[1] = (m > 0 && m < M) ? rel_gap(c[m - 1].a, c[m].a) : INFINITY;
    free(c);
    return m;
}

/*
 * Full-path search: K = argmax_m Theta_m over m = 0 .. B*g (ties -> smallest m),
 * with Theta_m = (B + sum of the m largest a) * SPS(B + m). Used for the
 * capacity of the lagged planner, and by tests as the retrospective
 * (non-early-stop) planner. margin = relative gap between the best and the
 * second-best Theta.
 */
int orc_plan_capacity(int B, int g, const float* conf, const double* sps, double* margin)
{
    orc_cand* c = sorted_candidates(B, g, conf);
    const int M = B * g;
    double tau = (double)B;
    double best = tau * sps[B], second = -INFINITY;
    int K = 0;
    for (int m = 1; m <= M; ++m) {
        tau += c[m - 1].a;
        double th = tau * sps[B + m];
        if (th > best) { second = best; best = th; K = m; }
        else if (th > second) second = th;
    }
    *margin = second == -INFINITY ? INFINITY : rel_gap(best, second);
    free(c);
    return K;
}

/* Theta_m = (B + sum of the m largest a) * SPS(B + m) for m = 0 .. B*g, the
   path the capacity search maximises (theta[B*g + 1]) */
void orc_plan_theta_path(int B, int g, const float* conf, const double* sps, double* theta)
{
    orc_cand* c = sorted_candidates(B, g, conf);
    const int M = B * g;
    double tau = (double)B;
    theta[0] = tau * sps[B];
    for (int m = 1; m <= M; ++m) {
        tau += c[m - 1].a;
        theta[m] = tau * sps[B + m];
    }
    free(c);
}

/* lengths from the K best current candidates; margin = relative a gap at the cut
   (the Theta margin does not apply: the capacity K is given) */
void orc_plan_topk(int B, int g, const float* conf, int K, int32_t* lengths, double* margin)
{
    orc_cand* c = sorted_candidates(B, g, conf);
    const int M = B * g;
    if (K > M) K = M;
    for (int b = 0; b < B; ++b) lengths[b] = 1;
    for (int i = 0; i < K; ++i) lengths[c[i].b] += 1;
    *margin = (K > 0 && K < M) ? rel_gap(c[K - 1].a, c[K].a) : INFINITY;
    free(c);
}

/* ------------------------------------------------------------------ */
/* Verify                                                              */
/* ------------------------------------------------------------------ */
/*
 * For each request b in reqs: rows P + row_off[b] .. + lengths[b]-1 of the
 * packed target logits (row j = target distribution after x_j, x_0 = anchor).
 * Draft tokens tokens[b][0..g) are x_1..x_g. The draft distribution p_d at
 * position j+1 is recomputed here in fp64 from (U, W1, W2, x_j) for the
 * Markov head, or from (U, ovec[b][j], W2) for the RNN head (ovec non-NULL:
 * the head vectors o_{j+1} of the draft).
 * Outputs: n_acc[b] (leading accepted drafts), next_anchor[b],
 *   acc_margin[b] = min |u - p_t/p_d| over the tests taken,
 *   smp_margin[b] = key-gap margin of the final draw (residual or bonus),
 *   resid[b] = 1 if the next anchor came from the residual distribution.
 */
void orc_verify_head(const orc_dims* d, const float* P, const int32_t* row_off,
                     const int32_t* lengths, const int32_t* anchor, const int32_t* tokens,
                     const float* U, const void* W1, const void* W2, const double* ovec,
                     uint64_t seed, uint64_t round, const int32_t* reqs, int n_req,
                     int32_t* n_acc, int32_t* next_anchor, double* acc_margin,
                     double* smp_margin, int32_t* resid)
{
    const long V = d->V, g = d->gamma;
#pragma omp parallel for schedule(dynamic, 1)
    for (int q = 0; q < n_req; ++q) {
        const long b = reqs[q];
        const int ell = lengths[b];
        double* lt = (double*)malloc(sizeof(double) * (size_t)V);   /* log p_t */
        double* z = (double*)malloc(sizeof(double) * (size_t)V);
        double* lw = (double*)malloc(sizeof(double) * (size_t)V);
        double* tol = (double*)malloc(sizeof(double) * (size_t)V);
        double* tm = (double*)malloc(sizeof(double) * (size_t)V);
        double am = INFINITY, sm = INFINITY;
        int n = ell - 1, out = -1, from_resid = 0;
        for (int j = 0; j < ell - 1; ++j) {
            const float* Prow = P + (long)(row_off[b] + j) * V;
            for (long v = 0; v < V; ++v) lt[v] = (double)Prow[v];
            double Lt = orc_logsumexp(lt, V);
            for (long v = 0; v < V; ++v) lt[v] -= Lt;
            const int x_prev = j == 0 ? anchor[b] : tokens[b * g + (j - 1)];
            const int x = tokens[b * g + j];
            if (ovec)
                head_logits(d, U + (b * g + j) * V, W2, ovec + (b * g + j) * d->r, z);
            else
                markov_logits(d, U + (b * g + j) * V, W1, W2, x_prev, z);
            double Ld = orc_logsumexp(z, V);
            double pt = exp(lt[x]), pd = exp(z[x] - Ld);
            double u = orc_uniform(seed, round, ORC_P_ACCEPT, (uint32_t)b, (uint32_t)j, 0u);
            double ratio_gap = fabs(u - pt / pd);
            if (ratio_gap < am) am = ratio_gap;
            if (u * pd < pt) continue;         /* accepted with prob min(1, p_t/p_d) */
            /* first rejection: resample from norm(max(0, p_t - p_d)) */
            n = j;
            for (long v = 0; v < V; ++v) {
                double lpd = z[v] - Ld;
                if (lt[v] > lpd) {
                    double c = -expm1(lpd - lt[v]);      /* (p_t - p_d) / p_t */
                    lw[v] = lt[v] + log(c);
                    /* an fp32 evaluation of lpd - lt carries about 4e-6 absolute
                       error, which moves log c by 4e-6 * (1 - c) / c */
                    tol[v] = 4e-6 * (1.0 - c) / c;
                    /* a block mass summed as max(0, p_t - p_d) in fp32 carries
                       about 4e-6 (p_t + p_d) absolute error per token */
                    tm[v] = 4e-6 * exp(lt[v]) * (2.0 - c);
                } else {
                    lw[v] = -INFINITY;
                    tol[v] = 0.0;
                    tm[v] = 0.0;
                }
            }
            out = sample_two_level(lw, tol, tm, V, seed, round, ORC_P_RESID_BLOCK,
                                   ORC_P_RESID_TOKEN, (uint32_t)b, (uint32_t)j, &sm);
            from_resid = 1;
            if (out < 0) {   /* no positive residual mass: sample p_t itself */
                out = sample_two_level(lt, NULL, NULL, V, seed, round, ORC_P_BONUS_BLOCK,
                                       ORC_P_BONUS_TOKEN, (uint32_t)b, (uint32_t)j, &sm);
                from_resid = 0;
            }
            break;
        }
        if (out < 0) {   /* every verified draft accepted: bonus from row ell-1 */
            const float* Prow = P + (long)(row_off[b] + n) * V;
            for (long v = 0; v < V; ++v) lt[v] = (double)Prow[v];
            out = sample_two_level(lt, NULL, NULL, V, seed, round, ORC_P_BONUS_BLOCK,
                                   ORC_P_BONUS_TOKEN, (uint32_t)b, (uint32_t)n, &sm);
        }
        n_acc[b] = n;
        next_anchor[b] = out;
        acc_margin[b] = am;
        smp_margin[b] = sm;
        resid[b] = from_resid;
        free(lt); free(z); free(lw); free(tol); free(tm);
    }
}

void orc_verify(const orc_dims* d, const float* P, const int32_t* row_off,
                const int32_t* lengths, const int32_t* anchor, const int32_t* tokens,
                const float* U, const void* W1, const void* W2,
                uint64_t seed, uint64_t round, const int32_t* reqs, int n_req,
                int32_t* n_acc, int32_t* next_anchor, double* acc_margin,
                double* smp_margin, int32_t* resid)
{
    orc_verify_head(d, P, row_off, lengths, anchor, tokens, U, W1, W2, NULL, seed, round, reqs, n_req,
                    n_acc, next_anchor, acc_margin, smp_margin, resid);
}

/* ------------------------------------------------------------------ */
/* PCTree: the chain made a tree ([V4.1 blog] "后续工作": the Markov     */
/* head already scores every child token under a parent token, so it   */
/* picks candidate children per parent node, and the most probable     */
/* paths are kept within a fixed verify budget; no retraining, no extra */
/* backbone pass). The pages only summarise it; the steps below are the */
/* plainest reading:                                                   */
/*  build: node 0 is the anchor (depth 0, log-probability 0). A node x  */
/*   at depth k < gamma proposes its c most probable children under    */
/*   p_d(. | x) = softmax(U_{k+1} + W1[x] W2) (U of the position, shared */
/*   by every node of that depth: no extra backbone pass), each with    */
/*   the path log-probability of its parent plus log p_d(child). Nodes  */
/*   are admitted best first (highest path log-probability; ties to the */
/*   smaller depth, parent index, token) until N nodes besides the root */
/*   are in: the N most probable paths' nodes. Children are kept in     */
/*   admission order, so siblings come in decreasing probability.       */
/*  verify (lossless): at a node with target p = softmax(P[node]), the  */
/*   children are tried in order; child i is accepted with the current  */
/*   (renormalised) p of its token, u < p(t_i) with u = uniform(purpose */
/*   8, b, node, i); a rejected child's token is removed from p and p is */
/*   renormalised. An accepted child becomes the node. When no child is */
/*   accepted (or there is none), the next anchor is drawn from p (the   */
/*   target with the rejected tokens removed) by the two-level sampler  */
/*   (purposes 9, 10; j = node). Each emitted token is then an exact    */
/*   draw from the target given its prefix.                             */
/* ------------------------------------------------------------------ */
typedef struct { double lp; int depth, parent, token; } orc_tcand;

/* a better than b: higher log-probability, then smaller depth, parent, token */
static int tcand_better(const orc_tcand* a, const orc_tcand* b)
{
    if (a->lp != b->lp) return a->lp > b->lp;
    if (a->depth != b->depth) return a->depth < b->depth;
    if (a->parent != b->parent) return a->parent < b->parent;
    return a->token < b->token;
}

/*
 * Per request b in reqs[0..n_req): tok, par, dep [b][N+1] (node 0 the root;
 * -1 past the last node), lp [b][N+1] the path log-probabilities; n_nodes[b]
 * the nodes besides the root (< N only when every path reaches depth gamma);
 * margin[b] = the smallest log-probability gap that decided an admission or a
 * top-c choice.
 */
void orc_pctree_build(const orc_dims* d, const float* U, const void* W1, const void* W2,
                      const int32_t* anchor, int c, int N, const int32_t* reqs, int n_req,
                      int32_t* tok, int32_t* par, int32_t* dep,
                      double* lp, int32_t* n_nodes, double* margin)
{
    const long V = d->V, g = d->gamma;
#pragma omp parallel for schedule(dynamic, 1)
    for (int q = 0; q < n_req; ++q) {
        const int b = reqs[q];
        double* z = (double*)malloc(sizeof(double) * (size_t)V);
        orc_tcand* fr = (orc_tcand*)malloc(sizeof(orc_tcand) * (size_t)(N + 1) * (size_t)(c > 0 ? c : 1));
        int nf = 0;
        double mg = INFINITY;
        int32_t* tk = tok + (long)b * (N + 1);
        int32_t* pa = par + (long)b * (N + 1);
        int32_t* de = dep + (long)b * (N + 1);
        double* l = lp + (long)b * (N + 1);
        for (int i = 0; i <= N; ++i) { tk[i] = -1; pa[i] = -1; de[i] = -1; l[i] = -INFINITY; }
        tk[0] = anchor[b]; de[0] = 0; l[0] = 0.0;
        int n = 0, last = 0;
        for (;;) {
            /* expand the node just admitted */
            if (de[last] < g && c > 0) {
                markov_logits(d, U + ((long)b * g + de[last]) * V, W1, W2, tk[last], z);
                const double L = orc_logsumexp(z, V);
                for (int t = 0; t < c && t < V; ++t) {
                    long best = -1;
                    for (long v = 0; v < V; ++v) {
                        if (z[v] == -INFINITY) continue;
                        if (best < 0 || z[v] > z[best]) best = v;
                    }
                    if (best < 0) break;
                    fr[nf].lp = l[last] + (z[best] - L);
                    fr[nf].depth = de[last] + 1;
                    fr[nf].parent = last;
                    fr[nf].token = (int)best;
                    ++nf;
                    z[best] = -INFINITY;
                    /* the gap to the next child decided this top-c choice */
                    if (t == c - 1) {
                        double nxt = -INFINITY;
                        for (long v = 0; v < V; ++v) if (z[v] > nxt) nxt = z[v];
                        if (nxt > -INFINITY) {
                            const double gap = (fr[nf - 1].lp - l[last]) - (nxt - L);
                            if (gap < mg) mg = gap;
                        }
                    }
                }
            }
            if (n == N || nf == 0) break;
            /* admit the best frontier candidate */
            int bi = 0;
            for (int i = 1; i < nf; ++i) if (tcand_better(&fr[i], &fr[bi])) bi = i;
            for (int i = 0; i < nf; ++i)
                if (i != bi && fr[bi].lp - fr[i].lp < mg) mg = fr[bi].lp - fr[i].lp;
            ++n;
            tk[n] = fr[bi].token; pa[n] = fr[bi].parent; de[n] = fr[bi].depth; l[n] = fr[bi].lp;
            last = n;
            fr[bi] = fr[nf - 1];
            --nf;
        }
        n_nodes[b] = n;
        margin[b] = mg;
        free(z); free(fr);
    }
}

/*
 * P holds [B][N+1][V] target logits, row i the target's distribution of the
 * token after node i's path; the requests in reqs[0..n_req) are walked (their
 * global indices keep their random streams). Outputs: path [b][gamma+1] the accepted nodes
 * (root first, -1 after the last), n_acc[b] the accepted draft tokens,
 * next_anchor[b], margin[b] = min |u - p| over the tests taken and the final
 * draw's key margin.
 */
void orc_pctree_verify(const orc_dims* d, int N, const int32_t* tok, const int32_t* par, const float* P,
                       uint64_t seed, uint64_t round, const int32_t* reqs, int n_req,
                       int32_t* path, int32_t* n_acc, int32_t* next_anchor, double* margin)
{
    const long V = d->V, g = d->gamma;
#pragma omp parallel for schedule(dynamic, 1)
    for (int q = 0; q < n_req; ++q) {
        const int b = reqs[q];
        double* lt = (double*)malloc(sizeof(double) * (size_t)V);
        double* pr = (double*)malloc(sizeof(double) * (size_t)V);
        const int32_t* tk = tok + (long)b * (N + 1);
        const int32_t* pa = par + (long)b * (N + 1);
        int32_t* ph = path + (long)b * (g + 1);
        for (long i = 0; i <= g; ++i) ph[i] = -1;
        int node = 0, n = 0;
        double mg = INFINITY;
        ph[0] = 0;
        for (;;) {
            const float* row = P + ((long)b * (N + 1) + node) * V;
            for (long v = 0; v < V; ++v) lt[v] = (double)row[v];
            const double L = orc_logsumexp(lt, V);
            for (long v = 0; v < V; ++v) pr[v] = exp(lt[v] - L);
            int next = -1, i = 0;
            for (int ch = node + 1; ch <= N && tk[ch] >= 0; ++ch) {
                if (pa[ch] != node) continue;
                const double q = pr[tk[ch]];
                const double u = orc_uniform(seed, round, ORC_P_TREE_ACCEPT, (uint32_t)b, (uint32_t)node,
                                             (uint32_t)i);
                if (fabs(u - q) < mg) mg = fabs(u - q);
                ++i;
                if (u < q) { next = ch; break; }
                pr[tk[ch]] = 0.0;                        /* removed, the rest renormalised */
                const double keep = 1.0 - q;
                for (long v = 0; v < V; ++v) pr[v] /= keep;
            }
            if (next >= 0) {
                node = next;
                ph[++n] = node;
                continue;
            }
            for (long v = 0; v < V; ++v) lt[v] = pr[v] > 0.0 ? log(pr[v]) : -INFINITY;
            double sm = INFINITY;
            next_anchor[b] = sample_two_level(lt, NULL, NULL, V, seed, round, ORC_P_TREE_BLOCK,
                                              ORC_P_TREE_TOKEN, (uint32_t)b, (uint32_t)node, &sm);
            if (sm < mg) mg = sm;
            break;
        }
        n_acc[b] = n;
        margin[b] = mg;
        free(lt); free(pr);
    }
}

/* ------------------------------------------------------------------ */
/* Training objective of the draft head ([V4.1 blog] "训练：直接优化接受 */
/* 率"; [csdn] section 6, eqs. (9)-(12); [ailearn] 07), teacher-forced:   */
/* position k (0-based) of request b drafts from x_prev = anchor[b] for   */
/* k = 0, else xstar[b][k-1], so every position is independent.          */
/*   z_d = U[b,k] + W1[x_prev] W2,  p_d = softmax(z_d)                    */
/*   p_t = softmax(P[b,k])  (the target's logits at that position)        */
/*   ce  = -log p_d(xstar[b][k])                                (9)       */
/*   l1  = sum_v |p_d(v) - p_t(v)|                              (10)      */
/*   c*  = 1 - l1 / 2 (the position's acceptance probability)             */
/*   bce = -(c* log c + (1 - c*) log(1 - c)),  c = conf[b][k]   (11)      */
/*   loss = (1/B) sum_b sum_k w_k (0.1 ce + 0.9 l1 + 1.0 bce),            */
/*   w_k = exp(-k / tau)                                        (12)      */
/* ------------------------------------------------------------------ */
void orc_train_loss(const orc_dims* d, const float* U, const void* W1, const void* W2,
                    const int32_t* anchor, const int32_t* xstar, const float* P, const float* conf,
                    double tau, double* ce, double* l1, double* bce, double* loss)
{
    const long V = d->V, g = d->gamma;
    double total = 0.0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : total)
    for (long o = 0; o < (long)d->B * g; ++o) {
        const long b = o / g, k = o % g;
        double* z = (double*)malloc(sizeof(double) * (size_t)V);
        double* zt = (double*)malloc(sizeof(double) * (size_t)V);
        const int x_prev = k == 0 ? anchor[b] : xstar[b * g + k - 1];
        markov_logits(d, U + o * V, W1, W2, x_prev, z);
        for (long v = 0; v < V; ++v) zt[v] = (double)P[o * V + v];
        const double Ld = orc_logsumexp(z, V), Lt = orc_logsumexp(zt, V);
        double s = 0.0;
        for (long v = 0; v < V; ++v) s += fabs(exp(z[v] - Ld) - exp(zt[v] - Lt));
        const double c = (double)conf[o], cs = 1.0 - 0.5 * s;
        ce[o] = Ld - z[xstar[o]];
        l1[o] = s;
        bce[o] = -(cs * log(c) + (1.0 - cs) * log(1.0 - c));
        total += exp(-(double)k / tau) * (0.1 * ce[o] + 0.9 * l1[o] + 1.0 * bce[o]);
        free(z); free(zt);
    }
    *loss = total / (double)d->B;
}

/* ------------------------------------------------------------------ */
/* STS: sequential temperature scaling of the confidence head          */
/* ([V4.1 blog] section "confidence head" (a temperature per position, */
/* fitted on held-out data); zdszero "spec_dspark" "STS 校准"; [ailearn] */
/* 05; [csdn] 5.2: left to right, a one-dimensional grid search per    */
/* position minimising the ECE of the cumulative product, earlier      */
/* positions kept fixed).                                              */
/*                                                                     */
/* For n < N held-out blocks and positions k = 1..g: raw[n][k] is the  */
/* confidence logit before the temperature and cstar[n][k] the soft    */
/* label (the position's acceptance probability). With                 */
/*   a_k(n) = prod_{i<=k} sigma(raw[n][i] / T_i),                      */
/*   y_k(n) = prod_{i<=k} cstar[n][i]                                  */
/* (the prefix's joint acceptance factorises by the chain rule), and   */
/* M equal-width bins of [0, 1] (bin floor(a M), a = 1 in the last),   */
/*   ECE_k(T) = (1/N) sum_m | sum_{n: a_k(n) in bin m}                   */
/*                             (a_k(n) - y_k(n)) |,                     */
/* T_k is the first grid value minimising ECE_k given T_1..T_{k-1}.    */
/* margin_out[k] = second-best ECE - best ECE (INFINITY if G == 1).    */
/* ------------------------------------------------------------------ */
void orc_sts_fit(int N, int g, const float* raw, const float* cstar, int G, const float* Tgrid,
                 int M, float* T_out, double* ece_out, double* margin_out)
{
    double* a = (double*)malloc(sizeof(double) * (size_t)N);
    double* y = (double*)malloc(sizeof(double) * (size_t)N);
    double* yk = (double*)malloc(sizeof(double) * (size_t)N);
    double* S = (double*)malloc(sizeof(double) * (size_t)M);
    for (int n = 0; n < N; ++n) { a[n] = 1.0; y[n] = 1.0; }
    for (int k = 0; k < g; ++k) {
        for (int n = 0; n < N; ++n) yk[n] = y[n] * (double)cstar[(size_t)n * g + k];
        double best = INFINITY, second = INFINITY;
        int gbest = 0;
        for (int gi = 0; gi < G; ++gi) {
            const double T = (double)Tgrid[gi];
            for (int m = 0; m < M; ++m) S[m] = 0.0;
            for (int n = 0; n < N; ++n) {
                const double c = 1.0 / (1.0 + exp(-(double)raw[(size_t)n * g + k] / T));
                const double an = a[n] * c;
                int m = (int)floor(an * M);
                if (m > M - 1) m = M - 1;
                if (m < 0) m = 0;
                S[m] += an - yk[n];
            }
            double e = 0.0;
            for (int m = 0; m < M; ++m) e += fabs(S[m]);
            e /= (double)N;
            if (e < best) { second = best; best = e; gbest = gi; }
            else if (e < second) second = e;
        }
        T_out[k] = Tgrid[gbest];
        ece_out[k] = best;
        margin_out[k] = second - best;
        const double Tk = (double)Tgrid[gbest];
        for (int n = 0; n < N; ++n) {
            a[n] *= 1.0 / (1.0 + exp(-(double)raw[(size_t)n * g + k] / Tk));
            y[n] = yk[n];
        }
    }
    free(a); free(y); free(yk); free(S);
}

/* ------------------------------------------------------------------ */
/* Generic helpers exposed for pin tests                               */
/* ------------------------------------------------------------------ */
/* one exact draw from weights exp(logw) with the two-level sampler */
int orc_sample(const double* logw, long V, uint64_t seed, uint64_t round,
               uint32_t pblk, uint32_t ptok, uint32_t b, uint32_t j, double* margin)
{
    return sample_two_level(logw, NULL, NULL, V, seed, round, pblk, ptok, b, j, margin);
}

/* one exact draw with the draft's stream (purposes draft block / draft token) */
int orc_sample_draft(const double* logw, long V, uint64_t seed, uint64_t round,
                     uint32_t b, uint32_t j, double* margin)
{
    return sample_two_level(logw, NULL, NULL, V, seed, round, ORC_P_DRAFT_BLOCK, ORC_P_DRAFT_TOKEN,
                            b, j, margin);
}

/* residual draw for explicit p_t, p_d (pin tests); returns -1 if no mass */
int orc_residual(const double* pt, const double* pd, long V, uint64_t seed,
                 uint64_t round, uint32_t b, uint32_t j, double* margin)
{
    double* lw = (double*)malloc(sizeof(double) * (size_t)V);
    for (long v = 0; v < V; ++v) lw[v] = pt[v] > pd[v] ? log(pt[v] - pd[v]) : -INFINITY;
    int out = sample_two_level(lw, NULL, NULL, V, seed, round, ORC_P_RESID_BLOCK,
                               ORC_P_RESID_TOKEN, b, j, margin);
    free(lw);
    return out;
}

/* the Markov logits of one position (bias GEMM pin) */
void orc_markov_logits(const orc_dims* d, const float* Urow, const void* W1,
                       const void* W2, int x_prev, double* z)
{
    markov_logits(d, Urow, W1, W2, x_prev, z);
}

int orc_block_width(void) { return ORC_BLOCK; }

void orc_set_threads(int n)
{
#ifdef _OPENMP
    extern void omp_set_num_threads(int);
    omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int orc_get_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
