/*
 * sv_oracle.c -- plain, slow, fp64 CPU oracle for the batched speculative-decoding verifier.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's CPU-baseline
 * leg load this library. The GPU library neither links nor calls it, and the two share no
 * source, header, table or helper: everything below is written from the pages' definitions.
 *
 * What it computes, and where each rule comes from:
 *   - p = softmax(logits / T) per position, in fp64 with the maximum subtracted.
 *     ("投机解码" [Speculative decoding], rustineverything, section 接受规则为什么不改变分布
 *     [why the acceptance rule keeps the distribution]: p already carries temperature.)
 *   - Standard rejection: accept draft x with probability min(1, p(x)/q(x)); on the first
 *     rejection draw from max(0, p - q) / Z; if all k drafts are accepted draw one bonus token
 *     from the (k+1)-th position.  (same page and section, subsection 采样：标准拒绝采样;
 *     also the page's opening conclusions: one round emits 1 to k+1 tokens.)
 *   - One-hot draft (target-only chain): q = delta_x, so the accept probability is p(x) and
 *     the residual is p with x zeroed. (same section, subsection 默认路径：草稿当 one-hot;
 *     "The speculative decoding zoo", mlinterviewnotes 06-06, verification-method section.)
 *   - Greedy: accept while the draft equals the target argmax; at the first mismatch (or after
 *     all k) emit the argmax. ("The speculative decoding zoo", DFlash section: matches /
 *     cumprod / bonus; "投机解码", subsection 贪心.)
 *   - Tree, target-only: one coin per tree level; children are tried in order with a running
 *     sum of their target probabilities; the first child with p > 0 and coin < running sum is
 *     accepted; if none is, draw from p with the tried children zeroed. (same section,
 *     subsection SGLang 默认：只看目标概率，可以验证一棵树.)  Tree, greedy: follow the child
 *     whose token equals the argmax.
 *   - q(x) = 0 accepts iff p(x) > 0 ("投机解码", section 对照：mistral.rs), which the strict
 *     test u*q < p reproduces.
 *
 *   - Block verification ("The speculative decoding zoo", mlinterviewnotes 06-06, the block
 *     branch of the rejection sampler, citing Sun et al. 2024, arXiv:2403.10444): the prefix of
 *     L drafts is judged by its joint weight w_L and the residual mass r_L at the next position,
 *     h_L = r_L / (r_L + 1 - w_L) (h = 1 when that denominator is 0), h_k = w_k for the last
 *     draft; the accepted length is the largest L with a passing test.
 *
 * Readings where the pages are silent:
 *   - Uniforms: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
 *     1, 2, 3", SC'11), counter = (slot, request, offset_lo, offset_hi), key = (seed_lo,
 *     seed_hi). Word 0 -> u (accept test / tree coin), word 1 -> v (the draw at the stop slot).
 *     u01(x) = (x >> 8) * 2^-24.  slot = draft position (chain) or depth (tree).
 *   - Accept iff u*q(x) < p(x) (strict), u in [0,1).
 *   - Draws: inverse CDF in ascending token order: the smallest y with C(y) > v*Z; if rounding
 *     leaves none, the last y with nonzero weight.  If Z <= 0 the draw falls back to p.
 *   - Argmax ties go to the lowest index.
 *   - A draft id of -1 ends the chain at that slot; the token there is drawn from p.
 *   - Tree: node 0 is the root, parents[0] = -1, 0 <= parents[j] < j; children are tried in
 *     ascending node index; a child whose token is -1 is absent (never tried).
 *   - Rows holding NaN or +inf, or no finite logit, are invalid (status 2).
 *   - Block verification (the pages print only h): w_0 = 1, w_{i+1} = min(1, w_i p_i(x)/q_i(x))
 *     (a q of 0 gives 1 when w_i p_i(x) > 0), r_L = sum_y max(w_L p_L(y) - q_L(y), 0) with
 *     q_L the one-hot of the next draft when there are no draft probabilities; candidate
 *     length L passes iff u_L < h_L, u_L being word 0 of slot L - 1; the token after the
 *     accepted prefix is drawn from max(w_j p_j - q_j, 0) / Z (from p_j when j reaches the
 *     last draft or an absent draft), with v of slot j.  These follow Sun et al.'s algorithm.
 *
 *   - Relaxed thresholds ("投机解码", section 接受规则为什么不改变分布, subsection SGLang 默认 and
 *     its closing remark on the two thresholds): in target-only decisions a candidate c with
 *     p(c) > 0 is accepted when coin < (running sum of the tried candidates' p) / threshold_acc,
 *     or when p(c) >= threshold_single.  Both default to 1, which is the exact rule; smaller values
 *     accept more and change the output distribution.  A chain without draft probabilities is
 *     the one-candidate case (running sum = p(x)).  With draft probabilities the thresholds do
 *     not apply (reading: the pages give them only for the target-only kernel).
 *   - Top-k / top-p: p is the target distribution after temperature and top-k / top-p ("投机解码",
 *     section 接受规则为什么不改变分布: p already carries temperature, top-k and top-p).  The pages do
 *     not define the filters; readings: top-k keeps every token whose logit reaches the k-th
 *     largest logit (ties at the boundary all kept; k <= 0 or k >= V: off); top-p then keeps,
 *     among those, the fewest whole value levels from the top whose probability (renormalised
 *     over the top-k set) reaches top_p (top_p >= 1: off); p is renormalised over what is kept.
 *     A top-p crossing within 1e-6 (relative) of its target is flagged as a boundary case.
 *   - Per-request temperature in one batch ("The speculative decoding zoo", DSpark section:
 *     accept_draft_tokens runs the greedy rule when the whole batch is greedy, the sampling rule
 *     when none is, and both, merged, when the batch is mixed): request b uses T_b; T_b = 0
 *     means greedy for that request (argmax rule), T_b > 0 the sampling rule with p at T_b.
 *
 * Boundary draws: a decision whose operands lie within 1e-6 (relative) of the decision
 * boundary is flagged, because an fp32 implementation may legitimately decide it the other way.
 *
 * Pinned by tests (not by re-typing these formulas): Philox against the Random123 known-answer
 * vectors; the decision functions by integrating them over a uniform grid (emitted distribution
 * equals p for any q, the toy acceptance rates printed on "投机解码" section 数学验证), by the
 * closed form E = (1 - a^(k+1)) / (1 - a), by a Markov-chain joint distribution, and by the
 * greedy argmax-prefix rule.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SVO_MAX_ROWS 64 /* rows per request (k + 1) the block verifier accepts */
#define SVO_DT_BF16 0
#define SVO_DT_FP32 1
#define SVO_DT_FP64 2

#define SVO_OK 0
#define SVO_BAD_TOKEN 1
#define SVO_BAD_ROW 2
#define SVO_BAD_TREE 3
#define SVO_DUP_SIBLING 4
#define SVO_ENOMEM 100
#define SVO_EINVAL 101

#define SVO_BOUNDARY_REL 1e-6

/* ------------------------------------------------------------------------------------------ */
/* Philox4x32-10, from Salmon et al. (SC'11): ten rounds of two 32x32->64 multiplies with the */
/* paper's multipliers, and a Weyl sequence on the key between rounds.                        */
/* ------------------------------------------------------------------------------------------ */
void svo_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u; /* golden-ratio Weyl increment */
            k1 += 0xBB67AE85u; /* sqrt(3) - 1 Weyl increment */
        }
        uint64_t prod0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
        uint64_t prod1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
        uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

/* The top 24 bits as a uniform on [0, 1): exact in both fp32 and fp64. */
double svo_u01(uint32_t x) { return (double)(x >> 8) * (1.0 / 16777216.0); }

/* The two uniforms of one (slot, request) pair. */
void svo_uniform_pair(uint64_t seed, uint64_t offset, uint32_t slot, uint32_t request,
                      double *u, double *v)
{
    uint32_t ctr[4] = {slot, request, (uint32_t)offset, (uint32_t)(offset >> 32)};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    svo_philox4x32_10(ctr, key, out);
    *u = svo_u01(out[0]);
    *v = svo_u01(out[1]);
}

/* ------------------------------------------------------------------------------------------ */
/* Loading logits: bf16 (bit patterns), fp32 or fp64, always widened exactly to fp64.         */
/* ------------------------------------------------------------------------------------------ */
static double svo_load(const void *base, int dtype, int64_t idx)
{
    if (dtype == SVO_DT_BF16) {
        uint32_t w = (uint32_t)((const uint16_t *)base)[idx] << 16;
        float f;
        memcpy(&f, &w, sizeof f);
        return (double)f;
    }
    if (dtype == SVO_DT_FP32) return (double)((const float *)base)[idx];
    return ((const double *)base)[idx];
}

/* A row is usable when it holds no NaN, no +inf, and at least one finite value. */
static int svo_row_status(const void *logits, int dtype, int64_t row, int64_t V)
{
    int any_finite = 0;
    for (int64_t y = 0; y < V; ++y) {
        double l = svo_load(logits, dtype, row * V + y);
        if (isnan(l) || l == INFINITY) return SVO_BAD_ROW;
        if (isfinite(l)) any_finite = 1;
    }
    return any_finite ? SVO_OK : SVO_BAD_ROW;
}

/* p = softmax(l / T): divide by T, subtract the maximum, exponentiate, normalise. */
int svo_softmax_row(const void *logits, int dtype, int64_t row, int64_t V, double T, double *p)
{
    int st = svo_row_status(logits, dtype, row, V);
    if (st != SVO_OK) return st;
    double zmax = -INFINITY;
    for (int64_t y = 0; y < V; ++y) {
        double z = svo_load(logits, dtype, row * V + y) / T;
        p[y] = z;
        if (z > zmax) zmax = z;
    }
    double sum = 0.0;
    for (int64_t y = 0; y < V; ++y) {
        p[y] = exp(p[y] - zmax);
        sum += p[y];
    }
    for (int64_t y = 0; y < V; ++y) p[y] /= sum;
    return SVO_OK;
}

/* Top-k then top-p on a row's probabilities p (from the logits of `row`), in place: zero what
 * is not kept, renormalise.  Sets *boundary when a top-p decision is within 1e-6 of its target. */
static int svo_cmp_desc(const void *a, const void *b)
{
    double x = *(const double *)a, y = *(const double *)b;
    return x < y ? 1 : (x > y ? -1 : 0);
}

int svo_filter_row(const void *logits, int dtype, int64_t row, int64_t V, int top_k, double top_p,
                   double *p, int32_t *boundary)
{
    int use_k = top_k >= 1 && top_k < V, use_p = top_p < 1.0;
    if (!use_k && !use_p) return SVO_OK;
    double *x = (double *)malloc(sizeof(double) * (size_t)V);
    double *srt = (double *)malloc(sizeof(double) * (size_t)V);
    if (!x || !srt) {
        free(x);
        free(srt);
        return SVO_ENOMEM;
    }
    for (int64_t y = 0; y < V; ++y) x[y] = srt[y] = svo_load(logits, dtype, row * V + y);
    qsort(srt, (size_t)V, sizeof(double), svo_cmp_desc);
    double tau = -INFINITY;
    if (use_k) tau = srt[top_k - 1]; /* the k-th largest logit */
    if (use_p) {
        /* Mass of the top-k set, then whole value levels from the top until top_p of it. */
        double zk = 0.0;
        for (int64_t y = 0; y < V; ++y)
            if (x[y] >= tau) zk += p[y];
        double target = top_p * zk, cum = 0.0;
        int64_t i = 0;
        double taup = tau;
        while (i < V && srt[i] >= tau) {
            double level = srt[i], m = 0.0;
            for (int64_t y = 0; y < V; ++y)
                if (x[y] == level) m += p[y];
            while (i < V && srt[i] == level) ++i;
            double before = cum;
            cum += m;
            if (fabs(cum - target) < 1e-6 * zk || fabs(before - target) < 1e-6 * zk) *boundary = 1;
            if (cum >= target) {
                taup = level;
                break;
            }
        }
        if (taup > tau) tau = taup;
    }
    double z = 0.0;
    for (int64_t y = 0; y < V; ++y) {
        if (!(x[y] >= tau)) p[y] = 0.0;
        z += p[y];
    }
    for (int64_t y = 0; y < V; ++y) p[y] /= z;
    free(x);
    free(srt);
    return SVO_OK;
}

/* Index of the largest logit, the lowest index on ties. */
int svo_argmax_row(const void *logits, int dtype, int64_t row, int64_t V, int32_t *idx)
{
    int st = svo_row_status(logits, dtype, row, V);
    if (st != SVO_OK) return st;
    double best = -INFINITY;
    int32_t arg = -1;
    for (int64_t y = 0; y < V; ++y) {
        double l = svo_load(logits, dtype, row * V + y);
        if (arg < 0 || l > best) {
            best = l;
            arg = (int32_t)y;
        }
    }
    *idx = arg;
    return SVO_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* Inverse-CDF draw from unnormalised weights r[0..V-1] in ascending token order.              */
/* Returns the smallest y with C(y) = r[0] + ... + r[y] > v * Z; when rounding leaves no such */
/* y, the last y with r[y] > 0.  Returns -1 when Z <= 0.  Flags a boundary draw when v*Z lies */
/* within 1e-6 * Z of either end of the chosen token's interval.                               */
/* ------------------------------------------------------------------------------------------ */
static int64_t svo_inverse_cdf(const double *r, int64_t V, double v, int32_t *boundary,
                               double *Z_out)
{
    double Z = 0.0;
    for (int64_t y = 0; y < V; ++y) Z += r[y];
    *Z_out = Z;
    if (!(Z > 0.0)) return -1;
    double t = v * Z, c = 0.0;
    int64_t last = -1;
    for (int64_t y = 0; y < V; ++y) {
        if (!(r[y] > 0.0)) continue;
        double c_before = c;
        c += r[y];
        last = y;
        if (c > t) {
            if (fabs(t - c) < SVO_BOUNDARY_REL * Z || fabs(t - c_before) < SVO_BOUNDARY_REL * Z)
                *boundary = 1;
            return y;
        }
    }
    *boundary = 1; /* v*Z reached the total: the draw sits on the top boundary */
    return last;
}

/* ------------------------------------------------------------------------------------------ */
/* Chain verification of one request with explicit uniforms.                                   */
/*   p      : (k+1) x V target probabilities (row i conditions on the prefix and drafts < i)  */
/*   q      : k x V draft probabilities, or NULL for a one-hot draft                           */
/*   drafts : k draft ids in [-1, V)                                                           */
/*   u, v   : k+1 uniforms each; u[i] tests draft i, v[j] draws the token at the stop slot j  */
/*   tokens : k+1 outputs (accepted drafts, then the drawn token, then -1)                     */
/*   probs  : (k+1) x 3 or NULL: p_i(x_i), q_i(x_i), and Z at the stop slot                    */
/*   work   : V doubles                                                                        */
/* ------------------------------------------------------------------------------------------ */
int svo_chain_core_t(const double *p, const double *q, const int32_t *drafts, int k, int64_t V,
                     const double *u, const double *v, double thr_single, double thr_acc,
                     int32_t *tokens, int32_t *accept_len, int32_t *boundary, double *probs,
                     double *work)
{
    for (int i = 0; i <= k; ++i) tokens[i] = -1;
    if (probs) memset(probs, 0, sizeof(double) * 3 * (size_t)(k + 1));
    *accept_len = -1;
    for (int i = 0; i < k; ++i)
        if (drafts[i] < -1 || drafts[i] >= V) return SVO_BAD_TOKEN;

    if (probs) {
        for (int i = 0; i < k; ++i) {
            if (drafts[i] < 0) continue;
            probs[3 * i + 0] = p[(int64_t)i * V + drafts[i]];
            probs[3 * i + 1] = q ? q[(int64_t)i * V + drafts[i]] : 1.0;
        }
    }

    /* Left to right: the first draft that is absent or rejected ends the chain. */
    int j = k;
    int residual = 0; /* 1: draw from max(0, p - q); 0: draw from p (bonus or absent draft) */
    for (int i = 0; i < k; ++i) {
        int32_t x = drafts[i];
        if (x < 0) {
            j = i;
            break;
        }
        double px = p[(int64_t)i * V + x];
        int accept;
        if (q) {
            double qx = q[(int64_t)i * V + x];
            double lhs = u[i] * qx;
            if (fabs(lhs - px) < SVO_BOUNDARY_REL * fmax(qx, px)) *boundary = 1;
            accept = lhs < px;
        } else {
            /* One candidate: running sum = p(x); thresholds of 1 give the exact test u < p(x). */
            double a = px / thr_acc;
            if (fabs(u[i] - a) < SVO_BOUNDARY_REL * fmax(1.0, a)) *boundary = 1;
            if (thr_single < 1.0 && fabs(px - thr_single) < SVO_BOUNDARY_REL) *boundary = 1;
            accept = px > 0.0 && (u[i] < a || px >= thr_single);
        }
        if (accept) {
            tokens[i] = x;
            continue;
        }
        j = i;
        residual = 1;
        break;
    }

    const double *pj = p + (int64_t)j * V;
    if (residual) {
        int32_t x = drafts[j];
        for (int64_t y = 0; y < V; ++y) {
            double qy = q ? q[(int64_t)j * V + y] : (y == x ? 1.0 : 0.0);
            work[y] = fmax(0.0, pj[y] - qy);
        }
    } else {
        for (int64_t y = 0; y < V; ++y) work[y] = pj[y];
    }
    double Z;
    int64_t tok = svo_inverse_cdf(work, V, v[j], boundary, &Z);
    if (tok < 0) { /* Z <= 0 in floating point: draw from p instead */
        for (int64_t y = 0; y < V; ++y) work[y] = pj[y];
        tok = svo_inverse_cdf(work, V, v[j], boundary, &Z);
    }
    tokens[j] = (int32_t)tok;
    *accept_len = j;
    if (probs) probs[3 * j + 2] = Z;
    return SVO_OK;
}

int svo_chain_core(const double *p, const double *q, const int32_t *drafts, int k, int64_t V,
                   const double *u, const double *v, int32_t *tokens, int32_t *accept_len,
                   int32_t *boundary, double *probs, double *work)
{
    return svo_chain_core_t(p, q, drafts, k, V, u, v, 1.0, 1.0, tokens, accept_len, boundary, probs,
                            work);
}

/* ------------------------------------------------------------------------------------------ */
/* Tree verification of one request with explicit uniforms.                                    */
/*   mode 0 (greedy): amax[n] is the argmax of node n's row; p is unused.                      */
/*   mode 1 (target-only): p is N x V; coin[d] and v[d] are the uniforms of depth d.           */
/*   out_tokens[0..L]  : accepted node tokens, then the token drawn at the stop node          */
/*   accept_index[0..L]: node 0, then the accepted nodes                                      */
/* ------------------------------------------------------------------------------------------ */
/* Structural checks of one request's tree; returns the largest fault code found (0 if none). */
int svo_tree_check(const int32_t *tokens, const int32_t *parents, int N, int64_t V, int mode)
{
    int st = SVO_OK;
    for (int j = 1; j < N; ++j)
        if (tokens[j] < -1 || tokens[j] >= V) st = SVO_BAD_TOKEN;
    if (parents[0] != -1) st = SVO_BAD_TREE;
    for (int j = 1; j < N; ++j)
        if (parents[j] < 0 || parents[j] >= j) st = SVO_BAD_TREE;
    if (mode == 1) {
        for (int a = 1; a < N; ++a)
            for (int b = a + 1; b < N; ++b)
                if (parents[a] == parents[b] && tokens[a] >= 0 && tokens[a] == tokens[b])
                    st = SVO_DUP_SIBLING;
    }
    return st;
}

int svo_tree_core_t(const double *p, const int32_t *amax, const int32_t *tokens,
                    const int32_t *parents, int N, int64_t V, int mode, const double *coin,
                    const double *v, double thr_single, double thr_acc, int32_t *out_tokens,
                    int32_t *accept_index, int32_t *accept_len, int32_t *boundary, double *work)
{
    for (int i = 0; i < N; ++i) {
        out_tokens[i] = -1;
        accept_index[i] = -1;
    }
    *accept_len = -1;
    int st = svo_tree_check(tokens, parents, N, V, mode);
    if (st != SVO_OK) return st;

    int cur = 0, depth = 0, L = 0;
    accept_index[0] = 0;
    for (;;) {
        int next = -1;
        if (mode == 0) {
            int32_t am = amax[cur];
            for (int ch = 1; ch < N; ++ch) {
                if (parents[ch] != cur || tokens[ch] < 0) continue;
                if (tokens[ch] == am) {
                    next = ch;
                    break;
                }
            }
            if (next < 0) {
                out_tokens[L] = am;
                break;
            }
        } else {
            const double *pc = p + (int64_t)cur * V;
            double c = coin[depth], acc = 0.0;
            for (int ch = 1; ch < N; ++ch) {
                if (parents[ch] != cur || tokens[ch] < 0) continue;
                double pt = pc[tokens[ch]];
                acc += pt;
                double a = acc / thr_acc;
                if (pt > 0.0 && fabs(c - a) < SVO_BOUNDARY_REL * fmax(1.0, a)) *boundary = 1;
                if (pt > 0.0 && thr_single < 1.0 && fabs(pt - thr_single) < SVO_BOUNDARY_REL) *boundary = 1;
                if (pt > 0.0 && (c < a || pt >= thr_single)) {
                    next = ch;
                    break;
                }
            }
            if (next < 0) {
                /* No child accepted: draw from p with every tried child's token zeroed. */
                for (int64_t y = 0; y < V; ++y) work[y] = pc[y];
                for (int ch = 1; ch < N; ++ch)
                    if (parents[ch] == cur && tokens[ch] >= 0) work[tokens[ch]] = 0.0;
                double Z;
                int64_t tok = svo_inverse_cdf(work, V, v[depth], boundary, &Z);
                if (tok < 0) {
                    for (int64_t y = 0; y < V; ++y) work[y] = pc[y];
                    tok = svo_inverse_cdf(work, V, v[depth], boundary, &Z);
                }
                out_tokens[L] = (int32_t)tok;
                break;
            }
        }
        out_tokens[L] = tokens[next];
        ++L;
        accept_index[L] = next;
        cur = next;
        ++depth;
    }
    *accept_len = L;
    return SVO_OK;
}

int svo_tree_core(const double *p, const int32_t *amax, const int32_t *tokens,
                  const int32_t *parents, int N, int64_t V, int mode, const double *coin,
                  const double *v, int32_t *out_tokens, int32_t *accept_index,
                  int32_t *accept_len, int32_t *boundary, double *work)
{
    return svo_tree_core_t(p, amax, tokens, parents, N, V, mode, coin, v, 1.0, 1.0, out_tokens,
                           accept_index, accept_len, boundary, work);
}

/* ------------------------------------------------------------------------------------------ */
/* Batched entry points over a [B][rows][V] logits array.  req_ids (n_req entries, or NULL   */
/* for 0..n_req-1) selects which requests to verify; the request index is also the Philox    */
/* counter's request word.  Outputs are indexed by position in req_ids.                       */
/* ------------------------------------------------------------------------------------------ */
int svo_verify_greedy(const void *logits, int dtype, const int32_t *drafts, int B, int k,
                      int64_t V, const int32_t *req_ids, int n_req, int32_t *out_tokens,
                      int32_t *accept_len, int32_t *status)
{
    if (B < 1 || k < 0 || V < 1 || n_req < 0) return SVO_EINVAL;
    int32_t *amax = (int32_t *)malloc(sizeof(int32_t) * (size_t)(k + 1));
    if (!amax) return SVO_ENOMEM;
    for (int i = 0; i < n_req; ++i) {
        int b = req_ids ? req_ids[i] : i;
        int32_t *tok = out_tokens + (int64_t)i * (k + 1);
        const int32_t *d = drafts + (int64_t)b * k;
        for (int r = 0; r <= k; ++r) tok[r] = -1;
        accept_len[i] = -1;
        status[i] = SVO_OK;
        if (b < 0 || b >= B) {
            free(amax);
            return SVO_EINVAL;
        }
        for (int r = 0; r < k; ++r)
            if (d[r] < -1 || d[r] >= V) status[i] = SVO_BAD_TOKEN;
        for (int r = 0; r <= k; ++r) {
            int st = svo_argmax_row(logits, dtype, (int64_t)b * (k + 1) + r, V, &amax[r]);
            if (st > status[i]) status[i] = st;
        }
        if (status[i] != SVO_OK) continue;
        int j = k;
        for (int r = 0; r < k; ++r) {
            if (d[r] < 0 || d[r] != amax[r]) {
                j = r;
                break;
            }
            tok[r] = d[r];
        }
        tok[j] = amax[j];
        accept_len[i] = j;
    }
    free(amax);
    return SVO_OK;
}

int svo_verify_rejection(const void *logits, int dtype, const int32_t *drafts, const float *q,
                         int B, int k, int64_t V, double T, uint64_t seed, uint64_t offset,
                         const int32_t *req_ids, int n_req, int32_t *out_tokens,
                         int32_t *accept_len, double *out_probs, int32_t *boundary,
                         int32_t *status)
{
    if (B < 1 || k < 0 || V < 1 || n_req < 0 || !(T > 0.0) || !isfinite(T)) return SVO_EINVAL;
    double *p = (double *)malloc(sizeof(double) * (size_t)(k + 1) * (size_t)V);
    double *qd = q ? (double *)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1) * (size_t)V) : NULL;
    double *work = (double *)malloc(sizeof(double) * (size_t)V);
    double *u = (double *)malloc(sizeof(double) * (size_t)(k + 1));
    double *v = (double *)malloc(sizeof(double) * (size_t)(k + 1));
    int rc = SVO_OK;
    if (!p || (q && !qd) || !work || !u || !v) {
        rc = SVO_ENOMEM;
        goto done;
    }
    for (int i = 0; i < n_req; ++i) {
        int b = req_ids ? req_ids[i] : i;
        int32_t *tok = out_tokens + (int64_t)i * (k + 1);
        double *probs = out_probs ? out_probs + (int64_t)i * (k + 1) * 3 : NULL;
        for (int r = 0; r <= k; ++r) tok[r] = -1;
        if (probs) memset(probs, 0, sizeof(double) * 3 * (size_t)(k + 1));
        accept_len[i] = -1;
        boundary[i] = 0;
        status[i] = SVO_OK;
        if (b < 0 || b >= B) {
            rc = SVO_EINVAL;
            goto done;
        }
        const int32_t *d = drafts + (int64_t)b * k;
        for (int r = 0; r < k; ++r)
            if (d[r] < -1 || d[r] >= V) status[i] = SVO_BAD_TOKEN;
        for (int r = 0; r <= k; ++r) {
            int st = svo_softmax_row(logits, dtype, (int64_t)b * (k + 1) + r, V, T,
                                     p + (int64_t)r * V);
            if (st > status[i]) status[i] = st;
        }
        if (status[i] != SVO_OK) continue;
        if (q) {
            const float *qb = q + (int64_t)b * k * V;
            for (int64_t e = 0; e < (int64_t)k * V; ++e) qd[e] = (double)qb[e];
        }
        for (int r = 0; r <= k; ++r) svo_uniform_pair(seed, offset, (uint32_t)r, (uint32_t)b, &u[r], &v[r]);
        status[i] = svo_chain_core(p, qd, d, k, V, u, v, tok, &accept_len[i], &boundary[i], probs,
                                   work);
    }
done:
    free(p);
    free(qd);
    free(work);
    free(u);
    free(v);
    return rc;
}

/* ------------------------------------------------------------------------------------------ */
/* Block verification of one request with explicit uniforms.                                   */
/*   p: (k+1) x V target probabilities; q: k x V draft probabilities, or NULL for one-hot drafts */
/*   u[L-1] judges candidate length L; v[j] draws the token after the accepted prefix j.         */
/* ------------------------------------------------------------------------------------------ */
static double svo_block_q(const double *q, const int32_t *drafts, int row, int64_t V, int64_t y)
{
    if (q) return q[(int64_t)row * V + y];
    return y == drafts[row] ? 1.0 : 0.0;
}

int svo_block_core(const double *p, const double *q, const int32_t *drafts, int k, int64_t V,
                   const double *u, const double *v, int32_t *tokens, int32_t *accept_len,
                   int32_t *boundary, double *work)
{
    if (k < 0 || k + 1 > SVO_MAX_ROWS) return SVO_EINVAL;
    for (int i = 0; i <= k; ++i) tokens[i] = -1;
    *accept_len = -1;
    for (int i = 0; i < k; ++i)
        if (drafts[i] < -1 || drafts[i] >= V) return SVO_BAD_TOKEN;
    int ke = k; /* drafts actually present: an absent draft ends the block */
    for (int i = 0; i < k; ++i)
        if (drafts[i] < 0) {
            ke = i;
            break;
        }

    /* Joint weight of each prefix. */
    double w[SVO_MAX_ROWS + 1];
    w[0] = 1.0;
    for (int i = 0; i < ke; ++i) {
        double px = p[(int64_t)i * V + drafts[i]];
        double qx = svo_block_q(q, drafts, i, V, drafts[i]);
        double next;
        if (w[i] * px <= 0.0) next = 0.0;
        else if (qx <= 0.0) next = 1.0;
        else next = fmin(1.0, w[i] * px / qx);
        w[i + 1] = next;
    }

    /* The largest candidate length whose test passes. */
    int j = 0;
    for (int L = 1; L <= ke; ++L) {
        double h;
        if (L < ke) {
            const double *pl = p + (int64_t)L * V;
            double r = 0.0;
            for (int64_t y = 0; y < V; ++y) r += fmax(0.0, w[L] * pl[y] - svo_block_q(q, drafts, L, V, y));
            double denom = r + 1.0 - w[L];
            h = denom > 0.0 ? r / denom : 1.0;
        } else {
            h = w[L];
        }
        if (fabs(u[L - 1] - h) < SVO_BOUNDARY_REL) *boundary = 1;
        if (u[L - 1] < h) j = L;
    }

    /* The token after the accepted prefix. */
    const double *pj = p + (int64_t)j * V;
    if (j < ke) {
        for (int64_t y = 0; y < V; ++y) work[y] = fmax(0.0, w[j] * pj[y] - svo_block_q(q, drafts, j, V, y));
    } else {
        for (int64_t y = 0; y < V; ++y) work[y] = pj[y];
    }
    double Z;
    int64_t tok = svo_inverse_cdf(work, V, v[j], boundary, &Z);
    if (tok < 0) { /* Z <= 0 in floating point: draw from p instead */
        for (int64_t y = 0; y < V; ++y) work[y] = pj[y];
        tok = svo_inverse_cdf(work, V, v[j], boundary, &Z);
    }
    for (int i = 0; i < j; ++i) tokens[i] = drafts[i];
    tokens[j] = (int32_t)tok;
    *accept_len = j;
    return SVO_OK;
}

int svo_verify_block(const void *logits, int dtype, const int32_t *drafts, const float *q, int B,
                     int k, int64_t V, double T, uint64_t seed, uint64_t offset,
                     const int32_t *req_ids, int n_req, int32_t *out_tokens, int32_t *accept_len,
                     int32_t *boundary, int32_t *status)
{
    if (B < 1 || k < 0 || k + 1 > SVO_MAX_ROWS || V < 1 || n_req < 0 || !(T > 0.0) || !isfinite(T))
        return SVO_EINVAL;
    double *p = (double *)malloc(sizeof(double) * (size_t)(k + 1) * (size_t)V);
    double *qd = q ? (double *)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1) * (size_t)V) : NULL;
    double *work = (double *)malloc(sizeof(double) * (size_t)V);
    double u[SVO_MAX_ROWS + 1], v[SVO_MAX_ROWS + 1];
    int rc = SVO_OK;
    if (!p || (q && !qd) || !work) {
        rc = SVO_ENOMEM;
        goto done;
    }
    for (int i = 0; i < n_req; ++i) {
        int b = req_ids ? req_ids[i] : i;
        int32_t *tok = out_tokens + (int64_t)i * (k + 1);
        for (int r = 0; r <= k; ++r) tok[r] = -1;
        accept_len[i] = -1;
        boundary[i] = 0;
        status[i] = SVO_OK;
        if (b < 0 || b >= B) {
            rc = SVO_EINVAL;
            goto done;
        }
        const int32_t *d = drafts + (int64_t)b * k;
        for (int r = 0; r < k; ++r)
            if (d[r] < -1 || d[r] >= V) status[i] = SVO_BAD_TOKEN;
        for (int r = 0; r <= k; ++r) {
            int st = svo_softmax_row(logits, dtype, (int64_t)b * (k + 1) + r, V, T, p + (int64_t)r * V);
            if (st > status[i]) status[i] = st;
        }
        if (status[i] != SVO_OK) continue;
        if (q) {
            const float *qb = q + (int64_t)b * k * V;
            for (int64_t e = 0; e < (int64_t)k * V; ++e) qd[e] = (double)qb[e];
        }
        for (int r = 0; r <= k; ++r) svo_uniform_pair(seed, offset, (uint32_t)r, (uint32_t)b, &u[r], &v[r]);
        status[i] = svo_block_core(p, qd, d, k, V, u, v, tok, &accept_len[i], &boundary[i], work);
    }
done:
    free(p);
    free(qd);
    free(work);
    return rc;
}

int svo_verify_tree(const void *logits, int dtype, const int32_t *tokens, const int32_t *parents,
                    int B, int N, int64_t V, int mode, double T, uint64_t seed, uint64_t offset,
                    const int32_t *req_ids, int n_req, int32_t *out_tokens,
                    int32_t *accept_index, int32_t *accept_len, int32_t *boundary,
                    int32_t *status)
{
    if (B < 1 || N < 1 || V < 1 || n_req < 0 || (mode != 0 && mode != 1)) return SVO_EINVAL;
    if (mode == 1 && (!(T > 0.0) || !isfinite(T))) return SVO_EINVAL;
    double *p = mode == 1 ? (double *)malloc(sizeof(double) * (size_t)N * (size_t)V) : NULL;
    int32_t *amax = (int32_t *)malloc(sizeof(int32_t) * (size_t)N);
    double *work = (double *)malloc(sizeof(double) * (size_t)V);
    double *coin = (double *)malloc(sizeof(double) * (size_t)N);
    double *v = (double *)malloc(sizeof(double) * (size_t)N);
    int rc = SVO_OK;
    if ((mode == 1 && !p) || !amax || !work || !coin || !v) {
        rc = SVO_ENOMEM;
        goto done;
    }
    for (int i = 0; i < n_req; ++i) {
        int b = req_ids ? req_ids[i] : i;
        int32_t *ot = out_tokens + (int64_t)i * N;
        int32_t *ai = accept_index + (int64_t)i * N;
        for (int r = 0; r < N; ++r) ot[r] = ai[r] = -1;
        accept_len[i] = -1;
        boundary[i] = 0;
        status[i] = SVO_OK;
        if (b < 0 || b >= B) {
            rc = SVO_EINVAL;
            goto done;
        }
        const int32_t *tk = tokens + (int64_t)b * N;
        const int32_t *pa = parents + (int64_t)b * N;
        for (int r = 0; r < N; ++r) {
            int64_t row = (int64_t)b * N + r;
            int st = mode == 1 ? svo_softmax_row(logits, dtype, row, V, T, p + (int64_t)r * V)
                               : svo_argmax_row(logits, dtype, row, V, &amax[r]);
            if (st > status[i]) status[i] = st;
        }
        if (status[i] != SVO_OK) {
            int st = svo_tree_check(tk, pa, N, V, mode);
            if (st > status[i]) status[i] = st;
            continue;
        }
        for (int d = 0; d < N; ++d) svo_uniform_pair(seed, offset, (uint32_t)d, (uint32_t)b, &coin[d], &v[d]);
        status[i] = svo_tree_core(p, amax, tk, pa, N, V, mode, coin, v, ot, ai, &accept_len[i],
                                  &boundary[i], work);
    }
done:
    free(p);
    free(amax);
    free(work);
    free(coin);
    free(v);
    return rc;
}

/* ------------------------------------------------------------------------------------------ */
/* Self-test support: integrate a decision function over a G x G midpoint grid of uniforms.   */
/* ------------------------------------------------------------------------------------------ */

/* One position (k = 1) of the chain: for every draft x with weight w[x] (the draft's own     */
/* distribution), run svo_chain_core at u = (a+1/2)/G, v = (c+1/2)/G and accumulate the first */
/* emitted token's distribution in dist[V] and the accepted mass in *accept_rate.             */
int svo_grid_chain_first_token(const double *p0, const double *q0, const double *w, int64_t V,
                               int G, double *dist, double *accept_rate)
{
    double *p = (double *)malloc(sizeof(double) * 2 * (size_t)V);
    double *work = (double *)malloc(sizeof(double) * (size_t)V);
    if (!p || !work) {
        free(p);
        free(work);
        return SVO_ENOMEM;
    }
    memcpy(p, p0, sizeof(double) * (size_t)V);
    memcpy(p + V, p0, sizeof(double) * (size_t)V);
    for (int64_t y = 0; y < V; ++y) dist[y] = 0.0;
    *accept_rate = 0.0;
    double cell = 1.0 / ((double)G * (double)G);
    for (int64_t x = 0; x < V; ++x) {
        if (!(w[x] > 0.0)) continue;
        int32_t draft = (int32_t)x;
        for (int a = 0; a < G; ++a) {
            double u[2] = {(a + 0.5) / G, 0.5};
            for (int c = 0; c < G; ++c) {
                double v[2] = {(c + 0.5) / G, (c + 0.5) / G};
                int32_t tok[2], len, bnd = 0;
                svo_chain_core(p, q0, &draft, 1, V, u, v, tok, &len, &bnd, NULL, work);
                dist[tok[0]] += w[x] * cell;
                if (len == 1) *accept_rate += w[x] * cell;
            }
        }
    }
    free(p);
    free(work);
    return SVO_OK;
}

/* One level of a target-only tree: the root (row p0) has n_child children with the given     */
/* tokens; integrate the first emitted token over (coin, v) on a G x G grid.                  */
int svo_grid_tree_first_token_t(const double *p0, const int32_t *child_tokens, int n_child,
                                int64_t V, int G, double thr_single, double thr_acc, double *dist,
                                double *accept_rate)
{
    int N = n_child + 1;
    double *p = (double *)malloc(sizeof(double) * (size_t)N * (size_t)V);
    double *work = (double *)malloc(sizeof(double) * (size_t)V);
    int32_t *tokens = (int32_t *)malloc(sizeof(int32_t) * (size_t)N);
    int32_t *parents = (int32_t *)malloc(sizeof(int32_t) * (size_t)N);
    int32_t *ot = (int32_t *)malloc(sizeof(int32_t) * (size_t)N);
    int32_t *ai = (int32_t *)malloc(sizeof(int32_t) * (size_t)N);
    double *coin = (double *)malloc(sizeof(double) * (size_t)N);
    double *v = (double *)malloc(sizeof(double) * (size_t)N);
    int rc = SVO_OK;
    if (!p || !work || !tokens || !parents || !ot || !ai || !coin || !v) {
        rc = SVO_ENOMEM;
        goto done;
    }
    for (int n = 0; n < N; ++n) memcpy(p + (int64_t)n * V, p0, sizeof(double) * (size_t)V);
    tokens[0] = -1;
    parents[0] = -1;
    for (int c = 0; c < n_child; ++c) {
        tokens[c + 1] = child_tokens[c];
        parents[c + 1] = 0;
    }
    for (int64_t y = 0; y < V; ++y) dist[y] = 0.0;
    *accept_rate = 0.0;
    double cell = 1.0 / ((double)G * (double)G);
    for (int a = 0; a < G; ++a) {
        for (int c = 0; c < G; ++c) {
            for (int d = 0; d < N; ++d) {
                coin[d] = (a + 0.5) / G;
                v[d] = (c + 0.5) / G;
            }
            int32_t len, bnd = 0;
            int st = svo_tree_core_t(p, NULL, tokens, parents, N, V, 1, coin, v, thr_single, thr_acc,
                                     ot, ai, &len, &bnd, work);
            if (st != SVO_OK) {
                rc = st;
                goto done;
            }
            dist[ot[0]] += cell;
            if (len >= 1) *accept_rate += cell;
        }
    }
done:
    free(p);
    free(work);
    free(tokens);
    free(parents);
    free(ot);
    free(ai);
    free(coin);
    free(v);
    return rc;
}

int svo_grid_tree_first_token(const double *p0, const int32_t *child_tokens, int n_child,
                              int64_t V, int G, double *dist, double *accept_rate)
{
    return svo_grid_tree_first_token_t(p0, child_tokens, n_child, V, G, 1.0, 1.0, dist, accept_rate);
}

/* ------------------------------------------------------------------------------------------ */
/* Batches with a temperature per request (T_b = 0: greedy for request b) and the relaxed      */
/* thresholds of target-only decisions.  Chain: drafts [B][k], q [B][k][V] or NULL; outputs as */
/* svo_verify_rejection (a greedy request's out_probs stay 0).  Tree: outputs as              */
/* svo_verify_tree; a greedy request walks by argmax, the others by the target-only rule.     */
/* ------------------------------------------------------------------------------------------ */
static int svo_temp_ok(double T) { return T == 0.0 || (T > 0.0 && isfinite(T)); }
static int svo_thr_ok(double t) { return t > 0.0 && t <= 1.0; }

int svo_verify_ex(const void *logits, int dtype, const int32_t *drafts, const float *q, int B,
                  int k, int64_t V, const double *temps, double thr_single, double thr_acc,
                  const int32_t *top_k, const double *top_p,
                  uint64_t seed, uint64_t offset, const int32_t *req_ids, int n_req,
                  int32_t *out_tokens, int32_t *accept_len, double *out_probs, int32_t *boundary,
                  int32_t *status)
{
    if (B < 1 || k < 0 || V < 1 || n_req < 0 || !temps) return SVO_EINVAL;
    if (!svo_thr_ok(thr_single) || !svo_thr_ok(thr_acc)) return SVO_EINVAL;
    if (q && (thr_single != 1.0 || thr_acc != 1.0)) return SVO_EINVAL;
    for (int b = 0; b < B; ++b)
        if (!svo_temp_ok(temps[b]) || (top_p && !(top_p[b] > 0.0))) return SVO_EINVAL;
    double *p = (double *)malloc(sizeof(double) * (size_t)(k + 1) * (size_t)V);
    double *qd = q ? (double *)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1) * (size_t)V) : NULL;
    double *work = (double *)malloc(sizeof(double) * (size_t)V);
    double *u = (double *)malloc(sizeof(double) * (size_t)(k + 1));
    double *v = (double *)malloc(sizeof(double) * (size_t)(k + 1));
    int32_t *amax = (int32_t *)malloc(sizeof(int32_t) * (size_t)(k + 1));
    int rc = SVO_OK;
    if (!p || (q && !qd) || !work || !u || !v || !amax) {
        rc = SVO_ENOMEM;
        goto done;
    }
    for (int i = 0; i < n_req; ++i) {
        int b = req_ids ? req_ids[i] : i;
        int32_t *tok = out_tokens + (int64_t)i * (k + 1);
        double *probs = out_probs ? out_probs + (int64_t)i * (k + 1) * 3 : NULL;
        for (int r = 0; r <= k; ++r) tok[r] = -1;
        if (probs) memset(probs, 0, sizeof(double) * 3 * (size_t)(k + 1));
        accept_len[i] = -1;
        boundary[i] = 0;
        status[i] = SVO_OK;
        if (b < 0 || b >= B) {
            rc = SVO_EINVAL;
            goto done;
        }
        const int32_t *d = drafts + (int64_t)b * k;
        for (int r = 0; r < k; ++r)
            if (d[r] < -1 || d[r] >= V) status[i] = SVO_BAD_TOKEN;
        const double T = temps[b];
        for (int r = 0; r <= k; ++r) {
            int64_t row = (int64_t)b * (k + 1) + r;
            int st = T == 0.0 ? svo_argmax_row(logits, dtype, row, V, &amax[r])
                              : svo_softmax_row(logits, dtype, row, V, T, p + (int64_t)r * V);
            if (st == SVO_OK && T != 0.0)
                st = svo_filter_row(logits, dtype, row, V, top_k ? top_k[b] : 0, top_p ? top_p[b] : 1.0,
                                    p + (int64_t)r * V, &boundary[i]);
            if (st > status[i]) status[i] = st;
        }
        if (status[i] != SVO_OK) continue;
        if (T == 0.0) {
            /* Greedy request: accept while the draft is the row's argmax, then emit the argmax. */
            int j = k;
            for (int r = 0; r < k; ++r) {
                if (d[r] < 0 || d[r] != amax[r]) {
                    j = r;
                    break;
                }
                tok[r] = d[r];
            }
            tok[j] = amax[j];
            accept_len[i] = j;
            continue;
        }
        if (q) {
            const float *qb = q + (int64_t)b * k * V;
            for (int64_t e = 0; e < (int64_t)k * V; ++e) qd[e] = (double)qb[e];
        }
        for (int r = 0; r <= k; ++r) svo_uniform_pair(seed, offset, (uint32_t)r, (uint32_t)b, &u[r], &v[r]);
        status[i] = svo_chain_core_t(p, qd, d, k, V, u, v, thr_single, thr_acc, tok, &accept_len[i],
                                     &boundary[i], probs, work);
    }
done:
    free(p);
    free(qd);
    free(work);
    free(u);
    free(v);
    free(amax);
    return rc;
}

int svo_verify_tree_ex(const void *logits, int dtype, const int32_t *tokens, const int32_t *parents,
                       int B, int N, int64_t V, const double *temps, double thr_single,
                       double thr_acc, const int32_t *top_k, const double *top_p, uint64_t seed,
                       uint64_t offset, const int32_t *req_ids,
                       int n_req, int32_t *out_tokens, int32_t *accept_index, int32_t *accept_len,
                       int32_t *boundary, int32_t *status)
{
    if (B < 1 || N < 1 || V < 1 || n_req < 0 || !temps) return SVO_EINVAL;
    if (!svo_thr_ok(thr_single) || !svo_thr_ok(thr_acc)) return SVO_EINVAL;
    for (int b = 0; b < B; ++b)
        if (!svo_temp_ok(temps[b]) || (top_p && !(top_p[b] > 0.0))) return SVO_EINVAL;
    double *p = (double *)malloc(sizeof(double) * (size_t)N * (size_t)V);
    int32_t *amax = (int32_t *)malloc(sizeof(int32_t) * (size_t)N);
    double *work = (double *)malloc(sizeof(double) * (size_t)V);
    double *coin = (double *)malloc(sizeof(double) * (size_t)N);
    double *v = (double *)malloc(sizeof(double) * (size_t)N);
    int rc = SVO_OK;
    if (!p || !amax || !work || !coin || !v) {
        rc = SVO_ENOMEM;
        goto done;
    }
    for (int i = 0; i < n_req; ++i) {
        int b = req_ids ? req_ids[i] : i;
        int32_t *ot = out_tokens + (int64_t)i * N;
        int32_t *ai = accept_index + (int64_t)i * N;
        for (int r = 0; r < N; ++r) ot[r] = ai[r] = -1;
        accept_len[i] = -1;
        boundary[i] = 0;
        status[i] = SVO_OK;
        if (b < 0 || b >= B) {
            rc = SVO_EINVAL;
            goto done;
        }
        const int mode = temps[b] == 0.0 ? 0 : 1;
        const int32_t *tk = tokens + (int64_t)b * N;
        const int32_t *pa = parents + (int64_t)b * N;
        for (int r = 0; r < N; ++r) {
            int64_t row = (int64_t)b * N + r;
            int st = mode == 1 ? svo_softmax_row(logits, dtype, row, V, temps[b], p + (int64_t)r * V)
                               : svo_argmax_row(logits, dtype, row, V, &amax[r]);
            if (st == SVO_OK && mode == 1)
                st = svo_filter_row(logits, dtype, row, V, top_k ? top_k[b] : 0, top_p ? top_p[b] : 1.0,
                                    p + (int64_t)r * V, &boundary[i]);
            if (st > status[i]) status[i] = st;
        }
        if (status[i] != SVO_OK) {
            int st = svo_tree_check(tk, pa, N, V, mode);
            if (st > status[i]) status[i] = st;
            continue;
        }
        for (int d = 0; d < N; ++d) svo_uniform_pair(seed, offset, (uint32_t)d, (uint32_t)b, &coin[d], &v[d]);
        status[i] = svo_tree_core_t(p, amax, tk, pa, N, V, mode, coin, v, thr_single, thr_acc, ot, ai,
                                    &accept_len[i], &boundary[i], work);
    }
done:
    free(p);
    free(amax);
    free(work);
    free(coin);
    free(v);
    return rc;
}
