/*
 * spec_oracle.c -- CPU oracle for the speculative-decoding verify-and-sample step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no code, header or constant with the CUDA
 * library; it has its own bf16 decoder and its own definitions of every step.
 *
 * What it computes, and where each step comes from:
 *
 *   "Beschleunigung von Sonar durch Spekulation" (Perplexity blog,
 *   English title "Accelerating Sonar through speculation"):
 *     - section "Spekulatives Decoding": a draft of n tokens is checked by the
 *       target, the longest acceptable prefix is kept, and the target gives
 *       one more token for free, so at most n + 1 tokens leave one step;
 *       phase "Akzeptanz" finds the length of the longest acceptable prefix,
 *       phase "Zielgenerierung" samples the target logits at the first
 *       mismatch, or at the end of the draft, for the extra token.
 *     - section "Ziel-Entwurf": acceptance compares the full draft and target
 *       probability distributions; the method cited for it in the page's
 *       reference list is "Fast Inference from Transformers via Speculative
 *       Decoding" (standard speculative sampling).
 *   "Speculative-Decoding / Medusa" blog, section 三 (Attention Tree): the
 *     target's choice (greedy or sampled) at a node is looked up among that
 *     node's candidate children, and verification continues along the child
 *     that matches, until no child matches.
 *
 * Readings taken where the pages are silent:
 *   - accept draft token x_i iff u_i < min(1, p_i(x_i) / q_i(x_i)) (strict),
 *     with p_i = softmax(target_i / T) and q_i = softmax(draft_i / T); for
 *     finite logits both are positive, and the quotient is evaluated as
 *     exp(((t_x - m_t) - (d_x - m_d)) / T) * S_d / S_t so that it stays
 *     defined where p and q both underflow in double;
 *   - at the first rejection j < K the extra token is drawn from the
 *     normalised residual max(0, p_j - q_j); if every draft token was
 *     accepted it is drawn from p_K;
 *   - inverse CDF: the first v whose inclusive cumulative weight C_v exceeds
 *     u_b * W; if rounding leaves none, the last v with nonzero weight;
 *     if W == 0 (possible only through rounding), fall back to p_j and flag;
 *   - greedy mode (T == 0): accept iff x_i == argmax target_i (lowest index on
 *     ties); the extra token is argmax target_j;
 *   - tree: among the children of the current node (increasing node index),
 *     take the first whose token equals argmax of the current node's target
 *     row; stop when none matches or max_depth nodes were accepted; the extra
 *     token is argmax at the last accepted node.
 *   - one token per row (the draft side's own choice of its next token, or
 *     any row a caller wants sampled): a draw from softmax(l / T) by inverse
 *     CDF with the row's uniform, or argmax (lowest index) when T == 0.
 *   - tree attention mask (same page, section 三: a causal-style mask under
 *     which no token attends to a token of another path): row i holds node
 *     i and every ancestor of node i; depth[i] is the number of edges from
 *     the root (the token's offset in position).
 *   - MTP token plug-in ("Beschleunigung von Sonar durch Spekulation",
 *     sections "MTP" and "MTP-Zeitplan für ein einzelnes Token"): the draft
 *     layer at position i reads the target's hidden state H_i together with
 *     the token that follows position i, so its input tokens are the target's
 *     input tokens of the step shifted left by one; after verification a
 *     kernel writes the target's next tokens into their places, and the
 *     draft runs over the same positions as the target (work past the
 *     accepted prefix is redundant).  Reading: row b of the target's input is
 *     (the token the step started from, x_0 .. x_{K-1}); the draft's input row
 *     is next[i] = in[i + 1] for i < K and next[K] = pad, and then the n_b
 *     emitted tokens (x_0 .. x_{j-1} and the extra token) overwrite positions
 *     0 .. n_b - 1; the sequence length grows by n_b, on the device, with no
 *     host round trip.  A count outside [0, K + 1] leaves the row shifted,
 *     the length unchanged, and is reported.
 *   - sparse candidate tree ("Speculative-Decoding / Medusa" blog, section
 *     四): with a_k^(i) the accuracy of head k's i-th ranked token, taken as
 *     independent, the node reached by the rank path [i_1 .. i_m] is accepted
 *     with probability prod_j a_j^(i_j), E[L] is the sum of that product over
 *     the tree's non-root nodes, and the tree is grown from the root by adding,
 *     one node at a time, the candidate (a child of a node already in the
 *     tree) whose product is largest, up to a fixed node count.  Readings:
 *     the product is taken left to right from 1; equal products go to the
 *     smaller depth, then to the lexicographically smaller rank path; nodes
 *     are numbered by (depth, rank path), so every parent precedes its
 *     children; a node count above the full tree's size gives the full tree.
 *   - tree, sampling mode (the page's "Greedy或者Sampling"): the target's
 *     choice at node n is a draw from softmax(target_n / T) by inverse CDF
 *     with the caller's uniform u[b, n]; the walk is the greedy walk with that
 *     draw in place of the argmax, and the extra token is the draw at the last
 *     accepted node.
 *
 * Precision: every logit is widened to double (fp32 directly; bf16 by placing
 * its 16 bits in the high half of an IEEE single), and all arithmetic is
 * double, summed sequentially in vocabulary order.  The temperature is taken
 * as the same single-precision value the GPU path receives, widened.
 *
 * Parallelism: sequences are independent problems; an OpenMP loop over them
 * changes no arithmetic inside a sequence.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F32 0
#define ORACLE_BF16 1

/* flag bits returned per sequence */
#define ORACLE_FLAG_ZERO_RESIDUAL 1u /* W == 0 at the first rejection: fell back to p_j */
#define ORACLE_FLAG_BAD_TOKEN 2u     /* a draft token outside [0, V) */

/* One logit, widened to double.  bf16 is the upper half of an IEEE single. */
static double logit_at(const void *base, int dtype, size_t idx) {
    if (dtype == ORACLE_F32) return (double)((const float *)base)[idx];
    uint16_t h = ((const uint16_t *)base)[idx];
    uint32_t w = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* p[v] = exp((l_v - m) / T) / S with m = max_v l_v and S = sum_v exp((l_v - m) / T),
 * summed sequentially; m and S are returned too. */
static void softmax_row(const void *logits, int dtype, size_t row, int V, double T, double *p,
                        double *m_out, double *S_out) {
    size_t off = row * (size_t)V;
    double m = -INFINITY;
    for (int v = 0; v < V; ++v) {
        double l = logit_at(logits, dtype, off + v);
        if (l > m) m = l;
    }
    double S = 0.0;
    for (int v = 0; v < V; ++v) {
        p[v] = exp((logit_at(logits, dtype, off + v) - m) / T);
        S += p[v];
    }
    for (int v = 0; v < V; ++v) p[v] /= S;
    if (m_out) *m_out = m;
    if (S_out) *S_out = S;
}

/* Lowest index of the maximum logit of one row. */
static int argmax_row(const void *logits, int dtype, size_t row, int V) {
    size_t off = row * (size_t)V;
    int best = 0;
    double bv = logit_at(logits, dtype, off);
    for (int v = 1; v < V; ++v) {
        double l = logit_at(logits, dtype, off + v);
        if (l > bv) { bv = l; best = v; }
    }
    return best;
}

/* Inverse-CDF draw from nonnegative weights w[0..V).  Returns the token and
 * writes the cumulative interval [lo, hi) of the chosen token, normalised by W. */
static int inverse_cdf(const double *w, int V, double u, double *lo, double *hi) {
    double W = 0.0;
    for (int v = 0; v < V; ++v) W += w[v];
    double target = u * W;
    double C = 0.0;
    for (int v = 0; v < V; ++v) {
        double Cprev = C;
        C += w[v];
        if (C > target) {
            *lo = Cprev / W;
            *hi = C / W;
            return v;
        }
    }
    /* rounding left no index: the last token with nonzero weight */
    int last = -1;
    for (int v = 0; v < V; ++v)
        if (w[v] > 0.0) last = v;
    if (last < 0) { *lo = *hi = 0.0; return 0; }
    double Cl = 0.0;
    for (int v = 0; v < last; ++v) Cl += w[v];
    *lo = Cl / W;
    *hi = (Cl + w[last]) / W;
    return last;
}

/* The extra token at row j of sequence b (sampling mode): residual
 * max(0, p_j - q_j) if j < K, else p_K.  Returns the token; lo/hi as above. */
static int extra_token_sampled(const void *target, const void *draft, int dtype, int b, int K, int V,
                               int j, double T, double u, double *w, double *pj, double *qj,
                               double *lo, double *hi, uint32_t *flag) {
    softmax_row(target, dtype, (size_t)b * (K + 1) + j, V, T, pj, NULL, NULL);
    if (j < K) {
        softmax_row(draft, dtype, (size_t)b * K + j, V, T, qj, NULL, NULL);
        double W = 0.0;
        for (int v = 0; v < V; ++v) {
            double d = pj[v] - qj[v];
            w[v] = d > 0.0 ? d : 0.0;
            W += w[v];
        }
        if (W > 0.0) return inverse_cdf(w, V, u, lo, hi);
        *flag |= ORACLE_FLAG_ZERO_RESIDUAL;
    }
    return inverse_cdf(pj, V, u, lo, hi);
}

/*
 * Linear verify of B sequences with K draft tokens each.
 *   target [B, K+1, V], draft [B, K, V] (ignored when T == 0), row-major.
 *   draft_tokens [B, K]; u_accept [B, K]; u_bonus [B] or NULL (no extra token).
 * Outputs: accept_len [B]; out_tokens [B, K+1] (accepted draft tokens, then the
 * extra token, then -1); num_emitted [B]; probs [B, K, 3] = (p_i(x_i),
 * q_i(x_i), min(1, ratio)) for every position, or NULL; bonus_cdf [B, 2] = the
 * chosen token's normalised cumulative interval, or NULL; flags [B] or NULL.
 */
int oracle_verify_linear(const void *target, const void *draft, int dtype, int B, int K, int V,
                         const int32_t *draft_tokens, const float *u_accept, const float *u_bonus,
                         float temperature, int32_t *accept_len, int32_t *out_tokens,
                         int32_t *num_emitted, double *probs, double *bonus_cdf, uint32_t *flags) {
    if (B < 0 || K < 0 || V < 1) return 1;
    const double T = (double)temperature;
    const int greedy = (temperature == 0.0f);
#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)V);
        double *q = (double *)malloc(sizeof(double) * (size_t)V);
        double *w = (double *)malloc(sizeof(double) * (size_t)V);
#pragma omp for schedule(dynamic, 1)
        for (int b = 0; b < B; ++b) {
            uint32_t flag = 0;
            int j = K;
            if (greedy) {
                for (int i = 0; i < K; ++i) {
                    int x = draft_tokens[(size_t)b * K + i];
                    int am = argmax_row(target, dtype, (size_t)b * (K + 1) + i, V);
                    if (x < 0 || x >= V) flag |= ORACLE_FLAG_BAD_TOKEN;
                    if (x != am) { j = i; break; }
                }
            } else {
                int decided = 0;
                for (int i = 0; i < K; ++i) {
                    int x = draft_tokens[(size_t)b * K + i];
                    double px = 0.0, qx = 0.0, thr = 0.0;
                    if (x >= 0 && x < V) {
                        double mt, St, md, Sd;
                        softmax_row(target, dtype, (size_t)b * (K + 1) + i, V, T, p, &mt, &St);
                        softmax_row(draft, dtype, (size_t)b * K + i, V, T, q, &md, &Sd);
                        px = p[x];
                        qx = q[x];
                        /* p_i(x) / q_i(x), written as one quotient of the two softmax
                         * terms so that it stays defined where p and q both underflow */
                        double tx = logit_at(target, dtype, ((size_t)b * (K + 1) + i) * (size_t)V + x);
                        double dx = logit_at(draft, dtype, ((size_t)b * K + i) * (size_t)V + x);
                        double ratio = exp(((tx - mt) - (dx - md)) / T) * (Sd / St);
                        thr = ratio < 1.0 ? ratio : 1.0;
                    } else {
                        flag |= ORACLE_FLAG_BAD_TOKEN;
                    }
                    if (probs) {
                        probs[((size_t)b * K + i) * 3 + 0] = px;
                        probs[((size_t)b * K + i) * 3 + 1] = qx;
                        probs[((size_t)b * K + i) * 3 + 2] = thr;
                    }
                    /* positions are tested in order; the first failure ends the prefix */
                    if (!decided && !((double)u_accept[(size_t)b * K + i] < thr)) {
                        j = i;
                        decided = 1;
                        if (!probs) break;
                    }
                }
            }
            accept_len[b] = j;
            int32_t *row_out = out_tokens ? out_tokens + (size_t)b * (K + 1) : NULL;
            if (row_out) {
                for (int i = 0; i <= K; ++i) row_out[i] = -1;
                for (int i = 0; i < j; ++i) row_out[i] = draft_tokens[(size_t)b * K + i];
            }
            if (u_bonus) {
                int tok;
                double lo = 0.0, hi = 0.0;
                if (greedy) {
                    tok = argmax_row(target, dtype, (size_t)b * (K + 1) + j, V);
                } else {
                    tok = extra_token_sampled(target, draft, dtype, b, K, V, j, T, (double)u_bonus[b],
                                              w, p, q, &lo, &hi, &flag);
                }
                if (row_out) row_out[j] = tok;
                if (bonus_cdf) {
                    bonus_cdf[(size_t)b * 2 + 0] = lo;
                    bonus_cdf[(size_t)b * 2 + 1] = hi;
                }
                num_emitted[b] = j + 1;
            } else {
                num_emitted[b] = j;
            }
            if (flags) flags[b] = flag;
        }
        free(p);
        free(q);
        free(w);
    }
    return 0;
}

/*
 * The extra token alone, for a caller that already holds accept_len:
 * residual at row j = accept_len[b] if j < K, else p_K; argmax of target row
 * j when T == 0.  bonus_cdf [B, 2] and flags [B] may be NULL.
 */
int oracle_sample_bonus(const void *target, const void *draft, int dtype, int B, int K, int V,
                        const int32_t *accept_len, const float *u_bonus, float temperature,
                        int32_t *bonus_token, double *bonus_cdf, uint32_t *flags) {
    if (B < 0 || K < 0 || V < 1) return 1;
    const double T = (double)temperature;
#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)V);
        double *q = (double *)malloc(sizeof(double) * (size_t)V);
        double *w = (double *)malloc(sizeof(double) * (size_t)V);
#pragma omp for schedule(dynamic, 1)
        for (int b = 0; b < B; ++b) {
            uint32_t flag = 0;
            int j = accept_len[b];
            double lo = 0.0, hi = 0.0;
            if (j < 0 || j > K) {
                bonus_token[b] = -1;
            } else if (temperature == 0.0f) {
                bonus_token[b] = argmax_row(target, dtype, (size_t)b * (K + 1) + j, V);
            } else {
                bonus_token[b] = extra_token_sampled(target, draft, dtype, b, K, V, j, T,
                                                     (double)u_bonus[b], w, p, q, &lo, &hi, &flag);
            }
            if (bonus_cdf) {
                bonus_cdf[(size_t)b * 2 + 0] = lo;
                bonus_cdf[(size_t)b * 2 + 1] = hi;
            }
            if (flags) flags[b] = flag;
        }
        free(p);
        free(q);
        free(w);
    }
    return 0;
}

/*
 * Greedy tree verify ("Speculative-Decoding / Medusa", section 三).
 *   target [B, N, V]: row n holds the target logits after node n (node 0 is
 *   the root, i.e. the last token already accepted).
 *   parents [N]: parents[0] = -1, 0 <= parents[c] < c otherwise.
 *   node_tokens [B, N]: the candidate token of each node (column 0 unused).
 * Outputs (max_depth + 1 columns, -1 padded): path_nodes = 0, n1, n2, ...;
 * path_len = number of accepted non-root nodes; out_tokens = accepted node
 * tokens followed by the extra token argmax(target row of the last node).
 */
int oracle_verify_tree(const void *target, int dtype, int B, int N, int V, const int32_t *parents,
                       const int32_t *node_tokens, int max_depth, int32_t *path_nodes,
                       int32_t *path_len, int32_t *out_tokens) {
    if (B < 0 || N < 1 || V < 1 || max_depth < 0) return 1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        int32_t *pn = path_nodes + (size_t)b * (max_depth + 1);
        int32_t *ot = out_tokens + (size_t)b * (max_depth + 1);
        for (int d = 0; d <= max_depth; ++d) pn[d] = ot[d] = -1;
        int cur = 0, depth = 0;
        pn[0] = 0;
        while (depth < max_depth) {
            int want = argmax_row(target, dtype, (size_t)b * N + cur, V);
            int next = -1;
            for (int c = 1; c < N; ++c) {
                if (parents[c] == cur && node_tokens[(size_t)b * N + c] == want) {
                    next = c;
                    break;
                }
            }
            if (next < 0) break;
            ot[depth] = node_tokens[(size_t)b * N + next];
            ++depth;
            pn[depth] = next;
            cur = next;
        }
        path_len[b] = depth;
        ot[depth] = argmax_row(target, dtype, (size_t)b * N + cur, V);
    }
    return 0;
}

/*
 * Tree verify in sampling mode ("Speculative-Decoding / Medusa", section 三,
 * the sampled variant of the walk).  Arguments as oracle_verify_tree, plus
 *   u_nodes [B, N]: the uniform for the target's draw at each node;
 *   temperature > 0;
 *   node_cdf [B, N, 2] or NULL: each node's draw as its normalised cumulative
 *   interval [lo, hi) (every node is drawn, visited or not).
 * The draw at node n is inverse_cdf(softmax(target_n / T), u[b, n]).
 */
int oracle_verify_tree_sample(const void *target, int dtype, int B, int N, int V, const int32_t *parents,
                              const int32_t *node_tokens, const float *u_nodes, float temperature,
                              int max_depth, int32_t *path_nodes, int32_t *path_len, int32_t *out_tokens,
                              double *node_cdf) {
    if (B < 0 || N < 1 || V < 1 || max_depth < 0 || !(temperature > 0.0f)) return 1;
    const double T = (double)temperature;
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        double *p = (double *)malloc(sizeof(double) * (size_t)V);
        int32_t *draw = (int32_t *)malloc(sizeof(int32_t) * (size_t)N);
        for (int n = 0; n < N; ++n) {
            double lo = 0.0, hi = 0.0;
            softmax_row(target, dtype, (size_t)b * N + n, V, T, p, NULL, NULL);
            draw[n] = inverse_cdf(p, V, (double)u_nodes[(size_t)b * N + n], &lo, &hi);
            if (node_cdf) {
                node_cdf[((size_t)b * N + n) * 2 + 0] = lo;
                node_cdf[((size_t)b * N + n) * 2 + 1] = hi;
            }
        }
        int32_t *pn = path_nodes + (size_t)b * (max_depth + 1);
        int32_t *ot = out_tokens + (size_t)b * (max_depth + 1);
        for (int d = 0; d <= max_depth; ++d) pn[d] = ot[d] = -1;
        int cur = 0, depth = 0;
        pn[0] = 0;
        while (depth < max_depth) {
            int next = -1;
            for (int c = 1; c < N; ++c) {
                if (parents[c] == cur && node_tokens[(size_t)b * N + c] == draw[cur]) {
                    next = c;
                    break;
                }
            }
            if (next < 0) break;
            ot[depth] = node_tokens[(size_t)b * N + next];
            ++depth;
            pn[depth] = next;
            cur = next;
        }
        path_len[b] = depth;
        ot[depth] = draw[cur];
        free(p);
        free(draw);
    }
    return 0;
}

/*
 * One token per row: logits [B, V]; u [B] (ignored when T == 0).
 *   T > 0: inverse_cdf(softmax(row / T), u[b]); T == 0: argmax, lowest index.
 * Outputs: tokens [B]; cdf [B, 2] (the draw's normalised cumulative interval;
 * zeros when greedy) or NULL.
 */
int oracle_sample_rows(const void *logits, int dtype, int B, int V, const float *u, float temperature,
                       int32_t *tokens, double *cdf) {
    if (B < 0 || V < 1 || !(temperature >= 0.0f)) return 1;
    const double T = (double)temperature;
#pragma omp parallel for schedule(dynamic, 4)
    for (int b = 0; b < B; ++b) {
        double lo = 0.0, hi = 0.0;
        if (temperature == 0.0f) {
            tokens[b] = argmax_row(logits, dtype, (size_t)b, V);
        } else {
            double *p = (double *)malloc(sizeof(double) * (size_t)V);
            softmax_row(logits, dtype, (size_t)b, V, T, p, NULL, NULL);
            tokens[b] = inverse_cdf(p, V, (double)u[b], &lo, &hi);
            free(p);
        }
        if (cdf) {
            cdf[(size_t)b * 2 + 0] = lo;
            cdf[(size_t)b * 2 + 1] = hi;
        }
    }
    return 0;
}

/*
 * Tree attention mask and depths from the parent array (parents[0] ignored;
 * a node c >= 1 needs 0 <= parents[c] < c).  mask [N, W] uint32 words,
 * W = ceil(N / 32): bit (j % 32) of word j / 32 of row i is set iff node j is
 * node i or one of its ancestors.  depth [N].  Returns 0, or 2 if some parent
 * breaks the rule (that node's walk stops there; its row and depth hold what
 * was walked).
 */
int oracle_tree_mask(const int32_t *parents, int N, uint32_t *mask, int32_t *depth) {
    if (N < 1) return 1;
    const int W = (N + 31) / 32;
    int bad = 0;
    memset(mask, 0, sizeof(uint32_t) * (size_t)N * (size_t)W);
    for (int i = 0; i < N; ++i) {
        int cur = i, d = 0;
        mask[(size_t)i * W + cur / 32] |= 1u << (cur % 32);
        while (cur != 0) {
            int par = parents[cur];
            if (par < 0 || par >= cur) {
                bad = 1;
                break;
            }
            cur = par;
            ++d;
            mask[(size_t)i * W + cur / 32] |= 1u << (cur % 32);
        }
        depth[i] = d;
    }
    return bad ? 2 : 0;
}

/*
 * MTP token plug-in (see the reading above).  in_tokens [B, K+1], out_tokens
 * [B, K+1] and num_emitted [B] (a linear verify's outputs), pad: the token
 * written at the last position when nothing is shifted into it.
 * Outputs: next_tokens [B, K+1]; seq_lens [B] (incremented in place; NULL to
 * skip).  Returns 0, or 2 if some num_emitted[b] was outside [0, K + 1].
 */
int oracle_mtp_plug(const int32_t *in_tokens, int B, int K, const int32_t *out_tokens, const int32_t *num_emitted,
                    int32_t pad, int32_t *next_tokens, int32_t *seq_lens) {
    if (B < 0 || K < 0) return 1;
    const int W = K + 1;
    int bad = 0;
    for (int b = 0; b < B; ++b) {
        const int32_t *in = in_tokens + (size_t)b * W;
        int32_t *nx = next_tokens + (size_t)b * W;
        /* shift left by one: position i takes the token that follows it */
        for (int i = 0; i < K; ++i) nx[i] = in[i + 1];
        nx[K] = pad;
        const int n = num_emitted[b];
        if (n < 0 || n > W) {
            bad = 1;
            continue;
        }
        /* the target's next tokens go to their places */
        for (int i = 0; i < n; ++i) nx[i] = out_tokens[(size_t)b * W + i];
        if (seq_lens) seq_lens[b] += n;
    }
    return bad ? 2 : 0;
}

/* prod_j a_j^(i_j) along a rank path, left to right from 1 (a: [K][S], ranks 1-based). */
static double path_product(const double *acc, int S, const int *path, int m) {
    double v = 1.0;
    for (int j = 0; j < m; ++j) v *= acc[(size_t)j * S + (path[j] - 1)];
    return v;
}

/* Is rank path a (length ma) before rank path b (length mb) in (depth, lexicographic) order? */
static int path_before(const int *a, int ma, const int *b, int mb) {
    if (ma != mb) return ma < mb;
    for (int j = 0; j < ma; ++j)
        if (a[j] != b[j]) return a[j] < b[j];
    return 0;
}

/*
 * Greedy sparse tree (see the reading above).  acc [K * S]: acc[(k-1) * S +
 * (i-1)] = a_k^(i).  n_nodes >= 1 counts the root.  Outputs (n_nodes entries,
 * the first *n_built used): parents (parents[0] = -1), depth, rank (1-based,
 * 0 for the root); *expected_len = E[L].  Returns 0 or 1 (bad arguments).
 */
int oracle_build_sparse_tree(const double *acc, int K, int S, int n_nodes, int32_t *parents, int32_t *depth,
                             int32_t *rank, int *n_built, double *expected_len) {
    if (K < 1 || S < 1 || n_nodes < 1) return 1;
    /* chosen rank paths, K ints each; the root is the empty path */
    int *paths = (int *)calloc((size_t)n_nodes * K, sizeof(int));
    int *len = (int *)calloc((size_t)n_nodes, sizeof(int));
    int *cand = (int *)malloc(sizeof(int) * (size_t)K);
    int *best = (int *)malloc(sizeof(int) * (size_t)K);
    int n = 1;
    while (n < n_nodes) {
        int found = 0, best_m = 0;
        double best_v = 0.0;
        /* every child of every chosen node that is not chosen yet */
        for (int p = 0; p < n; ++p) {
            const int m = len[p];
            if (m >= K) continue;
            for (int i = 1; i <= S; ++i) {
                memcpy(cand, paths + (size_t)p * K, sizeof(int) * (size_t)m);
                cand[m] = i;
                int taken = 0;
                for (int q = 0; q < n && !taken; ++q)
                    if (len[q] == m + 1 && memcmp(paths + (size_t)q * K, cand, sizeof(int) * (size_t)(m + 1)) == 0)
                        taken = 1;
                if (taken) continue;
                const double v = path_product(acc, S, cand, m + 1);
                if (!found || v > best_v || (v == best_v && path_before(cand, m + 1, best, best_m))) {
                    found = 1;
                    best_v = v;
                    best_m = m + 1;
                    memcpy(best, cand, sizeof(int) * (size_t)best_m);
                }
            }
        }
        if (!found) break; /* the full tree is smaller than n_nodes */
        memcpy(paths + (size_t)n * K, best, sizeof(int) * (size_t)best_m);
        len[n] = best_m;
        ++n;
    }
    /* number the nodes by (depth, rank path): a selection sort into order[] */
    int *order = (int *)malloc(sizeof(int) * (size_t)n);
    int *used = (int *)calloc((size_t)n, sizeof(int));
    for (int r = 0; r < n; ++r) {
        int pick = -1;
        for (int q = 0; q < n; ++q)
            if (!used[q] && (pick < 0 || path_before(paths + (size_t)q * K, len[q], paths + (size_t)pick * K, len[pick])))
                pick = q;
        used[pick] = 1;
        order[r] = pick;
    }
    double e = 0.0;
    for (int r = 0; r < n; ++r) {
        const int q = order[r];
        const int m = len[q];
        depth[r] = m;
        rank[r] = m > 0 ? paths[(size_t)q * K + m - 1] : 0;
        parents[r] = -1;
        if (m > 0) {
            /* the parent is the chosen node whose path is this one without its last rank */
            for (int t = 0; t < r; ++t) {
                const int pq = order[t];
                if (len[pq] == m - 1 && memcmp(paths + (size_t)pq * K, paths + (size_t)q * K, sizeof(int) * (size_t)(m - 1)) == 0) {
                    parents[r] = t;
                    break;
                }
            }
            e += path_product(acc, S, paths + (size_t)q * K, m);
        }
    }
    *n_built = n;
    if (expected_len) *expected_len = e;
    free(paths);
    free(len);
    free(cand);
    free(best);
    free(order);
    free(used);
    return 0;
}

/* Number of OpenMP threads the oracle runs with; n > 0 sets it first. */
int oracle_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}
