/*
 * oracle.c -- plain, slow, fp64 CPU definition of what the ring-chunked
 * attention path computes.  TEST INFRASTRUCTURE ONLY: the tests, the smoke
 * check and the bench's cpu_baseline / reference arm call it; the product
 * path never does.  It shares no code, header or constant with the CUDA
 * library.
 *
 * Sources (web pages, cited by title and section):
 *  [R1] diffusers issue #14265 "Ring attention backward uses stale
 *       iteration-0 KV from ctx.saved_tensors -- silent gradient corruption
 *       when training with context parallelism": sections "Root cause"
 *       (per-iteration forward op returning a partial with its LSE, K/V
 *       rotating each iteration), "How it surfaces per backend" (ring needs
 *       the LSE to merge partial results; GQA head rule), "Reproduction"
 *       (full-sequence SDPA reference, default scale) and "Expected
 *       behavior" (each backward iteration must see that iteration's K/V).
 *  [R2] DeepSpeed PR #8491 "[bugfix] _DimZeroAllToAll silently fails to
 *       send grads under torch.compile": the exchange is a permutation whose
 *       backward is the transposed exchange; section "Testing" (slot rule,
 *       gradient of sum(y^2) is 2x).
 *  [R3] diffusers PR #12443 "Fix Flux Context Parallel Bug (Incoherent Image
 *       Generation)": padding to a multiple of the world size, and the
 *       discussion that padded tokens must be masked.
 *  [R4] DeepSpeed issue #7842 "[BUG] DistributedAttention produces
 *       numerically incorrect results ... not divisible by world size":
 *       section "Testcase" (sequence-first [S,B,H,D], scatter heads / gather
 *       sequence) and the closing comment's shapes (5,8,8,64) -> (10,8,4,64).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - LSE merge: L = log sum_i exp(lse_i), O = sum_i exp(lse_i - L) O_i.
 *  - Ring order: at iteration i query chunk r meets KV chunk (r - i) mod P.
 *  - GQA: query head h reads kv head floor(h * Hkv / Hq).
 *  - Causal: key j visible to query i iff j <= i (global indices).
 *  - Exchange: rank rho = r*U + u holds rows [rho*Ssh, (rho+1)*Ssh) of the
 *    sequence padded at its end to W*Ssh, Ssh = ceil(S/W); after the
 *    exchange rank (r,u) holds the U shards of ring group r (slot u' from
 *    rank r*U+u') restricted to head group u.
 *
 * Tensors are addressed as [B,S,H,D] through element strides (sB,sS,sH);
 * the D stride is 1.  The same routine therefore reads [B,S,H,D] and
 * sequence-first [S,B,H,D] storage: the caller states the strides.
 * The log-sum-exp array is [B,H,S] contiguous.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Number of OpenMP threads of the calling thread's later parallel loops (a
 * launcher may have pinned OMP_NUM_THREADS before the runtime started);
 * no arithmetic depends on it. */
void oracle_set_threads(int n) {
    if (n > 0) omp_set_num_threads(n);
}

#define AT(p, st, b, s, h) ((p) + (long)(b) * (st)[0] + (long)(s) * (st)[1] + (long)(h) * (st)[2])

static int kv_head(int h, int Hq, int Hkv) { return (int)(((long)h * Hkv) / Hq); }

static double dot(const double* a, const double* b, int D) {
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += a[d] * b[d];
    return acc;
}

static int visible(int causal, int i, int j) { return !causal || j <= i; }

static int check_dims(int B, int S, int Hq, int Hkv, int D) {
    if (B < 1 || S < 1 || Hq < 1 || Hkv < 1 || D < 1) return 1;
    if (Hq % Hkv != 0) return 1; /* [R1] "How it surfaces": heads of K/V must divide heads of Q */
    return 0;
}

/* Log-sum-exp of the scores of query row (b,h,i) over keys [j0,j1) that are
 * visible; -inf when none is.  Max-subtracted for range, as any stable LSE. */
static double row_lse(int causal, int i, int j0, int j1, double scale, const double* qi,
                      const double* k, const long* ks, int b, int hk, int D) {
    double m = -INFINITY;
    for (int j = j0; j < j1; ++j) {
        if (!visible(causal, i, j)) continue;
        double s = scale * dot(qi, AT(k, ks, b, j, hk), D);
        if (s > m) m = s;
    }
    if (m == -INFINITY) return -INFINITY;
    double sum = 0.0;
    for (int j = j0; j < j1; ++j) {
        if (!visible(causal, i, j)) continue;
        sum += exp(scale * dot(qi, AT(k, ks, b, j, hk), D) - m);
    }
    return m + log(sum);
}

/* o_i = sum_{j in [j0,j1)} exp(s_ij - lse) v_j */
static void row_out(int causal, int i, int j0, int j1, double scale, double lse, const double* qi,
                    const double* k, const double* v, const long* ks, int b, int hk, int D,
                    double* o) {
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (lse == -INFINITY) return;
    for (int j = j0; j < j1; ++j) {
        if (!visible(causal, i, j)) continue;
        double p = exp(scale * dot(qi, AT(k, ks, b, j, hk), D) - lse);
        const double* vj = AT(v, ks, b, j, hk);
        for (int d = 0; d < D; ++d) o[d] += p * vj[d];
    }
}

/* Full-sequence softmax attention forward, the plain definition
 * ([R1] "Reproduction": the full-sequence SDPA the ring result must equal):
 *   s_ij = scale <q_i, k_j>,  lse_i = log sum_j exp(s_ij),
 *   o_i  = sum_j exp(s_ij - lse_i) v_j. */
int oracle_attn_fwd(int B, int S, int Hq, int Hkv, int D, double scale, int causal,
                    const double* q, const long* qs, const double* k, const double* v,
                    const long* ks, double* out, const long* os, double* lse) {
    if (check_dims(B, S, Hq, Hkv, D)) return 1;
    long rows = (long)B * Hq * S;
#pragma omp parallel for schedule(dynamic, 16)
    for (long r = 0; r < rows; ++r) {
        int i = (int)(r % S), h = (int)((r / S) % Hq), b = (int)(r / ((long)S * Hq));
        int hk = kv_head(h, Hq, Hkv);
        const double* qi = AT(q, qs, b, i, h);
        double L = row_lse(causal, i, 0, S, scale, qi, k, ks, b, hk, D);
        row_out(causal, i, 0, S, scale, L, qi, k, v, ks, b, hk, D, AT(out, os, b, i, h));
        lse[((long)b * Hq + h) * S + i] = L;
    }
    return 0;
}

/* Row statistics of the analytic backward for query row (b,h,i):
 * lse_i and Delta_i = sum_j P_ij dp_ij with P_ij = exp(s_ij - lse_i),
 * dp_ij = <do_i, v_j>. */
static void row_stats(int causal, int S, int i, double scale, const double* qi, const double* doi,
                      const double* k, const double* v, const long* ks, int b, int hk, int D,
                      double* lse_out, double* delta_out) {
    double L = row_lse(causal, i, 0, S, scale, qi, k, ks, b, hk, D);
    double delta = 0.0;
    if (L != -INFINITY) {
        for (int j = 0; j < S; ++j) {
            if (!visible(causal, i, j)) continue;
            double p = exp(scale * dot(qi, AT(k, ks, b, j, hk), D) - L);
            delta += p * dot(doi, AT(v, ks, b, j, hk), D);
        }
    }
    *lse_out = L;
    *delta_out = delta;
}

/* dq_i = scale sum_j ds_ij k_j, ds_ij = P_ij (dp_ij - Delta_i) */
static void row_dq(int causal, int S, int i, double scale, double L, double delta, const double* qi,
                   const double* doi, const double* k, const double* v, const long* ks, int b,
                   int hk, int D, double* dq) {
    for (int d = 0; d < D; ++d) dq[d] = 0.0;
    if (L == -INFINITY) return;
    for (int j = 0; j < S; ++j) {
        if (!visible(causal, i, j)) continue;
        const double* kj = AT(k, ks, b, j, hk);
        double p = exp(scale * dot(qi, kj, D) - L);
        double ds = p * (dot(doi, AT(v, ks, b, j, hk), D) - delta);
        for (int d = 0; d < D; ++d) dq[d] += scale * ds * kj[d];
    }
}

/* dk_j = scale sum_{h in group, i} ds_ij q_i ; dv_j = sum_{h in group, i} P_ij do_i.
 * lse/delta hold the statistics of every query row ([B,Hq,S]). */
static void key_row_grads(int causal, int S, int Hq, int Hkv, int j, double scale, const double* q,
                          const long* qs, const double* dout, const long* dos, const double* k,
                          const double* v, const long* ks, const double* lse, const double* delta,
                          int b, int hk, int D, double* dk, double* dv) {
    int G = Hq / Hkv;
    const double* kj = AT(k, ks, b, j, hk);
    const double* vj = AT(v, ks, b, j, hk);
    for (int d = 0; d < D; ++d) { dk[d] = 0.0; dv[d] = 0.0; }
    for (int h = hk * G; h < (hk + 1) * G; ++h) {
        for (int i = 0; i < S; ++i) {
            if (!visible(causal, i, j)) continue;
            double L = lse[((long)b * Hq + h) * S + i];
            if (L == -INFINITY) continue;
            const double* qi = AT(q, qs, b, i, h);
            const double* doi = AT(dout, dos, b, i, h);
            double p = exp(scale * dot(qi, kj, D) - L);
            double ds = p * (dot(doi, vj, D) - delta[((long)b * Hq + h) * S + i]);
            for (int d = 0; d < D; ++d) {
                dk[d] += scale * ds * qi[d];
                dv[d] += p * doi[d];
            }
        }
    }
}

/* Analytic backward of the full-sequence definition (the gradient the ring
 * backward must reproduce, [R1] "Expected behavior"):
 *   P = exp(S - lse), dV = P^T dO, dP = dO V^T, Delta = rowsum(P o dP),
 *   dS = P o (dP - Delta), dQ = scale dS K, dK = scale dS^T Q;
 * for GQA dK, dV sum over the query heads sharing a kv head. */
int oracle_attn_bwd(int B, int S, int Hq, int Hkv, int D, double scale, int causal,
                    const double* q, const long* qs, const double* k, const double* v,
                    const long* ks, const double* dout, const long* dos, double* dq,
                    const long* dqs, double* dk, double* dv, const long* dks) {
    if (check_dims(B, S, Hq, Hkv, D)) return 1;
    long rows = (long)B * Hq * S;
    double* lse = (double*)malloc(sizeof(double) * rows);
    double* delta = (double*)malloc(sizeof(double) * rows);
    if (!lse || !delta) { free(lse); free(delta); return 2; }
#pragma omp parallel for schedule(dynamic, 16)
    for (long r = 0; r < rows; ++r) {
        int i = (int)(r % S), h = (int)((r / S) % Hq), b = (int)(r / ((long)S * Hq));
        int hk = kv_head(h, Hq, Hkv);
        const double* qi = AT(q, qs, b, i, h);
        const double* doi = AT(dout, dos, b, i, h);
        row_stats(causal, S, i, scale, qi, doi, k, v, ks, b, hk, D, &lse[r], &delta[r]);
        row_dq(causal, S, i, scale, lse[r], delta[r], qi, doi, k, v, ks, b, hk, D,
               AT(dq, dqs, b, i, h));
    }
    long krows = (long)B * Hkv * S;
#pragma omp parallel for schedule(dynamic, 16)
    for (long r = 0; r < krows; ++r) {
        int j = (int)(r % S), hk = (int)((r / S) % Hkv), b = (int)(r / ((long)S * Hkv));
        key_row_grads(causal, S, Hq, Hkv, j, scale, q, qs, dout, dos, k, v, ks, lse, delta, b, hk,
                      D, AT(dk, dks, b, j, hk), AT(dv, dks, b, j, hk));
    }
    free(lse);
    free(delta);
    return 0;
}

/* Sampled forward: out and lse of n query rows (bi[t], hi[t], si[t]). */
int oracle_attn_fwd_rows(int B, int S, int Hq, int Hkv, int D, double scale, int causal,
                         const double* q, const long* qs, const double* k, const double* v,
                         const long* ks, int n, const int* bi, const int* hi, const int* si,
                         double* out_rows, double* lse_rows) {
    if (check_dims(B, S, Hq, Hkv, D)) return 1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < n; ++t) {
        int b = bi[t], h = hi[t], i = si[t], hk = kv_head(h, Hq, Hkv);
        const double* qi = AT(q, qs, b, i, h);
        double L = row_lse(causal, i, 0, S, scale, qi, k, ks, b, hk, D);
        row_out(causal, i, 0, S, scale, L, qi, k, v, ks, b, hk, D, out_rows + (long)t * D);
        lse_rows[t] = L;
    }
    return 0;
}

/* Sampled backward, query side: dq of n query rows. */
int oracle_attn_dq_rows(int B, int S, int Hq, int Hkv, int D, double scale, int causal,
                        const double* q, const long* qs, const double* k, const double* v,
                        const long* ks, const double* dout, const long* dos, int n, const int* bi,
                        const int* hi, const int* si, double* dq_rows) {
    if (check_dims(B, S, Hq, Hkv, D)) return 1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < n; ++t) {
        int b = bi[t], h = hi[t], i = si[t], hk = kv_head(h, Hq, Hkv);
        const double* qi = AT(q, qs, b, i, h);
        const double* doi = AT(dout, dos, b, i, h);
        double L, delta;
        row_stats(causal, S, i, scale, qi, doi, k, v, ks, b, hk, D, &L, &delta);
        row_dq(causal, S, i, scale, L, delta, qi, doi, k, v, ks, b, hk, D, dq_rows + (long)t * D);
    }
    return 0;
}

/* Sampled backward, key side: dk, dv of n key rows (bi[t], hki[t], sj[t]).
 * Every query row of the kv head's group enters each of them, so the row
 * statistics of those groups are computed in full first. */
int oracle_attn_dkv_rows(int B, int S, int Hq, int Hkv, int D, double scale, int causal,
                         const double* q, const long* qs, const double* k, const double* v,
                         const long* ks, const double* dout, const long* dos, int n,
                         const int* bi, const int* hki, const int* sj, double* dk_rows,
                         double* dv_rows) {
    if (check_dims(B, S, Hq, Hkv, D)) return 1;
    long rows = (long)B * Hq * S;
    double* lse = (double*)malloc(sizeof(double) * rows);
    double* delta = (double*)malloc(sizeof(double) * rows);
    char* need = (char*)calloc((size_t)B * Hkv, 1);
    if (!lse || !delta || !need) { free(lse); free(delta); free(need); return 2; }
    for (int t = 0; t < n; ++t) need[bi[t] * Hkv + hki[t]] = 1;
#pragma omp parallel for schedule(dynamic, 16)
    for (long r = 0; r < rows; ++r) {
        int i = (int)(r % S), h = (int)((r / S) % Hq), b = (int)(r / ((long)S * Hq));
        int hk = kv_head(h, Hq, Hkv);
        if (!need[b * Hkv + hk]) continue;
        row_stats(causal, S, i, scale, AT(q, qs, b, i, h), AT(dout, dos, b, i, h), k, v, ks, b,
                  hk, D, &lse[r], &delta[r]);
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < n; ++t)
        key_row_grads(causal, S, Hq, Hkv, sj[t], scale, q, qs, dout, dos, k, v, ks, lse, delta,
                      bi[t], hki[t], D, dk_rows + (long)t * D, dv_rows + (long)t * D);
    free(lse);
    free(delta);
    free(need);
    return 0;
}

/* ------------------------------------------------------------------------
 * Ring-structured forms, used to pin the chunked algorithm itself.
 * Chunk c holds sequence rows [off[c], off[c+1]).
 * ---------------------------------------------------------------------- */

static int check_offsets(int S, int P, const int* off) {
    if (P < 1 || off[0] != 0 || off[P] != S) return 1;
    for (int c = 0; c < P; ++c)
        if (off[c + 1] <= off[c]) return 1; /* empty chunks are rejected */
    return 0;
}

/* Ring forward ([R1] "Root cause"): the query chunk r stays put; at
 * iteration i it meets KV chunk c = (r - i) mod P, and the attention call of
 * that iteration returns a partial (O_i, LSE_i) over chunk c only.  The
 * partials are merged by LSE weighting ([R1] "How it surfaces": the ring
 * needs the LSE to merge partial results):
 *   L = log sum_i exp(LSE_i)   (max-subtracted),
 *   O = sum_i exp(LSE_i - L) O_i.
 * If part_o / part_lse are non-NULL they receive the partials, indexed
 * [i][b][h][s][d] and [i][b][h][s] (query row s of chunk r at iteration i). */
int oracle_ring_fwd(int B, int S, int Hq, int Hkv, int D, double scale, int causal, int P,
                    const int* off, const double* q, const long* qs, const double* k,
                    const double* v, const long* ks, double* out, const long* os, double* lse,
                    double* part_o, double* part_lse) {
    if (check_dims(B, S, Hq, Hkv, D) || check_offsets(S, P, off)) return 1;
    long rows = (long)B * Hq * S;
    int fail = 0;
#pragma omp parallel for schedule(dynamic, 16)
    for (long rr = 0; rr < rows; ++rr) {
        int s = (int)(rr % S), h = (int)((rr / S) % Hq), b = (int)(rr / ((long)S * Hq));
        int hk = kv_head(h, Hq, Hkv);
        int r = 0;
        while (off[r + 1] <= s) ++r;
        const double* qi = AT(q, qs, b, s, h);
        double* oi = (double*)malloc(sizeof(double) * (size_t)P * D);
        double* li = (double*)malloc(sizeof(double) * (size_t)P);
        if (!oi || !li) {
            free(oi); free(li);
#pragma omp atomic write
            fail = 1;
            continue;
        }
        for (int it = 0; it < P; ++it) {
            int c = ((r - it) % P + P) % P;
            li[it] = row_lse(causal, s, off[c], off[c + 1], scale, qi, k, ks, b, hk, D);
            row_out(causal, s, off[c], off[c + 1], scale, li[it], qi, k, v, ks, b, hk, D,
                    oi + (long)it * D);
            if (part_o) {
                long pidx = (((long)it * B + b) * Hq + h) * S + s;
                memcpy(part_o + pidx * D, oi + (long)it * D, sizeof(double) * D);
                part_lse[pidx] = li[it];
            }
        }
        /* merge */
        double m = -INFINITY;
        for (int it = 0; it < P; ++it) if (li[it] > m) m = li[it];
        double* o = AT(out, os, b, s, h);
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        double L = -INFINITY;
        if (m != -INFINITY) {
            double sum = 0.0;
            for (int it = 0; it < P; ++it) if (li[it] != -INFINITY) sum += exp(li[it] - m);
            L = m + log(sum);
            for (int it = 0; it < P; ++it) {
                if (li[it] == -INFINITY) continue;
                double w = exp(li[it] - L);
                for (int d = 0; d < D; ++d) o[d] += w * oi[(long)it * D + d];
            }
        }
        lse[((long)b * Hq + h) * S + s] = L;
        free(oi);
        free(li);
    }
    return fail ? 2 : 0;
}

/* Merge of materialised partials (the same LSE weighting as above), for
 * partials indexed [i][b][h][s][d] / [i][b][h][s]. */
int oracle_lse_merge(int B, int S, int H, int D, int P, const double* part_o,
                     const double* part_lse, double* out, const long* os, double* lse) {
    long rows = (long)B * H * S;
#pragma omp parallel for schedule(static)
    for (long rr = 0; rr < rows; ++rr) {
        int s = (int)(rr % S), h = (int)((rr / S) % H), b = (int)(rr / ((long)S * H));
        double m = -INFINITY;
        for (int it = 0; it < P; ++it) {
            double l = part_lse[(long)it * rows + rr];
            if (l > m) m = l;
        }
        double* o = AT(out, os, b, s, h);
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        double L = -INFINITY;
        if (m != -INFINITY) {
            double sum = 0.0;
            for (int it = 0; it < P; ++it) {
                double l = part_lse[(long)it * rows + rr];
                if (l != -INFINITY) sum += exp(l - m);
            }
            L = m + log(sum);
            for (int it = 0; it < P; ++it) {
                double l = part_lse[(long)it * rows + rr];
                if (l == -INFINITY) continue;
                double w = exp(l - L);
                const double* po = part_o + ((long)it * rows + rr) * D;
                for (int d = 0; d < D; ++d) o[d] += w * po[d];
            }
        }
        lse[rr] = L;
    }
    (void)B;
    return 0;
}

/* Ring backward ([R1] "Expected behavior"): for every pair (query chunk r,
 * iteration i) the probabilities are recomputed against that iteration's
 * own KV chunk c = (r - i) mod P with the merged (global) LSE of the query
 * row, P = exp(s - lse), and
 *   dV_c += P^T dO_r,  dS = P o (dO_r V_c^T - Delta_r),
 *   dQ_r += scale dS K_c,  dK_c += scale dS^T Q_r,
 * with Delta = rowsum(dO o O) from the merged forward output.
 * stale != 0 plants the defect the issue describes ("Root cause": every
 * iteration of the backward reads the iteration-0 tensors, i.e. the query's
 * own chunk K_r, V_r, while the gradients still travel to chunk c).  That
 * mode exists only as a negative control for the tests. */
int oracle_ring_bwd(int B, int S, int Hq, int Hkv, int D, double scale, int causal, int P,
                    const int* off, const double* q, const long* qs, const double* k,
                    const double* v, const long* ks, const double* out, const long* os,
                    const double* lse, const double* dout, const long* dos, int stale,
                    double* dq, const long* dqs, double* dk, double* dv, const long* dks) {
    if (check_dims(B, S, Hq, Hkv, D) || check_offsets(S, P, off)) return 1;
    int G = Hq / Hkv;
    /* zero the outputs */
    for (int b = 0; b < B; ++b)
        for (int s = 0; s < S; ++s) {
            for (int h = 0; h < Hq; ++h) memset(AT(dq, dqs, b, s, h), 0, sizeof(double) * D);
            for (int h = 0; h < Hkv; ++h) {
                memset(AT(dk, dks, b, s, h), 0, sizeof(double) * D);
                memset(AT(dv, dks, b, s, h), 0, sizeof(double) * D);
            }
        }
    /* one task per (b, kv head): it owns dK/dV of that head and dQ of the
     * group's query heads, so the accumulation needs no locking. */
#pragma omp parallel for schedule(dynamic, 1)
    for (long task = 0; task < (long)B * Hkv; ++task) {
        int b = (int)(task / Hkv), hk = (int)(task % Hkv);
        for (int h = hk * G; h < (hk + 1) * G; ++h) {
            for (int r = 0; r < P; ++r) {
                for (int it = 0; it < P; ++it) {
                    int c = ((r - it) % P + P) % P;     /* where the gradient goes */
                    int src = stale ? r : c;            /* which K/V the op reads */
                    for (int i = off[r]; i < off[r + 1]; ++i) {
                        double L = lse[((long)b * Hq + h) * S + i];
                        if (L == -INFINITY) continue;
                        const double* qi = AT(q, qs, b, i, h);
                        const double* doi = AT(dout, dos, b, i, h);
                        double delta = dot(doi, AT(out, os, b, i, h), D);
                        double* dqi = AT(dq, dqs, b, i, h);
                        for (int t = 0; t < off[c + 1] - off[c]; ++t) {
                            int j = off[c] + t;                       /* gradient row */
                            int js = off[src] + t;                    /* row actually read */
                            if (js >= off[src + 1]) continue;         /* stale chunk shorter */
                            if (!visible(causal, i, j)) continue;
                            const double* kj = AT(k, ks, b, js, hk);
                            const double* vj = AT(v, ks, b, js, hk);
                            double p = exp(scale * dot(qi, kj, D) - L);
                            double ds = p * (dot(doi, vj, D) - delta);
                            double* dkj = AT(dk, dks, b, j, hk);
                            double* dvj = AT(dv, dks, b, j, hk);
                            for (int d = 0; d < D; ++d) {
                                dqi[d] += scale * ds * kj[d];
                                dkj[d] += scale * ds * qi[d];
                                dvj[d] += p * doi[d];
                            }
                        }
                    }
                }
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * Ulysses sequence <-> head exchange ([R2], [R4]), on raw 16-bit words so
 * that the comparison is bitwise.
 *
 * x: the full sequence [B,S,H,D] at strides xs (either storage order).
 * W = ring * U emulated ranks.  Ssh = ceil(S / W).  Rank rho = r*U + u
 * holds rows [rho*Ssh, (rho+1)*Ssh) of the sequence padded with zero rows
 * at its end to W*Ssh ([R3]: pad to a multiple of the world size).
 *
 * All-to-all inside ulysses group r ([R2] "Testing": slot u' of a rank's
 * output holds the slot that rank owns in rank u''s input): rank (r,u)
 * ends up with [B, U*Ssh, H/U, D] = its group's U shards in slot order,
 * heads [u*H/U, (u+1)*H/U).
 *
 * Storage of the exchanged tensor y (every emulated rank at once):
 * [U][B][W*Ssh][H/U][D] for layout 0, [U][W*Ssh][B][H/U][D] for layout 1,
 * contiguous; rank (r,u)'s local tensor is rows [r*U*Ssh, (r+1)*U*Ssh) of
 * head group u.  dir 0: x -> y; dir 1: y -> x (the inverse, which is the
 * transpose, i.e. the backward of the exchange).
 * ---------------------------------------------------------------------- */
static long y_index(int layout, int B, long Sp, int Hu, int D, int u, int b, long s, int hh) {
    if (layout == 0) return ((((long)u * B + b) * Sp + s) * Hu + hh) * D;
    return ((((long)u * Sp + s) * B + b) * Hu + hh) * D;
}

int oracle_seq_head_exchange(int B, int S, int H, int D, int ring, int U, int dir, int layout,
                             const uint16_t* src, uint16_t* dst, const long* xs) {
    if (ring < 1 || U < 1 || H % U != 0 || B < 1 || S < 1 || D < 1) return 1;
    int W = ring * U, Hu = H / U;
    long Ssh = (S + W - 1) / W, Sp = Ssh * W;
    for (int r = 0; r < ring; ++r)
        for (int u = 0; u < U; ++u)            /* destination rank (r,u) */
            for (int up = 0; up < U; ++up) {   /* slot u': from source rank r*U+u' */
                int rho_src = r * U + up;
                for (int b = 0; b < B; ++b)
                    for (long t = 0; t < Ssh; ++t) {
                        long s = (long)rho_src * Ssh + t; /* global (padded) row */
                        for (int hh = 0; hh < Hu; ++hh) {
                            int h = u * Hu + hh;
                            long yi = y_index(layout, B, Sp, Hu, D, u, b, s, hh);
                            if (dir == 0) {
                                if (s < S) {
                                    long xi = (long)b * xs[0] + s * xs[1] + (long)h * xs[2];
                                    memcpy(dst + yi, src + xi, sizeof(uint16_t) * D);
                                } else {
                                    memset(dst + yi, 0, sizeof(uint16_t) * D);
                                }
                            } else if (s < S) {
                                long xi = (long)b * xs[0] + s * xs[1] + (long)h * xs[2];
                                memcpy(dst + xi, src + yi, sizeof(uint16_t) * D);
                            }
                        }
                    }
            }
    return 0;
}
