/*
 * oracle.c -- plain, slow, fp64 CPU oracle for exact attention and its
 * backward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: it is built into liboracle.so and used by the tests, by
 * the smoke check and by the benchmark's CPU-baseline leg.  It shares no
 * code, header, table or helper with the CUDA library.
 *
 * What it computes (the plain definition the fused kernel must reproduce):
 *
 *   Three-step form of attention ("Reading CMU 11-868 LLM Systems:
 *   FlashAttention", section "The scenario", slide page 5):
 *       S = scale * Q K^T,  A = softmax(S) row-wise,  O = A V.
 *   FlashAttention's output equals standard attention's exactly (same
 *   post, page 15 summary; quidproquo tag page "flashattention", Hung-yi
 *   Lee paragraph), so the oracle is that definition written out, with no
 *   tiling and no online rescaling.
 *
 *   Per row i (causal: keys j > i are masked out, top-left alignment):
 *       S_ij   = scale * sum_k q_ik k_jk
 *       m_i    = max_j S_ij                 (only to keep exp() finite;
 *                                            cs2680 Lecture 9, sec. 9.4)
 *       lse_i  = m_i + ln sum_j exp(S_ij - m_i)
 *       A_ij   = exp(S_ij - lse_i)
 *       O_i    = sum_j A_ij v_j
 *   lse is the per-row normalisation constant the forward pass keeps for
 *   the backward pass (CMU 11-868 post, "Recomputation", slide page 14;
 *   cs2680 Lecture 9, sec. 9.6).
 *
 *   Backward: the pages give no formulas; this is the textbook gradient of
 *   O = softmax(scale Q K^T) V with upstream gradient dO:
 *       dV   = A^T dO
 *       dA   = dO V^T
 *       D_i  = sum_j A_ij dA_ij
 *       dS   = A o (dA - D)      (o = elementwise product, D broadcast per row)
 *       dQ   = scale * dS K
 *       dK   = scale * dS^T Q
 *   lse receives no upstream gradient.
 *
 * Layout: every tensor is a dense row-major fp64 array [BH][N][d] (lse and
 * D are [BH][N]).
 *
 * General form (oracle_attn_fwd_gqa): N_q query rows per head against N_kv
 * keys, and H_q query heads sharing H_kv key/value heads in groups of
 * G = H_q / H_kv (query head h reads key/value head h / G).  The causal
 * mask is aligned bottom-right: query i is the (N_kv - N_q + i)-th position
 * of the key sequence and attends to keys j <= i + N_kv - N_q, which is the
 * square top-left mask when N_q = N_kv.  A row with no key has O = 0 and
 * lse = -inf.  The split-KV combine of cs2680 Lecture 9 sec. 9.8 merges
 * partial results (O_s, lse_s) over key ranges s by the same rescaling as
 * sec. 9.4: lse = ln sum_s exp(lse_s), O = sum_s exp(lse_s - lse) O_s
 * (oracle_combine_splits).
 *
 * Block-sparse form (oracle_attn_fwd_blockmask / oracle_attn_bwd_blockmask):
 * a 0/1 mask bm over (bs-row query block, bs-key block) pairs, shared by all
 * heads; key j is visible to query i when bm[i / bs][j / bs] is 1 (and
 * j <= i under the causal mask).  This is dense attention with the masked
 * scores at -inf, evaluated entry by entry; a row with no visible key has
 * O = 0, lse = -inf and takes no part in the gradients.
 *
 * FP8 form with incoherent processing (CMU 11-868 FlashAttention post,
 * FA3 section, slide page 24: quantisation outliers are spread by
 * multiplying Q and K by the same orthogonal Hadamard matrix, which leaves
 * Q K^T unchanged).  The steps, in order (oracle_attn_fwd_fp8):
 *   1. with `hadamard`, every row of Q and of K is multiplied by the
 *      Sylvester Hadamard matrix H_d (entries (-1)^popcount(i & j), so
 *      H H^T = d I and (Q H)(K H)^T = d Q K^T); V is not transformed;
 *   2. each head of each of Q, K, V is quantised to FP8 E4M3 with one
 *      scale: amax = max |x| over the head, code = E4M3(x * (448 / amax)),
 *      rounded to nearest-even and saturated to +-448; the dequantised
 *      value is decode(code) * (amax / 448).  The rounding decision is made
 *      in fp32 (x, amax, 448 / amax and the product each rounded to fp32),
 *      the precision of the GPU kernel that takes the same decision;
 *      amax = 0 gives code 0 and scale 1;
 *   3. exact attention (the three-step definition above) over the
 *      dequantised Q, K, V with scale / d under the rotation (scale
 *      otherwise).
 * Readings (the pages give none of these details): one scale per head and
 * tensor; E4M3 in its OCP "fn" form (bias 7, no infinities, largest finite
 * 448, S.1111.111 is NaN); the softmax probabilities are exact here (the GPU
 * rounds them to E4M3 as tensor-core operands, which its tolerance covers).
 *
 * Loops are parallelised with OpenMP over independent rows (forward, dQ) or
 * independent key rows (dK, dV); each output element is computed by one
 * thread with a plain sequential sum, so results do not depend on the thread
 * count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Number of keys row i may attend to. */
static int64_t row_len(int64_t i, int64_t N, int causal)
{
    return causal ? (i + 1 < N ? i + 1 : N) : N;
}

/* Scores of row i of head h into s[0..len), returns len. */
static int64_t scores_row(const double* q, const double* k, int64_t h, int64_t i,
                          int64_t N, int64_t d, int causal, double scale, double* s)
{
    const double* qi = q + (h * N + i) * d;
    const double* kh = k + h * N * d;
    int64_t len = row_len(i, N, causal);
    for (int64_t j = 0; j < len; ++j) {
        const double* kj = kh + j * d;
        double acc = 0.0;
        for (int64_t c = 0; c < d; ++c) acc += qi[c] * kj[c];
        s[j] = scale * acc;
    }
    return len;
}

/* lse of a row of scores: m + ln sum exp(s - m). */
static double logsumexp_row(const double* s, int64_t len)
{
    double m = -INFINITY;
    for (int64_t j = 0; j < len; ++j) if (s[j] > m) m = s[j];
    double l = 0.0;
    for (int64_t j = 0; j < len; ++j) l += exp(s[j] - m);
    return m + log(l);
}

/* Forward for one (head, row): fills o_row[0..d) and returns lse. */
static double fwd_row(const double* q, const double* k, const double* v, int64_t h,
                      int64_t i, int64_t N, int64_t d, int causal, double scale,
                      double* s, double* o_row)
{
    int64_t len = scores_row(q, k, h, i, N, d, causal, scale, s);
    double lse = logsumexp_row(s, len);
    const double* vh = v + h * N * d;
    for (int64_t c = 0; c < d; ++c) o_row[c] = 0.0;
    for (int64_t j = 0; j < len; ++j) {
        double a = exp(s[j] - lse);
        const double* vj = vh + j * d;
        for (int64_t c = 0; c < d; ++c) o_row[c] += a * vj[c];
    }
    return lse;
}

/* O and lse for all heads and rows. */
void oracle_attn_fwd(const double* q, const double* k, const double* v, int64_t BH,
                     int64_t N, int64_t d, int causal, double scale, double* o,
                     double* lse)
{
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < BH * N; ++r) {
            int64_t h = r / N, i = r % N;
            lse[r] = fwd_row(q, k, v, h, i, N, d, causal, scale, s, o + r * d);
        }
        free(s);
    }
}

/* O and lse for a selection of (head, row) pairs only: the sampled check of
 * large workloads.  o_sel is [nsel][d], lse_sel is [nsel]. */
void oracle_attn_fwd_rows(const double* q, const double* k, const double* v,
                          int64_t BH, int64_t N, int64_t d, int causal, double scale,
                          const int64_t* heads, const int64_t* rows, int64_t nsel,
                          double* o_sel, double* lse_sel)
{
    (void)BH;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < nsel; ++t)
            lse_sel[t] = fwd_row(q, k, v, heads[t], rows[t], N, d, causal, scale, s,
                                 o_sel + t * d);
        free(s);
    }
}

/* The full attention matrix A = softmax(S) of every head, [BH][N][N]; masked
 * entries are exactly 0.  For small cases only. */
void oracle_attn_probs(const double* q, const double* k, int64_t BH, int64_t N,
                       int64_t d, int causal, double scale, double* A)
{
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < BH * N; ++r) {
            int64_t h = r / N, i = r % N;
            int64_t len = scores_row(q, k, h, i, N, d, causal, scale, s);
            double lse = logsumexp_row(s, len);
            double* Ar = A + r * N;
            for (int64_t j = 0; j < N; ++j) Ar[j] = j < len ? exp(s[j] - lse) : 0.0;
        }
        free(s);
    }
}

/*
 * Backward.  Pass 1 (one thread per row i): scores, lse_i, A_i, dA_i,
 * D_i = sum_j A_ij dA_ij and dQ_i = scale sum_j dS_ij k_j.  Pass 2 (one
 * thread per key row j): A_ij and dS_ij from the same definitions, using
 * lse_i and D_i from pass 1, then dV_j = sum_i A_ij dO_i and
 * dK_j = scale sum_i dS_ij q_i.  Only O(N) per-row values cross between the
 * passes; no N x N matrix is stored.
 */
void oracle_attn_bwd(const double* q, const double* k, const double* v,
                     const double* dout, int64_t BH, int64_t N, int64_t d, int causal,
                     double scale, double* dq, double* dk, double* dv)
{
    double* lse = (double*)malloc(sizeof(double) * (size_t)(BH * N > 0 ? BH * N : 1));
    double* D = (double*)malloc(sizeof(double) * (size_t)(BH * N > 0 ? BH * N : 1));

#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        double* da = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < BH * N; ++r) {
            int64_t h = r / N, i = r % N;
            const double* vh = v + h * N * d;
            const double* kh = k + h * N * d;
            const double* doi = dout + r * d;
            int64_t len = scores_row(q, k, h, i, N, d, causal, scale, s);
            double l = logsumexp_row(s, len);
            lse[r] = l;
            double Di = 0.0;
            for (int64_t j = 0; j < len; ++j) {
                const double* vj = vh + j * d;
                double acc = 0.0;
                for (int64_t c = 0; c < d; ++c) acc += doi[c] * vj[c];
                da[j] = acc;
                Di += exp(s[j] - l) * acc;
            }
            D[r] = Di;
            double* dqi = dq + r * d;
            for (int64_t c = 0; c < d; ++c) dqi[c] = 0.0;
            for (int64_t j = 0; j < len; ++j) {
                double ds = exp(s[j] - l) * (da[j] - Di);
                const double* kj = kh + j * d;
                for (int64_t c = 0; c < d; ++c) dqi[c] += ds * kj[c];
            }
            for (int64_t c = 0; c < d; ++c) dqi[c] *= scale;
        }
        free(s);
        free(da);
    }

#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t r = 0; r < BH * N; ++r) {
        int64_t h = r / N, j = r % N;
        const double* qh = q + h * N * d;
        const double* kj = k + r * d;
        const double* vj = v + r * d;
        const double* doh = dout + h * N * d;
        double* dkj = dk + r * d;
        double* dvj = dv + r * d;
        for (int64_t c = 0; c < d; ++c) { dkj[c] = 0.0; dvj[c] = 0.0; }
        int64_t i0 = causal ? j : 0;
        for (int64_t i = i0; i < N; ++i) {
            const double* qi = qh + i * d;
            const double* doi = doh + i * d;
            double sdot = 0.0, ddot = 0.0;
            for (int64_t c = 0; c < d; ++c) { sdot += qi[c] * kj[c]; ddot += doi[c] * vj[c]; }
            double a = exp(scale * sdot - lse[h * N + i]);
            double ds = a * (ddot - D[h * N + i]);
            for (int64_t c = 0; c < d; ++c) { dvj[c] += a * doi[c]; dkj[c] += ds * qi[c]; }
        }
        for (int64_t c = 0; c < d; ++c) dkj[c] *= scale;
    }
    free(lse);
    free(D);
}

/* Floating-point operation counts of the method, as the pages count them:
 * the forward pass is two S x S x d matmuls, 4 S^2 d per head (cs2680
 * Lecture 9, sec. 9.2), half of that when causal; the recomputation of the
 * scores in the backward pass is one extra Q K^T, 2 S^2 d (sec. 9.6). */
double oracle_fwd_flops(int64_t BH, int64_t N, int64_t d, int causal)
{
    double f = 4.0 * (double)BH * (double)N * (double)N * (double)d;
    return causal ? 0.5 * f : f;
}

double oracle_recompute_flops(int64_t N, int64_t d)
{
    return 2.0 * (double)N * (double)N * (double)d;
}

/* General forward (see the header): q, o are [B][Hq][Nq][d], k, v are
 * [B][Hkv][Nkv][d], lse is [B][Hq][Nq]. */
void oracle_attn_fwd_gqa(const double* q, const double* k, const double* v, int64_t B,
                         int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nkv, int64_t d, int causal,
                         double scale, double* o, double* lse)
{
    const int64_t G = Hq / Hkv;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(Nkv > 0 ? Nkv : 1));
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < B * Hq * Nq; ++r) {
            const int64_t b = r / (Hq * Nq), h = (r / Nq) % Hq, i = r % Nq;
            const int64_t hk = h / G;
            const double* qi = q + r * d;
            const double* kh = k + (b * Hkv + hk) * Nkv * d;
            const double* vh = v + (b * Hkv + hk) * Nkv * d;
            int64_t len = Nkv;
            if (causal) {
                int64_t lim = i + Nkv - Nq + 1;  /* keys j < lim are visible */
                len = lim < 0 ? 0 : (lim < Nkv ? lim : Nkv);
            }
            double* orow = o + r * d;
            for (int64_t c = 0; c < d; ++c) orow[c] = 0.0;
            if (len == 0) { lse[r] = -INFINITY; continue; }
            for (int64_t j = 0; j < len; ++j) {
                const double* kj = kh + j * d;
                double acc = 0.0;
                for (int64_t c = 0; c < d; ++c) acc += qi[c] * kj[c];
                s[j] = scale * acc;
            }
            const double l = logsumexp_row(s, len);
            lse[r] = l;
            for (int64_t j = 0; j < len; ++j) {
                const double a = exp(s[j] - l);
                const double* vj = vh + j * d;
                for (int64_t c = 0; c < d; ++c) orow[c] += a * vj[c];
            }
        }
        free(s);
    }
}

/* Merge S partial results over disjoint key ranges: o_parts is [S][R][d],
 * lse_parts is [S][R] (a part with no key has lse = -inf and is ignored). */
void oracle_combine_splits(const double* o_parts, const double* lse_parts, int64_t S, int64_t R,
                           int64_t d, double* o, double* lse)
{
    for (int64_t r = 0; r < R; ++r) {
        double m = -INFINITY;
        for (int64_t t = 0; t < S; ++t) if (lse_parts[t * R + r] > m) m = lse_parts[t * R + r];
        double* orow = o + r * d;
        for (int64_t c = 0; c < d; ++c) orow[c] = 0.0;
        if (m == -INFINITY) { lse[r] = -INFINITY; continue; }
        double sum = 0.0;
        for (int64_t t = 0; t < S; ++t) sum += exp(lse_parts[t * R + r] - m);
        const double l = m + log(sum);
        lse[r] = l;
        for (int64_t t = 0; t < S; ++t) {
            const double w = exp(lse_parts[t * R + r] - l);
            if (w == 0.0) continue;
            const double* part = o_parts + (t * R + r) * d;
            for (int64_t c = 0; c < d; ++c) orow[c] += w * part[c];
        }
    }
}

static int visible(int64_t i, int64_t j, int causal, const unsigned char* bm, int64_t nb,
                   int64_t bs)
{
    if (causal && j > i) return 0;
    return bm[(i / bs) * nb + j / bs] != 0;
}

/* Block-sparse forward (see the header); q, k, v, o are [BH][N][d]. */
void oracle_attn_fwd_blockmask(const double* q, const double* k, const double* v, int64_t BH,
                               int64_t N, int64_t d, int causal, double scale,
                               const unsigned char* bm, int64_t bs, double* o, double* lse)
{
    const int64_t nb = (N + bs - 1) / bs;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < BH * N; ++r) {
            const int64_t h = r / N, i = r % N;
            const double* qi = q + r * d;
            double m = -INFINITY;
            for (int64_t j = 0; j < N; ++j) {
                if (!visible(i, j, causal, bm, nb, bs)) { s[j] = -INFINITY; continue; }
                const double* kj = k + (h * N + j) * d;
                double acc = 0.0;
                for (int64_t c = 0; c < d; ++c) acc += qi[c] * kj[c];
                s[j] = scale * acc;
                if (s[j] > m) m = s[j];
            }
            double* orow = o + r * d;
            for (int64_t c = 0; c < d; ++c) orow[c] = 0.0;
            if (m == -INFINITY) { lse[r] = -INFINITY; continue; }
            double l = 0.0;
            for (int64_t j = 0; j < N; ++j) if (s[j] > -INFINITY) l += exp(s[j] - m);
            const double ls = m + log(l);
            lse[r] = ls;
            for (int64_t j = 0; j < N; ++j) {
                if (s[j] == -INFINITY) continue;
                const double a = exp(s[j] - ls);
                const double* vj = v + (h * N + j) * d;
                for (int64_t c = 0; c < d; ++c) orow[c] += a * vj[c];
            }
        }
        free(s);
    }
}

/* Block-sparse backward: the textbook formulas over the visible entries
 * (A = 0 elsewhere), in the two passes of oracle_attn_bwd. */
void oracle_attn_bwd_blockmask(const double* q, const double* k, const double* v,
                               const double* dout, int64_t BH, int64_t N, int64_t d, int causal,
                               double scale, const unsigned char* bm, int64_t bs, double* dq,
                               double* dk, double* dv)
{
    const int64_t nb = (N + bs - 1) / bs;
    double* lse = (double*)malloc(sizeof(double) * (size_t)(BH * N > 0 ? BH * N : 1));
    double* D = (double*)malloc(sizeof(double) * (size_t)(BH * N > 0 ? BH * N : 1));
    double* o = (double*)malloc(sizeof(double) * (size_t)(BH * N * d > 0 ? BH * N * d : 1));
    oracle_attn_fwd_blockmask(q, k, v, BH, N, d, causal, scale, bm, bs, o, lse);
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t r = 0; r < BH * N; ++r) {
        const int64_t h = r / N, i = r % N;
        const double* qi = q + r * d;
        const double* doi = dout + r * d;
        double* dqi = dq + r * d;
        for (int64_t c = 0; c < d; ++c) dqi[c] = 0.0;
        double Di = 0.0;
        if (lse[r] == -INFINITY) { D[r] = 0.0; continue; }
        for (int64_t j = 0; j < N; ++j) {
            if (!visible(i, j, causal, bm, nb, bs)) continue;
            const double* kj = k + (h * N + j) * d;
            const double* vj = v + (h * N + j) * d;
            double sd = 0.0, dd = 0.0;
            for (int64_t c = 0; c < d; ++c) { sd += qi[c] * kj[c]; dd += doi[c] * vj[c]; }
            Di += exp(scale * sd - lse[r]) * dd;
        }
        D[r] = Di;
        for (int64_t j = 0; j < N; ++j) {
            if (!visible(i, j, causal, bm, nb, bs)) continue;
            const double* kj = k + (h * N + j) * d;
            const double* vj = v + (h * N + j) * d;
            double sd = 0.0, dd = 0.0;
            for (int64_t c = 0; c < d; ++c) { sd += qi[c] * kj[c]; dd += doi[c] * vj[c]; }
            const double ds = exp(scale * sd - lse[r]) * (dd - Di);
            for (int64_t c = 0; c < d; ++c) dqi[c] += ds * kj[c];
        }
        for (int64_t c = 0; c < d; ++c) dqi[c] *= scale;
    }
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t r = 0; r < BH * N; ++r) {
        const int64_t h = r / N, j = r % N;
        const double* kj = k + r * d;
        const double* vj = v + r * d;
        double* dkj = dk + r * d;
        double* dvj = dv + r * d;
        for (int64_t c = 0; c < d; ++c) { dkj[c] = 0.0; dvj[c] = 0.0; }
        for (int64_t i = 0; i < N; ++i) {
            if (!visible(i, j, causal, bm, nb, bs) || lse[h * N + i] == -INFINITY) continue;
            const double* qi = q + (h * N + i) * d;
            const double* doi = dout + (h * N + i) * d;
            double sd = 0.0, dd = 0.0;
            for (int64_t c = 0; c < d; ++c) { sd += qi[c] * kj[c]; dd += doi[c] * vj[c]; }
            const double a = exp(scale * sd - lse[h * N + i]);
            const double ds = a * (dd - D[h * N + i]);
            for (int64_t c = 0; c < d; ++c) { dvj[c] += a * doi[c]; dkj[c] += ds * qi[c]; }
        }
        for (int64_t c = 0; c < d; ++c) dkj[c] *= scale;
    }
    free(lse);
    free(D);
    free(o);
}

/* ------------------------------------------------------------------ FP8 */

/* Value of an E4M3 code: sign, 4 exponent bits with bias 7, 3 mantissa
 * bits; exponent field 0 is subnormal (mantissa / 8 * 2^-6); exponent 15
 * with mantissa 7 is NaN (there is no infinity). */
double oracle_e4m3_decode(unsigned char c)
{
    const int sgn = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sgn ? -v : v;
}

/* Nearest E4M3 code to x, ties to the even code (even mantissa), magnitudes
 * above the largest finite value 448 saturated to 448: a plain search over
 * the 127 non-negative finite codes. */
unsigned char oracle_e4m3_encode(double x)
{
    const int neg = signbit(x) != 0;
    const double a = fabs(x);
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        const double err = fabs(oracle_e4m3_decode((unsigned char)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0)) {
            best = c;
            best_err = err;
        }
    }
    if (a >= 448.0) best = 0x7E;
    return (unsigned char)(best | (neg ? 0x80 : 0));
}

/* y = x H_d row by row (rows x d), H_d[i][j] = (-1)^popcount(i & j). */
void oracle_hadamard(const double* x, int64_t rows, int64_t d, double* y)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t j = 0; j < d; ++j) {
            double acc = 0.0;
            for (int64_t i = 0; i < d; ++i) {
                const int odd = __builtin_popcountll((unsigned long long)(i & j)) & 1;
                acc += odd ? -x[r * d + i] : x[r * d + i];
            }
            y[r * d + j] = acc;
        }
    }
}

/* Quantise n values with one scale (step 2 of the FP8 form): codes[n] and
 * the dequantisation scale amax / 448 (fp32), returned. */
float oracle_quantize_e4m3(const double* x, int64_t n, unsigned char* codes)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        const float a = fabsf((float)x[i]);
        if (a > amax) amax = a;
    }
    if (amax == 0.0f) {
        for (int64_t i = 0; i < n; ++i) codes[i] = 0;
        return 1.0f;
    }
    const float inv = 448.0f / amax;
    for (int64_t i = 0; i < n; ++i) {
        const float y = (float)x[i] * inv;
        codes[i] = oracle_e4m3_encode((double)y);
    }
    return amax / 448.0f;
}

/* The FP8 forward pass (steps 1-3 of the FP8 form).  q, k, v, o are
 * [BH][N][d]; q8, k8, v8 receive the codes ([BH][N][d]) and descale the
 * scales, [3][BH] for Q, K, V. */
void oracle_attn_fwd_fp8(const double* q, const double* k, const double* v, int64_t BH,
                         int64_t N, int64_t d, int causal, double scale, int hadamard,
                         double* o, double* lse, unsigned char* q8, unsigned char* k8,
                         unsigned char* v8, float* descale)
{
    const int64_t n = BH * N * d, per = N * d;
    double* qh = (double*)malloc(sizeof(double) * (size_t)n);
    double* kh = (double*)malloc(sizeof(double) * (size_t)n);
    double* qd = (double*)malloc(sizeof(double) * (size_t)n);
    double* kd = (double*)malloc(sizeof(double) * (size_t)n);
    double* vd = (double*)malloc(sizeof(double) * (size_t)n);
    if (hadamard) {
        oracle_hadamard(q, BH * N, d, qh);
        oracle_hadamard(k, BH * N, d, kh);
    } else {
        for (int64_t i = 0; i < n; ++i) { qh[i] = q[i]; kh[i] = k[i]; }
    }
    for (int64_t h = 0; h < BH; ++h) {
        const float sq = oracle_quantize_e4m3(qh + h * per, per, q8 + h * per);
        const float sk = oracle_quantize_e4m3(kh + h * per, per, k8 + h * per);
        const float sv = oracle_quantize_e4m3(v + h * per, per, v8 + h * per);
        descale[h] = sq;
        descale[BH + h] = sk;
        descale[2 * BH + h] = sv;
        for (int64_t i = h * per; i < (h + 1) * per; ++i) {
            qd[i] = oracle_e4m3_decode(q8[i]) * (double)sq;
            kd[i] = oracle_e4m3_decode(k8[i]) * (double)sk;
            vd[i] = oracle_e4m3_decode(v8[i]) * (double)sv;
        }
    }
    oracle_attn_fwd(qd, kd, vd, BH, N, d, causal, hadamard ? scale / (double)d : scale, o, lse);
    free(qh);
    free(kh);
    free(qd);
    free(kd);
    free(vd);
}

/* Element-wise oracle_e4m3_encode / oracle_e4m3_decode over arrays. */
void oracle_e4m3_encode_array(const double* x, int64_t n, unsigned char* out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(x[i]);
}

void oracle_e4m3_decode_array(const unsigned char* c, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_decode(c[i]);
}
