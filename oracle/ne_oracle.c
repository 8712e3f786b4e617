/*
 * ne_oracle.c -- CPU oracle for causal grouped-query attention with rotary
 * position embeddings (RoPE), forward and backward, in double precision.
 *
 * TEST INFRASTRUCTURE ONLY.  The test suite, the package smoke check and the
 * benchmark's CPU-baseline leg are the only callers.  It shares no code with
 * the CUDA library and must never be used as a fallback for it.
 *
 * What it computes (the plain definition, no tiling, no online softmax):
 *
 *   "NanoEuler: GPT-2 scale LLM in C and CUDA", technical specification:
 *   RoPE is applied to the queries and keys; grouped-query attention shares a
 *   smaller set of key/value heads among the query heads; the model is
 *   decoder-only (causal).  "Building GPT-2 in a 100KB C/CUDA file" section
 *   3.4: the FlashAttention kernel is tiled attention with an online softmax
 *   that never stores the T x T matrix.  That is an exact reorganisation of
 *   softmax attention, so the oracle is softmax attention itself, with the
 *   T x T score matrix materialised.
 *
 *   RoPE (rotate-half pairing, positive angle, 0-based positions):
 *     theta_i = theta^(-2i/d),  a = pos * theta_i,  i = 0 .. d/2-1
 *     x'_i       = x_i cos a - x_{i+d/2} sin a
 *     x'_{i+d/2} = x_{i+d/2} cos a + x_i sin a
 *   GQA head map: query head h reads key/value head h / (Hq/Hkv).
 *   S[t,s] = <q'[t,h], k'[s,kv(h)]> / sqrt(d) for s <= t, -inf otherwise.
 *   Sliding window (window = W > 0): also -inf for s <= t - W, so query t
 *   sees the W keys t-W+1 .. t (the nanochat guide's per-layer window
 *   pattern); window = 0 is the plain causal mask.
 *   P = row softmax of S;  lse[t] = ln sum_s exp S[t,s];  O[t] = sum_s P v[s].
 *
 *   Backward for the loss L = sum(O * dO):
 *     dv[s]  = sum over heads of the group, sum_t P[t,s] dO[t]
 *     dP     = dO v^T,  D[t] = <dO[t], O[t]>,  dS = P * (dP - D)
 *     dq'[t] = sum_s dS[t,s] k'[s] / sqrt(d)
 *     dk'[s] = sum over heads, sum_t dS[t,s] q'[t] / sqrt(d)
 *     dq = R(t)^T dq',  dk = R(s)^T dk'    (rotation by -a)
 *   The pages validate every analytic gradient against a central finite
 *   difference in double precision ("Building GPT-2 ..." section 2.1); the
 *   test suite applies that check to this file.
 *
 * Layout: q, o, dO, dq are [B][T][Hq][d]; k, v, dk, dv are [B][T][Hkv][d];
 * lse and D are [B][Hq][T].  All arrays are contiguous float64.
 * window: 0 for the causal mask alone, W > 0 for a sliding window of W keys.
 * pos_offset shifts every position by a constant (a test hook for the
 * relative-position property of RoPE); the library itself always uses 0.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define IDX(b, t, h, c, T, H, d) ((((size_t)(b) * (T) + (t)) * (H) + (h)) * (d) + (c))

static void rope_row(const double *x, double *y, int d, double theta, long pos, int inverse)
{
    int half = d / 2;
    for (int i = 0; i < half; ++i) {
        double freq = pow(theta, -2.0 * (double)i / (double)d);
        double a = (double)pos * freq;
        double c = cos(a), s = sin(a);
        if (inverse)
            s = -s;
        double x0 = x[i], x1 = x[i + half];
        y[i] = x0 * c - x1 * s;
        y[i + half] = x1 * c + x0 * s;
    }
}

/* Rotate every row of a [B][T][H][d] array: y = R(pos) x (inverse: R(pos)^T x). */
int ne_oracle_rope(const double *x, double *y, int B, int T, int H, int d, double theta,
                   long pos_offset, int inverse)
{
    if (d <= 0 || d % 2)
        return 1;
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < T; ++t)
            for (int h = 0; h < H; ++h)
                rope_row(x + IDX(b, t, h, 0, T, H, d), y + IDX(b, t, h, 0, T, H, d), d, theta,
                         (long)t + pos_offset, inverse);
    return 0;
}

static int check_shape(int B, int T, int Hq, int Hkv, int d)
{
    if (B < 1 || T < 1 || Hq < 1 || Hkv < 1 || d < 2 || d % 2 || Hq % Hkv)
        return 1;
    return 0;
}

/*
 * Softmax probabilities of one (b, h): P is T x T, row-major, zero above the
 * diagonal.  qr and kr are the rotated query / key rows of this head (T x d).
 * Writes lse[t] (natural log) as well.
 */
static void probs(const double *qr, const double *kr, int T, int d, int window, double *P,
                  double *lse)
{
    double scale = 1.0 / sqrt((double)d);
    for (int t = 0; t < T; ++t) {
        double *S = P + (size_t)t * T;
        for (int s = 0; s < T; ++s) {
            if (s > t) {
                S[s] = -INFINITY;
                continue;
            }
            if (window > 0 && t - s >= window) {   /* outside the sliding window */
                S[s] = -INFINITY;
                continue;
            }
            double acc = 0.0;
            for (int c = 0; c < d; ++c)
                acc += qr[(size_t)t * d + c] * kr[(size_t)s * d + c];
            S[s] = acc * scale;
        }
        double mx = -INFINITY;
        for (int s = 0; s <= t; ++s)
            if (S[s] > mx)
                mx = S[s];
        double sum = 0.0;
        for (int s = 0; s <= t; ++s)
            sum += exp(S[s] - mx);
        double l = mx + log(sum);
        lse[t] = l;
        for (int s = 0; s < T; ++s)
            S[s] = (s <= t) ? exp(S[s] - l) : 0.0;
    }
}

static void gather_rotated(const double *x, double *xr, int b, int h, int T, int H, int d,
                           double theta, long pos_offset)
{
    for (int t = 0; t < T; ++t)
        rope_row(x + IDX(b, t, h, 0, T, H, d), xr + (size_t)t * d, d, theta,
                 (long)t + pos_offset, 0);
}

int ne_oracle_fwd(const double *q, const double *k, const double *v, double *o, double *lse,
                  int B, int T, int Hq, int Hkv, int d, double theta, long pos_offset,
                  int nthreads, int window)
{
    if (check_shape(B, T, Hq, Hkv, d))
        return 1;
    int G = Hq / Hkv;
    int nbh = B * Hq;
    int err = 0;
#ifdef _OPENMP
    if (nthreads < 1)
        nthreads = omp_get_max_threads();
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1)
#endif
    for (int bh = 0; bh < nbh; ++bh) {
        int b = bh / Hq, h = bh % Hq, j = h / G;
        double *qr = malloc(sizeof(double) * (size_t)T * d);
        double *kr = malloc(sizeof(double) * (size_t)T * d);
        double *P = malloc(sizeof(double) * (size_t)T * T);
        if (!qr || !kr || !P) {
            err = 2;
        } else {
            gather_rotated(q, qr, b, h, T, Hq, d, theta, pos_offset);
            gather_rotated(k, kr, b, j, T, Hkv, d, theta, pos_offset);
            probs(qr, kr, T, d, window, P, lse + ((size_t)b * Hq + h) * T);
            for (int t = 0; t < T; ++t) {
                double *orow = o + IDX(b, t, h, 0, T, Hq, d);
                for (int c = 0; c < d; ++c)
                    orow[c] = 0.0;
                for (int s = 0; s <= t; ++s) {
                    double p = P[(size_t)t * T + s];
                    const double *vrow = v + IDX(b, s, j, 0, T, Hkv, d);
                    for (int c = 0; c < d; ++c)
                        orow[c] += p * vrow[c];
                }
            }
        }
        free(qr);
        free(kr);
        free(P);
    }
    return err;
}

/*
 * Backward.  Writes dq, dk, dv; optionally (non-NULL) o, lse and D as the
 * oracle computes them.  Parallel over (b, kv head) groups so that dk and dv
 * are summed over the group's query heads without races.
 */
int ne_oracle_bwd(const double *q, const double *k, const double *v, const double *dO,
                  double *dq, double *dk, double *dv, double *o_out, double *lse_out,
                  double *D_out, int B, int T, int Hq, int Hkv, int d, double theta,
                  long pos_offset, int nthreads, int window)
{
    if (check_shape(B, T, Hq, Hkv, d))
        return 1;
    int G = Hq / Hkv;
    int ngroups = B * Hkv;
    double scale = 1.0 / sqrt((double)d);
    int err = 0;
#ifdef _OPENMP
    if (nthreads < 1)
        nthreads = omp_get_max_threads();
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1)
#endif
    for (int bj = 0; bj < ngroups; ++bj) {
        int b = bj / Hkv, j = bj % Hkv;
        size_t Td = (size_t)T * d;
        double *qr = malloc(sizeof(double) * Td);
        double *kr = malloc(sizeof(double) * Td);
        double *dqr = malloc(sizeof(double) * Td);
        double *dkr = calloc(Td, sizeof(double));
        double *orow = malloc(sizeof(double) * d);
        double *lse = malloc(sizeof(double) * T);
        double *Dv = malloc(sizeof(double) * T);
        double *P = malloc(sizeof(double) * (size_t)T * T);
        if (!qr || !kr || !dqr || !dkr || !orow || !lse || !Dv || !P) {
            err = 2;
            goto done;
        }
        gather_rotated(k, kr, b, j, T, Hkv, d, theta, pos_offset);
        for (int s = 0; s < T; ++s)
            memset(dv + IDX(b, s, j, 0, T, Hkv, d), 0, sizeof(double) * d);
        for (int h = j * G; h < (j + 1) * G; ++h) {
            gather_rotated(q, qr, b, h, T, Hq, d, theta, pos_offset);
            probs(qr, kr, T, d, window, P, lse);
            memset(dqr, 0, sizeof(double) * Td);
            for (int t = 0; t < T; ++t) {
                const double *dorow = dO + IDX(b, t, h, 0, T, Hq, d);
                /* O[t] and D[t] = <dO[t], O[t]> */
                for (int c = 0; c < d; ++c)
                    orow[c] = 0.0;
                for (int s = 0; s <= t; ++s) {
                    double p = P[(size_t)t * T + s];
                    const double *vrow = v + IDX(b, s, j, 0, T, Hkv, d);
                    for (int c = 0; c < d; ++c)
                        orow[c] += p * vrow[c];
                }
                double Dt = 0.0;
                for (int c = 0; c < d; ++c)
                    Dt += dorow[c] * orow[c];
                Dv[t] = Dt;
                if (o_out)
                    memcpy(o_out + IDX(b, t, h, 0, T, Hq, d), orow, sizeof(double) * d);
                for (int s = 0; s <= t; ++s) {
                    double p = P[(size_t)t * T + s];
                    const double *vrow = v + IDX(b, s, j, 0, T, Hkv, d);
                    double *dvrow = dv + IDX(b, s, j, 0, T, Hkv, d);
                    double dp = 0.0;
                    for (int c = 0; c < d; ++c)
                        dp += dorow[c] * vrow[c];
                    double ds = p * (dp - Dt);
                    for (int c = 0; c < d; ++c) {
                        dvrow[c] += p * dorow[c];
                        dqr[(size_t)t * d + c] += scale * ds * kr[(size_t)s * d + c];
                        dkr[(size_t)s * d + c] += scale * ds * qr[(size_t)t * d + c];
                    }
                }
            }
            for (int t = 0; t < T; ++t)
                rope_row(dqr + (size_t)t * d, dq + IDX(b, t, h, 0, T, Hq, d), d, theta,
                         (long)t + pos_offset, 1);
            if (lse_out)
                memcpy(lse_out + ((size_t)b * Hq + h) * T, lse, sizeof(double) * T);
            if (D_out)
                memcpy(D_out + ((size_t)b * Hq + h) * T, Dv, sizeof(double) * T);
        }
        for (int s = 0; s < T; ++s)
            rope_row(dkr + (size_t)s * d, dk + IDX(b, s, j, 0, T, Hkv, d), d, theta,
                     (long)s + pos_offset, 1);
    done:
        free(qr);
        free(kr);
        free(dqr);
        free(dkr);
        free(orow);
        free(lse);
        free(Dv);
        free(P);
    }
    return err;
}

/*
 * Variable-length (padded) batches: sequence b holds its first seqlen[b]
 * tokens, 0 <= seqlen[b] <= T, and the rows after them are padding.  The
 * NanoEuler SFT stage pads every instruction/response pair to the context
 * and masks the loss on prompt and padding ("Rebuilding GPT-2 in one 100KB
 * C/CUDA file" section 3.2, SFT stage; "NanoEuler: a GPT-2-scale LLM"
 * two-stage training, SFT).  Each sequence is its own causal problem over
 * its L = seqlen[b] tokens (positions 0 .. L-1), so the definition is the
 * attention above applied to every sequence's prefix; a padding row attends
 * to nothing: O = 0, lse = -inf.  In the backward only the valid rows carry
 * a loss, so dq, dk, dv are the prefix problem's gradients and 0 on padding
 * positions (dO of padding rows is never read).  A sequence's prefix rows are
 * contiguous in the [B][T][H][d] layout, so each call below is the B = 1,
 * T = L problem on a pointer into batch b.
 */
int ne_oracle_fwd_varlen(const double *q, const double *k, const double *v, double *o,
                         double *lse, const int *seqlen, int B, int T, int Hq, int Hkv, int d,
                         double theta, long pos_offset, int nthreads)
{
    if (check_shape(B, T, Hq, Hkv, d) || !seqlen)
        return 1;
    for (int b = 0; b < B; ++b)
        if (seqlen[b] < 0 || seqlen[b] > T)
            return 1;
    double *lse1 = malloc(sizeof(double) * (size_t)Hq * T);
    if (!lse1)
        return 2;
    int err = 0;
    for (int b = 0; b < B && !err; ++b) {
        int L = seqlen[b];
        for (int t = L; t < T; ++t)
            memset(o + IDX(b, t, 0, 0, T, Hq, d), 0, sizeof(double) * Hq * d);
        for (int h = 0; h < Hq; ++h)
            for (int t = L; t < T; ++t)
                lse[((size_t)b * Hq + h) * T + t] = -INFINITY;
        if (L == 0)
            continue;
        err = ne_oracle_fwd(q + IDX(b, 0, 0, 0, T, Hq, d), k + IDX(b, 0, 0, 0, T, Hkv, d),
                            v + IDX(b, 0, 0, 0, T, Hkv, d), o + IDX(b, 0, 0, 0, T, Hq, d), lse1,
                            1, L, Hq, Hkv, d, theta, pos_offset, nthreads, 0);
        for (int h = 0; h < Hq; ++h)
            memcpy(lse + ((size_t)b * Hq + h) * T, lse1 + (size_t)h * L, sizeof(double) * L);
    }
    free(lse1);
    return err;
}

int ne_oracle_bwd_varlen(const double *q, const double *k, const double *v, const double *dO,
                         double *dq, double *dk, double *dv, const int *seqlen, int B, int T,
                         int Hq, int Hkv, int d, double theta, long pos_offset, int nthreads)
{
    if (check_shape(B, T, Hq, Hkv, d) || !seqlen)
        return 1;
    for (int b = 0; b < B; ++b)
        if (seqlen[b] < 0 || seqlen[b] > T)
            return 1;
    int err = 0;
    for (int b = 0; b < B && !err; ++b) {
        int L = seqlen[b];
        for (int t = L; t < T; ++t) {
            memset(dq + IDX(b, t, 0, 0, T, Hq, d), 0, sizeof(double) * Hq * d);
            memset(dk + IDX(b, t, 0, 0, T, Hkv, d), 0, sizeof(double) * Hkv * d);
            memset(dv + IDX(b, t, 0, 0, T, Hkv, d), 0, sizeof(double) * Hkv * d);
        }
        if (L == 0)
            continue;
        err = ne_oracle_bwd(q + IDX(b, 0, 0, 0, T, Hq, d), k + IDX(b, 0, 0, 0, T, Hkv, d),
                            v + IDX(b, 0, 0, 0, T, Hkv, d), dO + IDX(b, 0, 0, 0, T, Hq, d),
                            dq + IDX(b, 0, 0, 0, T, Hq, d), dk + IDX(b, 0, 0, 0, T, Hkv, d),
                            dv + IDX(b, 0, 0, 0, T, Hkv, d), NULL, NULL, NULL, 1, L, Hq, Hkv, d,
                            theta, pos_offset, nthreads, 0);
    }
    return err;
}

/*
 * Packed variable-length batches: the B sequences are concatenated along the
 * token axis, sequence b holding tokens cu[b] .. cu[b+1]-1 of the pack
 * (cu[0] = 0, non-decreasing, cu[B] = total), with no padding between them.
 * Same definition as the padded form above: each sequence is a causal
 * problem of its own over positions 0 .. len-1.  q, o, dO, dq are
 * [total][Hq][d]; k, v, dk, dv are [total][Hkv][d]; lse is [Hq][total].
 * Every sequence's rows are contiguous, so each call is the B = 1, T = len
 * problem on a pointer into the pack.
 */
static int check_cu(const int *cu, int B)
{
    if (!cu || B < 1 || cu[0] != 0)
        return 1;
    for (int b = 0; b < B; ++b)
        if (cu[b + 1] < cu[b])
            return 1;
    return 0;
}

int ne_oracle_fwd_packed(const double *q, const double *k, const double *v, double *o,
                         double *lse, const int *cu, int B, int Hq, int Hkv, int d,
                         double theta, long pos_offset, int nthreads)
{
    if (check_cu(cu, B) || check_shape(1, 1, Hq, Hkv, d))
        return 1;
    const int total = cu[B];
    double *lse1 = malloc(sizeof(double) * (size_t)Hq * (total > 0 ? total : 1));
    if (!lse1)
        return 2;
    int err = 0;
    for (int b = 0; b < B && !err; ++b) {
        int L = cu[b + 1] - cu[b];
        if (L == 0)
            continue;
        err = ne_oracle_fwd(q + (size_t)cu[b] * Hq * d, k + (size_t)cu[b] * Hkv * d,
                            v + (size_t)cu[b] * Hkv * d, o + (size_t)cu[b] * Hq * d, lse1, 1, L,
                            Hq, Hkv, d, theta, pos_offset, nthreads, 0);
        for (int h = 0; h < Hq; ++h)
            memcpy(lse + (size_t)h * total + cu[b], lse1 + (size_t)h * L, sizeof(double) * L);
    }
    free(lse1);
    return err;
}

int ne_oracle_bwd_packed(const double *q, const double *k, const double *v, const double *dO,
                         double *dq, double *dk, double *dv, const int *cu, int B, int Hq,
                         int Hkv, int d, double theta, long pos_offset, int nthreads)
{
    if (check_cu(cu, B) || check_shape(1, 1, Hq, Hkv, d))
        return 1;
    int err = 0;
    for (int b = 0; b < B && !err; ++b) {
        int L = cu[b + 1] - cu[b];
        if (L == 0)
            continue;
        err = ne_oracle_bwd(q + (size_t)cu[b] * Hq * d, k + (size_t)cu[b] * Hkv * d,
                            v + (size_t)cu[b] * Hkv * d, dO + (size_t)cu[b] * Hq * d,
                            dq + (size_t)cu[b] * Hq * d, dk + (size_t)cu[b] * Hkv * d,
                            dv + (size_t)cu[b] * Hkv * d, NULL, NULL, NULL, 1, L, Hq, Hkv, d,
                            theta, pos_offset, nthreads, 0);
    }
    return err;
}

/*
 * Decode against a key/value cache (one new token per sequence).  The new
 * token is the last of Tk positions: its own key and value are the cache's
 * last rows, so every cached key is visible to it.  By definition this is the
 * last row (t = Tk - 1) of the causal attention above over the Tk positions:
 *   q1 is [B][Hq][d] (pre-RoPE; rotated at position Tk - 1 + pos_offset),
 *   k, v are [B][Tk][Hkv][d] (pre-RoPE keys, rotated at their positions),
 *   S[s] = <q1'[b,h], k'[b,s,kv(h)]> / sqrt(d) for s = 0 .. Tk-1,
 *   P = softmax(S), lse = ln sum_s exp S[s], o1[b,h] = sum_s P[s] v[b,s,kv(h)].
 * o1 is [B][Hq][d], lse1 is [B][Hq].
 */
int ne_oracle_decode(const double *q1, const double *k, const double *v, double *o1,
                     double *lse1, int B, int Tk, int Hq, int Hkv, int d, double theta,
                     long pos_offset)
{
    if (check_shape(B, Tk, Hq, Hkv, d))
        return 1;
    int G = Hq / Hkv;
    double scale = 1.0 / sqrt((double)d);
    double *qr = malloc(sizeof(double) * d);
    double *kr = malloc(sizeof(double) * d);
    double *S = malloc(sizeof(double) * Tk);
    if (!qr || !kr || !S) {
        free(qr);
        free(kr);
        free(S);
        return 2;
    }
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < Hq; ++h) {
            const int kvh = h / G;
            rope_row(q1 + ((size_t)b * Hq + h) * d, qr, d, theta, (long)(Tk - 1) + pos_offset, 0);
            double mx = -INFINITY;
            for (int s = 0; s < Tk; ++s) {
                rope_row(k + IDX(b, s, kvh, 0, Tk, Hkv, d), kr, d, theta, (long)s + pos_offset, 0);
                double acc = 0.0;
                for (int c = 0; c < d; ++c)
                    acc += qr[c] * kr[c];
                S[s] = acc * scale;
                if (S[s] > mx)
                    mx = S[s];
            }
            double sum = 0.0;
            for (int s = 0; s < Tk; ++s)
                sum += exp(S[s] - mx);
            const double lse_bh = mx + log(sum);
            lse1[(size_t)b * Hq + h] = lse_bh;
            double *orow = o1 + ((size_t)b * Hq + h) * d;
            for (int c = 0; c < d; ++c)
                orow[c] = 0.0;
            for (int s = 0; s < Tk; ++s) {
                double pr = exp(S[s] - lse_bh);
                const double *vrow = v + IDX(b, s, kvh, 0, Tk, Hkv, d);
                for (int c = 0; c < d; ++c)
                    orow[c] += pr * vrow[c];
            }
        }
    free(qr);
    free(kr);
    free(S);
    return 0;
}

int ne_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
