/*
 * TEST INFRASTRUCTURE -- NOT PART OF THE PRODUCT PATH.
 *
 * Plain, slow, float64 CPU oracle for the parallel Newton forward of a
 * diagonal-mix GRU.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load this code.  It shares nothing with
 * the CUDA library: no headers, no helpers, no constants.
 *
 * Sources (pararnn-torch pages):
 *   - FAQs, "Does parallel Newton match sequential unroll?" and the numerics
 *     contract page, "Invariant" and "Two thresholds": the sequential unroll
 *     (sequential_apply) is the definition of the result; Newton+scan must
 *     match it within tau = 1e-4 in float32; the residual gate is max|F(H)|.
 *   - shapes_layout page, "cu_seqlens" paragraph: a ragged pack is one row of
 *     length N split by cu_seqlens (length S+1); segment heads use J = 0 on
 *     the scan.
 *   - Cell of ParaGRU(mix='diag') (equations as stated for the diag-GRU
 *     benches): z = sig(P_z + a_z h + b_z), r = sig(P_r + a_r h + b_r),
 *     c = tanh(P_c + a_c (r h) + b_c), f = (1 - z) h + z c, where P = W_x x
 *     is the input projection (gate blocks [z | r | c] along the last axis).
 *
 * Readings where the pages are silent:
 *   - each segment of a pack is an independent sequence from h = 0, so the
 *     shifted state at a head is 0 as well as J = 0;
 *   - the residual is F evaluated at the returned iterate H^(K);
 *   - a NaN residual counts as +infinity.
 *
 * Layouts (all row-major, float64): P (B, T, 3 d_h); H (B, T, d_h); params
 * (6, d_h) in the order a_z, a_r, a_c, b_z, b_r, b_c.  cu_seqlens (S + 1
 * int64) is given only for a pack, where B must be 1.  Every function works on
 * the unit range [j0, j1) so that callers may split units across threads.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* One cell step f(h, P_t) and its derivative df/dh (chain rule on the cell). */
void oracle_cell(double h, double pz, double pr, double pc, const double prm[6],
                 double *f_out, double *J_out)
{
    const double a_z = prm[0], a_r = prm[1], a_c = prm[2];
    const double b_z = prm[3], b_r = prm[4], b_c = prm[5];
    const double z = sigmoid(pz + a_z * h + b_z);
    const double r = sigmoid(pr + a_r * h + b_r);
    const double q = r * h;
    const double c = tanh(pc + a_c * q + b_c);
    const double f = (1.0 - z) * h + z * c;
    if (f_out) *f_out = f;
    if (J_out) {
        const double dz = z * (1.0 - z) * a_z;        /* dz/dh */
        const double dr = r * (1.0 - r) * a_r;        /* dr/dh */
        const double dq = r + h * dr;                 /* d(r h)/dh */
        const double dc = (1.0 - c * c) * a_c * dq;   /* dc/dh */
        *J_out = (1.0 - z) + dz * (c - h) + z * dc;
    }
}

static void unit_params(const double *params, int64_t d_h, int64_t j, double prm[6])
{
    for (int g = 0; g < 6; ++g) prm[g] = params[g * d_h + j];
}

/* Segment boundaries of row b: a rectangular batch has one segment [0, T). */
static int64_t n_segments(const int64_t *cu, int64_t S) { return cu ? S : 1; }
static void segment(const int64_t *cu, int64_t T, int64_t i, int64_t *s0, int64_t *s1)
{
    if (cu) { *s0 = cu[i]; *s1 = cu[i + 1]; }
    else { *s0 = 0; *s1 = T; }
}

/*
 * Sequential unroll h_t = f(h_{t-1}, P_t), h = 0 before the first step of each
 * segment.  Writes H[b, t, j] for j in [j0, j1).
 */
void oracle_sequential(const double *P, const double *params, int64_t B, int64_t T,
                       int64_t d_h, const int64_t *cu, int64_t S, int64_t j0, int64_t j1,
                       double *H)
{
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t j = j0; j < j1; ++j) {
            double prm[6];
            unit_params(params, d_h, j, prm);
            for (int64_t i = 0; i < n_segments(cu, S); ++i) {
                int64_t s0, s1;
                segment(cu, T, i, &s0, &s1);
                double h = 0.0;
                for (int64_t t = s0; t < s1; ++t) {
                    const double *p = P + (b * T + t) * 3 * d_h;
                    oracle_cell(h, p[j], p[d_h + j], p[2 * d_h + j], prm, &h, NULL);
                    H[(b * T + t) * d_h + j] = h;
                }
            }
        }
    }
}

/* Marks t as a segment head: t = 0, or t = cu[i] with cu[i] < cu[i+1]. */
static void head_mask(const int64_t *cu, int64_t S, int64_t T, unsigned char *head)
{
    for (int64_t t = 0; t < T; ++t) head[t] = 0;
    if (T > 0) head[0] = 1;
    if (cu)
        for (int64_t i = 0; i < S; ++i)
            if (cu[i] < cu[i + 1]) head[cu[i]] = 1;
}

/* Residual of a trajectory G: F_t = G_t - f(G_{t-1}, P_t), G_{-1} = 0 at heads. */
static double residual_row(const double *P, const double prm[6], int64_t T, int64_t d_h,
                           int64_t j, const unsigned char *head, const double *G,
                           double *F, double *J)
{
    double rho = 0.0;
    for (int64_t t = 0; t < T; ++t) {
        const double *p = P + t * 3 * d_h;
        const double hs = head[t] ? 0.0 : G[t - 1];
        double f, dfdh;
        oracle_cell(hs, p[j], p[d_h + j], p[2 * d_h + j], prm, &f, &dfdh);
        const double Ft = G[t] - f;
        if (F) F[t] = Ft;
        if (J) J[t] = head[t] ? 0.0 : dfdh;
        const double a = fabs(Ft);
        if (isnan(a)) rho = INFINITY;
        else if (a > rho) rho = a;
    }
    return rho;
}

/*
 * Parallel-Newton algorithm, written sequentially:
 *   H^(0) = 0;  for k = 1..K:
 *     F_t = H_t - f(H_{t-1}, P_t),  J_t = df/dh at H_{t-1}   (J = 0, H_{-1} = 0 at heads)
 *     delta_t = J_t delta_{t-1} - F_t   (delta before the first step = 0)
 *     H <- H + delta
 *   rho = max |F(H^(K))|.
 * Writes H[b, t, j] for j in [j0, j1) and returns rho over those units.
 */
double oracle_newton(const double *P, const double *params, int64_t B, int64_t T,
                     int64_t d_h, const int64_t *cu, int64_t S, int64_t K,
                     int64_t j0, int64_t j1, double *H)
{
    unsigned char *head = (unsigned char *)malloc((size_t)(T > 0 ? T : 1));
    double *G = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    double *F = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    double *J = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    head_mask(cu, S, T, head);
    double rho = 0.0;
    for (int64_t b = 0; b < B; ++b) {
        const double *Pb = P + b * T * 3 * d_h;
        for (int64_t j = j0; j < j1; ++j) {
            double prm[6];
            unit_params(params, d_h, j, prm);
            for (int64_t t = 0; t < T; ++t) G[t] = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                residual_row(Pb, prm, T, d_h, j, head, G, F, J);
                double delta = 0.0;
                for (int64_t t = 0; t < T; ++t) {
                    delta = J[t] * delta - F[t];
                    G[t] += delta;
                }
            }
            const double r = residual_row(Pb, prm, T, d_h, j, head, G, NULL, NULL);
            if (!(r <= rho)) rho = r;   /* also takes +inf */
            for (int64_t t = 0; t < T; ++t) H[(b * T + t) * d_h + j] = G[t];
        }
    }
    free(head); free(G); free(F); free(J);
    return rho;
}

/* max |F(G)| over b, t and j in [j0, j1) for a given trajectory G (B, T, d_h). */
double oracle_residual(const double *P, const double *params, int64_t B, int64_t T,
                       int64_t d_h, const int64_t *cu, int64_t S, int64_t j0, int64_t j1,
                       const double *Gfull)
{
    unsigned char *head = (unsigned char *)malloc((size_t)(T > 0 ? T : 1));
    double *G = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    head_mask(cu, S, T, head);
    double rho = 0.0;
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t j = j0; j < j1; ++j) {
            double prm[6];
            unit_params(params, d_h, j, prm);
            for (int64_t t = 0; t < T; ++t) G[t] = Gfull[(b * T + t) * d_h + j];
            const double r = residual_row(P + b * T * 3 * d_h, prm, T, d_h, j, head, G,
                                          NULL, NULL);
            if (!(r <= rho)) rho = r;
        }
    }
    free(head); free(G);
    return rho;
}

/*
 * Picard (fixed-point) sweeps, the plainest reading of the FAQ's Picard warm
 * start ("How many Newton iterations should I use?": "try Picard warm-start
 * (picard_iters)"): starting from G = 0, each sweep sets G_t = f(G_{t-1}, P_t)
 * for every t at once from the previous sweep (shifted state 0 at heads).
 * Writes G[b, t, j] for j in [j0, j1).
 */
void oracle_picard(const double *P, const double *params, int64_t B, int64_t T, int64_t d_h,
                   const int64_t *cu, int64_t S, int64_t sweeps, int64_t j0, int64_t j1,
                   double *Gout)
{
    unsigned char *head = (unsigned char *)malloc((size_t)(T > 0 ? T : 1));
    double *G = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    double *Gn = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    head_mask(cu, S, T, head);
    for (int64_t b = 0; b < B; ++b) {
        const double *Pb = P + b * T * 3 * d_h;
        for (int64_t j = j0; j < j1; ++j) {
            double prm[6];
            unit_params(params, d_h, j, prm);
            for (int64_t t = 0; t < T; ++t) G[t] = 0.0;
            for (int64_t s = 0; s < sweeps; ++s) {
                for (int64_t t = 0; t < T; ++t) {
                    const double *p = Pb + t * 3 * d_h;
                    const double hs = head[t] ? 0.0 : G[t - 1];
                    oracle_cell(hs, p[j], p[d_h + j], p[2 * d_h + j], prm, &Gn[t], NULL);
                }
                for (int64_t t = 0; t < T; ++t) G[t] = Gn[t];
            }
            for (int64_t t = 0; t < T; ++t) Gout[(b * T + t) * d_h + j] = G[t];
        }
    }
    free(head); free(G); free(Gn);
}

/*
 * The parallel-Newton algorithm of oracle_newton started from a given iterate
 * H^(0) = H0 (B, T, d_h) instead of 0 (a warm start).  H and H0 may alias.
 */
double oracle_newton_init(const double *P, const double *params, int64_t B, int64_t T,
                          int64_t d_h, const int64_t *cu, int64_t S, int64_t K,
                          const double *H0, int64_t j0, int64_t j1, double *H)
{
    unsigned char *head = (unsigned char *)malloc((size_t)(T > 0 ? T : 1));
    double *G = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    double *F = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    double *J = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    head_mask(cu, S, T, head);
    double rho = 0.0;
    for (int64_t b = 0; b < B; ++b) {
        const double *Pb = P + b * T * 3 * d_h;
        for (int64_t j = j0; j < j1; ++j) {
            double prm[6];
            unit_params(params, d_h, j, prm);
            for (int64_t t = 0; t < T; ++t) G[t] = H0[(b * T + t) * d_h + j];
            for (int64_t k = 0; k < K; ++k) {
                residual_row(Pb, prm, T, d_h, j, head, G, F, J);
                double delta = 0.0;
                for (int64_t t = 0; t < T; ++t) {
                    delta = J[t] * delta - F[t];
                    G[t] += delta;
                }
            }
            const double r = residual_row(Pb, prm, T, d_h, j, head, G, NULL, NULL);
            if (!(r <= rho)) rho = r;
            for (int64_t t = 0; t < T; ++t) H[(b * T + t) * d_h + j] = G[t];
        }
    }
    free(head); free(G); free(F); free(J);
    return rho;
}

/*
 * Backward (adjoint) pass through the recurrence h_t = f(h_{t-1}, P_t), the
 * plainest reading of the pages' "train forward+backward surface" (shapes_layout
 * page): given the trajectory H and dL/dH, the total derivative
 *   lambda_t = dL/dh_t = dL/dH_t + J_{t+1} lambda_{t+1}   (lambda after the end = 0,
 *   J = 0 at segment heads, so nothing flows across a segment boundary)
 * gives dL/dP_{t,g} = lambda_t df/dP_g and dL/da_g, dL/db_g summed over (b, t).
 * Derivatives at (h~ = H_{t-1}, P_t):
 *   df/dP_z = z (1 - z) (c - h~),  df/dP_c = z (1 - c^2),
 *   df/dP_r = z (1 - c^2) a_c h~ r (1 - r);  df/db_g = df/dP_g;
 *   df/da_z = df/dP_z h~,  df/da_r = df/dP_r h~,  df/da_c = df/dP_c r h~.
 * Writes gP (B, T, 3 d_h) and adds into gprm (6, d_h) for units [j0, j1).
 */
void oracle_backward(const double *P, const double *params, int64_t B, int64_t T, int64_t d_h,
                     const int64_t *cu, int64_t S, const double *H, const double *gH,
                     int64_t j0, int64_t j1, double *gP, double *gprm)
{
    unsigned char *head = (unsigned char *)malloc((size_t)(T > 0 ? T : 1));
    head_mask(cu, S, T, head);
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t j = j0; j < j1; ++j) {
            double prm[6];
            unit_params(params, d_h, j, prm);
            double carry = 0.0;   /* J_{t+1} lambda_{t+1} */
            for (int64_t t = T - 1; t >= 0; --t) {
                const double *p = P + (b * T + t) * 3 * d_h;
                const double hs = head[t] ? 0.0 : H[(b * T + t - 1) * d_h + j];
                const double z = sigmoid(p[j] + prm[0] * hs + prm[3]);
                const double r = sigmoid(p[d_h + j] + prm[1] * hs + prm[4]);
                const double c = tanh(p[2 * d_h + j] + prm[2] * r * hs + prm[5]);
                const double lambda = gH[(b * T + t) * d_h + j] + carry;
                const double dPz = z * (1.0 - z) * (c - hs);
                const double dPc = z * (1.0 - c * c);
                const double dPr = dPc * prm[2] * hs * r * (1.0 - r);
                double *g = gP + (b * T + t) * 3 * d_h;
                g[j] = lambda * dPz;
                g[d_h + j] = lambda * dPr;
                g[2 * d_h + j] = lambda * dPc;
                gprm[0 * d_h + j] += lambda * dPz * hs;
                gprm[1 * d_h + j] += lambda * dPr * hs;
                gprm[2 * d_h + j] += lambda * dPc * r * hs;
                gprm[3 * d_h + j] += lambda * dPz;
                gprm[4 * d_h + j] += lambda * dPr;
                gprm[5 * d_h + j] += lambda * dPc;
                double J = 0.0;
                if (!head[t]) oracle_cell(hs, p[j], p[d_h + j], p[2 * d_h + j], prm, NULL, &J);
                carry = J * lambda;
            }
        }
    }
    free(head);
}
