/*
 * gs_oracle.c -- plain, slow CPU oracle for the forward rendering path of
 * 3D Gaussian Splatting.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library. It shares no code, header, table or
 * constant with the CUDA path; the two meet only in the seeded scene inputs.
 *
 * Source of the method: the lesson page "3D Gaussian Splatting à partir de
 * zéro" (and its Persian twin), sections
 *   "Ce qu'un Gaussien porte"        per-Gaussian parameters and activations,
 *                                    Sigma = R S S^T R^T
 *   "Rastérisation, non rayée"       project -> 16x16 tiles -> per-tile depth
 *                                    sort -> front-to-back composite
 *   "L'étape de projection"          mu' = project(mu), Sigma' = J W Sigma W^T J^T,
 *                                    weight exp(-0.5 (p-mu')^T Sigma'^-1 (p-mu'))
 *   "La règle de composition alpha"  C = sum alpha_i T_i c_i, T_i = prod (1-alpha_j)
 *   "Étape 2" (rasterise_2d)         integer pixel grid, alpha clamp at 0.99,
 *                                    depth-ordered front-to-back loop
 *   "Étape 5: De la 2D à la 3D"      quaternion rotation, camera-space depth
 *   "Étape 6" (eval_sh_degree_3)     SH basis and constants for bands 0..2
 *
 * Two arithmetic tracks:
 *   - the fp64 track (or_project_f64, or_composite*) follows the formulas in
 *     the pages' order and notation;
 *   - the fp32 decision program (or_decide_f32) fixes the integer results --
 *     culling, depth key bits, pixel and tile rectangles -- as an IEEE binary32
 *     program with a fixed operation order and no fused multiply-add. The pages'
 *     own code works in float32, so that is the precision the decisions are
 *     taken in. Build with -ffp-contract=off and without fast-math.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    float R[9];      /* world -> camera rotation, row-major */
    float t[3];      /* x_cam = R x_world + t */
    float fx, fy, cx, cy, near_z;
    int32_t width, height;
    float bg[3];
} or_camera;

enum { OR_EV_SKIP = 1, OR_EV_STOP = 2 };

/* thresholds of the compositing rule (section "Étape 2": clamp at 0.99;
 * the skip below 1/255 and the stop below 1e-4 are the tile renderer's cut-offs) */
static const double OR_ALPHA_MAX = 0.99;
static const double OR_ALPHA_MIN = 1.0 / 255.0;
static const double OR_T_MIN = 1e-4;

int or_version(void) { return 3; }

void or_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int or_get_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------- */
/* small fp64 matrix helpers (row-major, plain loops)                         */
/* ------------------------------------------------------------------------- */

static void mat_mul(const double *A, const double *B, double *C, int n, int k, int m) {
    /* C[n][m] = A[n][k] * B[k][m] */
    for (int i = 0; i < n; i++)
        for (int j = 0; j < m; j++) {
            double s = 0.0;
            for (int l = 0; l < k; l++) s += A[i * k + l] * B[l * m + j];
            C[i * m + j] = s;
        }
}

static void mat_T(const double *A, double *AT, int n, int m) {
    /* AT[m][n] = A[n][m]^T */
    for (int i = 0; i < n; i++)
        for (int j = 0; j < m; j++) AT[j * n + i] = A[i * m + j];
}

/* Textbook rotation matrix of a unit quaternion (w, x, y, z). */
static void quat_to_rot(double w, double x, double y, double z, double *G) {
    G[0] = 1 - 2 * (y * y + z * z); G[1] = 2 * (x * y - w * z);     G[2] = 2 * (x * z + w * y);
    G[3] = 2 * (x * y + w * z);     G[4] = 1 - 2 * (x * x + z * z); G[5] = 2 * (y * z - w * x);
    G[6] = 2 * (x * z - w * y);     G[7] = 2 * (y * z + w * x);     G[8] = 1 - 2 * (x * x + y * y);
}

/* Sigma = R S S^T R^T with R = rot(q) for a unit quaternion and
 * S = diag(exp(log_scale)) (section "Ce qu'un Gaussien porte"). */
static void covariance3d(double w, double x, double y, double z, const float *log_scale,
                         double *G, double *Sigma) {
    double S[9] = {0}, ST[9], GS[9], GSST[9], GT[9];
    quat_to_rot(w, x, y, z, G);
    for (int i = 0; i < 3; i++) S[i * 4] = exp((double)log_scale[i]);
    mat_T(S, ST, 3, 3);
    mat_T(G, GT, 3, 3);
    mat_mul(G, S, GS, 3, 3, 3);
    mat_mul(GS, ST, GSST, 3, 3, 3);
    mat_mul(GSST, GT, Sigma, 3, 3, 3);
}

/* Exported for the closed-form tests: R and Sigma per Gaussian (q normalised
 * first; rows of zeros for a zero quaternion). */
void or_covariance3d(int64_t n, const float *quats, const float *log_scales, double *R, double *Sigma) {
    for (int64_t g = 0; g < n; g++) {
        double qw = quats[4 * g], qx = quats[4 * g + 1], qy = quats[4 * g + 2], qz = quats[4 * g + 3];
        double qn = sqrt(qw * qw + qx * qx + qy * qy + qz * qz);
        if (!(qn > 0.0)) { for (int i = 0; i < 9; i++) R[9 * g + i] = Sigma[9 * g + i] = 0.0; continue; }
        covariance3d(qw / qn, qx / qn, qy / qn, qz / qn, log_scales + 3 * g, R + 9 * g, Sigma + 9 * g);
    }
}

/* ------------------------------------------------------------------------- */
/* spherical harmonics (section "Étape 6")                                    */
/* ------------------------------------------------------------------------- */

/* Real SH basis at unit direction (x, y, z), in the pages' sign convention.
 * Bands 0..2 are the printed ones: band 1 is -C1 y, +C1 z, -C1 x; band 2 is
 * +C2 xy, +C2 yz, +C2' (2z^2-x^2-y^2), +C2 xz, +C2'' (x^2-y^2).
 * Band 3 is left out of the printed code; it is taken here from the closed
 * forms of the real harmonics with the band-1 pattern (odd m negative). The
 * normalisation constants are computed from their closed forms, not typed in.
 * Parity unpinned for band 3's signs: the pages print no band-3 code, so only
 * its orthonormality, harmonicity and parity Y(-d) = (-1)^l Y(d) are pinned; its
 * sign convention is a reading. */
void or_sh_basis(double x, double y, double z, double *Y /* [16] */) {
    const double pi = 3.14159265358979323846;
    const double c0 = sqrt(1.0 / (4.0 * pi));
    const double c1 = sqrt(3.0 / (4.0 * pi));
    const double c2a = sqrt(15.0 / (4.0 * pi));   /* xy, yz, xz */
    const double c2b = sqrt(5.0 / (16.0 * pi));   /* 2z^2 - x^2 - y^2 */
    const double c2c = sqrt(15.0 / (16.0 * pi));  /* x^2 - y^2 */
    const double c3a = sqrt(35.0 / (32.0 * pi));  /* m = +-3 */
    const double c3b = sqrt(105.0 / (4.0 * pi));  /* m = -2: xyz */
    const double c3c = sqrt(21.0 / (32.0 * pi));  /* m = +-1 */
    const double c3d = sqrt(7.0 / (16.0 * pi));   /* m = 0 */
    const double c3e = sqrt(105.0 / (16.0 * pi)); /* m = +2 */
    const double xx = x * x, yy = y * y, zz = z * z;
    Y[0] = c0;
    Y[1] = -c1 * y;
    Y[2] = c1 * z;
    Y[3] = -c1 * x;
    Y[4] = c2a * x * y;
    Y[5] = c2a * y * z;
    Y[6] = c2b * (2.0 * zz - xx - yy);
    Y[7] = c2a * x * z;
    Y[8] = c2c * (xx - yy);
    Y[9] = -c3a * y * (3.0 * xx - yy);
    Y[10] = c3b * x * y * z;
    Y[11] = -c3c * y * (4.0 * zz - xx - yy);
    Y[12] = c3d * z * (2.0 * zz - 3.0 * xx - 3.0 * yy);
    Y[13] = -c3c * x * (4.0 * zz - xx - yy);
    Y[14] = c3e * z * (xx - yy);
    Y[15] = -c3a * x * (xx - 3.0 * yy);
}

/* colour = sum_k Y_k(dir) c_k (per channel) + 0.5, clamped at 0. */
static void eval_sh(const float *coeffs /* [(D+1)^2][3] */, int degree, const double *dir, double *rgb) {
    double Y[16];
    or_sh_basis(dir[0], dir[1], dir[2], Y);
    int nk = (degree + 1) * (degree + 1);
    for (int c = 0; c < 3; c++) {
        double s = 0.0;
        for (int k = 0; k < nk; k++) s += Y[k] * (double)coeffs[k * 3 + c];
        s += 0.5;
        rgb[c] = s > 0.0 ? s : 0.0;
    }
}

void or_eval_sh(int64_t n, const float *sh, int degree, const double *dirs, double *rgb) {
    int nk = (degree + 1) * (degree + 1);
    for (int64_t i = 0; i < n; i++) eval_sh(sh + i * nk * 3, degree, dirs + 3 * i, rgb + 3 * i);
}

/* ------------------------------------------------------------------------- */
/* fp64 projection track                                                     */
/* ------------------------------------------------------------------------- */

/* Per Gaussian, in fp64:
 *   q^ = q/|q|, R = rot(q^), S = diag(exp(s)), Sigma = R S S^T R^T
 *   x_c = W mu + t (W the camera rotation), depth = z_c, culled if z_c <= near
 *   mu' = (fx x/z + cx, fy y/z + cy)
 *   J = [[fx/z, 0, -fx x/z^2], [0, fy/z, -fy y/z^2]]
 *   Sigma' = J W Sigma W^T J^T  (2x2: a b; b c), culled if det <= 0
 *   conic = Sigma'^-1 = (c, -b, a)/det, lam_max, radius = ceil(3 sqrt(lam_max))
 *   opacity = sigmoid(logit); colour = SH(normalize(mu - camera centre)) + 0.5, >= 0
 * valid[i] = 0 for culled Gaussians (their other outputs are zero). */
void or_project_f64(int64_t n, const float *means, const float *quats, const float *log_scales,
                    const float *logits, const float *sh, int sh_degree, const or_camera *cam,
                    double *mean2d, double *conic, double *opacity, double *rgb, double *depth,
                    double *cov2d, double *lam_max, uint8_t *valid) {
    double Wm[9], WT[9], t[3], C[3];
    for (int i = 0; i < 9; i++) Wm[i] = cam->R[i];
    for (int i = 0; i < 3; i++) t[i] = cam->t[i];
    mat_T(Wm, WT, 3, 3);
    /* camera centre C = -W^T t */
    for (int i = 0; i < 3; i++) C[i] = -(WT[i * 3 + 0] * t[0] + WT[i * 3 + 1] * t[1] + WT[i * 3 + 2] * t[2]);
    const double fx = cam->fx, fy = cam->fy, cx = cam->cx, cy = cam->cy, nearz = cam->near_z;
    const int nk = (sh_degree + 1) * (sh_degree + 1);

#pragma omp parallel for schedule(static)
    for (int64_t g = 0; g < n; g++) {
        double mu[3] = {means[3 * g], means[3 * g + 1], means[3 * g + 2]};
        double xc[3];
        for (int i = 0; i < 3; i++) xc[i] = Wm[i * 3] * mu[0] + Wm[i * 3 + 1] * mu[1] + Wm[i * 3 + 2] * mu[2] + t[i];
        valid[g] = 0;
        mean2d[2 * g] = mean2d[2 * g + 1] = 0.0;
        conic[3 * g] = conic[3 * g + 1] = conic[3 * g + 2] = 0.0;
        cov2d[3 * g] = cov2d[3 * g + 1] = cov2d[3 * g + 2] = 0.0;
        rgb[3 * g] = rgb[3 * g + 1] = rgb[3 * g + 2] = 0.0;
        opacity[g] = 0.0;
        depth[g] = xc[2];
        lam_max[g] = 0.0;
        if (!(xc[2] > nearz)) continue;

        double qw = quats[4 * g], qx = quats[4 * g + 1], qy = quats[4 * g + 2], qz = quats[4 * g + 3];
        double qn = sqrt(qw * qw + qx * qx + qy * qy + qz * qz);
        if (!(qn > 0.0) || !isfinite(qn)) continue;
        double G[9], Sigma[9];
        covariance3d(qw / qn, qx / qn, qy / qn, qz / qn, log_scales + 3 * g, G, Sigma);

        const double z = xc[2];
        double J[6] = {fx / z, 0.0, -fx * xc[0] / (z * z),
                       0.0, fy / z, -fy * xc[1] / (z * z)};
        double JT[6], JW[6], JWS[6], WTJT[6], S2[4];
        mat_T(J, JT, 2, 3);
        mat_mul(J, Wm, JW, 2, 3, 3);         /* J W */
        mat_mul(JW, Sigma, JWS, 2, 3, 3);    /* J W Sigma */
        mat_mul(WT, JT, WTJT, 3, 3, 2);      /* W^T J^T */
        mat_mul(JWS, WTJT, S2, 2, 3, 2);     /* J W Sigma W^T J^T */
        double a = S2[0], b = 0.5 * (S2[1] + S2[2]), c = S2[3];
        double det = a * c - b * b;
        if (!(det > 0.0) || !isfinite(det)) continue;

        valid[g] = 1;
        mean2d[2 * g] = fx * xc[0] / z + cx;
        mean2d[2 * g + 1] = fy * xc[1] / z + cy;
        cov2d[3 * g] = a; cov2d[3 * g + 1] = b; cov2d[3 * g + 2] = c;
        conic[3 * g] = c / det;
        conic[3 * g + 1] = -b / det;
        conic[3 * g + 2] = a / det;
        double h = 0.5 * (a - c);
        lam_max[g] = 0.5 * (a + c) + sqrt(h * h + b * b);
        opacity[g] = 1.0 / (1.0 + exp(-(double)logits[g]));

        double d[3] = {mu[0] - C[0], mu[1] - C[1], mu[2] - C[2]};
        double dn = sqrt(d[0] * d[0] + d[1] * d[1] + d[2] * d[2]);
        d[0] /= dn; d[1] /= dn; d[2] /= dn;
        eval_sh(sh + g * nk * 3, sh_degree, d, rgb + 3 * g);
    }
}

/* ------------------------------------------------------------------------- */
/* fp32 decision program                                                      */
/* ------------------------------------------------------------------------- */

/* Scale activation of the decision program, scale = e^l ("Ce qu'un Gaussien
 * porte": log-scales exponentiated at render time), evaluated in binary32 by
 * Cody and Waite's range reduction (Software Manual for the Elementary
 * Functions, 1980): l = k ln2 + r with ln2 split into a 12-bit head (exact
 * products k*head) and a rounded tail, then e^r by its Taylor polynomial of
 * degree 7 (|r| <= ln2/2, truncation below 6e-9 relative) in Horner form,
 * then the exact scaling by 2^k. Every operation is rounded on its own; l is
 * clamped to [-80, 80] so that 2^k and the result stay normal numbers.
 * The constants are ln 2 and 1/j!, rounded to binary32. */
float or_exp32(float x) {
    if (x != x) return x;
    if (x > 80.0f) x = 80.0f;
    if (x < -80.0f) x = -80.0f;
    const float ln2_hi = 2839.0f / 4096.0f;
    const float ln2_lo = (float)(log(2.0) - 2839.0 / 4096.0);
    const float inv_ln2 = (float)(1.0 / log(2.0));
    float c[8];
    double f = 1.0;
    for (int j = 0; j < 8; j++) {
        if (j > 0) f *= j;
        c[j] = (float)(1.0 / f);
    }
    const float k = rintf(x * inv_ln2);
    const float r = (x - k * ln2_hi) - k * ln2_lo;
    float p = c[7];
    for (int j = 6; j >= 0; j--) p = c[j] + r * p;
    return ldexpf(p, (int)k);
}

void or_exp32_batch(int64_t n, const float *x, float *y) {
    for (int64_t i = 0; i < n; i++) y[i] = or_exp32(x[i]);
}

/* The decision program, step by step (binary32, each operation rounded to
 * nearest-even, no fused multiply-add, sums left to right as bracketed):
 *  D1  p_i = ((R_i0 m0 + R_i1 m1) + R_i2 m2) + t_i; depth = p_2
 *  D2  culled unless p_2 > near
 *  D3  n2 = ((qw^2 + qx^2) + qy^2) + qz^2, culled unless 0 < n2 <= FLT_MAX;
 *      r = sqrt(n2); (w,x,y,z) = q / r
 *  D4  G = textbook rotation of (w,x,y,z): e.g. G00 = 1 - 2 (yy + zz),
 *      G01 = 2 (xy - wz), each product rounded first
 *  D5  s_k = exp32(l_k)   (or_exp32: binary32 Cody-Waite + Taylor, above)
 *  D6  A_ij = (R_i0 G_0j + R_i1 G_1j) + R_i2 G_2j;  B_ij = A_ij s_j
 *  D7  j00 = fx/z, j11 = fy/z, zz = z z, j02 = -((fx p0)/zz), j12 = -((fy p1)/zz)
 *  D8  M_0k = j00 B_0k + j02 B_2k;  M_1k = j11 B_1k + j12 B_2k
 *  D9  a = (M00 M00 + M01 M01) + M02 M02; b = (M00 M10 + M01 M11) + M02 M12;
 *      c = (M10 M10 + M11 M11) + M12 M12          (Sigma' = M M^T)
 *  D10 det = a c - b b; culled unless 0 < det <= FLT_MAX
 *  D11 hm = 0.5 (a - c); mid = 0.5 (a + c); lam = mid + sqrt(hm hm + b b);
 *      rf = ceil(3 sqrt(lam))
 *  D12 u = (fx p0)/z + cx; v = (fy p1)/z + cy; culled unless u, v, rf finite
 *  D13 x0 = max(ceil(u - rf), 0), x1 = min(floor(u + rf), W - 1), same for y;
 *      no tiles unless x0 <= x1 and y0 <= y1
 *  D14 tiles [x0>>4 .. x1>>4] x [y0>>4 .. y1>>4]
 * Sigma' = M M^T with M = J W R S is the pages' J W Sigma W^T J^T with
 * Sigma = (R S)(R S)^T, re-associated.
 * Outputs per Gaussian: valid, depth, mean2d, cov2d (a, b, c), radius,
 * pixel rect, tile rect, tiles_touched. */
void or_decide_f32(int64_t n, const float *means, const float *quats, const float *log_scales,
                   const or_camera *cam, uint8_t *valid, float *depth, float *mean2d, float *cov2d,
                   int32_t *radius, int32_t *pix_rect /* [n][4] x0 y0 x1 y1 */,
                   int32_t *tile_rect /* [n][4] tx0 ty0 tx1 ty1 */, uint32_t *tiles_touched) {
    const float *R = cam->R, *t = cam->t;
    const float fx = cam->fx, fy = cam->fy, cx = cam->cx, cy = cam->cy, nearz = cam->near_z;
    const float Wm1 = (float)(cam->width - 1), Hm1 = (float)(cam->height - 1);

#pragma omp parallel for schedule(static)
    for (int64_t g = 0; g < n; g++) {
        const float m0 = means[3 * g], m1 = means[3 * g + 1], m2 = means[3 * g + 2];
        float p[3];
        for (int i = 0; i < 3; i++) {
            float s = R[3 * i] * m0;
            s = s + R[3 * i + 1] * m1;
            s = s + R[3 * i + 2] * m2;
            p[i] = s + t[i];
        }
        valid[g] = 0;
        depth[g] = p[2];
        mean2d[2 * g] = mean2d[2 * g + 1] = 0.0f;
        cov2d[3 * g] = cov2d[3 * g + 1] = cov2d[3 * g + 2] = 0.0f;
        radius[g] = 0;
        /* an empty rectangle is stored as (0, 0, -1, -1) */
        for (int k = 0; k < 4; k++) pix_rect[4 * g + k] = tile_rect[4 * g + k] = k < 2 ? 0 : -1;
        tiles_touched[g] = 0;
        const float z = p[2];
        if (!(z > nearz)) continue;                                  /* D2 */

        const float qw = quats[4 * g], qx = quats[4 * g + 1], qy = quats[4 * g + 2], qz = quats[4 * g + 3];
        float n2 = qw * qw;
        n2 = n2 + qx * qx;
        n2 = n2 + qy * qy;
        n2 = n2 + qz * qz;
        if (!(n2 > 0.0f && n2 <= FLT_MAX)) continue;                 /* D3 */
        const float r = sqrtf(n2);
        const float w = qw / r, x = qx / r, y = qy / r, zq = qz / r;

        float G[9];                                                  /* D4 */
        {
            const float xx = x * x, yy = y * y, zz = zq * zq;
            const float xy = x * y, xz = x * zq, yz = y * zq;
            const float wx = w * x, wy = w * y, wz = w * zq;
            G[0] = 1.0f - 2.0f * (yy + zz); G[1] = 2.0f * (xy - wz);        G[2] = 2.0f * (xz + wy);
            G[3] = 2.0f * (xy + wz);        G[4] = 1.0f - 2.0f * (xx + zz); G[5] = 2.0f * (yz - wx);
            G[6] = 2.0f * (xz - wy);        G[7] = 2.0f * (yz + wx);        G[8] = 1.0f - 2.0f * (xx + yy);
        }
        float s[3];                                                  /* D5 */
        for (int k = 0; k < 3; k++) s[k] = or_exp32(log_scales[3 * g + k]);
        float B[9];                                                  /* D6 */
        for (int i = 0; i < 3; i++)
            for (int j = 0; j < 3; j++) {
                float a_ij = R[3 * i] * G[j];
                a_ij = a_ij + R[3 * i + 1] * G[3 + j];
                a_ij = a_ij + R[3 * i + 2] * G[6 + j];
                B[3 * i + j] = a_ij * s[j];
            }
        const float j00 = fx / z, j11 = fy / z;                      /* D7 */
        const float zz2 = z * z;
        const float j02 = -((fx * p[0]) / zz2);
        const float j12 = -((fy * p[1]) / zz2);
        float M0[3], M1[3];                                          /* D8 */
        for (int k = 0; k < 3; k++) {
            M0[k] = j00 * B[k] + j02 * B[6 + k];
            M1[k] = j11 * B[3 + k] + j12 * B[6 + k];
        }
        float a = M0[0] * M0[0];                                     /* D9 */
        a = a + M0[1] * M0[1];
        a = a + M0[2] * M0[2];
        float b = M0[0] * M1[0];
        b = b + M0[1] * M1[1];
        b = b + M0[2] * M1[2];
        float c = M1[0] * M1[0];
        c = c + M1[1] * M1[1];
        c = c + M1[2] * M1[2];
        const float det = a * c - b * b;                             /* D10 */
        if (!(det > 0.0f && det <= FLT_MAX)) continue;
        const float hm = 0.5f * (a - c);                             /* D11 */
        const float mid = 0.5f * (a + c);
        const float lam = mid + sqrtf(hm * hm + b * b);
        const float rf = ceilf(3.0f * sqrtf(lam));
        const float u = (fx * p[0]) / z + cx;                        /* D12 */
        const float v = (fy * p[1]) / z + cy;
        if (!(fabsf(u) <= FLT_MAX && fabsf(v) <= FLT_MAX && rf <= FLT_MAX)) continue;

        valid[g] = 1;
        mean2d[2 * g] = u;
        mean2d[2 * g + 1] = v;
        cov2d[3 * g] = a; cov2d[3 * g + 1] = b; cov2d[3 * g + 2] = c;
        radius[g] = rf <= 1073741824.0f ? (int32_t)rf : 1073741824;

        float x0 = ceilf(u - rf), x1 = floorf(u + rf);               /* D13 */
        float y0 = ceilf(v - rf), y1 = floorf(v + rf);
        x0 = x0 > 0.0f ? x0 : 0.0f;
        y0 = y0 > 0.0f ? y0 : 0.0f;
        x1 = x1 < Wm1 ? x1 : Wm1;
        y1 = y1 < Hm1 ? y1 : Hm1;
        if (!(x0 <= x1 && y0 <= y1)) continue;
        const int32_t ix0 = (int32_t)x0, ix1 = (int32_t)x1, iy0 = (int32_t)y0, iy1 = (int32_t)y1;
        pix_rect[4 * g] = ix0; pix_rect[4 * g + 1] = iy0; pix_rect[4 * g + 2] = ix1; pix_rect[4 * g + 3] = iy1;
        const int32_t tx0 = ix0 >> 4, tx1 = ix1 >> 4, ty0 = iy0 >> 4, ty1 = iy1 >> 4;  /* D14 */
        tile_rect[4 * g] = tx0; tile_rect[4 * g + 1] = ty0; tile_rect[4 * g + 2] = tx1; tile_rect[4 * g + 3] = ty1;
        tiles_touched[g] = (uint32_t)((tx1 - tx0 + 1) * (ty1 - ty0 + 1));
    }
}

/* The same rectangle decision taken in fp64 from the fp64 track's mean2d and
 * lam_max, for cross-checking the fp32 program (disagreements must sit on a
 * rounding boundary). */
void or_rect_f64(int64_t n, const double *mean2d, const double *lam_max, const uint8_t *valid,
                 int32_t width, int32_t height, int32_t *radius, int32_t *pix_rect) {
    for (int64_t g = 0; g < n; g++) {
        radius[g] = 0;
        for (int k = 0; k < 4; k++) pix_rect[4 * g + k] = k < 2 ? 0 : -1;
        if (!valid[g]) continue;
        double rf = ceil(3.0 * sqrt(lam_max[g]));
        radius[g] = rf <= 1073741824.0 ? (int32_t)rf : 1073741824;
        double u = mean2d[2 * g], v = mean2d[2 * g + 1];
        double x0 = fmax(ceil(u - rf), 0.0), x1 = fmin(floor(u + rf), width - 1.0);
        double y0 = fmax(ceil(v - rf), 0.0), y1 = fmin(floor(v + rf), height - 1.0);
        if (!(x0 <= x1 && y0 <= y1)) continue;
        pix_rect[4 * g] = (int32_t)x0; pix_rect[4 * g + 1] = (int32_t)y0;
        pix_rect[4 * g + 2] = (int32_t)x1; pix_rect[4 * g + 3] = (int32_t)y1;
    }
}

/* ------------------------------------------------------------------------- */
/* binning, sort, ranges                                                      */
/* ------------------------------------------------------------------------- */

/* Inclusive prefix sum of tiles_touched; returns the total key count K. */
uint64_t or_scan(int64_t n, const uint32_t *tiles_touched, uint64_t *offsets_inclusive) {
    uint64_t acc = 0;
    for (int64_t g = 0; g < n; g++) {
        acc += tiles_touched[g];
        offsets_inclusive[g] = acc;
    }
    return acc;
}

/* One key per (Gaussian, touched tile): Gaussians in index order, tiles of a
 * Gaussian in row-major order over its tile rectangle;
 * key = (ty * tiles_x + tx) << 32 | bits(depth), value = Gaussian index. */
void or_duplicate(int64_t n, const uint32_t *tiles_touched, const int32_t *tile_rect,
                  const float *depth, int32_t tiles_x, uint64_t *keys, uint32_t *vals) {
    uint64_t pos = 0;
    for (int64_t g = 0; g < n; g++) {
        if (tiles_touched[g] == 0) continue;
        uint32_t dbits;
        memcpy(&dbits, &depth[g], 4);
        for (int32_t ty = tile_rect[4 * g + 1]; ty <= tile_rect[4 * g + 3]; ty++)
            for (int32_t tx = tile_rect[4 * g]; tx <= tile_rect[4 * g + 2]; tx++) {
                uint64_t tile = (uint64_t)ty * (uint64_t)tiles_x + (uint64_t)tx;
                keys[pos] = (tile << 32) | (uint64_t)dbits;
                vals[pos] = (uint32_t)g;
                pos++;
            }
    }
}

typedef struct { uint64_t key; uint32_t val; } or_pair;

static int pair_cmp(const void *pa, const void *pb) {
    const or_pair *a = (const or_pair *)pa, *b = (const or_pair *)pb;
    if (a->key != b->key) return a->key < b->key ? -1 : 1;
    if (a->val != b->val) return a->val < b->val ? -1 : 1;
    return 0;
}

/* Ascending sort by key, equal keys in Gaussian-index order (the order a
 * stable sort of the index-ordered key list gives). Library qsort on the
 * total order (key, index). */
void or_sort(int64_t k, uint64_t *keys, uint32_t *vals) {
    or_pair *p = (or_pair *)malloc((size_t)(k > 0 ? k : 1) * sizeof(or_pair));
    for (int64_t i = 0; i < k; i++) { p[i].key = keys[i]; p[i].val = vals[i]; }
    qsort(p, (size_t)k, sizeof(or_pair), pair_cmp);
    for (int64_t i = 0; i < k; i++) { keys[i] = p[i].key; vals[i] = p[i].val; }
    free(p);
}

/* ranges[t] = [first index with tile id t, one past the last) over the
 * sorted keys, by binary search; [0, 0) for tiles with no key. */
void or_tile_ranges(int64_t k, const uint64_t *sorted_keys, int64_t n_tiles, uint32_t *ranges) {
    for (int64_t t = 0; t < n_tiles; t++) {
        int64_t lo = 0, hi = k;
        while (lo < hi) { int64_t mid = (lo + hi) / 2; if ((int64_t)(sorted_keys[mid] >> 32) < t) lo = mid + 1; else hi = mid; }
        int64_t start = lo;
        hi = k;
        while (lo < hi) { int64_t mid = (lo + hi) / 2; if ((int64_t)(sorted_keys[mid] >> 32) <= t) lo = mid + 1; else hi = mid; }
        if (lo == start) { ranges[2 * t] = 0; ranges[2 * t + 1] = 0; }
        else { ranges[2 * t] = (uint32_t)start; ranges[2 * t + 1] = (uint32_t)lo; }
    }
}

/* ------------------------------------------------------------------------- */
/* compositing (section "La règle de composition alpha", "Étape 2")          */
/* ------------------------------------------------------------------------- */

typedef struct {
    double C[3], T;
    uint32_t n_contrib;      /* 1 + list position of the last contributor, 0 if none */
    uint32_t n_eval;         /* list entries taken before the pixel stopped */
    uint32_t n_used;         /* contributions (alpha >= 1/255) */
    int32_t n_events;        /* near-threshold decisions seen (may exceed the stored count) */
} or_pixel;

/* Front to back over one pixel's ordered list of Gaussian indices:
 *   d = p - mu', q = d^T conic d, alpha = min(0.99, o exp(-q/2));
 *   skip if alpha < 1/255; C += alpha T c; T *= (1 - alpha); stop once T < 1e-4.
 * flips: list positions (with the decision type) whose decision is inverted.
 * band > 0 records decisions whose alpha or T lies within a relative band of
 * the threshold into ev_pos/ev_type (up to max_ev). */
static void composite_pixel(double px, double py, const uint32_t *list, int64_t len,
                            const double *mean2d, const double *conic, const double *opacity,
                            const double *rgb, const int32_t *flip_pos, const int8_t *flip_type,
                            int n_flips, double band, int32_t *ev_pos, int8_t *ev_type, int max_ev,
                            or_pixel *out) {
    double T = 1.0, C[3] = {0.0, 0.0, 0.0};
    uint32_t last = 0, used = 0;
    int64_t j;
    int nev = 0;
    int64_t taken = len;
    for (j = 0; j < len; j++) {
        uint32_t g = list[j];
        double dx = px - mean2d[2 * g], dy = py - mean2d[2 * g + 1];
        double A = conic[3 * g], B = conic[3 * g + 1], Cc = conic[3 * g + 2];
        double q = A * dx * dx + 2.0 * B * dx * dy + Cc * dy * dy;
        double alpha = opacity[g] * exp(-0.5 * q);
        if (alpha > OR_ALPHA_MAX) alpha = OR_ALPHA_MAX;
        int skip = alpha < OR_ALPHA_MIN;
        if (band > 0.0 && fabs(alpha - OR_ALPHA_MIN) <= band * OR_ALPHA_MIN) {
            if (nev < max_ev) { ev_pos[nev] = (int32_t)j; ev_type[nev] = OR_EV_SKIP; }
            nev++;
        }
        for (int f = 0; f < n_flips; f++)
            if (flip_pos[f] == j && flip_type[f] == OR_EV_SKIP) skip = !skip;
        if (skip) continue;
        for (int c = 0; c < 3; c++) C[c] += alpha * T * rgb[3 * g + c];
        T = T * (1.0 - alpha);
        used++;
        last = (uint32_t)(j + 1);
        int stop = T < OR_T_MIN;
        if (band > 0.0 && fabs(T - OR_T_MIN) <= band * OR_T_MIN) {
            if (nev < max_ev) { ev_pos[nev] = (int32_t)j; ev_type[nev] = OR_EV_STOP; }
            nev++;
        }
        for (int f = 0; f < n_flips; f++)
            if (flip_pos[f] == j && flip_type[f] == OR_EV_STOP) stop = !stop;
        if (stop) { taken = j + 1; break; }
    }
    for (int c = 0; c < 3; c++) out->C[c] = C[c];
    out->T = T;
    out->n_contrib = last;
    out->n_eval = (uint32_t)taken;
    out->n_used = used;
    out->n_events = nev;
}

/* Tiled composite of the whole image. Each pixel walks the sorted list of its
 * 16x16 tile; image = C + T_final * bg (HWC). Outputs per pixel: final T,
 * n_contrib, n_eval, n_used, and the near-threshold decisions (max_ev per pixel). */
void or_composite(const or_camera *cam, const double *mean2d, const double *conic,
                  const double *opacity, const double *rgb, const uint32_t *sorted_vals,
                  const uint32_t *ranges, double band, int max_ev, double *image, double *final_T,
                  uint32_t *n_contrib, uint32_t *n_eval, uint32_t *n_used, int32_t *n_events,
                  int32_t *ev_pos, int8_t *ev_type) {
    const int W = cam->width, H = cam->height;
    const int TX = (W + 15) / 16, TY = (H + 15) / 16;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t tile = 0; tile < (int64_t)TX * TY; tile++) {
        const int tx = (int)(tile % TX), ty = (int)(tile / TX);
        const uint32_t start = ranges[2 * tile], end = ranges[2 * tile + 1];
        for (int yy = 0; yy < 16; yy++)
            for (int xx = 0; xx < 16; xx++) {
                const int x = tx * 16 + xx, y = ty * 16 + yy;
                if (x >= W || y >= H) continue;
                const int64_t p = (int64_t)y * W + x;
                or_pixel r;
                composite_pixel((double)x, (double)y, sorted_vals + start, (int64_t)end - start, mean2d,
                                conic, opacity, rgb, NULL, NULL, 0, band,
                                ev_pos ? ev_pos + p * max_ev : NULL, ev_type ? ev_type + p * max_ev : NULL,
                                (ev_pos && ev_type) ? max_ev : 0, &r);
                for (int c = 0; c < 3; c++) image[3 * p + c] = r.C[c] + r.T * (double)cam->bg[c];
                final_T[p] = r.T;
                n_contrib[p] = r.n_contrib;
                n_eval[p] = r.n_eval;
                n_used[p] = r.n_used;
                n_events[p] = r.n_events;
            }
    }
}

/* One pixel of the tiled composite with the given decisions inverted: each
 * (list position, decision type) in the flip list inverts the skip test or the
 * stop test taken at that position of the pixel's tile list; positions the walk
 * never reaches change nothing. Pinned on hand-made pixels with closed forms
 * (tests/test_oracle_flip_pins.py). */
void or_composite_pixel_flipped(const or_camera *cam, int32_t x, int32_t y, const double *mean2d,
                                const double *conic, const double *opacity, const double *rgb,
                                const uint32_t *sorted_vals, const uint32_t *ranges,
                                const int32_t *flip_pos, const int8_t *flip_type, int n_flips,
                                double *out_rgb, double *out_T) {
    const int TX = (cam->width + 15) / 16;
    const int64_t tile = (int64_t)(y / 16) * TX + (x / 16);
    const uint32_t start = ranges[2 * tile], end = ranges[2 * tile + 1];
    or_pixel r;
    composite_pixel((double)x, (double)y, sorted_vals + start, (int64_t)end - start, mean2d, conic,
                    opacity, rgb, flip_pos, flip_type, n_flips, 0.0, NULL, NULL, 0, &r);
    for (int c = 0; c < 3; c++) out_rgb[c] = r.C[c] + r.T * (double)cam->bg[c];
    *out_T = r.T;
}

typedef struct { float depth; uint32_t idx; } or_dpair;

static int dpair_cmp(const void *pa, const void *pb) {
    const or_dpair *a = (const or_dpair *)pa, *b = (const or_dpair *)pb;
    if (a->depth != b->depth) return a->depth < b->depth ? -1 : 1;
    if (a->idx != b->idx) return a->idx < b->idx ? -1 : 1;
    return 0;
}

/* Untiled brute force in the manner of the pages' rasterise_2d: one global
 * depth order (camera-space z, ties by index) over all Gaussians that survive
 * culling, every pixel walks the whole list. With tile_filter = 1 a Gaussian
 * is taken at a pixel only if the pixel's 16x16 tile lies in its tile
 * rectangle (which makes the result equal to the tiled composite); with 0
 * there is no 3-sigma truncation at all. Pixels are [y0, y1) x [x0, x1). */
void or_render_untiled(const or_camera *cam, int64_t n, const uint8_t *valid, const float *depth_f32,
                       const int32_t *tile_rect, const uint32_t *tiles_touched,
                       const double *mean2d, const double *conic, const double *opacity,
                       const double *rgb, int tile_filter, int32_t x0, int32_t y0, int32_t x1, int32_t y1,
                       double *image /* [(y1-y0)][(x1-x0)][3] */, double *final_T) {
    or_dpair *order = (or_dpair *)malloc((size_t)(n > 0 ? n : 1) * sizeof(or_dpair));
    int64_t m = 0;
    for (int64_t g = 0; g < n; g++)
        if (valid[g] && (!tile_filter || tiles_touched[g] > 0)) { order[m].depth = depth_f32[g]; order[m].idx = (uint32_t)g; m++; }
    qsort(order, (size_t)m, sizeof(or_dpair), dpair_cmp);
    const int64_t w = x1 - x0;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t p = 0; p < (int64_t)(y1 - y0) * w; p++) {
        const int x = x0 + (int)(p % w), y = y0 + (int)(p / w);
        const int tx = x / 16, ty = y / 16;
        double T = 1.0, C[3] = {0.0, 0.0, 0.0};
        for (int64_t j = 0; j < m; j++) {
            const uint32_t g = order[j].idx;
            if (tile_filter) {
                const int32_t *r = tile_rect + 4 * g;
                if (tx < r[0] || tx > r[2] || ty < r[1] || ty > r[3]) continue;
            }
            double dx = x - mean2d[2 * g], dy = y - mean2d[2 * g + 1];
            double q = conic[3 * g] * dx * dx + 2.0 * conic[3 * g + 1] * dx * dy + conic[3 * g + 2] * dy * dy;
            double alpha = opacity[g] * exp(-0.5 * q);
            if (alpha > OR_ALPHA_MAX) alpha = OR_ALPHA_MAX;
            if (alpha < OR_ALPHA_MIN) continue;
            for (int c = 0; c < 3; c++) C[c] += alpha * T * rgb[3 * g + c];
            T = T * (1.0 - alpha);
            if (T < OR_T_MIN) break;
        }
        for (int c = 0; c < 3; c++) image[3 * p + c] = C[c] + T * (double)cam->bg[c];
        final_T[p] = T;
    }
    free(order);
}
