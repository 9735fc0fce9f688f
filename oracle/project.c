/*
 * project.c -- oracle of the projection of 3-D Gaussians to Splat2D records
 * and of its backward.
 *
 * TEST INFRASTRUCTURE ONLY, like the rest of oracle/: nothing in the product
 * library links or calls it, and it shares no source with the CUDA path.
 *
 * This is the step on either side of the rasterizer in the 3D Gaussian
 * Splatting trainer the pages profile: it produces the Splat2D records and
 * depths the rasterizer bins, and it turns the rasterizer's per-splat
 * gradients into gradients of the 3-D parameters ("M3 per-splat backward",
 * section 3: the trainer's parity covers the downstream log_scales and
 * rot_quats gradients; "W1 warp sparse skip + exp-skip", body: color_a is the
 * sigmoid of the opacity logit).  The pages print no projection formula; this
 * is the standard perspective (EWA) projection of a Gaussian, written out in
 * double precision, one Gaussian at a time:
 *
 *   p      = W mu + t                      (camera space; depth = p.z)
 *   mean2  = (fx p.x / p.z + cx, fy p.y / p.z + cy)
 *   R      = rotation of q / |q|           (q = (w, x, y, z))
 *   M      = R diag(exp(log_scale)),  Sigma3 = M M^T
 *   J      = [[fx / p.z, 0, -fx p.x / p.z^2], [0, fy / p.z, -fy p.y / p.z^2]]
 *   Sigma2 = (J W) Sigma3 (J W)^T + eps I  (eps: a low-pass dilation)
 *   conic  = (a, b, c) with [[a, b], [b, c]] = Sigma2^-1
 *   color_a = 1 / (1 + exp(-logit)),  rgb passed through
 *
 * A Gaussian with p.z <= z_near, a non-finite value or det(Sigma2) <= 0 is not
 * visible: its Splat2D has mean and conic 0 (the binning culls a conic with
 * a <= 0) and depth 0, and it receives no gradient.
 *
 * Layouts (doubles):
 *   gaussian [14]: mean xyz, log_scale xyz, quat wxyz, logit_opacity, rgb
 *   camera   [18]: W row-major (9), t (3), fx, fy, cx, cy, z_near, eps
 *   splat    [9] : mean_x, mean_y, conic a, b, c, r, g, b, color_a
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "oracle.h"

/* Rotation matrix of the unit quaternion (w, x, y, z). */
static void quat_to_rot(const double *q, double *R)
{
    const double w = q[0], x = q[1], y = q[2], z = q[3];
    R[0] = 1.0 - 2.0 * (y * y + z * z);
    R[1] = 2.0 * (x * y - w * z);
    R[2] = 2.0 * (x * z + w * y);
    R[3] = 2.0 * (x * y + w * z);
    R[4] = 1.0 - 2.0 * (x * x + z * z);
    R[5] = 2.0 * (y * z - w * x);
    R[6] = 2.0 * (x * z - w * y);
    R[7] = 2.0 * (y * z + w * x);
    R[8] = 1.0 - 2.0 * (x * x + y * y);
}

/* Everything the forward computes for one Gaussian, kept for the backward. */
typedef struct {
    int visible;
    double p[3];        /* camera-space mean */
    double qn[4];       /* normalised quaternion */
    double qlen;        /* |q| */
    double s[3];        /* scales */
    double R[9];        /* rotation */
    double M[9];        /* R diag(s) */
    double S3[9];       /* Sigma3 */
    double J[6];        /* 2x3, row-major */
    double T[6];        /* J W, 2x3 */
    double s00, s01, s11;  /* Sigma2 */
    double a, b, c;     /* conic */
    double alpha;       /* color_a */
} proj_state;

static void project_one(const double *g, const double *cam, proj_state *st)
{
    memset(st, 0, sizeof *st);
    const double *W = cam, *t = cam + 9;
    const double fx = cam[12], fy = cam[13], z_near = cam[16], eps = cam[17];
    for (int k = 0; k < 14; ++k)
        if (!isfinite(g[k])) return;
    /* camera space */
    for (int i = 0; i < 3; ++i) st->p[i] = W[3 * i] * g[0] + W[3 * i + 1] * g[1] + W[3 * i + 2] * g[2] + t[i];
    if (!(st->p[2] > z_near)) return;
    /* rotation and scales */
    st->qlen = sqrt(g[6] * g[6] + g[7] * g[7] + g[8] * g[8] + g[9] * g[9]);
    if (!(st->qlen > 0.0)) return;
    for (int k = 0; k < 4; ++k) st->qn[k] = g[6 + k] / st->qlen;
    quat_to_rot(st->qn, st->R);
    for (int k = 0; k < 3; ++k) st->s[k] = exp(g[3 + k]);
    for (int i = 0; i < 3; ++i)
        for (int j = 0; j < 3; ++j) st->M[3 * i + j] = st->R[3 * i + j] * st->s[j];
    /* Sigma3 = M M^T */
    for (int i = 0; i < 3; ++i)
        for (int j = 0; j < 3; ++j) {
            double v = 0.0;
            for (int k = 0; k < 3; ++k) v += st->M[3 * i + k] * st->M[3 * j + k];
            st->S3[3 * i + j] = v;
        }
    /* Jacobian of the perspective division at p, and T = J W */
    const double x = st->p[0], y = st->p[1], z = st->p[2];
    st->J[0] = fx / z;
    st->J[1] = 0.0;
    st->J[2] = -fx * x / (z * z);
    st->J[3] = 0.0;
    st->J[4] = fy / z;
    st->J[5] = -fy * y / (z * z);
    for (int i = 0; i < 2; ++i)
        for (int j = 0; j < 3; ++j) {
            double v = 0.0;
            for (int k = 0; k < 3; ++k) v += st->J[3 * i + k] * W[3 * k + j];
            st->T[3 * i + j] = v;
        }
    /* Sigma2 = T Sigma3 T^T + eps I */
    double TS[6];
    for (int i = 0; i < 2; ++i)
        for (int j = 0; j < 3; ++j) {
            double v = 0.0;
            for (int k = 0; k < 3; ++k) v += st->T[3 * i + k] * st->S3[3 * k + j];
            TS[3 * i + j] = v;
        }
    double S2[4];
    for (int i = 0; i < 2; ++i)
        for (int j = 0; j < 2; ++j) {
            double v = 0.0;
            for (int k = 0; k < 3; ++k) v += TS[3 * i + k] * st->T[3 * j + k];
            S2[2 * i + j] = v;
        }
    st->s00 = S2[0] + eps;
    st->s01 = S2[1];
    st->s11 = S2[3] + eps;
    const double det = st->s00 * st->s11 - st->s01 * st->s01;
    if (!(det > 0.0) || !isfinite(det)) return;
    st->a = st->s11 / det;
    st->b = -st->s01 / det;
    st->c = st->s00 / det;
    st->alpha = 1.0 / (1.0 + exp(-g[10]));
    st->visible = 1;
}

void orc_project_forward(const double *g, int32_t n, const double *cam, double *splats, double *depths,
                         uint8_t *visible)
{
    const double fx = cam[12], fy = cam[13], cx = cam[14], cy = cam[15];
    for (int32_t i = 0; i < n; ++i) {
        const double *gi = g + 14 * (int64_t)i;
        double *sp = splats + 9 * (int64_t)i;
        proj_state st;
        project_one(gi, cam, &st);
        visible[i] = (uint8_t)st.visible;
        memset(sp, 0, 9 * sizeof(double));
        sp[5] = gi[11];
        sp[6] = gi[12];
        sp[7] = gi[13];
        depths[i] = 0.0;
        if (!st.visible) continue;
        sp[0] = fx * st.p[0] / st.p[2] + cx;
        sp[1] = fy * st.p[1] / st.p[2] + cy;
        sp[2] = st.a;
        sp[3] = st.b;
        sp[4] = st.c;
        sp[8] = st.alpha;
        depths[i] = st.p[2];
    }
}

/* gabs (optional): for each output, the sum of the absolute values of the
 * terms its last sum adds up (the rounding scale of that sum: an exact zero
 * such as the rotation gradient of an isotropic Gaussian is a sum of terms
 * that cancel, and a float evaluation leaves about u times this much). */
void orc_project_backward(const double *g, int32_t n, const double *cam, const double *dl_dsplat,
                          double *dl_dg, double *gabs)
{
    const double *W = cam;
    const double fx = cam[12], fy = cam[13];
    for (int32_t i = 0; i < n; ++i) {
        const double *gi = g + 14 * (int64_t)i;
        const double *G = dl_dsplat + 9 * (int64_t)i;
        double *out = dl_dg + 14 * (int64_t)i;
        double ab[14];
        memset(out, 0, 14 * sizeof(double));
        memset(ab, 0, sizeof ab);
        if (gabs) memset(gabs + 14 * (int64_t)i, 0, 14 * sizeof(double));
        proj_state st;
        project_one(gi, cam, &st);
        if (!st.visible) continue;
        /* rgb and opacity */
        out[11] = G[5];
        out[12] = G[6];
        out[13] = G[7];
        out[10] = G[8] * st.alpha * (1.0 - st.alpha);
        for (int k = 10; k < 14; ++k) ab[k] = fabs(out[k]);
        /* conic -> Sigma2: the entries of [[a, b], [b, c]] = Sigma2^-1 as
         * functions of s00, s01 (both off-diagonal entries), s11 */
        const double a = st.a, b = st.b, c = st.c;
        const double d00 = -G[2] * a * a - G[3] * a * b - G[4] * b * b;
        const double d11 = -G[2] * b * b - G[3] * b * c - G[4] * c * c;
        const double d01 = -2.0 * G[2] * a * b - G[3] * (a * c + b * b) - 2.0 * G[4] * b * c;
        /* G2: the symmetric gradient of Sigma2 (s01 counted in both entries) */
        const double G2[4] = {d00, 0.5 * d01, 0.5 * d01, d11};
        /* Sigma2 = T Sigma3 T^T: dSigma3 = T^T G2 T, dT = 2 G2 T Sigma3 */
        double G3[9];
        for (int r = 0; r < 3; ++r)
            for (int s = 0; s < 3; ++s) {
                double v = 0.0;
                for (int u = 0; u < 2; ++u)
                    for (int w = 0; w < 2; ++w) v += st.T[3 * u + r] * G2[2 * u + w] * st.T[3 * w + s];
                G3[3 * r + s] = v;
            }
        double GT[6];
        for (int u = 0; u < 2; ++u)
            for (int s = 0; s < 3; ++s) {
                double v = 0.0;
                for (int w = 0; w < 2; ++w)
                    for (int k = 0; k < 3; ++k) v += G2[2 * u + w] * st.T[3 * w + k] * st.S3[3 * k + s];
                GT[3 * u + s] = 2.0 * v;
            }
        /* T = J W: dJ = dT W^T */
        double GJ[6];
        for (int u = 0; u < 2; ++u)
            for (int k = 0; k < 3; ++k) {
                double v = 0.0;
                for (int s = 0; s < 3; ++s) v += GT[3 * u + s] * W[3 * k + s];
                GJ[3 * u + k] = v;
            }
        /* camera-space mean: through J and through the projected mean */
        const double x = st.p[0], y = st.p[1], z = st.p[2];
        double gp[3];
        gp[0] = GJ[2] * (-fx / (z * z)) + G[0] * fx / z;
        gp[1] = GJ[5] * (-fy / (z * z)) + G[1] * fy / z;
        gp[2] = GJ[0] * (-fx / (z * z)) + GJ[2] * (2.0 * fx * x / (z * z * z)) + GJ[4] * (-fy / (z * z)) +
                GJ[5] * (2.0 * fy * y / (z * z * z)) - G[0] * fx * x / (z * z) - G[1] * fy * y / (z * z);
        double gpa[3];
        gpa[0] = fabs(GJ[2] * fx / (z * z)) + fabs(G[0] * fx / z);
        gpa[1] = fabs(GJ[5] * fy / (z * z)) + fabs(G[1] * fy / z);
        gpa[2] = fabs(GJ[0] * fx / (z * z)) + fabs(GJ[2] * 2.0 * fx * x / (z * z * z)) + fabs(GJ[4] * fy / (z * z)) +
                 fabs(GJ[5] * 2.0 * fy * y / (z * z * z)) + fabs(G[0] * fx * x / (z * z)) +
                 fabs(G[1] * fy * y / (z * z));
        /* p = W mu + t: dmu = W^T dp */
        for (int k = 0; k < 3; ++k) {
            out[k] = W[k] * gp[0] + W[3 + k] * gp[1] + W[6 + k] * gp[2];
            ab[k] = fabs(W[k]) * gpa[0] + fabs(W[3 + k]) * gpa[1] + fabs(W[6 + k]) * gpa[2];
        }
        /* Sigma3 = M M^T: dM = 2 G3 M */
        double GM[9];
        for (int r = 0; r < 3; ++r)
            for (int s = 0; s < 3; ++s) {
                double v = 0.0;
                for (int k = 0; k < 3; ++k) v += G3[3 * r + k] * st.M[3 * k + s];
                GM[3 * r + s] = 2.0 * v;
            }
        /* M = R diag(s): ds_j = column j of R . column j of dM; dR = dM diag(s) */
        double GR[9];
        for (int j = 0; j < 3; ++j) {
            double v = 0.0, va = 0.0;
            for (int r = 0; r < 3; ++r) {
                v += st.R[3 * r + j] * GM[3 * r + j];
                va += fabs(st.R[3 * r + j] * GM[3 * r + j]);
                GR[3 * r + j] = GM[3 * r + j] * st.s[j];
            }
            out[3 + j] = v * st.s[j]; /* d log_scale = ds * s */
            ab[3 + j] = va * st.s[j];
        }
        /* R of the unit quaternion (w, x, y, z): dqn from the entries' partials */
        const double w = st.qn[0], qx = st.qn[1], qy = st.qn[2], qz = st.qn[3];
        double gq[4];
        gq[0] = 2.0 * (-qz * GR[1] + qy * GR[2] + qz * GR[3] - qx * GR[5] - qy * GR[6] + qx * GR[7]);
        gq[1] = 2.0 * (qy * GR[1] + qz * GR[2] + qy * GR[3] - w * GR[5] + qz * GR[6] + w * GR[7]) -
                4.0 * qx * (GR[4] + GR[8]);
        gq[2] = 2.0 * (qx * GR[1] + w * GR[2] + qx * GR[3] + qz * GR[5] - w * GR[6] + qz * GR[7]) -
                4.0 * qy * (GR[0] + GR[8]);
        gq[3] = 2.0 * (-w * GR[1] + qx * GR[2] + w * GR[3] + qy * GR[5] + qx * GR[6] + qy * GR[7]) -
                4.0 * qz * (GR[0] + GR[4]);
        double gqa[4];
        gqa[0] = 2.0 * (fabs(qz * GR[1]) + fabs(qy * GR[2]) + fabs(qz * GR[3]) + fabs(qx * GR[5]) +
                        fabs(qy * GR[6]) + fabs(qx * GR[7]));
        gqa[1] = 2.0 * (fabs(qy * GR[1]) + fabs(qz * GR[2]) + fabs(qy * GR[3]) + fabs(w * GR[5]) +
                        fabs(qz * GR[6]) + fabs(w * GR[7])) + 4.0 * fabs(qx) * (fabs(GR[4]) + fabs(GR[8]));
        gqa[2] = 2.0 * (fabs(qx * GR[1]) + fabs(w * GR[2]) + fabs(qx * GR[3]) + fabs(qz * GR[5]) +
                        fabs(w * GR[6]) + fabs(qz * GR[7])) + 4.0 * fabs(qy) * (fabs(GR[0]) + fabs(GR[8]));
        gqa[3] = 2.0 * (fabs(w * GR[1]) + fabs(qx * GR[2]) + fabs(w * GR[3]) + fabs(qy * GR[5]) +
                        fabs(qx * GR[6]) + fabs(qy * GR[7])) + 4.0 * fabs(qz) * (fabs(GR[0]) + fabs(GR[4]));
        /* qn = q / |q|: dq = (dqn - qn (qn . dqn)) / |q| */
        const double dot = w * gq[0] + qx * gq[1] + qy * gq[2] + qz * gq[3];
        double dota = 0.0;
        for (int k = 0; k < 4; ++k) dota += fabs(st.qn[k]) * gqa[k];
        for (int k = 0; k < 4; ++k) {
            out[6 + k] = (gq[k] - st.qn[k] * dot) / st.qlen;
            ab[6 + k] = (gqa[k] + fabs(st.qn[k]) * dota) / st.qlen;
        }
        if (gabs) memcpy(gabs + 14 * (int64_t)i, ab, sizeof ab);
    }
}
