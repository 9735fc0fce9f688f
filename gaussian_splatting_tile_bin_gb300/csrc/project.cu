// project.cu -- projection of 3-D Gaussians to Splat2D records and depths, and
// its backward: the steps on either side of the rasterizer in the 3D Gaussian
// Splatting trainer whose findings pages define the rasterizer ("M3 per-splat
// backward", section 3: the trainer differentiates through to log_scales and
// rot_quats; "W1 warp sparse skip + exp-skip", body: color_a is the sigmoid of
// the opacity logit).  The pages print no projection formula; this is the
// standard perspective (EWA) projection of a Gaussian:
//
//   p = W mu + t,   mean2 = (fx p.x / p.z + cx, fy p.y / p.z + cy),  depth = p.z
//   Sigma2 = V V^T + eps I,   V = J W R diag(exp(log_scale))  (2 x 3)
//   conic = Sigma2^-1,  color_a = sigmoid(logit)
//
// One thread per Gaussian; both kernels are bound by HBM bandwidth (56 B of
// Gaussian in, 36 B of Splat2D + 4 B of depth out; 56 + 36 in and 56 out for
// the backward).  Chunks of 256 records move through shared memory so that
// every global access is a contiguous, coalesced run of the chunk's bytes, and
// each block keeps its next chunk's copy in flight while it computes.
//
// Numerics.  det(Sigma2) is formed without cancellation: for the two rows
// v0, v1 of V, |v0|^2 |v1|^2 - (v0 . v1)^2 = |v0 x v1|^2 (Lagrange's identity),
// so det = |v0 x v1|^2 + eps (|v0|^2 + |v1|^2) + eps^2, a sum of non-negative
// terms.  The conic is therefore accurate to a few ulps relative to its own
// metric even for needle-thin splats, where a c - b^2 in fp32 would lose all
// its bits.
#include <math.h>
#include <string.h>

#include <algorithm>

#include "internal.cuh"

namespace gsr {
namespace {

constexpr int kProjBlock = 256;
constexpr int kG = GSR_GAUSSIAN_FLOATS;   // 14 floats per Gaussian
constexpr int kS = 9;                     // 9 floats per Splat2D / Splat2D gradient

struct Camera {
    float W[9];
    float t[3];
    float fx, fy, cx, cy, z_near, eps;
};
static_assert(sizeof(Camera) == sizeof(gsr_camera), "camera layout");

// Asynchronous global -> shared copies (cp.async): the copies of a chunk are
// committed as one group, and a wait on the group count lets the block compute
// one chunk while the next is in flight.
__device__ __forceinline__ void cp_async16(float *smem, const float *gmem)
{
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(__cvta_generic_to_global(gmem))
                 : "memory");
}
__device__ __forceinline__ void cp_async4(float *smem, const float *gmem)
{
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(s), "l"(__cvta_generic_to_global(gmem))
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Starts copying `count` floats from src + first into dst (shared memory).
// Vec: src + first and dst are 16-byte aligned.
template <bool Vec>
__device__ __forceinline__ void stage_in_async(float *__restrict__ dst, const float *__restrict__ src, size_t first,
                                               int count)
{
    int done = 0;
    if (Vec) {
        const int n4 = count >> 2;
        for (int i = threadIdx.x; i < n4; i += kProjBlock) cp_async16(dst + 4 * i, src + first + 4 * i);
        done = n4 << 2;
    }
    for (int i = done + threadIdx.x; i < count; i += kProjBlock) cp_async4(dst + i, src + first + i);
}

// Copies `count` floats from shared memory to dst + first, coalesced.
template <bool Vec>
__device__ __forceinline__ void stage_out(float *__restrict__ dst, const float *__restrict__ src, size_t first,
                                          int count)
{
    int done = 0;
    if (Vec) {
        float4 *d4 = reinterpret_cast<float4 *>(dst + first);
        const float4 *s4 = reinterpret_cast<const float4 *>(src);
        const int n4 = count >> 2;
        for (int i = threadIdx.x; i < n4; i += kProjBlock) d4[i] = s4[i];
        done = n4 << 2;
    }
    for (int i = done + threadIdx.x; i < count; i += kProjBlock) dst[first + i] = src[i];
}

// Forward quantities of one Gaussian, kept in registers for the backward.
struct Proj {
    bool visible;
    float x, y, z, iz;      // camera-space mean, 1 / z
    float qw, qx, qy, qz;   // normalised quaternion
    float rinv;             // 1 / |q|
    float s[3];             // scales
    float R[9];             // rotation, row-major
    float T[6];             // J W, 2 x 3
    float V[6];             // T R diag(s), 2 x 3
    float cr[3];            // v0 x v1 (rows of V)
    float idet;             // 1 / det(Sigma2)
    float a, b, c;          // conic
    float e;                // exp(-logit)
    float alpha;            // color_a = 1 / (1 + e)
};

__device__ __forceinline__ void project(const float *g, const Camera &cam, Proj &P)
{
    P.visible = false;
    bool finite = true;
#pragma unroll
    for (int k = 0; k < kG; ++k) finite &= isfinite(g[k]);
    const float *W = cam.W;
    P.x = fmaf(W[0], g[0], fmaf(W[1], g[1], fmaf(W[2], g[2], cam.t[0])));
    P.y = fmaf(W[3], g[0], fmaf(W[4], g[1], fmaf(W[5], g[2], cam.t[1])));
    P.z = fmaf(W[6], g[0], fmaf(W[7], g[1], fmaf(W[8], g[2], cam.t[2])));
    const float q2 = g[6] * g[6] + g[7] * g[7] + g[8] * g[8] + g[9] * g[9];
    if (!finite || !(P.z > cam.z_near) || !(q2 > 0.0f)) return;

    P.iz = 1.0f / P.z;
    P.rinv = rsqrtf(q2);
    P.qw = g[6] * P.rinv;
    P.qx = g[7] * P.rinv;
    P.qy = g[8] * P.rinv;
    P.qz = g[9] * P.rinv;
    const float w = P.qw, x = P.qx, y = P.qy, z = P.qz;
    P.R[0] = 1.0f - 2.0f * (y * y + z * z);
    P.R[1] = 2.0f * (x * y - w * z);
    P.R[2] = 2.0f * (x * z + w * y);
    P.R[3] = 2.0f * (x * y + w * z);
    P.R[4] = 1.0f - 2.0f * (x * x + z * z);
    P.R[5] = 2.0f * (y * z - w * x);
    P.R[6] = 2.0f * (x * z - w * y);
    P.R[7] = 2.0f * (y * z + w * x);
    P.R[8] = 1.0f - 2.0f * (x * x + y * y);
#pragma unroll
    for (int k = 0; k < 3; ++k) P.s[k] = expf(g[3 + k]);

    // T = J W with J = [[fx/z, 0, -fx x/z^2], [0, fy/z, -fy y/z^2]]:
    // row 0 = fx/z (W row 0 - x/z W row 2), row 1 = fy/z (W row 1 - y/z W row 2).
    const float ux = P.x * P.iz, uy = P.y * P.iz;
    const float jx = cam.fx * P.iz, jy = cam.fy * P.iz;
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        P.T[j] = jx * fmaf(-ux, W[6 + j], W[j]);
        P.T[3 + j] = jy * fmaf(-uy, W[6 + j], W[3 + j]);
    }
    // V = T R diag(s)
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int k = 0; k < 3; ++k)
            P.V[3 * i + k] =
                P.s[k] * fmaf(P.T[3 * i], P.R[k], fmaf(P.T[3 * i + 1], P.R[3 + k], P.T[3 * i + 2] * P.R[6 + k]));

    const float *v0 = P.V, *v1 = P.V + 3;
    const float n0 = fmaf(v0[0], v0[0], fmaf(v0[1], v0[1], v0[2] * v0[2]));
    const float n1 = fmaf(v1[0], v1[0], fmaf(v1[1], v1[1], v1[2] * v1[2]));
    const float d01 = fmaf(v0[0], v1[0], fmaf(v0[1], v1[1], v0[2] * v1[2]));
    P.cr[0] = v0[1] * v1[2] - v0[2] * v1[1];
    P.cr[1] = v0[2] * v1[0] - v0[0] * v1[2];
    P.cr[2] = v0[0] * v1[1] - v0[1] * v1[0];
    const float eps = cam.eps;
    const float det = fmaf(P.cr[0], P.cr[0], fmaf(P.cr[1], P.cr[1], P.cr[2] * P.cr[2])) + eps * (n0 + n1) + eps * eps;
    if (!(det > 0.0f) || !isfinite(det)) return;
    P.idet = 1.0f / det;
    P.a = (n1 + eps) * P.idet;
    P.b = -d01 * P.idet;
    P.c = (n0 + eps) * P.idet;
    P.e = expf(-g[10]);
    P.alpha = 1.0f / (1.0f + P.e);
    P.visible = true;
}

// Splat2D record and depth of the Gaussian g (shared memory).
__device__ __forceinline__ void forward_one(const float *g, const Camera &cam, float *o, float &depth)
{
    Proj P;
    project(g, cam, P);
    o[0] = P.visible ? fmaf(cam.fx, P.x * P.iz, cam.cx) : 0.0f;
    o[1] = P.visible ? fmaf(cam.fy, P.y * P.iz, cam.cy) : 0.0f;
    o[2] = P.visible ? P.a : 0.0f;
    o[3] = P.visible ? P.b : 0.0f;
    o[4] = P.visible ? P.c : 0.0f;
    o[5] = g[11];
    o[6] = g[12];
    o[7] = g[13];
    o[8] = P.visible ? P.alpha : 0.0f;
    depth = P.visible ? P.z : 0.0f;
}

// dL/dg for the Gaussian g given G = dL/d(its Splat2D fields).
__device__ __forceinline__ void backward_one(const float *g, const float *G, const Camera &cam, float (&out)[kG])
{
#pragma unroll
    for (int k = 0; k < kG; ++k) out[k] = 0.0f;
    Proj P;
    project(g, cam, P);
    if (!P.visible) return;
    out[11] = G[5];
    out[12] = G[6];
    out[13] = G[7];
    // d alpha / d logit = alpha (1 - alpha) = e alpha^2 (no cancellation near alpha = 1)
    out[10] = G[8] * P.e * P.alpha * P.alpha;

    // Q = Sigma2^-1 is the conic, G_Q = [[Ga, Gb/2], [Gb/2, Gc]] its
    // symmetric gradient.  With Sigma2 = V V^T + eps I,
    //   dL/dSigma2 = -Q G_Q Q  and  dL/dV = 2 dL/dSigma2 V = -2 Q G_Q (Q V).
    // Q V = adj(Sigma2) V / det is formed row by row from cross products,
    //   row 0: |v1|^2 v0 - (v0.v1) v1 + eps v0 = v1 x (v0 x v1) + eps v0,
    //   row 1: |v0|^2 v1 - (v0.v1) v0 + eps v1 = (v0 x v1) x v0 + eps v1,
    // so that a column of V along a long splat axis, which Q nearly
    // annihilates, keeps its relative accuracy (multiplying by the
    // rounded Q would leave only an absolute one).
    const float a = P.a, b = P.b, c = P.c;
    const float Ga = G[2], Gb = 0.5f * G[3], Gc = G[4];
    const float eps = cam.eps;
    const float *v0 = P.V, *v1 = P.V + 3, *cr = P.cr;
    float QV0[3], QV1[3];
    QV0[0] = fmaf(eps, v0[0], v1[1] * cr[2] - v1[2] * cr[1]) * P.idet;
    QV0[1] = fmaf(eps, v0[1], v1[2] * cr[0] - v1[0] * cr[2]) * P.idet;
    QV0[2] = fmaf(eps, v0[2], v1[0] * cr[1] - v1[1] * cr[0]) * P.idet;
    QV1[0] = fmaf(eps, v1[0], cr[1] * v0[2] - cr[2] * v0[1]) * P.idet;
    QV1[1] = fmaf(eps, v1[1], cr[2] * v0[0] - cr[0] * v0[2]) * P.idet;
    QV1[2] = fmaf(eps, v1[2], cr[0] * v0[1] - cr[1] * v0[0]) * P.idet;
    float dV[6];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        const float h0 = fmaf(Ga, QV0[k], Gb * QV1[k]);   // (G_Q Q V)_0k
        const float h1 = fmaf(Gb, QV0[k], Gc * QV1[k]);   // (G_Q Q V)_1k
        dV[k] = -2.0f * fmaf(a, h0, b * h1);
        dV[3 + k] = -2.0f * fmaf(b, h0, c * h1);
        // dL/dlog_scale_k = sum_i dV_ik V_ik = -2 (Q V)_k . (G_Q Q V)_k
        out[3 + k] = -2.0f * fmaf(QV0[k], h0, QV1[k] * h1);
    }
    // V_ik = s_k sum_j T_ij R_jk: dL/dT_ij = sum_k dV_ik s_k R_jk,
    // dL/dR_jk = s_k sum_i T_ij dV_ik.
    float dT[6], dR[9];
#pragma unroll
    for (int i2 = 0; i2 < 2; ++i2)
#pragma unroll
        for (int j = 0; j < 3; ++j)
            dT[3 * i2 + j] = fmaf(dV[3 * i2] * P.s[0], P.R[3 * j],
                                  fmaf(dV[3 * i2 + 1] * P.s[1], P.R[3 * j + 1],
                                       dV[3 * i2 + 2] * P.s[2] * P.R[3 * j + 2]));
#pragma unroll
    for (int j = 0; j < 3; ++j)
#pragma unroll
        for (int k = 0; k < 3; ++k)
            dR[3 * j + k] = P.s[k] * fmaf(P.T[j], dV[k], P.T[3 + j] * dV[3 + k]);

    // R(q) for the unit quaternion (w, x, y, z): partial derivatives of
    // each entry, contracted with dR.
    const float w = P.qw, x = P.qx, y = P.qy, z = P.qz;
    const float gw = 2.0f * (-z * dR[1] + y * dR[2] + z * dR[3] - x * dR[5] - y * dR[6] + x * dR[7]);
    const float gx = 2.0f * (y * dR[1] + z * dR[2] + y * dR[3] - 2.0f * x * dR[4] - w * dR[5] +
                             z * dR[6] + w * dR[7] - 2.0f * x * dR[8]);
    const float gy = 2.0f * (-2.0f * y * dR[0] + x * dR[1] + w * dR[2] + x * dR[3] + z * dR[5] -
                             w * dR[6] + z * dR[7] - 2.0f * y * dR[8]);
    const float gz = 2.0f * (-2.0f * z * dR[0] - w * dR[1] + x * dR[2] + w * dR[3] - 2.0f * z * dR[4] +
                             y * dR[5] + x * dR[6] + y * dR[7]);
    // q -> q / |q|: the gradient loses its component along q and scales by 1/|q|.
    const float dot = w * gw + x * gx + y * gy + z * gz;
    out[6] = (gw - w * dot) * P.rinv;
    out[7] = (gx - x * dot) * P.rinv;
    out[8] = (gy - y * dot) * P.rinv;
    out[9] = (gz - z * dot) * P.rinv;

    // T = J(p) W: dL/dJ = dT W^T; J depends on p through
    // J00 = fx/z, J02 = -fx x/z^2, J11 = fy/z, J12 = -fy y/z^2.
    const float *Wm = cam.W;
    const float dJ00 = fmaf(dT[0], Wm[0], fmaf(dT[1], Wm[1], dT[2] * Wm[2]));
    const float dJ02 = fmaf(dT[0], Wm[6], fmaf(dT[1], Wm[7], dT[2] * Wm[8]));
    const float dJ11 = fmaf(dT[3], Wm[3], fmaf(dT[4], Wm[4], dT[5] * Wm[5]));
    const float dJ12 = fmaf(dT[3], Wm[6], fmaf(dT[4], Wm[7], dT[5] * Wm[8]));
    const float iz = P.iz, ux = P.x * iz, uy = P.y * iz;
    const float fxz = cam.fx * iz, fyz = cam.fy * iz;
    // mean2 = (fx x/z + cx, fy y/z + cy) plus the J terms
    const float dpx = fxz * (G[0] - dJ02 * iz);
    const float dpy = fyz * (G[1] - dJ12 * iz);
    const float dpz = -iz * (fxz * fmaf(G[0], P.x, dJ00 - 2.0f * dJ02 * ux) +
                             fyz * fmaf(G[1], P.y, dJ11 - 2.0f * dJ12 * uy));
    // p = W mu + t
    out[0] = fmaf(Wm[0], dpx, fmaf(Wm[3], dpy, Wm[6] * dpz));
    out[1] = fmaf(Wm[1], dpx, fmaf(Wm[4], dpy, Wm[7] * dpz));
    out[2] = fmaf(Wm[2], dpx, fmaf(Wm[5], dpy, Wm[8] * dpz));
}

// Chunks of 256 Gaussians, one per thread.  A block takes chunks blockIdx.x,
// blockIdx.x + gridDim.x, ... with the grid a few blocks per SM, and keeps the
// next chunk's copy in flight while it computes the current one (two buffers),
// so the loads of the whole launch are issued early instead of wave by wave.
constexpr int kStages = 2;
// Resident blocks per SM the kernels are compiled for, and the grid's blocks per SM.
#ifndef GSR_PROJ_FWD_BLOCKS
#define GSR_PROJ_FWD_BLOCKS 4
#endif
constexpr int kProjFwdBlocksPerSM = GSR_PROJ_FWD_BLOCKS;
constexpr int kProjBwdBlocksPerSM = 4;

template <bool Vec>
__global__ void __launch_bounds__(kProjBlock, kProjFwdBlocksPerSM) k_project_forward(const float *__restrict__ gauss, int n, Camera cam,
                                                                float *__restrict__ splats,
                                                                float *__restrict__ depths)
{
    __shared__ __align__(16) float sg[kStages][kProjBlock * kG];
    __shared__ __align__(16) float ss[kProjBlock * kS];
    grid_dependency_begin();
    const int chunks = (n + kProjBlock - 1) / kProjBlock;
#pragma unroll
    for (int d = 0; d < kStages; ++d) {
        const int c = blockIdx.x + d * gridDim.x;
        if (c < chunks) stage_in_async<Vec>(sg[d], gauss, (size_t)c * kProjBlock * kG,
                                            min(kProjBlock, n - c * kProjBlock) * kG);
        cp_async_commit();
    }
    int buf = 0;
    for (int c = blockIdx.x; c < chunks; c += gridDim.x) {
        const int base = c * kProjBlock;
        const int cnt = min(kProjBlock, n - base);
        cp_async_wait<kStages - 1>();   // this chunk's group has landed
        __syncthreads();
        const int i = threadIdx.x;
        if (i < cnt) {
            float depth;
            forward_one(sg[buf] + i * kG, cam, ss + i * kS, depth);
            depths[base + i] = depth;
        }
        __syncthreads();   // sg[buf] is read; ss is written
        stage_out<Vec>(splats, ss, (size_t)base * kS, cnt * kS);
        const int cn = c + kStages * gridDim.x;
        if (cn < chunks) stage_in_async<Vec>(sg[buf], gauss, (size_t)cn * kProjBlock * kG,
                                             min(kProjBlock, n - cn * kProjBlock) * kG);
        cp_async_commit();
        buf = (buf + 1) % kStages;
    }
    cp_async_wait<0>();
}

template <bool Vec>
__global__ void __launch_bounds__(kProjBlock, kProjBwdBlocksPerSM) k_project_backward(const float *__restrict__ gauss, int n, Camera cam,
                                                                 const float *__restrict__ dl_dsplat,
                                                                 float *__restrict__ dl_dg)
{
    __shared__ __align__(16) float sg[kStages][kProjBlock * kG];
    __shared__ __align__(16) float sd[kStages][kProjBlock * kS];
    grid_dependency_begin();
    const int chunks = (n + kProjBlock - 1) / kProjBlock;
#pragma unroll
    for (int d = 0; d < kStages; ++d) {
        const int c = blockIdx.x + d * gridDim.x;
        if (c < chunks) {
            const int cnt = min(kProjBlock, n - c * kProjBlock);
            stage_in_async<Vec>(sg[d], gauss, (size_t)c * kProjBlock * kG, cnt * kG);
            stage_in_async<Vec>(sd[d], dl_dsplat, (size_t)c * kProjBlock * kS, cnt * kS);
        }
        cp_async_commit();
    }
    int buf = 0;
    for (int c = blockIdx.x; c < chunks; c += gridDim.x) {
        const int base = c * kProjBlock;
        const int cnt = min(kProjBlock, n - base);
        cp_async_wait<kStages - 1>();
        __syncthreads();
        const int i = threadIdx.x;
        float out[kG];
        if (i < cnt) backward_one(sg[buf] + i * kG, sd[buf] + i * kS, cam, out);
        __syncthreads();   // every thread has read its Gaussian: sg[buf] can take the gradients
        if (i < cnt) {
#pragma unroll
            for (int k = 0; k < kG; ++k) sg[buf][i * kG + k] = out[k];
        }
        __syncthreads();
        stage_out<Vec>(dl_dg, sg[buf], (size_t)base * kG, cnt * kG);
        __syncthreads();   // the gradients are out: the buffers can take the next chunk
        const int cn = c + kStages * gridDim.x;
        if (cn < chunks) {
            const int cnt2 = min(kProjBlock, n - cn * kProjBlock);
            stage_in_async<Vec>(sg[buf], gauss, (size_t)cn * kProjBlock * kG, cnt2 * kG);
            stage_in_async<Vec>(sd[buf], dl_dsplat, (size_t)cn * kProjBlock * kS, cnt2 * kS);
        }
        cp_async_commit();
        buf = (buf + 1) % kStages;
    }
    cp_async_wait<0>();
}

Camera to_camera(const gsr_camera &c)
{
    Camera k;
    static_assert(sizeof(k) == sizeof(c), "camera layout");
    memcpy(&k, &c, sizeof k);
    return k;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15) == 0; }

}  // namespace

int projection_grid(gsr_ctx *ctx, int32_t n, int blocks_per_sm)
{
    const int64_t chunks = ((int64_t)n + kProjBlock - 1) / kProjBlock;
    return (int)std::min<int64_t>(chunks, (int64_t)ctx->num_sms * blocks_per_sm);
}

int project_forward(gsr_ctx *ctx, const float *gauss, int32_t n, const gsr_camera &camera, float *splats,
                    float *depths, cudaStream_t stream)
{
    const Camera cam = to_camera(camera);
    const dim3 grid((unsigned)projection_grid(ctx, n, kProjFwdBlocksPerSM));
    // Every chunk starts at a multiple of 256 records: 16-byte aligned whenever the arrays are.
    const bool vec = aligned16(gauss) && aligned16(splats);
    const cudaError_t e =
        vec ? launch_kernel(ctx, k_project_forward<true>, grid, dim3(kProjBlock), stream, gauss, (int)n, cam,
                            splats, depths)
            : launch_kernel(ctx, k_project_forward<false>, grid, dim3(kProjBlock), stream, gauss, (int)n, cam,
                            splats, depths);
    return cuda_check(ctx, e, "projection forward launch");
}

int project_backward(gsr_ctx *ctx, const float *gauss, int32_t n, const gsr_camera &camera,
                     const float *dl_dsplat, float *dl_dg, cudaStream_t stream)
{
    const Camera cam = to_camera(camera);
    const dim3 grid((unsigned)projection_grid(ctx, n, kProjBwdBlocksPerSM));
    const bool vec = aligned16(gauss) && aligned16(dl_dsplat) && aligned16(dl_dg);
    const cudaError_t e =
        vec ? launch_kernel(ctx, k_project_backward<true>, grid, dim3(kProjBlock), stream, gauss, (int)n, cam,
                            dl_dsplat, dl_dg)
            : launch_kernel(ctx, k_project_backward<false>, grid, dim3(kProjBlock), stream, gauss, (int)n, cam,
                            dl_dsplat, dl_dg);
    return cuda_check(ctx, e, "projection backward launch");
}

}  // namespace gsr
