// Preprocessing phase and its backward: one thread per Gaussian.
//
// Forward (3D Gaussian splatting's per-Gaussian preprocessing, the first stage of the
// rasterization pipeline named in DISTWAR: Fast Differentiable Rendering on Raster-based
// Rendering Pipelines, Abstract): view-space position, EWA projection of the 3D covariance to a
// 2D conic, 3-sigma radius and tile rectangle, sigmoid opacity, spherical-harmonic colour.
// Backward: the chain rule of that forward, recomputing its intermediates.
#include <atomic>

#include "gs_common.cuh"
#include "gs_internal.h"
#include "sh.cuh"

namespace gs {

struct Geo {
    float p[3];        // view-space position (p[2] is the float32 depth)
    float qn[4];       // normalised quaternion
    float qinv;        // 1 / |q|
    float Rq[9];       // rotation of the Gaussian
    float s[3];        // scales
    float M3[9];       // Rq diag(s): Sigma = M3 M3^T
    float J00, J02, J11, J12;
    bool clx, cly;     // x/z, y/z were clamped
    float T[6];        // J W, 2x3 row-major
    float K[6];        // T M3, 2x3: the 2D covariance before dilation is K K^T
    float n[3];        // K0 x K1 (rows of K), its components are the 2x2 minors of K
    float a, b, c;     // dilated 2D covariance
    float det;         // a c - b^2
    float A, B, C;     // conic
    float mx, my;
};

// a d - b c with one rounding error (fma-based difference of products)
__device__ __forceinline__ float diff_of_products(float a, float d, float b, float c) {
    const float w = b * c;
    const float e = __fmaf_rn(-b, c, w);
    const float f = __fmaf_rn(a, d, -w);
    return f + e;
}

// Shared forward geometry of one Gaussian; false when it is culled by depth or determinant.
__device__ __forceinline__ bool geometry(const float* m, const float* ls, const float* q,
                                         const KernelCamera& cam, Geo& g) {
    const float* R = cam.R;
    const float* t = cam.t;
    // view-space position; the depth is the fixed fused multiply-add chain used as sort key
    g.p[2] = __fmaf_rn(R[6], m[0], __fmaf_rn(R[7], m[1], __fmaf_rn(R[8], m[2], t[2])));
    if (!(g.p[2] > cam.near_z)) return false;
    g.p[0] = __fmaf_rn(R[0], m[0], __fmaf_rn(R[1], m[1], __fmaf_rn(R[2], m[2], t[0])));
    g.p[1] = __fmaf_rn(R[3], m[0], __fmaf_rn(R[4], m[1], __fmaf_rn(R[5], m[2], t[1])));

    const float qq = q[0] * q[0] + q[1] * q[1] + q[2] * q[2] + q[3] * q[3];
    g.qinv = 1.f / sqrtf(qq);
    const float w = q[0] * g.qinv, x = q[1] * g.qinv, y = q[2] * g.qinv, z = q[3] * g.qinv;
    g.qn[0] = w; g.qn[1] = x; g.qn[2] = y; g.qn[3] = z;
    float* Rq = g.Rq;
    Rq[0] = 1.f - 2.f * (y * y + z * z); Rq[1] = 2.f * (x * y - w * z);       Rq[2] = 2.f * (x * z + w * y);
    Rq[3] = 2.f * (x * y + w * z);       Rq[4] = 1.f - 2.f * (x * x + z * z); Rq[5] = 2.f * (y * z - w * x);
    Rq[6] = 2.f * (x * z - w * y);       Rq[7] = 2.f * (y * z + w * x);       Rq[8] = 1.f - 2.f * (x * x + y * y);
    for (int k = 0; k < 3; ++k) g.s[k] = expf(ls[k]);
    for (int i = 0; i < 3; ++i)
        for (int k = 0; k < 3; ++k) g.M3[3 * i + k] = Rq[3 * i + k] * g.s[k];

    // pinhole Jacobian at p with x/z, y/z clamped to the widened field of view
    const float zi = 1.f / g.p[2];
    float u = g.p[0] * zi, v = g.p[1] * zi;
    g.clx = fabsf(u) > cam.limx;
    g.cly = fabsf(v) > cam.limy;
    if (g.clx) u = copysignf(cam.limx, u);
    if (g.cly) v = copysignf(cam.limy, v);
    g.J00 = cam.fx * zi;
    g.J02 = -cam.fx * u * zi;
    g.J11 = cam.fy * zi;
    g.J12 = -cam.fy * v * zi;
    // T = J W (W = camera rotation), K = T M3
    for (int j = 0; j < 3; ++j) {
        g.T[j] = g.J00 * R[j] + g.J02 * R[6 + j];
        g.T[3 + j] = g.J11 * R[3 + j] + g.J12 * R[6 + j];
    }
    for (int r = 0; r < 2; ++r)
        for (int k = 0; k < 3; ++k)
            g.K[3 * r + k] = g.T[3 * r] * g.M3[k] + g.T[3 * r + 1] * g.M3[3 + k] + g.T[3 * r + 2] * g.M3[6 + k];
    const float* K = g.K;
    const float a0 = K[0] * K[0] + K[1] * K[1] + K[2] * K[2];
    const float c0 = K[3] * K[3] + K[4] * K[4] + K[5] * K[5];
    g.b = K[0] * K[3] + K[1] * K[4] + K[2] * K[5];
    // det(K K^T) as the sum of the squared 2x2 minors of K (Cauchy-Binet): no cancellation
    const float m01 = diff_of_products(K[0], K[4], K[1], K[3]);
    const float m02 = diff_of_products(K[0], K[5], K[2], K[3]);
    const float m12 = diff_of_products(K[1], K[5], K[2], K[4]);
    const float det0 = m01 * m01 + m02 * m02 + m12 * m12;
    g.n[0] = m12; g.n[1] = -m02; g.n[2] = m01;
    const float lp = cam.lowpass;
    g.a = a0 + lp;
    g.c = c0 + lp;
    const float det = det0 + lp * (a0 + c0) + lp * lp;
    g.det = det;
    if (!(det > 0.f)) return false;
    const float di = 1.f / det;
    g.A = g.c * di;
    g.B = -g.b * di;
    g.C = g.a * di;
    g.mx = cam.fx * g.p[0] * zi + cam.cx;
    g.my = cam.fy * g.p[1] * zi + cam.cy;
    return true;
}

constexpr int kFwdThreads = 128;

// SH rows moved by the bulk-copy engine (one copy per Gaussian's row) need rows of a multiple of
// 16 bytes (degrees 1 and 3) and 16-byte aligned arrays; the shared row stride is then an odd
// number of 16-byte chunks, so that each thread's float4 reads of its own row are conflict-free.
// Otherwise the rows move as coalesced 4-byte asynchronous copies into rows of K3 + 1 floats.
template <int K3>
struct ShRows {
    static constexpr bool kBulkable = K3 % 4 == 0;
    static constexpr int bulk_stride = ((K3 / 4) & 1) ? K3 : K3 + 4;
    template <bool BULK>
    static constexpr int stride = BULK ? bulk_stride : K3 + 1;
};

// colour = 0.5 + sum_k Y_k sh_k per channel, k in increasing order (one fused multiply-add per
// term, so both forms round alike), from a thread's row of K3 floats (coefficient-major,
// channel-minor) read as float4 chunks or as floats.
template <int K, bool VEC>
__device__ __forceinline__ void sh_colour(const float* row, const float* Y, float* col) {
    col[0] = col[1] = col[2] = 0.5f;
    if constexpr (VEC) {
        const float4* r4 = reinterpret_cast<const float4*>(row);
#pragma unroll
        for (int j = 0; j < 3 * K / 4; ++j) {
            const float4 v = r4[j];
            const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) col[(4 * j + t) % 3] = __fmaf_rn(Y[(4 * j + t) / 3], e[t], col[(4 * j + t) % 3]);
        }
    } else {
#pragma unroll
        for (int k = 0; k < K; ++k) {
            col[0] = __fmaf_rn(Y[k], row[3 * k], col[0]);
            col[1] = __fmaf_rn(Y[k], row[3 * k + 1], col[1]);
            col[2] = __fmaf_rn(Y[k], row[3 * k + 2], col[2]);
        }
    }
}

// Projection of one Gaussian: geometry, radius and tile rectangle; writes its depth, and zeros for
// its record, radius and tile count when it is culled. Returns whether it is visible.
__device__ __forceinline__ bool project_one(int i, const float* m, const float* ls, const float* q,
                                            const KernelCamera& cam, Geo& g, int& r, unsigned& tt,
                                            float4* __restrict__ rec, float* __restrict__ depth,
                                            int* __restrict__ radius, unsigned* __restrict__ tiles_touched) {
    bool ok = geometry(m, ls, q, cam, g);
    depth[i] = g.p[2];
    r = 0;
    tt = 0;
    if (ok) {
        // largest eigenvalue of the 2D covariance in the cancellation-free form
        const float hd = 0.5f * (g.a - g.c);
        const float lam = 0.5f * (g.a + g.c) + sqrtf(hd * hd + g.b * g.b);
        const float rf = ceilf(3.f * sqrtf(lam));
        ok = isfinite(g.mx) && isfinite(g.my) && rf < 16777216.0f;  // radius < 2^24 px (also rejects NaN)
        if (ok) {
            r = (int)rf;
            const Rect R = tile_rect(g.mx, g.my, r, cam.tiles_x, cam.tiles_y);
            ok = R.x0 <= R.x1;
            if (ok) tt = (unsigned)((R.x1 - R.x0 + 1) * (R.y1 - R.y0 + 1));
        }
    }
    if (!ok) {
        radius[i] = 0;
        tiles_touched[i] = 0;
        const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
        rec[3 * i] = z4;
        rec[3 * i + 1] = z4;
        rec[3 * i + 2] = z4;
    }
    return ok;
}

// Sigmoid opacity and view-dependent colour of a visible Gaussian; writes its record, radius and
// tile count.
template <int DEG, bool VEC>
__device__ __forceinline__ void shade_one(int i, const float* m, const Geo& g, int r, unsigned tt, float lg,
                                          const float* row, const KernelCamera& cam, float4* __restrict__ rec,
                                          int* __restrict__ radius, unsigned* __restrict__ tiles_touched) {
    const float op = 1.f / (1.f + expf(-lg));
    // view direction from the camera centre to the mean
    float dx = m[0] - cam.campos[0], dy = m[1] - cam.campos[1], dz = m[2] - cam.campos[2];
    const float dinv = rsqrtf(dx * dx + dy * dy + dz * dz);
    dx *= dinv; dy *= dinv; dz *= dinv;
    float Y[16];
    sh_basis<DEG>(dx, dy, dz, Y);
    float col[3];
    sh_colour<(DEG + 1) * (DEG + 1), VEC>(row, Y, col);
    rec[3 * i] = make_float4(g.mx, g.my, g.A, g.B);
    rec[3 * i + 1] = make_float4(g.C, op, fmaxf(col[0], 0.f), fmaxf(col[1], 0.f));
    rec[3 * i + 2] = make_float4(fmaxf(col[2], 0.f), 0.f, 0.f, 0.f);
    radius[i] = r;
    tiles_touched[i] = tt;
}

// One thread per Gaussian, SH rows as coalesced 4-byte asynchronous copies (any SH degree and
// alignment).
template <int DEG>
__global__ void __launch_bounds__(kFwdThreads) k_preprocess(int n, const float* __restrict__ mean3d,
                                                            const float* __restrict__ log_scale,
                                                            const float* __restrict__ quat,
                                                            const float* __restrict__ logit,
                                                            const float* __restrict__ sh, const KernelCamera cam,
                                                            float4* __restrict__ rec, float* __restrict__ depth,
                                                            int* __restrict__ radius,
                                                            unsigned* __restrict__ tiles_touched) {
    pdl_entry();
    constexpr int K3 = 3 * (DEG + 1) * (DEG + 1);
    constexpr int S = ShRows<K3>::template stride<false>;
    __shared__ float tile_all[kFwdThreads / 32][32 * S];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int warp_first = blockIdx.x * kFwdThreads + warp * 32;
    if (warp_first >= n) return;  // whole warp
    const int i = warp_first + lane;
    float m[3] = {0.f, 0.f, 0.f};
    Geo g;
    bool ok = false;
    int r = 0;
    unsigned tt = 0;
    if (i < n) {
        m[0] = mean3d[3 * i]; m[1] = mean3d[3 * i + 1]; m[2] = mean3d[3 * i + 2];
        const float ls[3] = {log_scale[3 * i], log_scale[3 * i + 1], log_scale[3 * i + 2]};
        const float q[4] = {quat[4 * i], quat[4 * i + 1], quat[4 * i + 2], quat[4 * i + 3]};
        ok = project_one(i, m, ls, q, cam, g, r, tt, rec, depth, radius, tiles_touched);
    }
    // SH coefficients of the warp's visible Gaussians only, with coalesced loads (the opacity
    // logit is loaded while they are in flight)
    float* tile = tile_all[warp];
    sh_tile_copy<K3, true, false, false>(tile, const_cast<float*>(sh), warp_first, n, lane,
                                         __ballot_sync(0xffffffffu, ok));
    const float lg = ok ? logit[i] : 0.f;
    cp_async_wait_all();
    __syncwarp();
    if (ok) shade_one<DEG, false>(i, m, g, r, tt, lg, tile + lane * S, cam, rec, radius, tiles_touched);
}

// Persistent, pipelined form for bulk SH rows (degrees 1 and 3, 16-byte aligned SH array): each
// warp walks 32-Gaussian groups with a stride of the grid's warp count. A group's SH rows can only
// be requested once its geometry says which Gaussians are visible, so the warp loads the geometry
// of its next group before it waits for the rows of the current one: the two dependent round trips
// of consecutive groups overlap. One bulk copy per visible row, completing on the warp's mbarrier.
template <int DEG>
__global__ void __launch_bounds__(kFwdThreads) k_preprocess_pipe(int n, const float* __restrict__ mean3d,
                                                                 const float* __restrict__ log_scale,
                                                                 const float* __restrict__ quat,
                                                                 const float* __restrict__ logit,
                                                                 const float* __restrict__ sh,
                                                                 const KernelCamera cam, float4* __restrict__ rec,
                                                                 float* __restrict__ depth, int* __restrict__ radius,
                                                                 unsigned* __restrict__ tiles_touched,
                                                                 unsigned spin_limit, unsigned* __restrict__ err) {
    pdl_entry();
    constexpr int K3 = 3 * (DEG + 1) * (DEG + 1);
    static_assert(ShRows<K3>::kBulkable, "bulk SH rows need a multiple of 16 bytes");
    constexpr int S = ShRows<K3>::template stride<true>;
    constexpr int W = kFwdThreads / 32;
    __shared__ __align__(16) float tile_all[W][32 * S];
    __shared__ uint64_t bars[W];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int groups = (n + 31) >> 5;
    const int wstride = gridDim.x * W;
    int grp = blockIdx.x * W + warp;
    if (grp >= groups) return;  // whole warp
    float* tile = tile_all[warp];
    uint64_t* bar = &bars[warp];
    if (lane == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    unsigned parity = 0;
    // the first group's geometry
    float m[3] = {0.f, 0.f, 0.f}, ls[3] = {0.f, 0.f, 0.f}, q[4] = {1.f, 0.f, 0.f, 0.f};
    {
        const int i = grp * 32 + lane;
        if (i < n) {
            m[0] = mean3d[3 * i]; m[1] = mean3d[3 * i + 1]; m[2] = mean3d[3 * i + 2];
            ls[0] = log_scale[3 * i]; ls[1] = log_scale[3 * i + 1]; ls[2] = log_scale[3 * i + 2];
            q[0] = quat[4 * i]; q[1] = quat[4 * i + 1]; q[2] = quat[4 * i + 2]; q[3] = quat[4 * i + 3];
        }
    }
    for (; grp < groups; grp += wstride) {
        const int i = grp * 32 + lane;
        Geo g;
        int r = 0;
        unsigned tt = 0;
        const bool ok = i < n && project_one(i, m, ls, q, cam, g, r, tt, rec, depth, radius, tiles_touched);
        const unsigned vis = __ballot_sync(0xffffffffu, ok);
        if (vis) {
            // the rows of the previous group have been read by every lane (the warp synchronised
            // at the end of the last iteration) before the copies overwrite them
            if (lane == 0) mbar_arrive_expect_tx(bar, (unsigned)(K3 * 4) * __popc(vis));
            __syncwarp();
            if (ok) {
                fence_proxy_async_smem();
                bulk_copy_g2s(tile + lane * S, sh + (size_t)i * K3, K3 * 4, bar);
            }
        }
        const float lg = ok ? logit[i] : 0.f;
        const float mc[3] = {m[0], m[1], m[2]};
        const int nxt = grp + wstride;
        if (nxt < groups) {  // the next group's geometry, in flight while this group's rows land
            const int j = nxt * 32 + lane;
            if (j < n) {
                m[0] = mean3d[3 * j]; m[1] = mean3d[3 * j + 1]; m[2] = mean3d[3 * j + 2];
                ls[0] = log_scale[3 * j]; ls[1] = log_scale[3 * j + 1]; ls[2] = log_scale[3 * j + 2];
                q[0] = quat[4 * j]; q[1] = quat[4 * j + 1]; q[2] = quat[4 * j + 2]; q[3] = quat[4 * j + 3];
            }
        }
        if (vis) {
            if (!mbar_wait_bounded(bar, parity, spin_limit, err)) {
                mbar_wait_bounded(bar, parity, kDrainLimit, err);  // let the copies land, then give up
                return;
            }
            parity ^= 1u;
        }
        if (ok) shade_one<DEG, true>(i, mc, g, r, tt, lg, tile + lane * S, cam, rec, radius, tiles_touched);
        __syncwarp();
    }
}

constexpr int kBwdThreads = 128;

// Gradients of one Gaussian with radius > 0 from its parameters and 2D gradient record (g0..g2):
// dm, dls, dq, dlg, and its SH row `my` (coefficients on entry, read as float4 chunks when VEC)
// overwritten with dL/dsh. False when the recomputed geometry culls it (nothing written then).
template <int DEG, bool VEC>
__device__ __forceinline__ bool grad_one(const float* m, const float* ls, const float* q, float lg, float4 g0,
                                         float4 g1, float4 g2, const KernelCamera& cam, float* my, float* dm,
                                         float* dls, float* dq, float& dlg) {
    constexpr int K = (DEG + 1) * (DEG + 1);
    constexpr int K3 = 3 * K;
    Geo g;
    if (!geometry(m, ls, q, cam, g)) return false;
    const float dmx = g0.x, dmy = g0.y, dA = g0.z, dB = g0.w, dC = g1.x, dop = g1.y;
    const float drgb[3] = {g1.z, g1.w, g2.x};

    // opacity = sigmoid(logit)
    const float op = 1.f / (1.f + expf(-lg));
    dlg = dop * op * (1.f - op);

    // Conic M = Sigma'^-1 with Sigma' = K K^T + lp I. With G = [[dA, dB/2], [dB/2, dC]] (B sits in both
    // off-diagonal slots), dL/dSigma' = -M G M and dL/dK = -2 M G M K. Forming M G M and then
    // multiplying by K cancels catastrophically for elongated Gaussians, so the chain is evaluated as
    //   Y = M K = [lp K0 + K1 x n ; lp K1 - K0 x n] / det    (n = K0 x K1; from a K0 - b K1 expanded with
    //                                                          the vector triple product, no cancellation)
    //   W = G Y,   dL/dK = -2 M W (M applied through the adjugate),
    //   dL/dlog s_k = -2 y_k^T G y_k = -2 (Y0_k W0_k + Y1_k W1_k)   (y_k = column k of Y).
    const float* Kp = g.K;
    const float* nv = g.n;
    const float lp = cam.lowpass, idet = 1.f / g.det;
    float Y0[3], Y1[3];
    {
        const float c0x = diff_of_products(Kp[4], nv[2], Kp[5], nv[1]);  // K1 x n
        const float c0y = diff_of_products(Kp[5], nv[0], Kp[3], nv[2]);
        const float c0z = diff_of_products(Kp[3], nv[1], Kp[4], nv[0]);
        const float c1x = diff_of_products(Kp[1], nv[2], Kp[2], nv[1]);  // K0 x n
        const float c1y = diff_of_products(Kp[2], nv[0], Kp[0], nv[2]);
        const float c1z = diff_of_products(Kp[0], nv[1], Kp[1], nv[0]);
        Y0[0] = (lp * Kp[0] + c0x) * idet; Y0[1] = (lp * Kp[1] + c0y) * idet; Y0[2] = (lp * Kp[2] + c0z) * idet;
        Y1[0] = (lp * Kp[3] - c1x) * idet; Y1[1] = (lp * Kp[4] - c1y) * idet; Y1[2] = (lp * Kp[5] - c1z) * idet;
    }
    const float hb = 0.5f * dB;
    float dK[6];
    for (int j = 0; j < 3; ++j) {
        const float W0 = dA * Y0[j] + hb * Y1[j];
        const float W1 = hb * Y0[j] + dC * Y1[j];
        dK[j] = -2.f * (g.c * W0 - g.b * W1) * idet;
        dK[3 + j] = -2.f * (g.a * W1 - g.b * W0) * idet;
        dls[j] = -2.f * (Y0[j] * W0 + Y1[j] * W1);
    }
    const float* T = g.T;
    const float* M3 = g.M3;
    float dT[6];
    for (int r0 = 0; r0 < 2; ++r0)
        for (int c0 = 0; c0 < 3; ++c0)
            dT[3 * r0 + c0] = dK[3 * r0] * M3[3 * c0] + dK[3 * r0 + 1] * M3[3 * c0 + 1] + dK[3 * r0 + 2] * M3[3 * c0 + 2];
    // T = J W: dJ = dT W^T (only the non-zero entries of J are needed)
    const float* R = cam.R;
    const float dJ00 = dT[0] * R[0] + dT[1] * R[1] + dT[2] * R[2];
    const float dJ02 = dT[0] * R[6] + dT[1] * R[7] + dT[2] * R[8];
    const float dJ11 = dT[3] * R[3] + dT[4] * R[4] + dT[5] * R[5];
    const float dJ12 = dT[3] * R[6] + dT[4] * R[7] + dT[5] * R[8];
    const float zi = 1.f / g.p[2];
    const float zi2 = zi * zi;
    const float u = g.clx ? copysignf(cam.limx, g.p[0]) : g.p[0] * zi;
    const float v = g.cly ? copysignf(cam.limy, g.p[1]) : g.p[1] * zi;
    float dp[3];
    // mean2d = (fx x / z + cx, fy y / z + cy)
    dp[0] = cam.fx * zi * dmx;
    dp[1] = cam.fy * zi * dmy;
    dp[2] = -(cam.fx * g.p[0] * dmx + cam.fy * g.p[1] * dmy) * zi2;
    // J00 = fx / z, J11 = fy / z, J02 = -fx u / z, J12 = -fy v / z with u = x / z unless clamped
    dp[2] -= (cam.fx * dJ00 + cam.fy * dJ11) * zi2;
    dp[2] += (g.clx ? 1.f : 2.f) * cam.fx * u * zi2 * dJ02 + (g.cly ? 1.f : 2.f) * cam.fy * v * zi2 * dJ12;
    if (!g.clx) dp[0] -= cam.fx * zi2 * dJ02;
    if (!g.cly) dp[1] -= cam.fy * zi2 * dJ12;
    // p = W mean + t
    for (int k = 0; k < 3; ++k) dm[k] += R[k] * dp[0] + R[3 + k] * dp[1] + R[6 + k] * dp[2];

    // M3 = Rq diag(s): dL/dM3 = T^T dL/dK, dRq = dL/dM3 diag(s)
    float dRq[9];
    for (int r0 = 0; r0 < 3; ++r0)
        for (int k = 0; k < 3; ++k) dRq[3 * r0 + k] = (T[r0] * dK[k] + T[3 + r0] * dK[3 + k]) * g.s[k];
    // rotation of the normalised quaternion (w, x, y, z)
    const float w = g.qn[0], x = g.qn[1], y = g.qn[2], z = g.qn[3];
    const float* G = dRq;
    float dqn[4];
    dqn[0] = 2.f * (-z * G[1] + y * G[2] + z * G[3] - x * G[5] - y * G[6] + x * G[7]);
    dqn[1] = 2.f * (y * G[1] + z * G[2] + y * G[3] - 2.f * x * G[4] - w * G[5] + z * G[6] + w * G[7] - 2.f * x * G[8]);
    dqn[2] = 2.f * (-2.f * y * G[0] + x * G[1] + w * G[2] + x * G[3] + z * G[5] - w * G[6] + z * G[7] - 2.f * y * G[8]);
    dqn[3] = 2.f * (-2.f * z * G[0] - w * G[1] + x * G[2] + w * G[3] - 2.f * z * G[4] + y * G[5] + x * G[6] + y * G[7]);
    const float dotq = dqn[0] * w + dqn[1] * x + dqn[2] * y + dqn[3] * z;
    for (int k = 0; k < 4; ++k) dq[k] = (dqn[k] - dotq * g.qn[k]) * g.qinv;

    // colour = sum_k Y_k sh_k + 0.5, clamped at 0 (last: the geometry is no longer live here)
    float vx = m[0] - cam.campos[0], vy = m[1] - cam.campos[1], vz = m[2] - cam.campos[2];
    const float vinv = rsqrtf(vx * vx + vy * vy + vz * vz);
    const float ux = vx * vinv, uy = vy * vinv, uz = vz * vinv;
    float Y[16];
    sh_basis<DEG>(ux, uy, uz, Y);
    float col[3];
    sh_colour<K, VEC>(my, Y, col);
    float dc[3];
    for (int ch = 0; ch < 3; ++ch) dc[ch] = (col[ch] < 0.f) ? 0.f : drgb[ch];
    // w_k = sum_c sh_kc dc_c (c in increasing order, fused multiply-adds), and the row now holds
    // dL/dsh_kc = Y_k dc_c
    float wk[16];
    if constexpr (VEC) {
        float4* r4 = reinterpret_cast<float4*>(my);
#pragma unroll
        for (int j = 0; j < K3 / 4; ++j) {
            const float4 v = r4[j];
            const float e[4] = {v.x, v.y, v.z, v.w};
            float o[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int f = 4 * j + t, k = f / 3, c = f % 3;
                wk[k] = c == 0 ? e[t] * dc[0] : __fmaf_rn(e[t], dc[c], wk[k]);
                o[t] = Y[k] * dc[c];
            }
            r4[j] = make_float4(o[0], o[1], o[2], o[3]);
        }
    } else {
#pragma unroll
        for (int k = 0; k < K; ++k) {
            wk[k] = __fmaf_rn(my[3 * k + 2], dc[2], __fmaf_rn(my[3 * k + 1], dc[1], my[3 * k] * dc[0]));
            my[3 * k] = Y[k] * dc[0];
            my[3 * k + 1] = Y[k] * dc[1];
            my[3 * k + 2] = Y[k] * dc[2];
        }
    }
    if (DEG > 0) {
        float gd[3] = {0.f, 0.f, 0.f};
        sh_basis_grad<DEG>(ux, uy, uz, wk, gd);
        // through the normalisation: (I - u u^T) / |v|
        const float dot = gd[0] * ux + gd[1] * uy + gd[2] * uz;
        dm[0] += (gd[0] - dot * ux) * vinv;
        dm[1] += (gd[1] - dot * uy) * vinv;
        dm[2] += (gd[2] - dot * uz) * vinv;
    }

    return true;
}

// Statistics (when stats.accum is set) and the parameter gradients of Gaussian i (radius rad; `my`
// holds its SH gradients) written or, when accumulating, added to the outputs; the SH row is stored
// by the caller. The statistics are a run-time choice, so that the gradients come from the same
// machine code with and without them (bit-identical results).
template <int K3, bool VEC>
__device__ __forceinline__ void finish_one(int i, int rad, float4 g0, const float* dm, const float* dls,
                                           const float* dq, float dlg, const float* my, const DensifyArgs& stats,
                                           int accumulate, float* __restrict__ d_mean3d,
                                           float* __restrict__ d_log_scale, float* __restrict__ d_quat,
                                           float* __restrict__ d_logit) {
    if (stats.accum) {
    // 3D Gaussian splatting's densification statistics and the 2-norm of this view's parameter
    // gradients (the tile row holds this view's SH gradients), as gs_densify_stats computes them
    if (rad > 0) {
        const float gx = stats.sx * g0.x, gy = stats.sy * g0.y;
        stats.accum[i] += sqrtf(__fmaf_rn(gx, gx, gy * gy));
        stats.count[i] += 1;
        stats.max_radius[i] = max(stats.max_radius[i], rad);
    }
    if (stats.grad_mag) {
        float ss = 0.f;
        if (rad > 0) {  // the summation order of gs_densify_stats
            for (int k = 0; k < 3; ++k) ss = __fmaf_rn(dm[k], dm[k], __fmaf_rn(dls[k], dls[k], ss));
            ss = __fmaf_rn(dq[0], dq[0], __fmaf_rn(dq[1], dq[1], __fmaf_rn(dq[2], dq[2], __fmaf_rn(dq[3], dq[3], ss))));
            ss = __fmaf_rn(dlg, dlg, ss);
            if constexpr (K3 % 4 == 0) {
                for (int k = 0; k < K3; k += 4) {
                    const float4 v = VEC ? reinterpret_cast<const float4*>(my)[k / 4]
                                          : make_float4(my[k], my[k + 1], my[k + 2], my[k + 3]);
                    ss = __fmaf_rn(v.x, v.x, __fmaf_rn(v.y, v.y, __fmaf_rn(v.z, v.z, __fmaf_rn(v.w, v.w, ss))));
                }
            } else {
                for (int k = 0; k < K3; ++k) ss = __fmaf_rn(my[k], my[k], ss);
            }
        }
        stats.grad_mag[i] = sqrtf(ss);
    }
    }
    if (accumulate) {
        for (int k = 0; k < 3; ++k) { d_mean3d[3 * i + k] += dm[k]; d_log_scale[3 * i + k] += dls[k]; }
        for (int k = 0; k < 4; ++k) d_quat[4 * i + k] += dq[k];
        d_logit[i] += dlg;
    } else {
        for (int k = 0; k < 3; ++k) { d_mean3d[3 * i + k] = dm[k]; d_log_scale[3 * i + k] = dls[k]; }
        for (int k = 0; k < 4; ++k) d_quat[4 * i + k] = dq[k];
        d_logit[i] = dlg;
    }
}

// One thread per Gaussian, SH rows by coalesced 4-byte asynchronous copies (any SH degree and
// alignment). With stats.accum set, also the post-backward statistics of the view (see
// DensifyArgs), from the gradients this call computes.
template <int DEG>
__global__ void __launch_bounds__(kBwdThreads, 5) k_preprocess_bwd(
    int n, const float* __restrict__ mean3d, const float* __restrict__ log_scale,
    const float* __restrict__ quat, const float* __restrict__ logit, const float* __restrict__ sh,
    const KernelCamera cam, const int* __restrict__ radius, const float4* __restrict__ grad2d,
    float* __restrict__ d_mean3d, float* __restrict__ d_log_scale, float* __restrict__ d_quat,
    float* __restrict__ d_logit, float* __restrict__ d_sh, int accumulate, const DensifyArgs stats) {
    pdl_entry();
    constexpr int K3 = 3 * (DEG + 1) * (DEG + 1);
    constexpr int S = ShRows<K3>::template stride<false>;
    __shared__ float tile_all[kBwdThreads / 32][32 * S];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float* tile = tile_all[warp];
    const int warp_first = blockIdx.x * kBwdThreads + warp * 32;
    const int i = warp_first + lane;
    // only Gaussians with radius > 0 have non-zero gradients: load their SH rows only. The rows'
    // copies, the geometry and the 2D gradients are all in flight before the first wait.
    const int rad = i < n ? radius[i] : 0;
    const unsigned seen = __ballot_sync(0xffffffffu, rad > 0);
    sh_tile_copy<K3, true, false, false>(tile, const_cast<float*>(sh), warp_first, n, lane, seen);
    float* my = tile + lane * S;   // this thread's coefficients, then its SH gradients
    float m[3] = {0.f, 0.f, 0.f}, ls[3] = {0.f, 0.f, 0.f}, q[4] = {1.f, 0.f, 0.f, 0.f}, lg = 0.f;
    float4 g0 = make_float4(0.f, 0.f, 0.f, 0.f), g1 = g0, g2 = g0;
    if (rad > 0) {
        m[0] = mean3d[3 * i]; m[1] = mean3d[3 * i + 1]; m[2] = mean3d[3 * i + 2];
        ls[0] = log_scale[3 * i]; ls[1] = log_scale[3 * i + 1]; ls[2] = log_scale[3 * i + 2];
        q[0] = quat[4 * i]; q[1] = quat[4 * i + 1]; q[2] = quat[4 * i + 2]; q[3] = quat[4 * i + 3];
        g0 = grad2d[3 * i]; g1 = grad2d[3 * i + 1]; g2 = grad2d[3 * i + 2];
        lg = logit[i];
    }
    cp_async_wait_all();
    __syncwarp();
    if (i < n) {
        float dm[3] = {0.f, 0.f, 0.f}, dls[3] = {0.f, 0.f, 0.f}, dq[4] = {0.f, 0.f, 0.f, 0.f}, dlg = 0.f;
        if (!(rad > 0 && grad_one<DEG, false>(m, ls, q, lg, g0, g1, g2, cam, my, dm, dls, dq, dlg)))
            for (int k = 0; k < K3; ++k) my[k] = 0.f;
        finish_one<K3, false>(i, rad, g0, dm, dls, dq, dlg, my, stats, accumulate, d_mean3d, d_log_scale,
                                     d_quat, d_logit);
    }
    __syncwarp();
    // accumulating: rows of Gaussians with radius 0 add nothing and are skipped
    if (accumulate) sh_tile_copy<K3, false, true>(tile, d_sh, warp_first, n, lane, seen);
    else sh_tile_copy<K3, false, false>(tile, d_sh, warp_first, n, lane, 0xffffffffu);
}

// Persistent, pipelined form for bulk SH rows (degrees 1 and 3, sh and d_sh 16-byte aligned): each
// warp walks 32-Gaussian groups with a stride of the grid's warp count. It loads the radii of its
// next group before waiting for the current group's rows, and each group's gradient rows leave by
// bulk copies (bulk additions when accumulating) that complete while the warp goes on; a lane
// refills its row only after its own copy out of it has read it.
template <int DEG>
__global__ void __launch_bounds__(kBwdThreads, 5) k_preprocess_bwd_pipe(
    int n, const float* __restrict__ mean3d, const float* __restrict__ log_scale,
    const float* __restrict__ quat, const float* __restrict__ logit, const float* __restrict__ sh,
    const KernelCamera cam, const int* __restrict__ radius, const float4* __restrict__ grad2d,
    float* __restrict__ d_mean3d, float* __restrict__ d_log_scale, float* __restrict__ d_quat,
    float* __restrict__ d_logit, float* __restrict__ d_sh, int accumulate, const DensifyArgs stats,
    unsigned spin_limit, unsigned* __restrict__ err) {
    pdl_entry();
    constexpr int K3 = 3 * (DEG + 1) * (DEG + 1);
    static_assert(ShRows<K3>::kBulkable, "bulk SH rows need a multiple of 16 bytes");
    constexpr int S = ShRows<K3>::template stride<true>;
    constexpr int W = kBwdThreads / 32;
    __shared__ __align__(16) float tile_all[W][32 * S];
    __shared__ uint64_t bars[W];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int groups = (n + 31) >> 5;
    const int wstride = gridDim.x * W;
    int grp = blockIdx.x * W + warp;
    if (grp >= groups) return;  // whole warp
    float* my = tile_all[warp] + lane * S;   // this thread's coefficients, then its SH gradients
    uint64_t* bar = &bars[warp];
    if (lane == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    unsigned parity = 0;
    int rad = grp * 32 + lane < n ? radius[grp * 32 + lane] : 0;
    for (; grp < groups; grp += wstride) {
        const int i = grp * 32 + lane;
        // only Gaussians with radius > 0 have non-zero gradients: load their SH rows only, with
        // their geometry and 2D gradients in flight at the same time
        const unsigned seen = __ballot_sync(0xffffffffu, rad > 0);
        bulk_wait_read();  // the previous group's copy out of this row has read it
        if (seen) {
            if (lane == 0) mbar_arrive_expect_tx(bar, (unsigned)(K3 * 4) * __popc(seen));
            __syncwarp();
            if (rad > 0) bulk_copy_g2s(my, sh + (size_t)i * K3, K3 * 4, bar);
        }
        float m[3] = {0.f, 0.f, 0.f}, ls[3] = {0.f, 0.f, 0.f}, q[4] = {1.f, 0.f, 0.f, 0.f}, lg = 0.f;
        float4 g0 = make_float4(0.f, 0.f, 0.f, 0.f), g1 = g0, g2 = g0;
        if (rad > 0) {
            m[0] = mean3d[3 * i]; m[1] = mean3d[3 * i + 1]; m[2] = mean3d[3 * i + 2];
            ls[0] = log_scale[3 * i]; ls[1] = log_scale[3 * i + 1]; ls[2] = log_scale[3 * i + 2];
            q[0] = quat[4 * i]; q[1] = quat[4 * i + 1]; q[2] = quat[4 * i + 2]; q[3] = quat[4 * i + 3];
            g0 = grad2d[3 * i]; g1 = grad2d[3 * i + 1]; g2 = grad2d[3 * i + 2];
            lg = logit[i];
        }
        const int nxt = grp + wstride, j = nxt * 32 + lane;
        const int rad_next = nxt < groups && j < n ? radius[j] : 0;
        if (seen) {
            if (!mbar_wait_bounded(bar, parity, spin_limit, err)) {
                mbar_wait_bounded(bar, parity, kDrainLimit, err);  // let the copies land, then give up
                return;
            }
            parity ^= 1u;
        }
        if (i < n) {
            float dm[3] = {0.f, 0.f, 0.f}, dls[3] = {0.f, 0.f, 0.f}, dq[4] = {0.f, 0.f, 0.f, 0.f}, dlg = 0.f;
            if (!(rad > 0 && grad_one<DEG, true>(m, ls, q, lg, g0, g1, g2, cam, my, dm, dls, dq, dlg)))
                for (int k = 0; k < K3 / 4; ++k) reinterpret_cast<float4*>(my)[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            finish_one<K3, true>(i, rad, g0, dm, dls, dq, dlg, my, stats, accumulate, d_mean3d, d_log_scale,
                                        d_quat, d_logit);
            // accumulating: rows of Gaussians with radius 0 add nothing and are skipped
            if (!accumulate || rad > 0) {
                fence_proxy_async_smem();
                if (accumulate) bulk_add_s2g(d_sh + (size_t)i * K3, my, K3 * 4);
                else bulk_copy_s2g(d_sh + (size_t)i * K3, my, K3 * 4);
            }
        }
        rad = rad_next;
    }
    bulk_wait_read();  // every copy out of shared memory has read it before the block exits
}

// ---- host-side launchers ------------------------------------------------------------------------

namespace {
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

cudaError_t launch_preprocess(int deg, int n, const gs_params& p, const KernelCamera& cam, const gs_proj& out,
                              unsigned spin_limit, unsigned* err, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const int blocks = (n + kFwdThreads - 1) / kFwdThreads;
    float4* rec = reinterpret_cast<float4*>(out.rec);
    unsigned* tt = out.tiles_touched;
    count_launches(1);
    if ((deg == 1 || deg == 3) && aligned16(p.sh)) {
        static std::atomic<int> cache1[256], cache3[256];
        auto k = deg == 1 ? k_preprocess_pipe<1> : k_preprocess_pipe<3>;
        const int res = resident_blocks(k, kFwdThreads, 0, deg == 1 ? cache1 : cache3);
        const int grid = res > 0 && res < blocks ? res : blocks;
        return launch_pdl(k, dim3(grid), dim3(kFwdThreads), 0, st, n, p.mean3d, p.log_scale, p.quat,
                          p.opacity_logit, p.sh, cam, rec, out.depth, out.radius, tt, spin_limit, err);
    }
    void (*k)(int, const float*, const float*, const float*, const float*, const float*, const KernelCamera, float4*,
              float*, int*, unsigned*) = deg == 0 ? k_preprocess<0> : deg == 1 ? k_preprocess<1>
                                                : deg == 2 ? k_preprocess<2> : k_preprocess<3>;
    return launch_pdl(k, dim3(blocks), dim3(kFwdThreads), 0, st, n, p.mean3d, p.log_scale, p.quat, p.opacity_logit,
                      p.sh, cam, rec, out.depth, out.radius, tt);
}

template <int DEG>
cudaError_t launch_bwd_pipe(int n, const gs_params& p, const KernelCamera& cam, const int* radius, const float4* g2,
                            float* dm, float* dls, float* dq, float* dlg, float* dsh, int accumulate,
                            const DensifyArgs& stats, unsigned spin_limit, unsigned* err, cudaStream_t st) {
    static std::atomic<int> cache[256];
    const int blocks = (n + kBwdThreads - 1) / kBwdThreads;
    const int res = resident_blocks(k_preprocess_bwd_pipe<DEG>, kBwdThreads, 0, cache);
    return launch_pdl(k_preprocess_bwd_pipe<DEG>, dim3(res > 0 && res < blocks ? res : blocks), dim3(kBwdThreads), 0,
                      st, n, p.mean3d, p.log_scale, p.quat, p.opacity_logit, p.sh, cam, radius, g2, dm, dls, dq, dlg,
                      dsh, accumulate, stats, spin_limit, err);
}

template <int DEG>
cudaError_t launch_bwd_plain(int n, const gs_params& p, const KernelCamera& cam, const int* radius, const float4* g2,
                             float* dm, float* dls, float* dq, float* dlg, float* dsh, int accumulate,
                             const DensifyArgs& stats, cudaStream_t st) {
    return launch_pdl(k_preprocess_bwd<DEG>, dim3((n + kBwdThreads - 1) / kBwdThreads), dim3(kBwdThreads), 0, st, n,
                      p.mean3d, p.log_scale, p.quat, p.opacity_logit, p.sh, cam, radius, g2, dm, dls, dq, dlg, dsh,
                      accumulate, stats);
}

cudaError_t launch_preprocess_bwd(int deg, int n, const gs_params& p, const KernelCamera& cam, const int* radius,
                                  const float* grad2d, float* dm, float* dls, float* dq, float* dlg, float* dsh,
                                  int accumulate, const DensifyArgs* stats, unsigned spin_limit, unsigned* err,
                                  cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const float4* g2 = reinterpret_cast<const float4*>(grad2d);
    const DensifyArgs none{};
    const DensifyArgs& sa = stats ? *stats : none;   // none.accum == nullptr: no statistics
    count_launches(1);
    if ((deg == 1 || deg == 3) && aligned16(p.sh) && aligned16(dsh))
        return deg == 1 ? launch_bwd_pipe<1>(n, p, cam, radius, g2, dm, dls, dq, dlg, dsh, accumulate, sa, spin_limit,
                                             err, st)
                        : launch_bwd_pipe<3>(n, p, cam, radius, g2, dm, dls, dq, dlg, dsh, accumulate, sa, spin_limit,
                                             err, st);
    switch (deg) {
        case 0: return launch_bwd_plain<0>(n, p, cam, radius, g2, dm, dls, dq, dlg, dsh, accumulate, sa, st);
        case 1: return launch_bwd_plain<1>(n, p, cam, radius, g2, dm, dls, dq, dlg, dsh, accumulate, sa, st);
        case 2: return launch_bwd_plain<2>(n, p, cam, radius, g2, dm, dls, dq, dlg, dsh, accumulate, sa, st);
        default: return launch_bwd_plain<3>(n, p, cam, radius, g2, dm, dls, dq, dlg, dsh, accumulate, sa, st);
    }
}

}  // namespace gs
