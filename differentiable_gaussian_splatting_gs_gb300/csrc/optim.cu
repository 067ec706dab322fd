// Optimizer update phase: sparse Adam over the Gaussians a view made visible (Odin: Primitive-Level
// Synchronization for Distributed Point-Based Neural Rendering, Figure 7, phase U; Abstract: a view
// updates only the primitives it sees; Review, item 1: Adam).
//
// One launch covers the five parameter tensors. The threads walk the concatenation of the tensors
// in units of four consecutive floats (one 16-byte load of each of parameter, gradient and both
// moments), so every access is a coalesced vector access; a unit whose Gaussians are all hidden
// reads only their radii. Elements of hidden Gaussians inside a partly visible unit are written
// back unchanged.
#include <cmath>

#include "gs_common.cuh"
#include "gs_internal.h"

namespace gs {

struct AdamSegment {
    float *p, *m, *v;
    const float* g;
    long long len;    // floats in the tensor
    long long units;  // ceil(len / 4)
    float lr, lr_rest;  // lr_rest: sh elements after the first 3 (k >= 1)
};

struct AdamArgs {
    AdamSegment seg[5];
    const int* radius;
    float beta1, beta2, one_m_beta1, one_m_beta2, inv_bc1, inv_bc2, eps;
};

__device__ __forceinline__ void adam_elem(float& p, float& m, float& v, float g, float lr, const AdamArgs& a) {
    m = __fmaf_rn(a.beta1, m, a.one_m_beta1 * g);
    v = __fmaf_rn(a.beta2, v, a.one_m_beta2 * g * g);
    // step lr m^ / (sqrt(v^) + eps); the division to 2 ulps (the step's tolerance is far wider)
    p -= __fdividef(lr * (m * a.inv_bc1), sqrtf(v * a.inv_bc2) + a.eps);
}

// Unit r (floats 4r .. 4r + 3) of a tensor with W floats per Gaussian (W a compile-time constant,
// so the Gaussian index is a multiply-shift; units are counted in 32 bits, which the launcher
// guarantees). SH: the sh tensor, whose first 3 floats per Gaussian take lr and the rest lr_rest.
template <int W, bool SH>
__device__ __forceinline__ void adam_unit(const AdamSegment& q, unsigned r, const AdamArgs& a) {
    const unsigned e0 = 4u * r;
    const unsigned len = (unsigned)q.len;
    const int cnt = (int)min(4u, len - e0);
    bool vis[4];
    bool any = false;
    if (W % 4 == 0) {  // the unit lies inside one Gaussian
        const bool v = a.radius[e0 / W] > 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) vis[k] = v;
        any = v;
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            vis[k] = k < cnt && a.radius[(e0 + k) / W] > 0;
            any |= vis[k];
        }
    }
    if (!any) return;
    float p[4], m[4], v[4], g[4];
    if (cnt == 4) {
        const float4 p4 = *reinterpret_cast<const float4*>(q.p + e0), m4 = *reinterpret_cast<const float4*>(q.m + e0);
        const float4 v4 = *reinterpret_cast<const float4*>(q.v + e0), g4 = *reinterpret_cast<const float4*>(q.g + e0);
        p[0] = p4.x; p[1] = p4.y; p[2] = p4.z; p[3] = p4.w;
        m[0] = m4.x; m[1] = m4.y; m[2] = m4.z; m[3] = m4.w;
        v[0] = v4.x; v[1] = v4.y; v[2] = v4.z; v[3] = v4.w;
        g[0] = g4.x; g[1] = g4.y; g[2] = g4.z; g[3] = g4.w;
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            p[k] = k < cnt ? q.p[e0 + k] : 0.f;
            m[k] = k < cnt ? q.m[e0 + k] : 0.f;
            v[k] = k < cnt ? q.v[e0 + k] : 0.f;
            g[k] = k < cnt ? q.g[e0 + k] : 0.f;
        }
    }
    const unsigned col0 = SH ? e0 % W : 0u;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if (!vis[k]) continue;
        const float lr = (SH && col0 + k >= 3u) ? q.lr_rest : q.lr;
        adam_elem(p[k], m[k], v[k], g[k], lr, a);
    }
    if (cnt == 4) {
        *reinterpret_cast<float4*>(q.p + e0) = make_float4(p[0], p[1], p[2], p[3]);
        *reinterpret_cast<float4*>(q.m + e0) = make_float4(m[0], m[1], m[2], m[3]);
        *reinterpret_cast<float4*>(q.v + e0) = make_float4(v[0], v[1], v[2], v[3]);
    } else {
        for (int k = 0; k < cnt; ++k) {
            if (!vis[k]) continue;
            q.p[e0 + k] = p[k];
            q.m[e0 + k] = m[k];
            q.v[e0 + k] = v[k];
        }
    }
}

template <int K3>
__global__ void __launch_bounds__(256) k_adam(const AdamArgs a, unsigned total_units) {
    const unsigned u = blockIdx.x * blockDim.x + threadIdx.x;
    if (u >= total_units) return;
    unsigned r = u;
    int s = 0;
    while (s < 4 && r >= (unsigned)a.seg[s].units) {
        r -= (unsigned)a.seg[s].units;
        ++s;
    }
    switch (s) {
        case 0: adam_unit<3, false>(a.seg[0], r, a); break;
        case 1: adam_unit<3, false>(a.seg[1], r, a); break;
        case 2: adam_unit<4, false>(a.seg[2], r, a); break;
        case 3: adam_unit<1, false>(a.seg[3], r, a); break;
        default: adam_unit<K3, true>(a.seg[4], r, a); break;
    }
}

cudaError_t launch_adam(const gs_tensors& P, const gs_tensors& G, const gs_tensors& M, const gs_tensors& V,
                        const int* radius, const gs_adam_options& o, int deg, float beta1, float beta2, float eps,
                        cudaStream_t st) {
    const long long n = P.n;
    if (n == 0) return cudaSuccess;
    const int K3 = 3 * (deg + 1) * (deg + 1);
    AdamArgs a{};
    const long long widths[5] = {3, 3, 4, 1, K3};
    float* ps[5] = {P.mean3d, P.log_scale, P.quat, P.opacity_logit, P.sh};
    float* ms[5] = {M.mean3d, M.log_scale, M.quat, M.opacity_logit, M.sh};
    float* vs[5] = {V.mean3d, V.log_scale, V.quat, V.opacity_logit, V.sh};
    const float* gs_[5] = {G.mean3d, G.log_scale, G.quat, G.opacity_logit, G.sh};
    const float lrs[5] = {o.lr_mean3d, o.lr_log_scale, o.lr_quat, o.lr_opacity, o.lr_sh_dc};
    long long total = 0;
    for (int s = 0; s < 5; ++s) {
        AdamSegment& q = a.seg[s];
        q.p = ps[s]; q.m = ms[s]; q.v = vs[s]; q.g = gs_[s];
        q.len = n * widths[s];
        q.units = (q.len + 3) / 4;
        q.lr = lrs[s];
        q.lr_rest = s == 4 ? o.lr_sh_rest : lrs[s];
        total += q.units;
    }
    a.radius = radius;
    a.beta1 = beta1;
    a.beta2 = beta2;
    a.one_m_beta1 = (float)(1.0 - (double)beta1);
    a.one_m_beta2 = (float)(1.0 - (double)beta2);
    a.inv_bc1 = (float)(1.0 / (1.0 - std::pow((double)beta1, (double)o.step)));
    a.inv_bc2 = (float)(1.0 / (1.0 - std::pow((double)beta2, (double)o.step)));
    a.eps = eps;
    // element and unit indices are 32-bit: the largest tensor must hold fewer than 2^32 floats
    if (a.seg[4].len >= (1ll << 32) || total >= (1ll << 32)) return cudaErrorInvalidValue;
    count_launches(1);
    const unsigned blocks = (unsigned)((total + 255) / 256);
    const unsigned tu = (unsigned)total;
    switch (deg) {
        case 0: k_adam<3><<<blocks, 256, 0, st>>>(a, tu); break;
        case 1: k_adam<12><<<blocks, 256, 0, st>>>(a, tu); break;
        case 2: k_adam<27><<<blocks, 256, 0, st>>>(a, tu); break;
        default: k_adam<48><<<blocks, 256, 0, st>>>(a, tu); break;
    }
    return cudaGetLastError();
}

}  // namespace gs

namespace gs {

// ---- post-backward statistics ------------------------------------------------------------------
// One thread per Gaussian: the 2D-mean gradient norm, view count and largest radius for
// densification, and optionally the 2-norm of all the Gaussian's parameter gradients.
template <int DEG>
__global__ void __launch_bounds__(256) k_densify_stats(int n, const int* __restrict__ radius,
                                                       const float* __restrict__ grad2d, float sx, float sy,
                                                       float* __restrict__ accum, int* __restrict__ count,
                                                       int* __restrict__ max_radius, gs_tensors pg,
                                                       float* __restrict__ grad_mag) {
    constexpr int K3 = 3 * (DEG + 1) * (DEG + 1);
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int r = radius[i];
    if (r > 0) {
        const float2 g = *reinterpret_cast<const float2*>(grad2d + 12 * (size_t)i);
        const float gx = sx * g.x, gy = sy * g.y;
        accum[i] += sqrtf(__fmaf_rn(gx, gx, gy * gy));
        count[i] += 1;
        max_radius[i] = max(max_radius[i], r);
    }
    if (!grad_mag) return;
    float ss = 0.f;
    if (r > 0) {
        for (int k = 0; k < 3; ++k) {
            const float a = pg.mean3d[3 * (size_t)i + k], b = pg.log_scale[3 * (size_t)i + k];
            ss = __fmaf_rn(a, a, __fmaf_rn(b, b, ss));
        }
        const float4 q = *reinterpret_cast<const float4*>(pg.quat + 4 * (size_t)i);
        ss = __fmaf_rn(q.x, q.x, __fmaf_rn(q.y, q.y, __fmaf_rn(q.z, q.z, __fmaf_rn(q.w, q.w, ss))));
        const float o = pg.opacity_logit[i];
        ss = __fmaf_rn(o, o, ss);
        const float* sh = pg.sh + (size_t)i * K3;
        if (K3 % 4 == 0) {
#pragma unroll
            for (int k = 0; k < K3 / 4; ++k) {
                const float4 c = reinterpret_cast<const float4*>(sh)[k];
                ss = __fmaf_rn(c.x, c.x, __fmaf_rn(c.y, c.y, __fmaf_rn(c.z, c.z, __fmaf_rn(c.w, c.w, ss))));
            }
        } else {
#pragma unroll
            for (int k = 0; k < K3; ++k) ss = __fmaf_rn(sh[k], sh[k], ss);
        }
    }
    grad_mag[i] = sqrtf(ss);
}

cudaError_t launch_densify_stats(int deg, int n, const int* radius, const float* grad2d, float sx, float sy,
                                 float* accum, int* count, int* max_radius, const gs_tensors* pg, float* grad_mag,
                                 cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    gs_tensors t{};
    if (pg) t = *pg;
    float* gm = pg ? grad_mag : nullptr;
    const int blocks = (n + 255) / 256;
    count_launches(1);
    switch (deg) {
        case 0: k_densify_stats<0><<<blocks, 256, 0, st>>>(n, radius, grad2d, sx, sy, accum, count, max_radius, t, gm); break;
        case 1: k_densify_stats<1><<<blocks, 256, 0, st>>>(n, radius, grad2d, sx, sy, accum, count, max_radius, t, gm); break;
        case 2: k_densify_stats<2><<<blocks, 256, 0, st>>>(n, radius, grad2d, sx, sy, accum, count, max_radius, t, gm); break;
        default: k_densify_stats<3><<<blocks, 256, 0, st>>>(n, radius, grad2d, sx, sy, accum, count, max_radius, t, gm); break;
    }
    return cudaGetLastError();
}

}  // namespace gs
