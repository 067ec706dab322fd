// Surfel variant of the training step: 2D Gaussian splatting, one of the four rendering pipelines
// Odin trains (Odin: Primitive-Level Synchronization for Distributed Point-Based Neural Rendering,
// Summary). Each Gaussian is a flat disk in 3D, P(u, v) = mean + s_u u t_u + s_v v t_v with t_u, t_v
// the first two columns of its rotation; a pixel weighs it by the disk's Gaussian at the point
// where the pixel's ray meets the disk's plane, or by a screen-space filter of variance 1/2 px^2
// around the disk's bounding-box centre, whichever is larger. Blending, thresholds, termination
// and the backward replay are those of the 3D rasterizer; the binning is the same tile sort.
//
// Record of a projected surfel (16 floats, 64 bytes): the 11 geometric fields
//   A_u = s_u fx (W t_u)_x, B_u = s_u fy (W t_u)_y, C_u = s_u (W t_u)_z, likewise A_v, B_v, C_v,
//   m = projected mean (px), z_c its depth, c = centre of the screen box of the 3-sigma disk,
// then opacity, r, g, b and one unused float. With K the intrinsics and T = [K W s_u t_u |
// K W s_v t_v | K p_c], the pixel (x, y) constrains (u, v) by the planes h_x = T_0 - x T_2 and
// h_y = T_1 - y T_2; written from the record, h_x = (A_u + (cx - x) C_u, A_v + (cx - x) C_v,
// z_c (m_x - x)), which keeps float32 free of the cancellation of T_0 - x T_2 near the mean.
#include <cmath>

#include "gs_common.cuh"
#include "gs_internal.h"
#include "sh.cuh"

namespace gs {

constexpr int kS2 = 16;  // floats per surfel record

// ---- forward-mode dual numbers (float) for the surfel preprocess backward --------------------
template <int NV>
struct Df {
    float v;
    float d[NV];
    __device__ Df() {}
    __device__ Df(float x) : v(x) {
#pragma unroll
        for (int i = 0; i < NV; ++i) d[i] = 0.f;
    }
    __device__ static Df var(float x, int i) {
        Df r(x);
        r.d[i] = 1.f;
        return r;
    }
};
template <int NV> __device__ Df<NV> operator+(const Df<NV>& a, const Df<NV>& b) {
    Df<NV> r(a.v + b.v);
#pragma unroll
    for (int i = 0; i < NV; ++i) r.d[i] = a.d[i] + b.d[i];
    return r;
}
template <int NV> __device__ Df<NV> operator-(const Df<NV>& a, const Df<NV>& b) {
    Df<NV> r(a.v - b.v);
#pragma unroll
    for (int i = 0; i < NV; ++i) r.d[i] = a.d[i] - b.d[i];
    return r;
}
template <int NV> __device__ Df<NV> operator*(const Df<NV>& a, const Df<NV>& b) {
    Df<NV> r(a.v * b.v);
#pragma unroll
    for (int i = 0; i < NV; ++i) r.d[i] = a.d[i] * b.v + a.v * b.d[i];
    return r;
}
template <int NV> __device__ Df<NV> operator/(const Df<NV>& a, const Df<NV>& b) {
    const float ib = 1.f / b.v;
    Df<NV> r(a.v * ib);
#pragma unroll
    for (int i = 0; i < NV; ++i) r.d[i] = (a.d[i] - r.v * b.d[i]) * ib;
    return r;
}
template <int NV> __device__ Df<NV> operator*(float a, const Df<NV>& b) {
    Df<NV> r(a * b.v);
#pragma unroll
    for (int i = 0; i < NV; ++i) r.d[i] = a * b.d[i];
    return r;
}
template <int NV> __device__ Df<NV> operator/(float a, const Df<NV>& b) {
    const float ib = 1.f / b.v;
    Df<NV> r(a * ib);
#pragma unroll
    for (int i = 0; i < NV; ++i) r.d[i] = -r.v * b.d[i] * ib;
    return r;
}
template <int NV> __device__ Df<NV> operator+(const Df<NV>& a, float b) {
    Df<NV> r = a;
    r.v += b;
    return r;
}
template <int NV> __device__ Df<NV> operator-(float a, const Df<NV>& b) {
    Df<NV> r(a - b.v);
#pragma unroll
    for (int i = 0; i < NV; ++i) r.d[i] = -b.d[i];
    return r;
}
template <int NV> __device__ Df<NV> dexp(const Df<NV>& a) {
    Df<NV> r(expf(a.v));
#pragma unroll
    for (int i = 0; i < NV; ++i) r.d[i] = r.v * a.d[i];
    return r;
}
template <int NV> __device__ Df<NV> dsqrt(const Df<NV>& a) {
    Df<NV> r(sqrtf(a.v));
    const float h = 0.5f / r.v;
#pragma unroll
    for (int i = 0; i < NV; ++i) r.d[i] = h * a.d[i];
    return r;
}
__device__ __forceinline__ float dexp(float a) { return expf(a); }
__device__ __forceinline__ float dsqrt(float a) { return sqrtf(a); }
__device__ __forceinline__ float fv(float a) { return a; }
template <int NV> __device__ __forceinline__ float fv(const Df<NV>& a) { return a.v; }

// r . m + t for a row r of the camera rotation; in float the fused chain the depth key uses
__device__ __forceinline__ float row_dot(const float* r, const float m[3], float t) {
    return __fmaf_rn(r[0], m[0], __fmaf_rn(r[1], m[1], __fmaf_rn(r[2], m[2], t)));
}
template <int NV> __device__ Df<NV> row_dot(const float* r, const Df<NV> m[3], float t) {
    return r[0] * m[0] + r[1] * m[1] + r[2] * m[2] + t;
}

// Geometric record of one surfel (fields 0..10) and the half extents of the screen box of its
// 3-sigma disk; false when the mean is behind the near plane or the disk reaches the camera plane.
// The box uses screen coordinates relative to the projected mean, where the dual conic of the disk
// has no cancelling terms: with e = first two entries of T_0 - m_x T_2 (and f for y), the box
// centre is m + (9 e.(C_u, C_v), 9 f.(C_u, C_v)) / c22 and its half width is
// sqrt(c02^2 - c00 c22) / |c22|, c22 = 9 (C_u^2 + C_v^2) - z_c^2 < 0.
template <class S>
__device__ __forceinline__ bool surfel_geometry(const S m[3], const S& lsu, const S& lsv, const S q[4],
                                                const KernelCamera& cam, S rec[11], float half[2]) {
    const float* R = cam.R;
    const S z = row_dot(R + 6, m, cam.t[2]);
    if (!(fv(z) > cam.near_z)) return false;
    const S px = row_dot(R, m, cam.t[0]), py = row_dot(R + 3, m, cam.t[1]);
    const S qn = dsqrt(q[0] * q[0] + q[1] * q[1] + q[2] * q[2] + q[3] * q[3]);
    const S w = q[0] / qn, x = q[1] / qn, y = q[2] / qn, zq = q[3] / qn;
    // first two columns of the rotation of the normalised quaternion
    const S a0 = 1.f - 2.f * (y * y + zq * zq), a1 = 2.f * (x * y + w * zq), a2 = 2.f * (x * zq - w * y);
    const S b0 = 2.f * (x * y - w * zq), b1 = 1.f - 2.f * (x * x + zq * zq), b2 = 2.f * (y * zq + w * x);
    const S su = dexp(lsu), sv = dexp(lsv);
    S wu[3], wv[3];
    for (int i = 0; i < 3; ++i) {
        wu[i] = R[3 * i] * a0 + R[3 * i + 1] * a1 + R[3 * i + 2] * a2;
        wv[i] = R[3 * i] * b0 + R[3 * i + 1] * b1 + R[3 * i + 2] * b2;
    }
    rec[0] = cam.fx * (su * wu[0]);
    rec[1] = cam.fy * (su * wu[1]);
    rec[2] = su * wu[2];
    rec[3] = cam.fx * (sv * wv[0]);
    rec[4] = cam.fy * (sv * wv[1]);
    rec[5] = sv * wv[2];
    const S zi = 1.f / z;
    rec[6] = cam.fx * (px * zi) + cam.cx;
    rec[7] = cam.fy * (py * zi) + cam.cy;
    rec[8] = z;
    const S e0 = rec[0] + (cam.cx - rec[6]) * rec[2], e1 = rec[3] + (cam.cx - rec[6]) * rec[5];
    const S f0 = rec[1] + (cam.cy - rec[7]) * rec[2], f1 = rec[4] + (cam.cy - rec[7]) * rec[5];
    const S c22 = 9.f * (rec[2] * rec[2] + rec[5] * rec[5]) - z * z;
    if (!(fv(c22) < 0.f)) return false;
    const S c02 = 9.f * (e0 * rec[2] + e1 * rec[5]), c12 = 9.f * (f0 * rec[2] + f1 * rec[5]);
    rec[9] = rec[6] + c02 / c22;
    rec[10] = rec[7] + c12 / c22;
    const float c00 = 9.f * (fv(e0) * fv(e0) + fv(e1) * fv(e1)), c11 = 9.f * (fv(f0) * fv(f0) + fv(f1) * fv(f1));
    const float nc22 = -fv(c22);
    half[0] = sqrtf(fv(c02) * fv(c02) + c00 * nc22) / nc22;
    half[1] = sqrtf(fv(c12) * fv(c12) + c11 * nc22) / nc22;
    for (int i = 0; i < 11; ++i)
        if (!isfinite(fv(rec[i]))) return false;
    return isfinite(half[0]) && isfinite(half[1]);
}

// Binning radius: the larger half extent, at least the 3-sigma extent of the screen filter.
__device__ __forceinline__ int surfel_radius(const float half[2]) {
    const float r = ceilf(fmaxf(fmaxf(half[0], half[1]), 3.f * 0.70710678118654752f));
    return r < 16777216.f ? (int)r : 0;
}

template <int DEG>
__global__ void __launch_bounds__(128) k_preprocess2d(int n, const float* __restrict__ mean3d,
                                                      const float* __restrict__ log_scale,
                                                      const float* __restrict__ quat, const float* __restrict__ logit,
                                                      const float* __restrict__ sh, const KernelCamera cam,
                                                      float4* __restrict__ proj_rec, float* __restrict__ depth,
                                                      int* __restrict__ radius, unsigned* __restrict__ tiles_touched,
                                                      float4* __restrict__ rec2d) {
    constexpr int K = (DEG + 1) * (DEG + 1);
    constexpr int K3 = 3 * K;
    __shared__ float tile_all[4][32 * (K3 + 1)];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int warp_first = blockIdx.x * 128 + warp * 32;
    if (warp_first >= n) return;  // whole warp
    const int i = warp_first + lane;
    float m[3] = {0.f, 0.f, 0.f}, rec[11], half[2];
    bool ok = false;
    int r = 0;
    unsigned tt = 0;
    if (i < n) {
        m[0] = mean3d[3 * i]; m[1] = mean3d[3 * i + 1]; m[2] = mean3d[3 * i + 2];
        const float q[4] = {quat[4 * i], quat[4 * i + 1], quat[4 * i + 2], quat[4 * i + 3]};
        depth[i] = row_dot(cam.R + 6, m, cam.t[2]);
        ok = surfel_geometry<float>(m, log_scale[3 * i], log_scale[3 * i + 1], q, cam, rec, half);
        if (ok) {
            r = surfel_radius(half);
            const Rect R = tile_rect(rec[9], rec[10], r, cam.tiles_x, cam.tiles_y);
            ok = r > 0 && R.x0 <= R.x1;
            if (ok) tt = (unsigned)((R.x1 - R.x0 + 1) * (R.y1 - R.y0 + 1));
        }
        if (!ok) {
            const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
            float4* o4 = rec2d + 4 * (size_t)i;
            radius[i] = 0;
            tiles_touched[i] = 0;
            proj_rec[3 * (size_t)i] = z4;
            proj_rec[3 * (size_t)i + 1] = z4;
            proj_rec[3 * (size_t)i + 2] = z4;
            o4[0] = z4; o4[1] = z4; o4[2] = z4; o4[3] = z4;
        }
    }
    // SH coefficients of the warp's visible surfels only, with coalesced loads
    float* tile = tile_all[warp];
    sh_tile_copy<K3, true, false, false>(tile, const_cast<float*>(sh), warp_first, n, lane,
                                         __ballot_sync(0xffffffffu, ok));
    const float lg = ok ? logit[i] : 0.f;
    cp_async_wait_all();
    __syncwarp();
    if (!ok) return;
    const float op = 1.f / (1.f + expf(-lg));
    float dx = m[0] - cam.campos[0], dy = m[1] - cam.campos[1], dz = m[2] - cam.campos[2];
    const float dinv = rsqrtf(dx * dx + dy * dy + dz * dz);
    float Y[16];
    sh_basis<DEG>(dx * dinv, dy * dinv, dz * dinv, Y);
    const float* shg = tile + lane * (K3 + 1);
    float col[3] = {0.5f, 0.5f, 0.5f};
#pragma unroll
    for (int k = 0; k < K; ++k) {
        col[0] += Y[k] * shg[3 * k];
        col[1] += Y[k] * shg[3 * k + 1];
        col[2] += Y[k] * shg[3 * k + 2];
    }
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    proj_rec[3 * (size_t)i] = make_float4(rec[9], rec[10], 0.f, 0.f);  // the binning reads the box centre
    proj_rec[3 * (size_t)i + 1] = z4;
    proj_rec[3 * (size_t)i + 2] = z4;
    radius[i] = r;
    tiles_touched[i] = tt;
    float4* o4 = rec2d + 4 * (size_t)i;
    o4[0] = make_float4(rec[0], rec[1], rec[2], rec[3]);
    o4[1] = make_float4(rec[4], rec[5], rec[6], rec[7]);
    o4[2] = make_float4(rec[8], rec[9], rec[10], op);
    o4[3] = make_float4(fmaxf(col[0], 0.f), fmaxf(col[1], 0.f), fmaxf(col[2], 0.f), 0.f);
}

// ---- render ------------------------------------------------------------------------------------
//
// Plane form. With dx = x - m_x, dy = y - m_y the two planes of a pixel are h_x = (e0 - C_u dx,
// e1 - C_v dx, -z dx) and h_y = (f0 - C_u dy, f1 - C_v dy, -z dy), where (e0, e1) and (f0, f1) are
// the planes' first two entries at the projected mean. Solving them by Cramer's rule, the dx dy
// terms of the 2x2 determinant cancel and the intersection is a projective map of the pixel:
//   (u, v) = z (f1 dx - e1 dy, e0 dy - f0 dx) / det,   det = d0 + dq dx + dp dy,
//   d0 = e0 f1 - e1 f0, dq = C_v f0 - C_u f1, dp = e1 C_u - e0 C_v.
// Each staged record is rewritten once per tile into this form, so that a pixel costs a few
// multiply-adds, one reciprocal and the squares; the same algebra gives the backward its sums
// (see k_render2d_bwd) and k_render2d_grad_fields turns them into record gradients.
//
// Precision. For a surfel seen nearly edge-on the numerators cancel: far from the mean along the
// ellipse's long axis |f1 dx| and |e1 dy| are hundreds of times |f1 dx - e1 dy|, so float32
// coefficients would cost that factor in relative accuracy (1e-5 in alpha on the test scenes).
// The coefficients z (f1, -e1, -f0, e0) are therefore kept as double-floats (head + tail) and each
// numerator is formed with exact products, and d0, dq, dp are formed from unrounded plane entries;
// alpha then agrees with a float64 evaluation of the same record to about 2e-7.

constexpr int kB2 = 128;  // threads per tile (two pixels each) and records per batch
constexpr float kAMin2 = 1.0f / 255.0f, kTMin2 = 1e-4f, kAMax2 = 0.99f;
constexpr float kNegLog2e = -1.4426950408889634f;
// kappa = sqrt(log2(e) / 2): det is stored divided by kappa, so that -(N_u^2 + N_v^2) / det'^2 is
// the disk term in base 2
constexpr float kInvKappa = 1.1774100225154747f;   // 1 / kappa
constexpr float kInvKappa2 = 1.3862943611198906f;  // 1 / kappa^2 = 2 ln 2
constexpr float kInvKappa3 = 1.6322368749392457f;  // 1 / kappa^3

struct Stage2 {
    // record, then the tails of its numerator coefficients; the 80-byte stride makes the
    // per-thread float4 accesses of the rewrite conflict-free (64 bytes would be 4-way)
    float4 rec[2][kB2][5];
    unsigned gidx[2][kB2];
    float4 cull_a[kB2];  // (o_x, o_y, B / C, B / A) of the disk's alpha ellipse (conic A, B, C)
    float4 cull_b[kB2];  // (D / A, L / A) of that ellipse, filter centre (c_x, c_y)
    float cull_tau[kB2]; // squared radius of the filter's alpha disk
    unsigned short list[4][kB2];
    uint64_t bar[2];
};

struct Stage2Bwd {
    Stage2 st;
    unsigned wmax[4];
};

// Double-float values (h + l, |l| <= ulp(h) / 2) for the plane form: the determinants d0, dq, dp
// cancel for surfels seen nearly edge-on, so they are formed from unrounded plane entries
// (Knuth's two-sum, the fused multiply-add exact product) and rounded once.
struct F2 {
    float h, l;
};

__device__ __forceinline__ F2 two_sum(float a, float b) {
    const float s = a + b;
    const float bb = s - a;
    return {s, (a - (s - bb)) + (b - bb)};
}

// a + b c with b a double-float.
__device__ __forceinline__ F2 plane_entry(float a, F2 b, float c) {
    const float ph = b.h * c;
    const float pl = __fmaf_rn(b.h, c, -ph) + b.l * c;
    const F2 t = two_sum(a, ph);
    const float l = t.l + pl;
    const float h = t.h + l;
    return {h, l - (h - t.h)};
}

// x y - z w of double-floats, rounded once up to the tails' second-order terms.
__device__ __forceinline__ float det2(F2 x, F2 y, F2 z, F2 w) {
    const float p = x.h * y.h, q = z.h * w.h;
    const float pe = __fmaf_rn(x.h, y.h, -p), qe = __fmaf_rn(z.h, w.h, -q);
    const float tail = (pe - qe) + (x.h * y.l + x.l * y.h) - (z.h * w.l + z.l * w.h);
    return (p - q) + tail;
}

struct SurfelPlanes {
    F2 e0, e1, f0, f1;
    float d0, dq, dp;
};

// The plane form of a record (fields A_u, B_u, C_u, A_v, B_v, C_v, m_x, m_y), (pcx, pcy) the
// principal point.
__device__ __forceinline__ SurfelPlanes surfel_planes(float Au, float Bu, float Cu, float Av, float Bv, float Cv,
                                                      float mx, float my, float pcx, float pcy) {
    const F2 ax = two_sum(pcx, -mx), ay = two_sum(pcy, -my);
    const F2 e0 = plane_entry(Au, ax, Cu), e1 = plane_entry(Av, ax, Cv);
    const F2 f0 = plane_entry(Bu, ay, Cu), f1 = plane_entry(Bv, ay, Cv);
    const F2 cu = {Cu, 0.f}, cv = {Cv, 0.f};
    SurfelPlanes p;
    p.e0 = e0;
    p.e1 = e1;
    p.f0 = f0;
    p.f1 = f1;
    p.d0 = det2(e0, f1, e1, f0);
    p.dq = det2(cv, f0, cu, f1);
    p.dp = det2(e1, cu, e0, cv);
    return p;
}

// z times a double-float, as a double-float.
__device__ __forceinline__ F2 scale_f2(float z, F2 a) {
    const float p = z * a.h;
    return {p, __fmaf_rn(z, a.h, -p) + z * a.l};
}

// Rewrites a staged record into its evaluation form and fills its culling entries:
//   r[0] = z (f1, -e1, -f0, e0) (heads; tails in r[4]), so that N_u = r[0].x dx + r[0].y dy and
//          N_v = r[0].z dx + r[0].w dy;
//   r[1] = (d0, dq, dp) / kappa and opacity;  r[2] = (m_x, m_y, c_x, c_y);  r[3] = colour, unchanged.
// The disk term in base 2 is then -(N_u^2 + N_v^2) / det'^2 with det' = r[1].x + r[1].y dx + r[1].z dy.
// Culling: alpha >= 1/255 where the disk term reaches -tau (tau = ln(255 opacity)), i.e. inside the
// screen image of the circle u^2 + v^2 <= 2 tau. When that circle lies in front of the camera its
// image is the ellipse (p - o)^T S^-1 (p - o) <= 1 read off the dual conic C* = T diag(2 tau,
// 2 tau, -1) T^T: o = m - (C*_02, C*_12) / n, S = C*_2x2 / n + (o - m)(o - m)^T with n = -C*_22,
// and det S = (d0 2 tau z)^2 / n^3. The filter term reaches -tau inside the disk |p - c|^2 <= tau.
// tau is widened by 0.1 % + 0.001 and the ellipse by 0.2 % so that rounding cannot drop a pair
// the per-pixel test blends; a circle that reaches the camera plane gives no bound (kept).
__device__ __forceinline__ void prepare2d(float4 (&r)[5], float pcx, float pcy, float4& ca, float4& cb, float& ct) {
    const float Au = r[0].x, Bu = r[0].y, Cu = r[0].z, Av = r[0].w, Bv = r[1].x, Cv = r[1].y;
    const float mx = r[1].z, my = r[1].w, z = r[2].x, cx = r[2].y, cy = r[2].z, o = r[2].w;
    const SurfelPlanes p = surfel_planes(Au, Bu, Cu, Av, Bv, Cv, mx, my, pcx, pcy);
    const F2 a1 = scale_f2(z, p.f1), a2 = scale_f2(-z, p.e1), b1 = scale_f2(-z, p.f0), b2 = scale_f2(z, p.e0);
    r[0] = make_float4(a1.h, a2.h, b1.h, b2.h);
    r[4] = make_float4(a1.l, a2.l, b1.l, b2.l);
    r[1] = make_float4(kInvKappa * p.d0, kInvKappa * p.dq, kInvKappa * p.dp, o);
    r[2] = make_float4(mx, my, cx, cy);
    const float e0 = p.e0.h, e1 = p.e1.h, f0 = p.f0.h, f1 = p.f1.h;
    const float inf = __int_as_float(0x7f800000);
    ca = make_float4(mx, my, 0.f, 0.f);
    cb = make_float4(0.f, -1.f, cx, cy);
    ct = -1.f;
    if (!(o * 1.00001f >= kAMin2)) return;  // alpha <= opacity < 1/255: never blended
    // culling values only (they carry margins): fast logarithm and hardware reciprocals
    const float tau = __logf(255.f * o * 1.00001f) * 1.001f + 0.001f;
    ct = tau;
    const float rr = 2.f * tau;
    const float n = __fmaf_rn(-rr, __fmaf_rn(Cu, Cu, Cv * Cv), z * z);
    const float in = rcp_approx(n);
    const float ox = -rr * __fmaf_rn(e0, Cu, e1 * Cv) * in, oy = -rr * __fmaf_rn(f0, Cu, f1 * Cv) * in;
    const float sxx = __fmaf_rn(rr * __fmaf_rn(e0, e0, e1 * e1), in, ox * ox);
    const float sxy = __fmaf_rn(rr * __fmaf_rn(e0, f0, e1 * f1), in, ox * oy);
    const float syy = __fmaf_rn(rr * __fmaf_rn(f0, f0, f1 * f1), in, oy * oy);
    const float t = p.d0 * rr * z * in;
    const float dets = t * t * in;
    const float isyy = rcp_approx(syy);
    const float ra = -sxy * isyy, rc = -sxy * rcp_approx(sxx), da = dets * isyy * isyy, la = dets * isyy * 1.002f;
    if (n > 0.f && dets > 0.f && ra == ra && rc == rc && da < inf && la < inf && fabsf(ox) < inf && fabsf(oy) < inf) {
        ca = make_float4(mx + ox, my + oy, rc, ra);
        cb.x = da;
        cb.y = la;
    } else {
        cb.y = inf;  // no bound on the disk term: every warp keeps the pair
    }
}

__device__ __forceinline__ void stage2_issue(Stage2& s, int slot, const float4* __restrict__ rec,
                                             const unsigned* __restrict__ vals, int first, int n_in, unsigned n_gauss,
                                             unsigned* err) {
    const int t = threadIdx.x;
    if (t < n_in) {
        unsigned g = vals[first + t];
        if (g >= n_gauss) {
            atomicOr(err, kErrCheck);
            g = 0;
        }
        s.gidx[slot][t] = g;
        bulk_copy_g2s(&s.rec[slot][t][0], rec + 4 * (size_t)g, 64u, &s.bar[slot]);
    }
}

// Keeps the staged records whose alpha can reach 1/255 in the warp's 8x8 block: the minimum of the
// ellipse's quadratic form over the block's rectangle of pixel centres (three clamps, as for the
// 3D conic), or the distance from the filter centre to the rectangle.
__device__ __forceinline__ int compact2(Stage2& s, int n_in, int pos_limit, float wx0, float wx1, float wy0, float wy1,
                                        int warp, int lane) {
    int cnt = 0;
    const int lim = min(n_in, pos_limit);
    const float x0 = wx0 - 0.01f, x1 = wx1 + 0.01f, y0 = wy0 - 0.01f, y1 = wy1 + 0.01f;
#pragma unroll
    for (int c = 0; c < kB2 / 32; ++c) {
        const int j = c * 32 + lane;
        bool hit = false;
        if (j < lim) {
            const float4 a = s.cull_a[j], b = s.cull_b[j];
            const float ax = x0 - a.x, bx = x1 - a.x, ay = y0 - a.y, by = y1 - a.y;
            const float cx = fminf(fmaxf(0.f, ax), bx);
            const float dy = fminf(fmaxf(-a.z * cx, ay), by);
            const float dx = fminf(fmaxf(-a.w * dy, ax), bx);
            const float u = __fmaf_rn(a.w, dy, dx);
            const bool disk = !(__fmaf_rn(u, u, b.x * dy * dy) > b.y);  // NaN keeps the pair
            const float qx = fminf(fmaxf(b.z, x0), x1) - b.z, qy = fminf(fmaxf(b.w, y0), y1) - b.w;
            hit = disk || __fmaf_rn(qx, qx, qy * qy) <= s.cull_tau[j];
        }
        const unsigned m = __ballot_sync(0xffffffffu, hit);
        if (hit) s.list[warp][cnt + __popc(m & lanemask_lt())] = (unsigned short)j;
        cnt += __popc(m);
    }
    __syncwarp();
    return cnt;
}

// Parts of a record's evaluation shared by a lane's two pixels (same x): the numerators' dx
// terms as exact head + tail, det's dx part, the base-2 filter term's dx part.
struct Col2 {
    float dx, fx, uh, ut, vh, vt, dex, fxx;
};

__device__ __forceinline__ Col2 column2(const float4& r0, const float4& tl, const float4& r1, const float4& r2,
                                        float x) {
    Col2 c;
    c.dx = x - r2.x;
    c.fx = r2.z - x;
    c.uh = r0.x * c.dx;
    c.ut = __fmaf_rn(tl.x, c.dx, __fmaf_rn(r0.x, c.dx, -c.uh));
    c.vh = r0.z * c.dx;
    c.vt = __fmaf_rn(tl.z, c.dx, __fmaf_rn(r0.z, c.dx, -c.vh));
    c.dex = __fmaf_rn(r1.y, c.dx, r1.x);
    c.fxx = kNegLog2e * c.fx * c.fx;
    return c;
}

// Base-2 exponents of the two terms at one pixel and the intermediates of their derivatives
// (dy = y - m_y, fy = c_y - y).
struct Pix2 {
    float p3, plp, id, nu, nv;
};

__device__ __forceinline__ Pix2 eval2(const float4& r0, const float4& tl, const float4& r1, const Col2& c, float dy,
                                      float fy) {
    Pix2 e;
    e.nu = __fmaf_rn(r0.y, dy, c.uh) + __fmaf_rn(tl.y, dy, c.ut);
    e.nv = __fmaf_rn(r0.w, dy, c.vh) + __fmaf_rn(tl.w, dy, c.vt);
    e.id = rcp_approx(__fmaf_rn(r1.z, dy, c.dex));
    e.p3 = -__fmaf_rn(e.nu, e.nu, e.nv * e.nv) * (e.id * e.id);  // det = 0: -inf, or NaN that fmaxf drops
    e.plp = __fmaf_rn(kNegLog2e * fy, fy, c.fxx);
    return e;
}

__device__ __forceinline__ void blend2(float pw, float o, const float4& col, unsigned pos1, float& T, float& c0,
                                       float& c1, float& c2, unsigned& last, bool& done) {
    const float alpha = fminf(kAMax2, o * ex2_approx(pw));
    if (alpha >= kAMin2) {
        const float test_T = T * (1.f - alpha);
        if (test_T < kTMin2) {
            done = true;
        } else {
            const float w = alpha * T;
            c0 = __fmaf_rn(col.x, w, c0);
            c1 = __fmaf_rn(col.y, w, c1);
            c2 = __fmaf_rn(col.z, w, c2);
            T = test_T;
            last = pos1;
        }
    }
}

// Makes a staged batch usable: plane form and culling entries of every record.
__device__ __forceinline__ void prepare_batch(Stage2& s, int slot, int n_in, const KernelCamera& cam) {
    const int t = threadIdx.x;
    if (t < n_in) prepare2d(s.rec[slot][t], cam.cx, cam.cy, s.cull_a[t], s.cull_b[t], s.cull_tau[t]);
}

__global__ void __launch_bounds__(kB2) k_render2d_fwd(const float4* __restrict__ rec, const unsigned* __restrict__ vals,
                                                      const uint2* __restrict__ ranges, const KernelCamera cam,
                                                      unsigned n_gauss, float* __restrict__ image,
                                                      float* __restrict__ t_final, unsigned* __restrict__ n_contrib,
                                                      unsigned spin_limit, unsigned* __restrict__ err) {
    __shared__ Stage2 s;
    const int tile = blockIdx.x;
    const int tx = tile % cam.tiles_x, ty = tile / cam.tiles_x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bx = tx * kTile + 8 * (warp & 1), by = ty * kTile + 8 * (warp >> 1);
    const int px = bx + (lane & 7), py0 = by + (lane >> 3), py1 = py0 + 4;
    const bool in0 = px < cam.width && py0 < cam.height, in1 = px < cam.width && py1 < cam.height;
    const float fpx = (float)px + 0.5f, fpy0 = (float)py0 + 0.5f, fpy1 = (float)py1 + 0.5f;
    const float wx0 = (float)bx + 0.5f, wx1 = wx0 + 7.f, wy0 = (float)by + 0.5f, wy1 = wy0 + 7.f;
    const uint2 rg = ranges[tile];
    const int start = (int)rg.x;
    const int count = (int)(rg.y > rg.x ? rg.y - rg.x : 0);
    const int nb = (count + kB2 - 1) / kB2;
    float T0 = 1.f, c00 = 0.f, c01 = 0.f, c02 = 0.f, T1 = 1.f, c10 = 0.f, c11 = 0.f, c12 = 0.f;
    unsigned last0 = 0, last1 = 0;
    bool done0 = !in0, done1 = !in1;
    if (nb > 0) {
        if (threadIdx.x == 0) {
            mbar_init(&s.bar[0], 1);
            mbar_init(&s.bar[1], 1);
            fence_mbar_init();
            mbar_arrive_expect_tx(&s.bar[0], (unsigned)min(kB2, count) * 64u);
            if (nb > 1) mbar_arrive_expect_tx(&s.bar[1], (unsigned)min(kB2, count - kB2) * 64u);
        }
        __syncthreads();
        stage2_issue(s, 0, rec, vals, start, min(kB2, count), n_gauss, err);
    }
    int issued = nb > 0 ? 0 : -1, consumed = -1;
    for (int b = 0; b < nb; ++b) {
        const int slot = b & 1;
        const int n_in = min(kB2, count - b * kB2);
        if (b + 1 < nb) {
            stage2_issue(s, slot ^ 1, rec, vals, start + (b + 1) * kB2, min(kB2, count - (b + 1) * kB2), n_gauss, err);
            issued = b + 1;
        }
        const bool ok = mbar_wait_bounded(&s.bar[slot], (unsigned)(b >> 1) & 1u, spin_limit, err);
        if (ok) consumed = b;
        if (ok) prepare_batch(s, slot, n_in, cam);
        if (__syncthreads_or(!ok)) break;
        const int nl = compact2(s, n_in, kB2, wx0, wx1, wy0, wy1, warp, lane);
        for (int k = 0; k < nl; ++k) {
            if (__all_sync(0xffffffffu, done0 && done1)) break;
            const int j = s.list[warp][k];
            const float4 r0 = s.rec[slot][j][0], r1 = s.rec[slot][j][1], r2 = s.rec[slot][j][2];
            const float4 tl = s.rec[slot][j][4];
            const Col2 c = column2(r0, tl, r1, r2, fpx);
            const unsigned pos1 = (unsigned)(b * kB2 + j + 1);
            if (!done0) {
                const Pix2 e = eval2(r0, tl, r1, c, fpy0 - r2.y, r2.w - fpy0);
                blend2(fmaxf(e.p3, e.plp), r1.w, s.rec[slot][j][3], pos1, T0, c00, c01, c02, last0, done0);
            }
            if (!done1) {
                const Pix2 e = eval2(r0, tl, r1, c, fpy1 - r2.y, r2.w - fpy1);
                blend2(fmaxf(e.p3, e.plp), r1.w, s.rec[slot][j][3], pos1, T1, c10, c11, c12, last1, done1);
            }
        }
        if (threadIdx.x == 0 && b + 2 < nb)
            mbar_arrive_expect_tx(&s.bar[slot], (unsigned)min(kB2, count - (b + 2) * kB2) * 64u);
        if (__syncthreads_count(!(done0 && done1)) == 0) break;
    }
    for (int k = consumed + 1; k <= issued; ++k) mbar_wait_bounded(&s.bar[k & 1], (unsigned)(k >> 1) & 1u, 1u << 22, err);
    const size_t plane = (size_t)cam.width * cam.height;
    if (in0) {
        const size_t pix = (size_t)py0 * cam.width + px;
        image[pix] = c00 + T0 * cam.bg[0];
        image[plane + pix] = c01 + T0 * cam.bg[1];
        image[2 * plane + pix] = c02 + T0 * cam.bg[2];
        t_final[pix] = T0;
        n_contrib[pix] = last0;
    }
    if (in1) {
        const size_t pix = (size_t)py1 * cam.width + px;
        image[pix] = c10 + T1 * cam.bg[0];
        image[plane + pix] = c11 + T1 * cam.bg[1];
        image[2 * plane + pix] = c12 + T1 * cam.bg[2];
        t_final[pix] = T1;
        n_contrib[pix] = last1;
    }
}

// One pixel's contribution to a record's 15 backward sums and the step of its backward state.
// Sums (dpow = dL/dpower in natural units, id = 1 / det', tN = dpow N id^2, tdet = dpow p3 id,
// base-2 p3):
//   0..2 tN_u (1, dx, dy), 3..5 tN_v (1, dx, dy), 6..8 tdet (1, dx, dy), 9, 10 dpow (c - x) of the
//   filter term, 11 dL/dopacity, 12..14 dL/dcolour.
__device__ __forceinline__ void add_pixel2(float (&v)[16], const Pix2& e, float dx, float dy, float fx, float fy,
                                           float alpha, float oG, float G, const float4& col, float& T, float& gS,
                                           float g0, float g1, float g2) {
    const float inv = rcp_approx(1.f - alpha);
    T *= inv;
    const float aT = alpha * T;
    v[12] = __fmaf_rn(aT, g0, v[12]);
    v[13] = __fmaf_rn(aT, g1, v[13]);
    v[14] = __fmaf_rn(aT, g2, v[14]);
    const float gc = __fmaf_rn(g0, col.x, __fmaf_rn(g1, col.y, g2 * col.z));
    const float dalpha = __fmaf_rn(T, gc, -inv * gS);
    gS = __fmaf_rn(aT, gc, gS);
    if (!(oG <= kAMax2)) return;
    const float dpow = oG * dalpha;
    v[11] = __fmaf_rn(G, dalpha, v[11]);
    if (!(e.p3 >= e.plp)) {  // the filter term is the larger
        v[9] = __fmaf_rn(dpow, fx, v[9]);
        v[10] = __fmaf_rn(dpow, fy, v[10]);
        return;
    }
    const float w2 = dpow * (e.id * e.id);
    const float tu = w2 * e.nu, tv = w2 * e.nv, td = dpow * e.p3 * e.id;
    v[0] += tu;
    v[1] = __fmaf_rn(tu, dx, v[1]);
    v[2] = __fmaf_rn(tu, dy, v[2]);
    v[3] += tv;
    v[4] = __fmaf_rn(tv, dx, v[4]);
    v[5] = __fmaf_rn(tv, dy, v[5]);
    v[6] += td;
    v[7] = __fmaf_rn(td, dx, v[7]);
    v[8] = __fmaf_rn(td, dy, v[8]);
}

// Transpose reduction of 16 components over the warp: after levels 16, 8, 4, 2 a lane keeps one
// component summed over 16 lanes, and level 1 completes the sum; lanes 2k and 2k + 1 then hold
// component k.
__device__ __forceinline__ float warp_reduce16(const float (&v)[16], int lane) {
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = (b4 ? v[i + 8] : v[i]) + __shfl_xor_sync(0xffffffffu, b4 ? v[i] : v[i + 8], 16);
    float c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = (b3 ? a[i + 4] : a[i]) + __shfl_xor_sync(0xffffffffu, b3 ? a[i] : a[i + 4], 8);
    float d[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) d[i] = (b2 ? c[i + 2] : c[i]) + __shfl_xor_sync(0xffffffffu, b2 ? c[i] : c[i + 2], 4);
    float x = (b1 ? d[1] : d[0]) + __shfl_xor_sync(0xffffffffu, b1 ? d[0] : d[1], 2);
    return x + __shfl_xor_sync(0xffffffffu, x, 1);
}

// Backward replay. Each record's 15 sums (add_pixel2) are accumulated in `grad`; a second kernel
// (k_render2d_grad_fields) turns them into gradients of the record fields.
template <int MODE>
__global__ void __launch_bounds__(kB2) k_render2d_bwd(const float4* __restrict__ rec, const unsigned* __restrict__ vals,
                                                      const uint2* __restrict__ ranges, const KernelCamera cam,
                                                      unsigned n_gauss, const float* __restrict__ dl_dimage,
                                                      const float* __restrict__ t_final,
                                                      const unsigned* __restrict__ n_contrib, float* __restrict__ grad,
                                                      int thr, unsigned spin_limit, unsigned* __restrict__ err) {
    __shared__ Stage2Bwd sm;
    Stage2& s = sm.st;
    const int tile = blockIdx.x;
    const int tx = tile % cam.tiles_x, ty = tile / cam.tiles_x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bx = tx * kTile + 8 * (warp & 1), by = ty * kTile + 8 * (warp >> 1);
    const int px = bx + (lane & 7), py0 = by + (lane >> 3), py1 = py0 + 4;
    const float fpx = (float)px + 0.5f, fpy0 = (float)py0 + 0.5f, fpy1 = (float)py1 + 0.5f;
    const float wx0 = (float)bx + 0.5f, wx1 = wx0 + 7.f, wy0 = (float)by + 0.5f, wy1 = wy0 + 7.f;
    const uint2 rg = ranges[tile];
    const int start = (int)rg.x;
    const int count = (int)(rg.y > rg.x ? rg.y - rg.x : 0);
    const size_t plane = (size_t)cam.width * cam.height;
    unsigned last0 = 0, last1 = 0;
    float T0 = 1.f, T1 = 1.f, a0 = 0.f, a1 = 0.f, a2 = 0.f, b0 = 0.f, b1 = 0.f, b2 = 0.f;
    if (px < cam.width && py0 < cam.height) {
        const size_t pix = (size_t)py0 * cam.width + px;
        last0 = min(n_contrib[pix], (unsigned)count);
        T0 = t_final[pix];
        a0 = dl_dimage[pix]; a1 = dl_dimage[plane + pix]; a2 = dl_dimage[2 * plane + pix];
    }
    if (px < cam.width && py1 < cam.height) {
        const size_t pix = (size_t)py1 * cam.width + px;
        last1 = min(n_contrib[pix], (unsigned)count);
        T1 = t_final[pix];
        b0 = dl_dimage[pix]; b1 = dl_dimage[plane + pix]; b2 = dl_dimage[2 * plane + pix];
    }
    float gS0 = T0 * (a0 * cam.bg[0] + a1 * cam.bg[1] + a2 * cam.bg[2]);
    float gS1 = T1 * (b0 * cam.bg[0] + b1 * cam.bg[1] + b2 * cam.bg[2]);
    const unsigned wmax = __reduce_max_sync(0xffffffffu, max(last0, last1));
    if (lane == 0) sm.wmax[warp] = wmax;
    __syncthreads();
    const unsigned tmax = max(max(sm.wmax[0], sm.wmax[1]), max(sm.wmax[2], sm.wmax[3]));
    const int nb = ((int)tmax + kB2 - 1) / kB2;
    if (nb > 0) {
        const int bl = nb - 1;
        if (threadIdx.x == 0) {
            mbar_init(&s.bar[0], 1);
            mbar_init(&s.bar[1], 1);
            fence_mbar_init();
            mbar_arrive_expect_tx(&s.bar[0], (unsigned)min(kB2, count - bl * kB2) * 64u);
            if (nb > 1) mbar_arrive_expect_tx(&s.bar[1], (unsigned)kB2 * 64u);
        }
        __syncthreads();
        stage2_issue(s, 0, rec, vals, start + bl * kB2, min(kB2, count - bl * kB2), n_gauss, err);
    }
    int issued = nb > 0 ? 0 : -1, consumed = -1;
    for (int it = 0; it < nb; ++it) {
        const int b = nb - 1 - it;
        const int slot = it & 1;
        const int n_in = min(kB2, count - b * kB2);
        if (b > 0) {
            stage2_issue(s, slot ^ 1, rec, vals, start + (b - 1) * kB2, kB2, n_gauss, err);
            issued = it + 1;
        }
        const bool ok = mbar_wait_bounded(&s.bar[slot], (unsigned)(it >> 1) & 1u, spin_limit, err);
        if (ok) consumed = it;
        if (ok) prepare_batch(s, slot, n_in, cam);
        if (__syncthreads_or(!ok)) break;
        const int pos_limit = (int)wmax - b * kB2;
        const int nl = compact2(s, n_in, pos_limit, wx0, wx1, wy0, wy1, warp, lane);
        for (int k = nl - 1; k >= 0; --k) {
            const int j = s.list[warp][k];
            const unsigned pos = (unsigned)(b * kB2 + j);
            const float4 r0 = s.rec[slot][j][0], r1 = s.rec[slot][j][1], r2 = s.rec[slot][j][2];
            const float4 tl = s.rec[slot][j][4];
            const Col2 c = column2(r0, tl, r1, r2, fpx);
            const float dy0 = fpy0 - r2.y, dy1 = fpy1 - r2.y, fy0 = r2.w - fpy0, fy1 = r2.w - fpy1;
            const Pix2 e0 = eval2(r0, tl, r1, c, dy0, fy0);
            const Pix2 e1 = eval2(r0, tl, r1, c, dy1, fy1);
            const float G0 = ex2_approx(fmaxf(e0.p3, e0.plp)), G1 = ex2_approx(fmaxf(e1.p3, e1.plp));
            const float oG0 = r1.w * G0, oG1 = r1.w * G1;
            const float al0 = fminf(kAMax2, oG0), al1 = fminf(kAMax2, oG1);
            const bool c0 = pos < last0 && al0 >= kAMin2;
            const bool c1 = pos < last1 && al1 >= kAMin2;
            const unsigned ballot = __ballot_sync(0xffffffffu, c0 || c1);
            if (ballot == 0u) continue;
            const float4 col = s.rec[slot][j][3];
            float v[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) v[c] = 0.f;
            if (c0) add_pixel2(v, e0, c.dx, dy0, c.fx, fy0, al0, oG0, G0, col, T0, gS0, a0, a1, a2);
            if (c1) add_pixel2(v, e1, c.dx, dy1, c.fx, fy1, al1, oG1, G1, col, T1, gS1, b0, b1, b2);
            float* gp = grad + kS2 * (size_t)s.gidx[slot][j];
            if (MODE == GS_BWD_DIRECT || (MODE == GS_BWD_ADAPTIVE && __popc(ballot) < thr)) {
                if (c0 || c1) {
                    red_add_global_v4(gp, v[0], v[1], v[2], v[3]);
                    red_add_global_v4(gp + 4, v[4], v[5], v[6], v[7]);
                    red_add_global_v4(gp + 8, v[8], v[9], v[10], v[11]);
                    red_add_global_v4(gp + 12, v[12], v[13], v[14], 0.f);
                }
            } else {
                const float x = warp_reduce16(v, lane);
                if ((lane & 1) == 0 && (lane >> 1) < 15) red_add_global(gp + (lane >> 1), x);
            }
        }
        __syncthreads();
        if (threadIdx.x == 0 && b >= 2) mbar_arrive_expect_tx(&s.bar[slot], (unsigned)kB2 * 64u);
        __syncthreads();
    }
    for (int k = consumed + 1; k <= issued; ++k) mbar_wait_bounded(&s.bar[k & 1], (unsigned)(k >> 1) & 1u, 1u << 22, err);
}

// Gradients of the record fields from the backward sums, in place. With the natural-unit sums
// G_N = -t_N / kappa^2 and G_det = -t_det / kappa^3 (t as in add_pixel2), each field's gradient is
// the sum over pixels of its per-pixel derivative through the planes h_x, h_y, which is linear in
// those sums: A_u, A_v, B_u, B_v through the planes' first two entries, C_u, C_v through the same
// entries times (cx - x) and (cy - y), m and z through the third entries z (m - x), z (m - y).
// The m terms use only the N sums (the det parts cancel exactly and are left out). The filter term
// gives dL/dc = -2 sum dpow (c - x).
__global__ void __launch_bounds__(256) k_render2d_grad_fields(unsigned n, const float4* __restrict__ rec,
                                                              float4* __restrict__ grad, float pcx, float pcy) {
    const unsigned i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    float4* g = grad + 4 * (size_t)i;
    const float4 s0 = g[0], s1 = g[1], s2 = g[2];
    if (s0.x == 0.f && s0.y == 0.f && s0.z == 0.f && s0.w == 0.f && s1.x == 0.f && s1.y == 0.f && s1.z == 0.f &&
        s1.w == 0.f && s2.x == 0.f && s2.y == 0.f && s2.z == 0.f)
        return;  // no geometric gradient; opacity and colour are final
    const float4 r0 = rec[4 * (size_t)i], r1 = rec[4 * (size_t)i + 1], r2 = rec[4 * (size_t)i + 2];
    const float Cu = r0.z, Cv = r1.y, mx = r1.z, my = r1.w, z = r2.x;
    const SurfelPlanes p = surfel_planes(r0.x, r0.y, Cu, r0.w, r1.x, Cv, mx, my, pcx, pcy);
    const float gnu = -kInvKappa2 * s0.x, gnu_x = -kInvKappa2 * s0.y, gnu_y = -kInvKappa2 * s0.z;
    const float gnv = -kInvKappa2 * s0.w, gnv_x = -kInvKappa2 * s1.x, gnv_y = -kInvKappa2 * s1.y;
    const float gd = -kInvKappa3 * s1.z, gd_x = -kInvKappa3 * s1.w, gd_y = -kInvKappa3 * s2.x;
    const float e0 = p.e0.h, e1 = p.e1.h, f0 = p.f0.h, f1 = p.f1.h;
    const float gz = f1 * gnu_x - e1 * gnu_y + e0 * gnv_y - f0 * gnv_x;
    const float gf1 = z * gnu_x + e0 * gd - Cu * gd_x;
    const float ge1 = -z * gnu_y - f0 * gd + Cu * gd_y;
    const float ge0 = z * gnv_y + f1 * gd - Cv * gd_y;
    const float gf0 = -z * gnv_x - e1 * gd + Cv * gd_x;
    const float ax = pcx - mx, ay = pcy - my;
    const float gcu = -f1 * gd_x + e1 * gd_y + ax * ge0 + ay * gf0;
    const float gcv = f0 * gd_x - e0 * gd_y + ax * ge1 + ay * gf1;
    const float gmx = z * (Cv * gnu_y - Cu * gnv_y + f0 * gnv - f1 * gnu);
    const float gmy = z * (Cu * gnv_x - Cv * gnu_x + e1 * gnu - e0 * gnv);
    g[0] = make_float4(ge0, gf0, gcu, ge1);
    g[1] = make_float4(gf1, gcv, gmx, gmy);
    g[2] = make_float4(gz, -2.f * s2.y, -2.f * s2.z, s2.w);
}

// ---- preprocess backward -------------------------------------------------------------------------
// The Jacobian of the geometric record with respect to (mean, log-scale u, log-scale v, quaternion)
// by running surfel_geometry on dual numbers; opacity and colour as in the 3D preprocess backward.
template <int DEG>
__global__ void __launch_bounds__(128) k_preprocess2d_bwd(int n, const float* __restrict__ mean3d,
                                                          const float* __restrict__ log_scale,
                                                          const float* __restrict__ quat,
                                                          const float* __restrict__ logit,
                                                          const float* __restrict__ sh, const KernelCamera cam,
                                                          const int* __restrict__ radius,
                                                          const float* __restrict__ grad, float* __restrict__ d_mean3d,
                                                          float* __restrict__ d_log_scale, float* __restrict__ d_quat,
                                                          float* __restrict__ d_logit, float* __restrict__ d_sh,
                                                          int accumulate) {
    constexpr int K = (DEG + 1) * (DEG + 1);
    constexpr int K3 = 3 * K;
    using D = Df<9>;
    __shared__ float tile_all[4][32 * (K3 + 1)];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int warp_first = blockIdx.x * 128 + warp * 32;
    if (warp_first >= n) return;  // whole warp
    const int i = warp_first + lane;
    // only surfels with radius > 0 have non-zero gradients: load their SH rows only. The rows'
    // copies, the parameters and the record gradient are all in flight before the first wait.
    const unsigned seen = __ballot_sync(0xffffffffu, i < n && radius[i] > 0);
    float* tile = tile_all[warp];
    sh_tile_copy<K3, true, false, false>(tile, const_cast<float*>(sh), warp_first, n, lane, seen);
    const bool live = i < n && ((seen >> lane) & 1u);
    float pm[3] = {0.f, 0.f, 0.f}, pq[4] = {1.f, 0.f, 0.f, 0.f}, ls0 = 0.f, ls1 = 0.f, lg = 0.f;
    float4 gi4[4] = {};
    if (live) {
        pm[0] = mean3d[3 * i]; pm[1] = mean3d[3 * i + 1]; pm[2] = mean3d[3 * i + 2];
        pq[0] = quat[4 * i]; pq[1] = quat[4 * i + 1]; pq[2] = quat[4 * i + 2]; pq[3] = quat[4 * i + 3];
        ls0 = log_scale[3 * i];
        ls1 = log_scale[3 * i + 1];
        lg = logit[i];
        const float4* g4 = reinterpret_cast<const float4*>(grad) + 4 * (size_t)i;
        gi4[0] = g4[0]; gi4[1] = g4[1]; gi4[2] = g4[2]; gi4[3] = g4[3];
    }
    cp_async_wait_all();
    __syncwarp();
    float* my = tile + lane * (K3 + 1);  // this thread's coefficients, then its SH gradients
    float gr[9] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float dlg = 0.f;
    if (live) {
        const float gi[16] = {gi4[0].x, gi4[0].y, gi4[0].z, gi4[0].w, gi4[1].x, gi4[1].y, gi4[1].z, gi4[1].w,
                              gi4[2].x, gi4[2].y, gi4[2].z, gi4[2].w, gi4[3].x, gi4[3].y, gi4[3].z, gi4[3].w};
        D m[3], q[4];
        for (int k = 0; k < 3; ++k) m[k] = D::var(pm[k], k);
        const D lsu = D::var(ls0, 3), lsv = D::var(ls1, 4);
        for (int k = 0; k < 4; ++k) q[k] = D::var(pq[k], 5 + k);
        D rec[11];
        float half[2];
        if (surfel_geometry<D>(m, lsu, lsv, q, cam, rec, half)) {
            for (int f = 0; f < 11; ++f) {
                const float gf = gi[f];
#pragma unroll
                for (int v = 0; v < 9; ++v) gr[v] = __fmaf_rn(gf, rec[f].d[v], gr[v]);
            }
        }
        const float op = 1.f / (1.f + expf(-lg));
        dlg = gi[11] * op * (1.f - op);
        // colour = sum_k Y_k sh_k + 0.5 clamped at 0; the direction depends on the mean
        float vx = pm[0] - cam.campos[0], vy = pm[1] - cam.campos[1];
        float vz = pm[2] - cam.campos[2];
        const float vinv = rsqrtf(vx * vx + vy * vy + vz * vz);
        const float ux = vx * vinv, uy = vy * vinv, uz = vz * vinv;
        float Y[16];
        sh_basis<DEG>(ux, uy, uz, Y);
        float col[3] = {0.5f, 0.5f, 0.5f};
#pragma unroll
        for (int k = 0; k < K; ++k)
            for (int c = 0; c < 3; ++c) col[c] += Y[k] * my[3 * k + c];
        float dc[3];
        for (int c = 0; c < 3; ++c) dc[c] = col[c] < 0.f ? 0.f : gi[12 + c];
        float wk[16];
#pragma unroll
        for (int k = 0; k < K; ++k) {
            wk[k] = my[3 * k] * dc[0] + my[3 * k + 1] * dc[1] + my[3 * k + 2] * dc[2];
            for (int c = 0; c < 3; ++c) my[3 * k + c] = Y[k] * dc[c];  // the row now holds dL/dsh
        }
        if (DEG > 0) {
            float gd[3] = {0.f, 0.f, 0.f};
            sh_basis_grad<DEG>(ux, uy, uz, wk, gd);
            const float dot = gd[0] * ux + gd[1] * uy + gd[2] * uz;
            gr[0] += (gd[0] - dot * ux) * vinv;
            gr[1] += (gd[1] - dot * uy) * vinv;
            gr[2] += (gd[2] - dot * uz) * vinv;
        }
    } else if (i < n) {
        for (int k = 0; k < K3; ++k) my[k] = 0.f;
    }
    if (i < n) {
        float* dm = d_mean3d + 3 * (size_t)i;
        float* dl = d_log_scale + 3 * (size_t)i;
        float* dq = d_quat + 4 * (size_t)i;
        if (accumulate) {
            for (int k = 0; k < 3; ++k) dm[k] += gr[k];
            dl[0] += gr[3];
            dl[1] += gr[4];
            for (int k = 0; k < 4; ++k) dq[k] += gr[5 + k];
            d_logit[i] += dlg;
        } else {
            for (int k = 0; k < 3; ++k) dm[k] = gr[k];
            dl[0] = gr[3];
            dl[1] = gr[4];
            dl[2] = 0.f;
            for (int k = 0; k < 4; ++k) dq[k] = gr[5 + k];
            d_logit[i] = dlg;
        }
    }
    __syncwarp();
    // accumulating: rows of surfels with radius 0 add nothing and are skipped
    if (accumulate) sh_tile_copy<K3, false, true>(tile, d_sh, warp_first, n, lane, seen);
    else sh_tile_copy<K3, false, false>(tile, d_sh, warp_first, n, lane, 0xffffffffu);
}

// ---- launchers -------------------------------------------------------------------------------------

cudaError_t launch_preprocess2d(int deg, int n, const gs_params& p, const KernelCamera& cam, const gs_proj& out,
                                float* rec2d, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const int blocks = (n + 127) / 128;
    float4* pr = reinterpret_cast<float4*>(out.rec);
    float4* r2 = reinterpret_cast<float4*>(rec2d);
    unsigned* tt = out.tiles_touched;
    count_launches(1);
    switch (deg) {
        case 0: k_preprocess2d<0><<<blocks, 128, 0, st>>>(n, p.mean3d, p.log_scale, p.quat, p.opacity_logit, p.sh, cam, pr, out.depth, out.radius, tt, r2); break;
        case 1: k_preprocess2d<1><<<blocks, 128, 0, st>>>(n, p.mean3d, p.log_scale, p.quat, p.opacity_logit, p.sh, cam, pr, out.depth, out.radius, tt, r2); break;
        case 2: k_preprocess2d<2><<<blocks, 128, 0, st>>>(n, p.mean3d, p.log_scale, p.quat, p.opacity_logit, p.sh, cam, pr, out.depth, out.radius, tt, r2); break;
        default: k_preprocess2d<3><<<blocks, 128, 0, st>>>(n, p.mean3d, p.log_scale, p.quat, p.opacity_logit, p.sh, cam, pr, out.depth, out.radius, tt, r2); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_render2d_fwd(const float* rec2d, unsigned n, const unsigned* vals, const unsigned* ranges,
                                const KernelCamera& cam, float* image, float* t_final, unsigned* n_contrib,
                                unsigned spin_limit, unsigned* err, cudaStream_t st) {
    const int tiles = cam.tiles_x * cam.tiles_y;
    count_launches(1);
    k_render2d_fwd<<<tiles, kB2, 0, st>>>(reinterpret_cast<const float4*>(rec2d), vals,
                                          reinterpret_cast<const uint2*>(ranges), cam, n, image, t_final, n_contrib,
                                          spin_limit, err);
    return cudaGetLastError();
}

cudaError_t launch_render2d_bwd(int mode, int thr, const float* rec2d, unsigned n, const unsigned* vals,
                                const unsigned* ranges, const KernelCamera& cam, const float* dl_dimage,
                                const float* t_final, const unsigned* n_contrib, float* grad, unsigned spin_limit,
                                unsigned* err, cudaStream_t st) {
    const int tiles = cam.tiles_x * cam.tiles_y;
    const float4* r = reinterpret_cast<const float4*>(rec2d);
    const uint2* rg = reinterpret_cast<const uint2*>(ranges);
    count_launches(1);
    if (mode == GS_BWD_DIRECT)
        k_render2d_bwd<GS_BWD_DIRECT><<<tiles, kB2, 0, st>>>(r, vals, rg, cam, n, dl_dimage, t_final, n_contrib, grad, thr, spin_limit, err);
    else if (mode == GS_BWD_WARP)
        k_render2d_bwd<GS_BWD_WARP><<<tiles, kB2, 0, st>>>(r, vals, rg, cam, n, dl_dimage, t_final, n_contrib, grad, thr, spin_limit, err);
    else
        k_render2d_bwd<GS_BWD_ADAPTIVE><<<tiles, kB2, 0, st>>>(r, vals, rg, cam, n, dl_dimage, t_final, n_contrib, grad, thr, spin_limit, err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || n == 0) return e;
    count_launches(1);
    k_render2d_grad_fields<<<(n + 255) / 256, 256, 0, st>>>(n, r, reinterpret_cast<float4*>(grad), cam.cx, cam.cy);
    return cudaGetLastError();
}

cudaError_t launch_preprocess2d_bwd(int deg, int n, const gs_params& p, const KernelCamera& cam, const int* radius,
                                    const float* grad, float* dm, float* dls, float* dq, float* dlg, float* dsh,
                                    int accumulate, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const int blocks = (n + 127) / 128;
    count_launches(1);
    switch (deg) {
        case 0: k_preprocess2d_bwd<0><<<blocks, 128, 0, st>>>(n, p.mean3d, p.log_scale, p.quat, p.opacity_logit, p.sh, cam, radius, grad, dm, dls, dq, dlg, dsh, accumulate); break;
        case 1: k_preprocess2d_bwd<1><<<blocks, 128, 0, st>>>(n, p.mean3d, p.log_scale, p.quat, p.opacity_logit, p.sh, cam, radius, grad, dm, dls, dq, dlg, dsh, accumulate); break;
        case 2: k_preprocess2d_bwd<2><<<blocks, 128, 0, st>>>(n, p.mean3d, p.log_scale, p.quat, p.opacity_logit, p.sh, cam, radius, grad, dm, dls, dq, dlg, dsh, accumulate); break;
        default: k_preprocess2d_bwd<3><<<blocks, 128, 0, st>>>(n, p.mean3d, p.log_scale, p.quat, p.opacity_logit, p.sh, cam, radius, grad, dm, dls, dq, dlg, dsh, accumulate); break;
    }
    return cudaGetLastError();
}

}  // namespace gs
