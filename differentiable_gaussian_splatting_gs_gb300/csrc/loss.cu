// Image loss of the training step and its gradient, the input of the gradient computation phase
// (Odin: Primitive-Level Synchronization for Distributed Point-Based Neural Rendering, Figure 7:
// rendering R, then backward B). The loss is the 3D Gaussian splatting training loss
// L = (1 - lambda) mean|x - y| + lambda (1 - mean SSIM(x, y)), SSIM per channel with an 11x11
// Gaussian window (sigma 1.5, normalised), constants C1 = 0.01^2 and C2 = 0.03^2, and zero padding
// outside the image.
//
// With mu = w * x, Exx = w * x^2, Exy = w * (x y) (w * . the windowed sum) and the SSIM map
// S = (2 mu_x mu_y + C1)(2 s_xy + C2) / ((mu_x^2 + mu_y^2 + C1)(s_xx + s_yy + C2)), the gradient of
// sum(S) with respect to x is w * dS/dmu_x + 2 x (w * dS/dExx) + y (w * dS/dExy) (w is symmetric,
// so the adjoint of the zero-padded window sum is the same window sum). Pass 1 computes the five
// windowed moments, S and the three partial derivatives per pixel; pass 2 takes their windowed sums.
// Both passes stage a 16x32 tile plus a 5-pixel halo in shared memory and filter rows, then columns.
#include <cmath>

#include "gs_common.cuh"
#include "gs_internal.h"

namespace gs {

constexpr int kLW = 32, kLH = 16, kHalo = 5, kTapN = 11;
constexpr int kInW = kLW + 2 * kHalo, kInH = kLH + 2 * kHalo;

struct LossArgs {
    float w[kTapN];     // window taps
    float c1, c2, lam, inv_n;
    int width, height;
};

__global__ void __launch_bounds__(256) k_ssim_fwd(const LossArgs a, const float* __restrict__ img,
                                                  const float* __restrict__ tgt, float* __restrict__ p_mu,
                                                  float* __restrict__ p_xx, float* __restrict__ p_xy,
                                                  double* __restrict__ sums) {
    __shared__ float sx[kInH][kInW], sy[kInH][kInW];
    __shared__ float hs[5][kInH][kLW];
    __shared__ double red[2][8];
    const int W = a.width, H = a.height;
    const int x0 = blockIdx.x * kLW, y0 = blockIdx.y * kLH, ch = blockIdx.z;
    const size_t plane = (size_t)W * H;
    const float* X = img + ch * plane;
    const float* Y = tgt + ch * plane;
    const int tid = threadIdx.y * blockDim.x + threadIdx.x;
    for (int i = tid; i < kInH * kInW; i += 256) {
        const int r = i / kInW, c = i - r * kInW;
        const int gy = y0 - kHalo + r, gx = x0 - kHalo + c;
        const bool in = gx >= 0 && gx < W && gy >= 0 && gy < H;
        sx[r][c] = in ? X[(size_t)gy * W + gx] : 0.f;
        sy[r][c] = in ? Y[(size_t)gy * W + gx] : 0.f;
    }
    __syncthreads();
    for (int i = tid; i < kInH * kLW; i += 256) {
        const int r = i / kLW, c = i - r * kLW;
        float m0 = 0.f, m1 = 0.f, m2 = 0.f, m3 = 0.f, m4 = 0.f;
#pragma unroll
        for (int k = 0; k < kTapN; ++k) {
            const float u = sx[r][c + k], v = sy[r][c + k], wk = a.w[k];
            m0 = __fmaf_rn(wk, u, m0);
            m1 = __fmaf_rn(wk, v, m1);
            m2 = __fmaf_rn(wk, u * u, m2);
            m3 = __fmaf_rn(wk, v * v, m3);
            m4 = __fmaf_rn(wk, u * v, m4);
        }
        hs[0][r][c] = m0; hs[1][r][c] = m1; hs[2][r][c] = m2; hs[3][r][c] = m3; hs[4][r][c] = m4;
    }
    __syncthreads();
    float l1f = 0.f, ssf = 0.f;
    const int c = threadIdx.x;
    for (int rr = threadIdx.y; rr < kLH; rr += blockDim.y) {
        const int gx = x0 + c, gy = y0 + rr;
        if (gx >= W || gy >= H) continue;
        float mx = 0.f, my = 0.f, exx = 0.f, eyy = 0.f, exy = 0.f;
#pragma unroll
        for (int k = 0; k < kTapN; ++k) {
            const float wk = a.w[k];
            mx = __fmaf_rn(wk, hs[0][rr + k][c], mx);
            my = __fmaf_rn(wk, hs[1][rr + k][c], my);
            exx = __fmaf_rn(wk, hs[2][rr + k][c], exx);
            eyy = __fmaf_rn(wk, hs[3][rr + k][c], eyy);
            exy = __fmaf_rn(wk, hs[4][rr + k][c], exy);
        }
        const float A = __fmaf_rn(2.f * mx, my, a.c1);
        const float B = __fmaf_rn(2.f, exy - mx * my, a.c2);
        const float Cc = __fmaf_rn(mx, mx, __fmaf_rn(my, my, a.c1));
        const float D = (exx - mx * mx) + (eyy - my * my) + a.c2;
        const float iC = __frcp_rn(Cc), iD = __frcp_rn(D);
        const float inv = iC * iD;
        const float S = A * B * inv;
        const size_t o = ch * plane + (size_t)gy * W + gx;
        p_mu[o] = 2.f * my * (B - A) * inv - 2.f * mx * S * (iC - iD);
        p_xx[o] = -S * iD;
        p_xy[o] = 2.f * A * inv;
        l1f += fabsf(sx[rr + kHalo][c + kHalo] - sy[rr + kHalo][c + kHalo]);
        ssf += S;
    }
    double l1 = (double)l1f, ss = (double)ssf;  // at most 2 terms per thread: float is exact enough
    // block sums of |x - y| and S
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        ss += __shfl_xor_sync(0xffffffffu, ss, off);
    }
    const int warp = tid >> 5;
    if ((tid & 31) == 0) {
        red[0][warp] = l1;
        red[1][warp] = ss;
    }
    __syncthreads();
    if (tid == 0) {
        double t0 = 0.0, t1 = 0.0;
        for (int w = 0; w < 8; ++w) {
            t0 += red[0][w];
            t1 += red[1][w];
        }
        atomicAdd(&sums[0], t0);
        atomicAdd(&sums[1], t1);
    }
}

__global__ void __launch_bounds__(256) k_ssim_bwd(const LossArgs a, const float* __restrict__ img,
                                                  const float* __restrict__ tgt, const float* __restrict__ p_mu,
                                                  const float* __restrict__ p_xx, const float* __restrict__ p_xy,
                                                  const double* __restrict__ sums, float* __restrict__ loss,
                                                  float* __restrict__ dl) {
    __shared__ float sp[3][kInH][kInW];
    __shared__ float hs[3][kInH][kLW];
    const int W = a.width, H = a.height;
    const int x0 = blockIdx.x * kLW, y0 = blockIdx.y * kLH, ch = blockIdx.z;
    const size_t plane = (size_t)W * H;
    const int tid = threadIdx.y * blockDim.x + threadIdx.x;
    if (tid == 0 && blockIdx.x == 0 && blockIdx.y == 0 && ch == 0)
        *loss = (float)((1.0 - a.lam) * sums[0] * a.inv_n + a.lam * (1.0 - sums[1] * a.inv_n));
    for (int i = tid; i < kInH * kInW; i += 256) {
        const int r = i / kInW, c = i - r * kInW;
        const int gy = y0 - kHalo + r, gx = x0 - kHalo + c;
        const bool in = gx >= 0 && gx < W && gy >= 0 && gy < H;
        const size_t o = ch * plane + (size_t)gy * W + gx;
        sp[0][r][c] = in ? p_mu[o] : 0.f;
        sp[1][r][c] = in ? p_xx[o] : 0.f;
        sp[2][r][c] = in ? p_xy[o] : 0.f;
    }
    __syncthreads();
    for (int i = tid; i < kInH * kLW; i += 256) {
        const int r = i / kLW, c = i - r * kLW;
        float m0 = 0.f, m1 = 0.f, m2 = 0.f;
#pragma unroll
        for (int k = 0; k < kTapN; ++k) {
            const float wk = a.w[k];
            m0 = __fmaf_rn(wk, sp[0][r][c + k], m0);
            m1 = __fmaf_rn(wk, sp[1][r][c + k], m1);
            m2 = __fmaf_rn(wk, sp[2][r][c + k], m2);
        }
        hs[0][r][c] = m0; hs[1][r][c] = m1; hs[2][r][c] = m2;
    }
    __syncthreads();
    const int c = threadIdx.x;
    for (int rr = threadIdx.y; rr < kLH; rr += blockDim.y) {
        const int gx = x0 + c, gy = y0 + rr;
        if (gx >= W || gy >= H) continue;
        float g0 = 0.f, g1 = 0.f, g2 = 0.f;
#pragma unroll
        for (int k = 0; k < kTapN; ++k) {
            const float wk = a.w[k];
            g0 = __fmaf_rn(wk, hs[0][rr + k][c], g0);
            g1 = __fmaf_rn(wk, hs[1][rr + k][c], g1);
            g2 = __fmaf_rn(wk, hs[2][rr + k][c], g2);
        }
        const size_t o = ch * plane + (size_t)gy * W + gx;
        const float x = img[o], y = tgt[o];
        const float dssim = __fmaf_rn(2.f * x, g1, __fmaf_rn(y, g2, g0));
        const float sgn = x > y ? 1.f : (x < y ? -1.f : 0.f);
        dl[o] = a.inv_n * ((1.f - a.lam) * sgn - a.lam * dssim);
    }
}

size_t loss_workspace_bytes(int width, int height) { return (size_t)3 * 3 * width * height * 4 + 256; }

cudaError_t launch_loss_l1_dssim(const float* img, const float* tgt, int width, int height, float lam, void* ws,
                                 float* loss, float* dl, cudaStream_t st) {
    LossArgs a{};
    double w[kTapN], sum = 0.0;
    for (int k = 0; k < kTapN; ++k) {
        const double d = k - kHalo;
        w[k] = std::exp(-d * d / (2.0 * 1.5 * 1.5));
        sum += w[k];
    }
    for (int k = 0; k < kTapN; ++k) a.w[k] = (float)(w[k] / sum);
    a.c1 = 0.01f * 0.01f;
    a.c2 = 0.03f * 0.03f;
    a.lam = lam;
    a.inv_n = (float)(1.0 / (3.0 * width * height));
    a.width = width;
    a.height = height;
    const size_t plane3 = (size_t)3 * width * height;
    double* sums = reinterpret_cast<double*>(ws);
    float* p_mu = reinterpret_cast<float*>(static_cast<char*>(ws) + 256);
    float* p_xx = p_mu + plane3;
    float* p_xy = p_xx + plane3;
    cudaError_t e = cudaMemsetAsync(sums, 0, 2 * sizeof(double), st);
    if (e) return e;
    const dim3 grid((width + kLW - 1) / kLW, (height + kLH - 1) / kLH, 3), block(32, 8);
    count_launches(2);
    k_ssim_fwd<<<grid, block, 0, st>>>(a, img, tgt, p_mu, p_xx, p_xy, sums);
    k_ssim_bwd<<<grid, block, 0, st>>>(a, img, tgt, p_mu, p_xx, p_xy, sums, loss, dl);
    return cudaGetLastError();
}

}  // namespace gs
