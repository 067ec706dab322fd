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
// Both passes stage a 128x34 tile plus a 5-pixel halo in shared memory.
#include <cmath>

#include "gs_common.cuh"
#include "gs_internal.h"

namespace gs {

// Tiles of kLW columns x kLH output rows, one column per thread. A thread takes the horizontal
// 11-tap sums of its column for each of the kLH + 10 input rows of the tile and adds each into
// the vertical sums of the 11 output rows it reaches, kept in an 11-slot ring of registers (input
// row r adds w[t] x its sums to output row r - t); with the row loop unrolled by 11 every ring
// index is a constant. Output row o is complete after input row o + 10.
constexpr int kLW = 128, kLH = 34, kHalo = 5, kTapN = 11;
constexpr int kInW = kLW + 2 * kHalo, kInH = kLH + 2 * kHalo;  // kInH = 44 = 4 x 11
static_assert(kInH % kTapN == 0, "the input rows of a tile are a multiple of the window");

struct LossArgs {
    float w[kTapN];     // window taps
    float c1, c2, lam, inv_n;
    int width, height;
};

// Stages NM maps of the tile (rows y0 - 5 .., columns x0 - 5 ..) with zeros outside the image:
// asynchronous copies, all in flight at once, waited for before returning (the caller then
// synchronises the block).
template <int NM>
__device__ __forceinline__ void stage_tile(float (*sm)[kInH][kInW], const float* const (&src)[NM], int x0, int y0,
                                           int W, int H) {
    for (int i = threadIdx.x; i < kInH * kInW; i += kLW) {
        const int r = i / kInW, c = i - r * kInW;
        const int gy = y0 - kHalo + r, gx = x0 - kHalo + c;
        const bool in = gx >= 0 && gx < W && gy >= 0 && gy < H;
#pragma unroll
        for (int m = 0; m < NM; ++m) {
            if (in) cp_async4(&sm[m][r][c], src[m] + (size_t)gy * W + gx);
            else sm[m][r][c] = 0.f;
        }
    }
    cp_async_wait_all();
}

__global__ void __launch_bounds__(kLW) k_ssim_fwd(const LossArgs a, const float* __restrict__ img,
                                                  const float* __restrict__ tgt, float* __restrict__ p_mu,
                                                  float* __restrict__ p_xx, float* __restrict__ p_xy,
                                                  double* __restrict__ sums) {
    extern __shared__ float smem_loss[];
    float (*sm)[kInH][kInW] = reinterpret_cast<float (*)[kInH][kInW]>(smem_loss);  // x, y
    __shared__ double red[2][kLW / 32];
    const int W = a.width, H = a.height;
    const int x0 = blockIdx.x * kLW, y0 = blockIdx.y * kLH, ch = blockIdx.z;
    const size_t plane = (size_t)W * H;
    const float* const src[2] = {img + ch * plane, tgt + ch * plane};
    stage_tile<2>(sm, src, x0, y0, W, H);
    __syncthreads();
    const int c = threadIdx.x, gx = x0 + c;
    float acc[kTapN][5];
#pragma unroll
    for (int s2 = 0; s2 < kTapN; ++s2)
#pragma unroll
        for (int m = 0; m < 5; ++m) acc[s2][m] = 0.f;
    float l1f = 0.f, ssf = 0.f;
    for (int q = 0; q < kInH / kTapN; ++q) {
#pragma unroll
        for (int j = 0; j < kTapN; ++j) {
            const int r = q * kTapN + j;
            float h[5] = {0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k = 0; k < kTapN; ++k) {
                const float u = sm[0][r][c + k], v = sm[1][r][c + k], wk = a.w[k];
                h[0] = __fmaf_rn(wk, u, h[0]);
                h[1] = __fmaf_rn(wk, v, h[1]);
                h[2] = __fmaf_rn(wk, u * u, h[2]);
                h[3] = __fmaf_rn(wk, v * v, h[3]);
                h[4] = __fmaf_rn(wk, u * v, h[4]);
            }
#pragma unroll
            for (int t = 0; t < kTapN; ++t)
#pragma unroll
                for (int m = 0; m < 5; ++m) acc[(j - t + kTapN) % kTapN][m] = __fmaf_rn(a.w[t], h[m], acc[(j - t + kTapN) % kTapN][m]);
            // output row o = r - 10 is complete
            const int slot = (j + 1) % kTapN;
            const int o = r - (kTapN - 1), gy = y0 + o;
            if (o >= 0 && gx < W && gy < H) {
                const float mx = acc[slot][0], my = acc[slot][1], exx = acc[slot][2], eyy = acc[slot][3];
                const float exy = acc[slot][4];
                const float A = __fmaf_rn(2.f * mx, my, a.c1);
                const float B = __fmaf_rn(2.f, exy - mx * my, a.c2);
                const float Cc = __fmaf_rn(mx, mx, __fmaf_rn(my, my, a.c1));
                const float D = (exx - mx * mx) + (eyy - my * my) + a.c2;
                const float iC = __frcp_rn(Cc), iD = __frcp_rn(D);
                const float inv = iC * iD;
                const float S = A * B * inv;
                const size_t oo = ch * plane + (size_t)gy * W + gx;
                p_mu[oo] = 2.f * my * (B - A) * inv - 2.f * mx * S * (iC - iD);
                p_xx[oo] = -S * iD;
                p_xy[oo] = 2.f * A * inv;
                l1f += fabsf(sm[0][o + kHalo][c + kHalo] - sm[1][o + kHalo][c + kHalo]);
                ssf += S;
            }
#pragma unroll
            for (int m = 0; m < 5; ++m) acc[slot][m] = 0.f;
        }
    }
    // block sums of |x - y| and S (float per thread, float64 across threads)
    double l1 = (double)l1f, ss = (double)ssf;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        ss += __shfl_xor_sync(0xffffffffu, ss, off);
    }
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        red[0][warp] = l1;
        red[1][warp] = ss;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double t0 = 0.0, t1 = 0.0;
        for (int w = 0; w < kLW / 32; ++w) {
            t0 += red[0][w];
            t1 += red[1][w];
        }
        atomicAdd(&sums[0], t0);
        atomicAdd(&sums[1], t1);
    }
}

__global__ void __launch_bounds__(kLW) k_ssim_bwd(const LossArgs a, const float* __restrict__ img,
                                                  const float* __restrict__ tgt, const float* __restrict__ p_mu,
                                                  const float* __restrict__ p_xx, const float* __restrict__ p_xy,
                                                  const double* __restrict__ sums, float* __restrict__ loss,
                                                  float* __restrict__ dl) {
    extern __shared__ float smem_loss[];
    float (*sm)[kInH][kInW] = reinterpret_cast<float (*)[kInH][kInW]>(smem_loss);  // the 3 partial maps
    const int W = a.width, H = a.height;
    const int x0 = blockIdx.x * kLW, y0 = blockIdx.y * kLH, ch = blockIdx.z;
    const size_t plane = (size_t)W * H;
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0 && ch == 0)
        *loss = (float)((1.0 - a.lam) * sums[0] * a.inv_n + a.lam * (1.0 - sums[1] * a.inv_n));
    const float* const src[3] = {p_mu + ch * plane, p_xx + ch * plane, p_xy + ch * plane};
    stage_tile<3>(sm, src, x0, y0, W, H);
    __syncthreads();
    const int c = threadIdx.x, gx = x0 + c;
    float acc[kTapN][3];
#pragma unroll
    for (int s2 = 0; s2 < kTapN; ++s2)
#pragma unroll
        for (int m = 0; m < 3; ++m) acc[s2][m] = 0.f;
    for (int q = 0; q < kInH / kTapN; ++q) {
        // image and target at the 11 outputs this group of rows completes, loaded ahead of use
        float xs[kTapN], ys[kTapN];
#pragma unroll
        for (int j = 0; j < kTapN; ++j) {
            const int o = q * kTapN + j - (kTapN - 1), gy = y0 + o;
            const bool ok = o >= 0 && gx < W && gy < H;
            const size_t oo = ch * plane + (size_t)(ok ? gy : 0) * W + (ok ? gx : 0);
            xs[j] = ok ? img[oo] : 0.f;
            ys[j] = ok ? tgt[oo] : 0.f;
        }
#pragma unroll
        for (int j = 0; j < kTapN; ++j) {
            const int r = q * kTapN + j;
            float h[3] = {0.f, 0.f, 0.f};
#pragma unroll
            for (int k = 0; k < kTapN; ++k) {
                const float wk = a.w[k];
                h[0] = __fmaf_rn(wk, sm[0][r][c + k], h[0]);
                h[1] = __fmaf_rn(wk, sm[1][r][c + k], h[1]);
                h[2] = __fmaf_rn(wk, sm[2][r][c + k], h[2]);
            }
#pragma unroll
            for (int t = 0; t < kTapN; ++t)
#pragma unroll
                for (int m = 0; m < 3; ++m) acc[(j - t + kTapN) % kTapN][m] = __fmaf_rn(a.w[t], h[m], acc[(j - t + kTapN) % kTapN][m]);
            const int slot = (j + 1) % kTapN;
            const int o = r - (kTapN - 1), gy = y0 + o;
            if (o >= 0 && gx < W && gy < H) {
                const size_t oo = ch * plane + (size_t)gy * W + gx;
                const float x = xs[j], y = ys[j];
                const float dssim = __fmaf_rn(2.f * x, acc[slot][1], __fmaf_rn(y, acc[slot][2], acc[slot][0]));
                const float sgn = x > y ? 1.f : (x < y ? -1.f : 0.f);
                dl[oo] = a.inv_n * ((1.f - a.lam) * sgn - a.lam * dssim);
            }
#pragma unroll
            for (int m = 0; m < 3; ++m) acc[slot][m] = 0.f;
        }
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
    const dim3 grid((width + kLW - 1) / kLW, (height + kLH - 1) / kLH, 3);
    const int smem2 = 2 * kInH * kInW * 4, smem3 = 3 * kInH * kInW * 4;
    if ((e = cudaFuncSetAttribute(k_ssim_fwd, cudaFuncAttributeMaxDynamicSharedMemorySize, smem2))) return e;
    if ((e = cudaFuncSetAttribute(k_ssim_bwd, cudaFuncAttributeMaxDynamicSharedMemorySize, smem3))) return e;
    count_launches(2);
    k_ssim_fwd<<<grid, kLW, smem2, st>>>(a, img, tgt, p_mu, p_xx, p_xy, sums);
    k_ssim_bwd<<<grid, kLW, smem3, st>>>(a, img, tgt, p_mu, p_xx, p_xy, sums, loss, dl);
    return cudaGetLastError();
}

}  // namespace gs
