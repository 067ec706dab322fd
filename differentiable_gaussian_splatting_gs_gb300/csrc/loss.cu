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
// Both passes stage a 128x34 tile plus a 5-pixel halo in shared memory, with the maps summed
// together held as pairs so that packed float32 pair instructions do two sums at once.
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

// Stages the tile (rows y0 - 5 .., columns x0 - 5 ..) of the maps a and b (b may be NULL) with zeros
// outside the image: PAIR stores them interleaved, sm2[r][c] = (a, b); otherwise a alone into sm1.
// Asynchronous copies, all in flight at once, waited for before returning (the caller then
// synchronises the block).
template <bool PAIR>
__device__ __forceinline__ void stage_tile(float2 (*sm2)[kInW], float (*sm1)[kInW], const float* a, const float* b,
                                           int x0, int y0, int W, int H) {
    for (int i = threadIdx.x; i < kInH * kInW; i += kLW) {
        const int r = i / kInW, c = i - r * kInW;
        const int gy = y0 - kHalo + r, gx = x0 - kHalo + c;
        const bool in = gx >= 0 && gx < W && gy >= 0 && gy < H;
        const size_t g = (size_t)gy * W + gx;
        if (PAIR) {
            if (in) {
                cp_async4(&sm2[r][c].x, a + g);
                cp_async4(&sm2[r][c].y, b + g);
            } else {
                sm2[r][c] = make_float2(0.f, 0.f);
            }
        } else {
            if (in) cp_async4(&sm1[r][c], a + g);
            else sm1[r][c] = 0.f;
        }
    }
    cp_async_wait_all();
}

// Pass 1: the five windowed moments of (x, y) per pixel, the SSIM map S and its partial
// derivatives with respect to mu_x, E[x^2] and E[xy]. x and y are staged as pairs, so that the
// moments run as packed pairs (mu_x, mu_y), (E[x^2], E[y^2]) and the scalar E[xy]: every sum takes
// its terms in the same order and rounding as scalar code would.
__global__ void __launch_bounds__(kLW) k_ssim_fwd(const LossArgs a, const float* __restrict__ img,
                                                  const float* __restrict__ tgt, float2* __restrict__ p_mx,
                                                  float* __restrict__ p_xy, double* __restrict__ sums) {
    extern __shared__ float4 smem_loss4[];
    float2 (*sm)[kInW] = reinterpret_cast<float2 (*)[kInW]>(smem_loss4);  // (x, y)
    __shared__ double red[2][kLW / 32];
    const int W = a.width, H = a.height;
    const int x0 = blockIdx.x * kLW, y0 = blockIdx.y * kLH, ch = blockIdx.z;
    const size_t plane = (size_t)W * H;
    stage_tile<true>(sm, nullptr, img + ch * plane, tgt + ch * plane, x0, y0, W, H);
    __syncthreads();
    const int c = threadIdx.x, gx = x0 + c;
    f32x2 w2[kTapN];
#pragma unroll
    for (int k = 0; k < kTapN; ++k) w2[k] = f2_pack(a.w[k], a.w[k]);
    f32x2 acc_m[kTapN], acc_s[kTapN];   // (mu_x, mu_y), (E[x^2], E[y^2]) of the 11 rows in flight
    float acc_c[kTapN];                 // E[xy]
#pragma unroll
    for (int s2 = 0; s2 < kTapN; ++s2) {
        acc_m[s2] = acc_s[s2] = 0ull;
        acc_c[s2] = 0.f;
    }
    float l1f = 0.f, ssf = 0.f;
    for (int q = 0; q < kInH / kTapN; ++q) {
#pragma unroll
        for (int j = 0; j < kTapN; ++j) {
            const int r = q * kTapN + j;
            f32x2 hm = 0ull, hs = 0ull;
            float hc = 0.f;
#pragma unroll
            for (int k = 0; k < kTapN; ++k) {
                const float2 p = sm[r][c + k];
                const f32x2 uv = f2_pack(p.x, p.y);
                hm = f2_fma(w2[k], uv, hm);
                hs = f2_fma(w2[k], f2_mul(uv, uv), hs);
                hc = __fmaf_rn(a.w[k], p.x * p.y, hc);
            }
#pragma unroll
            for (int t = 0; t < kTapN; ++t) {
                const int o = (j - t + kTapN) % kTapN;
                acc_m[o] = f2_fma(w2[t], hm, acc_m[o]);
                acc_s[o] = f2_fma(w2[t], hs, acc_s[o]);
                acc_c[o] = __fmaf_rn(a.w[t], hc, acc_c[o]);
            }
            // output row o = r - 10 is complete
            const int slot = (j + 1) % kTapN;
            const int o = r - (kTapN - 1), gy = y0 + o;
            if (o >= 0 && gx < W && gy < H) {
                const float2 mu = f2_unpack(acc_m[slot]), e2 = f2_unpack(acc_s[slot]);
                const float mx = mu.x, my = mu.y, exx = e2.x, eyy = e2.y, exy = acc_c[slot];
                const float A = __fmaf_rn(2.f * mx, my, a.c1);
                const float B = __fmaf_rn(2.f, exy - mx * my, a.c2);
                const float Cc = __fmaf_rn(mx, mx, __fmaf_rn(my, my, a.c1));
                const float D = (exx - mx * mx) + (eyy - my * my) + a.c2;
                const float iC = __frcp_rn(Cc), iD = __frcp_rn(D);
                const float inv = iC * iD;
                const float S = A * B * inv;
                const size_t oo = ch * plane + (size_t)gy * W + gx;
                p_mx[oo] = make_float2(2.f * my * (B - A) * inv - 2.f * mx * S * (iC - iD), -S * iD);
                p_xy[oo] = 2.f * A * inv;
                const float2 xy = sm[o + kHalo][c + kHalo];
                l1f += fabsf(xy.x - xy.y);
                ssf += S;
            }
            acc_m[slot] = acc_s[slot] = 0ull;
            acc_c[slot] = 0.f;
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

// Pass 2: dL/dx from the windowed sums of the three partial maps (dS/dmu_x and dS/dE[x^2] staged
// as pairs, summed as packed pairs; dS/dE[xy] alone), and the L1 term.
__global__ void __launch_bounds__(kLW) k_ssim_bwd(const LossArgs a, const float* __restrict__ img,
                                                  const float* __restrict__ tgt, const float2* __restrict__ p_mx,
                                                  const float* __restrict__ p_xy, const double* __restrict__ sums,
                                                  float* __restrict__ loss, float* __restrict__ dl) {
    extern __shared__ float4 smem_loss4[];
    float2 (*sm2)[kInW] = reinterpret_cast<float2 (*)[kInW]>(smem_loss4);                   // (d mu, d xx)
    float (*sm1)[kInW] = reinterpret_cast<float (*)[kInW]>(sm2 + kInH);                     // d xy
    const int W = a.width, H = a.height;
    const int x0 = blockIdx.x * kLW, y0 = blockIdx.y * kLH, ch = blockIdx.z;
    const size_t plane = (size_t)W * H;
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0 && ch == 0)
        *loss = (float)((1.0 - a.lam) * sums[0] * a.inv_n + a.lam * (1.0 - sums[1] * a.inv_n));
    {
        // the pair map: 8-byte copies of (d mu, d xx)
        const float2* src = p_mx + ch * plane;
        for (int i = threadIdx.x; i < kInH * kInW; i += kLW) {
            const int r = i / kInW, c = i - r * kInW;
            const int gy = y0 - kHalo + r, gx = x0 - kHalo + c;
            if (gx >= 0 && gx < W && gy >= 0 && gy < H) cp_async8(&sm2[r][c], src + (size_t)gy * W + gx);
            else sm2[r][c] = make_float2(0.f, 0.f);
        }
    }
    stage_tile<false>(nullptr, sm1, p_xy + ch * plane, nullptr, x0, y0, W, H);
    __syncthreads();
    const int c = threadIdx.x, gx = x0 + c;
    f32x2 w2[kTapN];
#pragma unroll
    for (int k = 0; k < kTapN; ++k) w2[k] = f2_pack(a.w[k], a.w[k]);
    f32x2 acc_p[kTapN];
    float acc_c[kTapN];
#pragma unroll
    for (int s2 = 0; s2 < kTapN; ++s2) {
        acc_p[s2] = 0ull;
        acc_c[s2] = 0.f;
    }
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
            f32x2 hp = 0ull;
            float hc = 0.f;
#pragma unroll
            for (int k = 0; k < kTapN; ++k) {
                const float2 p = sm2[r][c + k];
                hp = f2_fma(w2[k], f2_pack(p.x, p.y), hp);
                hc = __fmaf_rn(a.w[k], sm1[r][c + k], hc);
            }
#pragma unroll
            for (int t = 0; t < kTapN; ++t) {
                const int o = (j - t + kTapN) % kTapN;
                acc_p[o] = f2_fma(w2[t], hp, acc_p[o]);
                acc_c[o] = __fmaf_rn(a.w[t], hc, acc_c[o]);
            }
            const int slot = (j + 1) % kTapN;
            const int o = r - (kTapN - 1), gy = y0 + o;
            if (o >= 0 && gx < W && gy < H) {
                const size_t oo = ch * plane + (size_t)gy * W + gx;
                const float x = xs[j], y = ys[j];
                const float2 pm = f2_unpack(acc_p[slot]);
                const float dssim = __fmaf_rn(2.f * x, pm.y, __fmaf_rn(y, acc_c[slot], pm.x));
                const float sgn = x > y ? 1.f : (x < y ? -1.f : 0.f);
                dl[oo] = a.inv_n * ((1.f - a.lam) * sgn - a.lam * dssim);
            }
            acc_p[slot] = 0ull;
            acc_c[slot] = 0.f;
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
    float2* p_mx = reinterpret_cast<float2*>(static_cast<char*>(ws) + 256);   // (d mu, d xx) pairs
    float* p_xy = reinterpret_cast<float*>(p_mx + plane3);
    cudaError_t e = cudaMemsetAsync(sums, 0, 2 * sizeof(double), st);
    if (e) return e;
    const dim3 grid((width + kLW - 1) / kLW, (height + kLH - 1) / kLH, 3);
    const int smem2 = kInH * kInW * 8, smem3 = kInH * kInW * 12;
    if ((e = cudaFuncSetAttribute(k_ssim_fwd, cudaFuncAttributeMaxDynamicSharedMemorySize, smem2))) return e;
    if ((e = cudaFuncSetAttribute(k_ssim_bwd, cudaFuncAttributeMaxDynamicSharedMemorySize, smem3))) return e;
    count_launches(2);
    k_ssim_fwd<<<grid, kLW, smem2, st>>>(a, img, tgt, p_mx, p_xy, sums);
    k_ssim_bwd<<<grid, kLW, smem3, st>>>(a, img, tgt, p_mx, p_xy, sums, loss, dl);
    return cudaGetLastError();
}

}  // namespace gs
