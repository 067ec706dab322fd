// Rendering phase (forward alpha blending) and gradient computation phase (backward) of the tile
// rasterizer: one block per 16x16-pixel tile, the tile's sorted list staged in shared memory in
// batches of one record per thread. The forward uses 128 threads with two pixels each; the
// backward 64 threads with four pixels each (or the forward's layout on images of fewer than two
// tiles per SM).
//
// The backward accumulates each Gaussian's gradient over all pixels with atomics; that
// accumulation is the bottleneck that DISTWAR (Fast Differentiable Rendering on Raster-based
// Rendering Pipelines, Abstract) and ARC (Warp-level Adaptive Atomic Reduction in GPUs to
// Accelerate Differentiable Rendering, Abstract) identify, and the reason for the GS_BWD_* modes.
//
// Warp layout: warp w covers the 8x8 pixel block at (8 (w & 1), 8 (w >> 1)) of the tile; lane l
// holds pixels (l & 7, l >> 3) and (l & 7, (l >> 3) + 4), so that a Gaussian's record loads and
// culling test serve 64 pixels. The backward's 16x8 layout (BwdLayout) has its record loads,
// culling test, warp reduction and atomics serve 128 pixels.
//
// Warp-level culling. Before blending a batch, each warp keeps only the staged Gaussians whose
// alpha can reach 1/255 somewhere in its 8x8 block: the set alpha >= 1/255 is the ellipse
// q(d) = A dx^2 + 2 B dx dy + C dy^2 <= L = 2 tau, tau = ln(255 opacity), and the test is whether
// the minimum of q over the block's rectangle of pixel centres is <= L. q is convex, so for a fixed
// dy its minimum over dx in [ax, bx] is at dx = clamp(-(B/A) dy, ax, bx); what remains is a convex
// function of dy whose minimiser over the real line is dy = -(B/C) clamp(0, ax, bx), and over
// [ay, by] its clamp. Three clamps give the minimising point, and q there decides. The rectangle
// is widened by 0.01 px and tau by 0.1 % + 0.001 so that rounding cannot drop a pair the per-pixel
// test would blend; dropped pairs are exactly ones the per-pixel test skips, so the results do not
// change.
//
// The "skip when power > 0" rule never fires here: power is evaluated as a sum of non-negative
// terms times -1/2 (see prepare_record), which cannot be positive.
#include "gs_common.cuh"
#include "gs_internal.h"

namespace gs {

constexpr float kAlphaMin = 1.0f / 255.0f;
constexpr float kTMin = 1e-4f;
constexpr float kAlphaMax = 0.99f;
constexpr float kNegHalfLog2e = -0.72134752044448170f;  // -log2(e) / 2

// Shared-memory staging ring of BATCH records for a block of WARPS warps (one record per thread).
template <int BATCH, int WARPS>
struct StageSmemT {
    static constexpr int kB = BATCH;
    float4 rec[2][BATCH][3];       // double-buffered records
    unsigned gidx[2][BATCH];       // Gaussian index of each staged record
    float4 cull[BATCH];            // (mean_x, mean_y, B / C, B / A) for the warp culling test
    float2 cull2[BATCH];           // (D / A, L / A) with D = det / A and L = 2 tau
    unsigned short list[WARPS][BATCH];
    uint64_t bar[2];
};

// Both passes: 128 threads per tile, two pixels each; warp w covers the 8x8 block at
// (8 (w & 1), 8 (w >> 1)), lane l the pixels (l & 7, l >> 3) and (l & 7, (l >> 3) + 4) of it.
constexpr int kFwdBlock = 128;
constexpr int kFwdBatch = 128;
using FwdStage = StageSmemT<kFwdBatch, 4>;

// The forward's per-batch form of each staged record, built from the prepared record: the
// per-Gaussian constants of the alpha evaluation duplicated into pairs, so that a lane evaluates its
// two pixels with packed float32 pair instructions (f32x2, rounding each half as the scalar
// instruction would): (mx, mx, my, my), (r, r, A', A'), (D', D', o, red), (green, blue, -, -).
struct FwdSmem {
    FwdStage st;
    float4 pair[4][kFwdBatch];   // [field][record]: conflict-free writes by consecutive threads
};
// Backward layouts, PX pixels per lane: PX = 2 is the forward's layout (128 threads, 8x8 warp
// blocks); PX = 4 gives each warp a 16x8 block (64 threads per tile; warp w covers rows 8w..8w+7,
// lane l the column l & 15 and the rows (l >> 4) + 2q, q = 0..3). A larger warp block meets each
// Gaussian fewer times per tile, so the per-Gaussian work of a warp (record loads, culling, the
// gradient reduction and its atomics) is shared by twice as many pixels. One staged record per
// thread and batch.
template <int PX>
struct BwdLayout {
    static constexpr int kThreads = PX == 2 ? 128 : 64;
    static constexpr int kWarps = kThreads / 32;
    static constexpr int kBatch = kThreads;
    static constexpr int kBlockW = PX == 2 ? 8 : 16;   // warp block width; its height is 8
    static constexpr int kRowStep = 32 / kBlockW;      // rows between a lane's pixels
};

template <int PX>
struct BwdSmemT {
    StageSmemT<BwdLayout<PX>::kBatch, BwdLayout<PX>::kWarps> st;
    float acc[BwdLayout<PX>::kBatch * 9];   // per-batch gradient accumulators (GS_BWD_SM)
    unsigned wmax[BwdLayout<PX>::kWarps];
};

// Prepares a staged record for evaluation and returns its culling record.
//
// The quadratic form -power = (A dx^2 + C dy^2)/2 + B dx dy is evaluated by completing the square,
// (A u^2 + D dy^2) / 2 with u = dx + r dy, r = B / A and D = det / A, det = A C - B^2: both terms
// are non-negative, so the evaluation has no cancellation even for very elongated Gaussians
// (where the three terms of the plain form are large and nearly cancel). det is computed with
// one rounding error. The record's C slot is replaced by D and slot 9 receives r; A and B stay.
// A record whose conic is not positive definite is never blended (culled by every warp). Slots 10 and 11
// receive A and D scaled by -log2(e)/2, so that the kernels take exp(power) as 2^(A' u^2 + D' dy^2)
// with the hardware base-2 exponential.
//
// Culling record: the quantities of the warp test (see the file header) with q divided by A,
// q / A = (dx + (B/A) dy)^2 + (D/A) dy^2 <= L / A. Records that are never blended get L / A = -1.
__device__ __forceinline__ float4 prepare_record(float4& r0, float4& r1, float4& r2, float2& cull2) {
    const float mx = r0.x, my = r0.y, A = r0.z, B = r0.w, C = r1.x, o = r1.y;
    const float inf = __int_as_float(0x7f800000);
    cull2 = make_float2(0.f, -1.f);
    const float w = B * B;
    const float e = __fmaf_rn(-B, B, w);
    const float f = __fmaf_rn(A, C, -w);
    const float det = f + e;
    if (!(A > 0.f) || !(det > 0.f) || !(det < inf)) {
        r1.x = 0.f;
        r2.y = 0.f;
        r2.z = 0.f;
        r2.w = 0.f;
        return make_float4(mx, my, 0.f, 0.f);
    }
    // one hardware reciprocal of A (and of C) instead of five divisions: each quotient is within
    // about 2 ulps, well inside the float32 error bound the parity tests allow for the power, and
    // the culling values carry margins of their own
    const float iA = rcp_approx(A);
    const float D = det * iA;
    const float r = B * iA;
    r1.x = D;
    r2.y = r;
    r2.z = kNegHalfLog2e * A;
    r2.w = kNegHalfLog2e * D;
    if (!(o * 1.00001f >= kAlphaMin)) return make_float4(mx, my, 0.f, 0.f);  // alpha <= o < 1/255: never
    const float tau = __logf(255.0f * o * 1.00001f) * 1.001f + 0.001f;
    cull2 = make_float2(D * iA, 2.f * tau * iA);
    return make_float4(mx, my, B * rcp_approx(C), r);
}

// ---- batch staging ----------------------------------------------------------------------------

// Registers the transaction bytes of batch `b` on its barrier (thread 0 only, before any copy of
// that batch is issued).
template <int STAGING, class S>
__device__ __forceinline__ void stage_expect(S& s, int slot, int n_in) {
    if (STAGING == GS_STAGE_BULK) mbar_arrive_expect_tx(&s.bar[slot], (unsigned)n_in * 48u);
}

template <int STAGING, class S>
__device__ __forceinline__ void stage_issue(S& s, int slot, const float4* __restrict__ rec,
                                            const unsigned* __restrict__ vals, int first, int n_in,
                                            unsigned n_gauss, float4 (&pre)[3], unsigned* err) {
    const int t = threadIdx.x;
    if (t < n_in) {
        unsigned g = vals[first + t];
        if (g >= n_gauss) {
            atomicOr(err, kErrCheck);
            g = 0;
        }
        s.gidx[slot][t] = g;
        if (STAGING == GS_STAGE_BULK) {
            bulk_copy_g2s(&s.rec[slot][t][0], rec + 3 * (size_t)g, 48u, &s.bar[slot]);
        } else {
            pre[0] = __ldg(rec + 3 * (size_t)g);
            pre[1] = __ldg(rec + 3 * (size_t)g + 1);
            pre[2] = __ldg(rec + 3 * (size_t)g + 2);
        }
    }
}

// Makes batch `slot` visible in shared memory. For register staging the loads issued by
// stage_issue are stored here; the caller synchronises the block afterwards.
template <int STAGING, class S>
__device__ __forceinline__ bool stage_wait(S& s, int slot, unsigned parity, int n_in, const float4 (&pre)[3],
                                           unsigned spin_limit, unsigned* err) {
    if (STAGING == GS_STAGE_BULK) {
        return mbar_wait_bounded(&s.bar[slot], parity, spin_limit, err);
    } else {
        const int t = threadIdx.x;
        if (t < n_in) {
            s.rec[slot][t][0] = pre[0];
            s.rec[slot][t][1] = pre[1];
            s.rec[slot][t][2] = pre[2];
        }
        return true;
    }
}

// Compacts the staged entries [0, n_in) that may be blended in this warp's block (and whose
// batch position is below `pos_limit`) into s.list[warp], in increasing order. Returns the count.
template <class S>
__device__ __forceinline__ int compact_warp(S& s, int n_in, int pos_limit, float wx0, float wx1,
                                            float wy0, float wy1, int warp, int lane) {
    int cnt = 0;
    const int lim = min(n_in, pos_limit);
    const float x0 = wx0 - 0.01f, x1 = wx1 + 0.01f, y0 = wy0 - 0.01f, y1 = wy1 + 0.01f;
#pragma unroll
    for (int c = 0; c < S::kB / 32; ++c) {
        if (c * 32 >= lim) break;  // warp-uniform: the rest of the batch is empty or past the limit
        const int j = c * 32 + lane;
        bool hit = false;
        if (j < lim) {
            const float4 q = s.cull[j];
            const float2 q2 = s.cull2[j];
            const float ax = x0 - q.x, bx = x1 - q.x, ay = y0 - q.y, by = y1 - q.y;
            const float cx = fminf(fmaxf(0.f, ax), bx);
            const float dy = fminf(fmaxf(-q.z * cx, ay), by);
            const float dx = fminf(fmaxf(-q.w * dy, ax), bx);
            const float u = __fmaf_rn(q.w, dy, dx);
            hit = !(__fmaf_rn(u, u, q2.x * dy * dy) > q2.y);  // NaN keeps the pair
        }
        const unsigned m = __ballot_sync(0xffffffffu, hit);
        if (hit) s.list[warp][cnt + __popc(m & lanemask_lt())] = (unsigned short)j;
        cnt += __popc(m);
    }
    __syncwarp();
    return cnt;
}

// ---- forward ---------------------------------------------------------------------------------

// Front-to-back blending of one record, whose alpha at the pixel is given, into one pixel; sets
// `done` when the pixel terminates.
__device__ __forceinline__ void blend_pixel(float alpha, float cr, float cg, float cb, unsigned pos1, float& T,
                                            float& c0, float& c1, float& c2, unsigned& last, bool& done) {
    if (alpha >= kAlphaMin) {
        const float test_T = T * (1.f - alpha);
        if (test_T < kTMin) {
            done = true;
        } else {
            const float w = alpha * T;
            c0 = __fmaf_rn(cr, w, c0);
            c1 = __fmaf_rn(cg, w, c1);
            c2 = __fmaf_rn(cb, w, c2);
            T = test_T;
            last = pos1;
        }
    }
}

// Alphas of one staged Gaussian at a lane's two pixels from its pair record (FwdSmem::pair):
// o 2^(A' u^2 + D' dy^2) with u = dx + r dy, each half computed in the same order and rounding as
// the scalar form. fpx2 = (px, px) and fpy2 = (py0, py1) are the pixel centres. Also returns
// (o, red) and (green, blue).
__device__ __forceinline__ float2 pair_alphas(const float4 (&pr)[4][kFwdBatch], int j, f32x2 fpx2, f32x2 fpy2,
                                              float2& ored, float2& gb) {
    const ulonglong2 p0 = *reinterpret_cast<const ulonglong2*>(&pr[0][j]);   // (mx, mx), (my, my)
    const ulonglong2 p1 = *reinterpret_cast<const ulonglong2*>(&pr[1][j]);   // (r, r), (A', A')
    const ulonglong2 p2 = *reinterpret_cast<const ulonglong2*>(&pr[2][j]);   // (D', D'), (o, red)
    gb = *reinterpret_cast<const float2*>(&pr[3][j]);
    const f32x2 dx = f2_sub(p0.x, fpx2), dy = f2_sub(p0.y, fpy2);
    const f32x2 u = f2_fma(p1.x, dy, dx);
    const float2 e = f2_unpack(f2_fma(f2_mul(p1.y, u), u, f2_mul(f2_mul(p2.x, dy), dy)));
    ored = f2_unpack(p2.y);
    return make_float2(fminf(kAlphaMax, ored.x * ex2_approx(e.x)), fminf(kAlphaMax, ored.x * ex2_approx(e.y)));
}

template <int STAGING>
__global__ void __launch_bounds__(kFwdBlock) k_render_fwd(const float4* __restrict__ rec,
                                                          const unsigned* __restrict__ vals,
                                                          const uint2* __restrict__ ranges, const KernelCamera cam,
                                                          unsigned n_gauss, float* __restrict__ image,
                                                          float* __restrict__ t_final, unsigned* __restrict__ n_contrib,
                                                          unsigned spin_limit, unsigned* __restrict__ err) {
    pdl_entry();
    constexpr int kB = kFwdBatch;
    __shared__ FwdSmem sm;
    FwdStage& s = sm.st;
    const int tile = blockIdx.x;
    const int tx = tile % cam.tiles_x, ty = tile / cam.tiles_x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bx = tx * kTile + 8 * (warp & 1), by = ty * kTile + 8 * (warp >> 1);
    const int px = bx + (lane & 7), py0 = by + (lane >> 3), py1 = py0 + 4;
    const bool in0 = px < cam.width && py0 < cam.height, in1 = px < cam.width && py1 < cam.height;
    const float fpx = (float)px + 0.5f, fpy0 = (float)py0 + 0.5f, fpy1 = (float)py1 + 0.5f;
    const f32x2 fpx2 = f2_pack(fpx, fpx), fpy2 = f2_pack(fpy0, fpy1);
    const float wx0 = (float)bx + 0.5f, wx1 = wx0 + 7.f, wy0 = (float)by + 0.5f, wy1 = wy0 + 7.f;

    const uint2 rg = ranges[tile];
    const int start = (int)rg.x;
    const int count = (int)(rg.y > rg.x ? rg.y - rg.x : 0);
    const int nb = (count + kB - 1) / kB;

    float T0 = 1.f, c00 = 0.f, c01 = 0.f, c02 = 0.f, T1 = 1.f, c10 = 0.f, c11 = 0.f, c12 = 0.f;
    unsigned last0 = 0, last1 = 0;
    bool done0 = !in0, done1 = !in1;
    float4 pre[3];

    if (nb > 0) {
        if (threadIdx.x == 0 && STAGING == GS_STAGE_BULK) {
            mbar_init(&s.bar[0], 1);
            mbar_init(&s.bar[1], 1);
            fence_mbar_init();
            stage_expect<STAGING>(s, 0, min(kB, count));
            if (nb > 1) stage_expect<STAGING>(s, 1, min(kB, count - kB));
        }
        __syncthreads();
        stage_issue<STAGING>(s, 0, rec, vals, start, min(kB, count), n_gauss, pre, err);
    }
    bool ok = true;
    int issued = nb > 0 ? 0 : -1, consumed = -1;  // batches whose copies were issued / waited for
    for (int b = 0; b < nb; ++b) {
        const int slot = b & 1;
        const int n_in = min(kB, count - b * kB);
        float4 nxt[3];
        if (STAGING == GS_STAGE_LOADS) {
            // the loads of this batch were issued one iteration earlier (or above)
            ok = stage_wait<STAGING>(s, slot, 0, n_in, pre, spin_limit, err);
            if (b + 1 < nb) stage_issue<STAGING>(s, slot ^ 1, rec, vals, start + (b + 1) * kB,
                                                 min(kB, count - (b + 1) * kB), n_gauss, nxt, err);
        } else {
            if (b + 1 < nb) {
                stage_issue<STAGING>(s, slot ^ 1, rec, vals, start + (b + 1) * kB, min(kB, count - (b + 1) * kB),
                                     n_gauss, nxt, err);
                issued = b + 1;
            }
            ok = stage_wait<STAGING>(s, slot, (unsigned)(b >> 1) & 1u, n_in, pre, spin_limit, err);
            if (ok) consumed = b;
        }
        if (threadIdx.x < n_in) {
            float4 q0 = s.rec[slot][threadIdx.x][0], q1 = s.rec[slot][threadIdx.x][1], q2 = s.rec[slot][threadIdx.x][2];
            s.cull[threadIdx.x] = prepare_record(q0, q1, q2, s.cull2[threadIdx.x]);
            const int t = threadIdx.x;
            sm.pair[0][t] = make_float4(q0.x, q0.x, q0.y, q0.y);
            sm.pair[1][t] = make_float4(q2.y, q2.y, q2.z, q2.z);
            sm.pair[2][t] = make_float4(q2.w, q2.w, q1.y, q1.z);
            sm.pair[3][t] = make_float4(q1.w, q2.x, 0.f, 0.f);
        }
        if (__syncthreads_or(!ok)) break;
        const int nl = compact_warp(s, n_in, kB, wx0, wx1, wy0, wy1, warp, lane);
        // two listed Gaussians per iteration: their alphas do not depend on the transmittance, so
        // the four exponentials are computed together and only the blending stays in order
        for (int k = 0; k < nl; k += 2) {
            if (__all_sync(0xffffffffu, done0 && done1)) break;
            const bool two = k + 1 < nl;  // warp-uniform
            const int ja = s.list[warp][k], jb = two ? s.list[warp][k + 1] : ja;
            float2 oa, ga, ob, gb2;
            const float2 al_a = pair_alphas(sm.pair, ja, fpx2, fpy2, oa, ga);
            const float2 al_b = pair_alphas(sm.pair, jb, fpx2, fpy2, ob, gb2);
            const unsigned posa = (unsigned)(b * kB + ja + 1), posb = (unsigned)(b * kB + jb + 1);
            if (!done0) blend_pixel(al_a.x, oa.y, ga.x, ga.y, posa, T0, c00, c01, c02, last0, done0);
            if (!done1) blend_pixel(al_a.y, oa.y, ga.x, ga.y, posa, T1, c10, c11, c12, last1, done1);
            if (two) {
                if (!done0) blend_pixel(al_b.x, ob.y, gb2.x, gb2.y, posb, T0, c00, c01, c02, last0, done0);
                if (!done1) blend_pixel(al_b.y, ob.y, gb2.x, gb2.y, posb, T1, c10, c11, c12, last1, done1);
            }
        }
        if (STAGING == GS_STAGE_LOADS) {
            pre[0] = nxt[0]; pre[1] = nxt[1]; pre[2] = nxt[2];
        }
        if (threadIdx.x == 0 && b + 2 < nb) stage_expect<STAGING>(s, slot, min(kB, count - (b + 2) * kB));
        if (__syncthreads_count(!(done0 && done1)) == 0) break;
    }
    // bulk copies issued but not waited for (early termination or a wait that gave up) must land
    // before the block exits
    if (STAGING == GS_STAGE_BULK)
        for (int k = consumed + 1; k <= issued; ++k) mbar_wait_bounded(&s.bar[k & 1], (unsigned)(k >> 1) & 1u, kDrainLimit, err);
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

// ---- backward --------------------------------------------------------------------------------

// Sum over the 32 lanes of v[0..8]. Afterwards lane l with (l & 3) == 0 holds the total of
// component l >> 2 (0..7) and every lane holds the total of component 8. A transpose reduction:
// at each of the first three levels a lane keeps half of its components and sends the other
// half to its partner, so 9 shuffles reduce 8 components instead of 40.
__device__ __forceinline__ float warp_reduce9(const float (&v)[9], int lane, float& v8) {
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float u[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = b4 ? v[i] : v[i + 4];
        const float keep = b4 ? v[i + 4] : v[i];
        u[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
    float w[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = b3 ? u[i] : u[i + 2];
        const float keep = b3 ? u[i + 2] : u[i];
        w[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    const float send = b2 ? w[0] : w[1];
    float x = (b2 ? w[1] : w[0]) + __shfl_xor_sync(0xffffffffu, send, 4);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    float y = v[8];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) y += __shfl_xor_sync(0xffffffffu, y, o);
    v8 = y;
    return x;
}

// Steps one pixel's backward state past a Gaussian it blends (alpha, o G at the pixel): T becomes
// the transmittance in front of the Gaussian and gS gains its colour (gS = sum over channels of
// dL/dpixel_c x the colour blended behind, background included). Returns alpha T (the weight of
// the Gaussian's colour) in aT and dL/dpower in dp (0 where alpha was clamped at 0.99).
// r1, r2: the prepared record; g0..g2: dL/dpixel.
__device__ __forceinline__ void pixel_step(float alpha, float oG, const float4& r1, const float4& r2, float& T,
                                           float& gS, float g0, float g1, float g2, float& aT, float& dp) {
    const float inv = rcp_approx(1.f - alpha);
    T *= inv;
    aT = alpha * T;
    const float gc = __fmaf_rn(g0, r1.z, __fmaf_rn(g1, r1.w, g2 * r2.x));
    const float dalpha = __fmaf_rn(T, gc, -inv * gS);
    gS = __fmaf_rn(aT, gc, gS);
    dp = oG <= kAlphaMax ? oG * dalpha : 0.f;
}

// dl_dimage: dL/dpixel, or with `target` the rendered image, and dL/dpixel = image - target (the
// gradient of the squared error 0.5 |image - target|^2, whose sum is added to *loss when given).
template <int MODE, int STAGING, int PX>
__global__ void __launch_bounds__(BwdLayout<PX>::kThreads) k_render_bwd(
    const float4* __restrict__ rec, const unsigned* __restrict__ vals, const uint2* __restrict__ ranges,
    const KernelCamera cam, unsigned n_gauss, const float* __restrict__ dl_dimage, const float* __restrict__ target,
    float* __restrict__ loss, const float* __restrict__ t_final, const unsigned* __restrict__ n_contrib,
    float* __restrict__ grad2d, int thr, unsigned spin_limit, unsigned* __restrict__ err) {
    pdl_entry();
    using L = BwdLayout<PX>;
    constexpr int kB = L::kBatch;
    __shared__ BwdSmemT<PX> sm;
    auto& s = sm.st;
    const int tile = blockIdx.x;
    const int tx = tile % cam.tiles_x, ty = tile / cam.tiles_x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bx = tx * kTile + (PX == 2 ? 8 * (warp & 1) : 0);
    const int by = ty * kTile + (PX == 2 ? 8 * (warp >> 1) : 8 * warp);
    const int px = bx + lane % L::kBlockW, py = by + lane / L::kBlockW;
    const float fpx = (float)px + 0.5f;
    const float wx0 = (float)bx + 0.5f, wx1 = wx0 + (float)(L::kBlockW - 1), wy0 = (float)by + 0.5f, wy1 = wy0 + 7.f;

    const uint2 rg = ranges[tile];
    const int start = (int)rg.x;
    const int count = (int)(rg.y > rg.x ? rg.y - rg.x : 0);

    const size_t plane = (size_t)cam.width * cam.height;
    // per pixel q of the lane: its row offset dyo, contributor count, transmittance (from T_final
    // backwards), dL/dpixel and the sum over channels of dL/dpixel_c x (colour blended behind the
    // current Gaussian, background included), the only form in which that colour enters dL/dalpha
    float fpy[PX], T[PX], gS[PX], ga[PX][3];
    unsigned last[PX];
    float lsum = 0.f;
    unsigned lmax = 0;
#pragma unroll
    for (int q = 0; q < PX; ++q) {
        const int y = py + q * L::kRowStep;
        fpy[q] = (float)y + 0.5f;
        last[q] = 0;
        T[q] = 1.f;
        ga[q][0] = ga[q][1] = ga[q][2] = 0.f;
        if (px < cam.width && y < cam.height) {
            const size_t pix = (size_t)y * cam.width + px;
            last[q] = min(n_contrib[pix], (unsigned)count);
            T[q] = t_final[pix];
#pragma unroll
            for (int c = 0; c < 3; ++c) {
                ga[q][c] = dl_dimage[c * plane + pix];
                if (target) ga[q][c] -= target[c * plane + pix];
            }
        }
        lsum += __fmaf_rn(ga[q][0], ga[q][0], __fmaf_rn(ga[q][1], ga[q][1], ga[q][2] * ga[q][2]));
        gS[q] = T[q] * (ga[q][0] * cam.bg[0] + ga[q][1] * cam.bg[1] + ga[q][2] * cam.bg[2]);
        lmax = max(lmax, last[q]);
    }
    if (loss) {
        float l = 0.5f * lsum;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) red_add_global(loss, l);
    }
    const unsigned wmax = __reduce_max_sync(0xffffffffu, lmax);
    if (lane == 0) sm.wmax[warp] = wmax;
    __syncthreads();
    unsigned tmax = 0;
#pragma unroll
    for (int w = 0; w < L::kWarps; ++w) tmax = max(tmax, sm.wmax[w]);
    const int nb = ((int)tmax + kB - 1) / kB;
    float4 pre[3];

    if (nb > 0) {
        const int bl = nb - 1;
        if (threadIdx.x == 0 && STAGING == GS_STAGE_BULK) {
            mbar_init(&s.bar[0], 1);
            mbar_init(&s.bar[1], 1);
            fence_mbar_init();
            stage_expect<STAGING>(s, 0, min(kB, count - bl * kB));
            if (nb > 1) stage_expect<STAGING>(s, 1, kB);
        }
        __syncthreads();
        stage_issue<STAGING>(s, 0, rec, vals, start + bl * kB, min(kB, count - bl * kB), n_gauss, pre, err);
    }
    bool ok = true;
    int issued = nb > 0 ? 0 : -1, consumed = -1;  // iterations whose copies were issued / waited for
    for (int it = 0; it < nb; ++it) {
        const int b = nb - 1 - it;          // batches back to front
        const int slot = it & 1;
        const int n_in = min(kB, count - b * kB);
        float4 nxt[3];
        if (STAGING == GS_STAGE_LOADS) {
            ok = stage_wait<STAGING>(s, slot, 0, n_in, pre, spin_limit, err);
            if (b > 0) stage_issue<STAGING>(s, slot ^ 1, rec, vals, start + (b - 1) * kB, kB, n_gauss, nxt, err);
        } else {
            if (b > 0) {
                stage_issue<STAGING>(s, slot ^ 1, rec, vals, start + (b - 1) * kB, kB, n_gauss, nxt, err);
                issued = it + 1;
            }
            ok = stage_wait<STAGING>(s, slot, (unsigned)(it >> 1) & 1u, n_in, pre, spin_limit, err);
            if (ok) consumed = it;
        }
        if (threadIdx.x < n_in)
            s.cull[threadIdx.x] = prepare_record(s.rec[slot][threadIdx.x][0], s.rec[slot][threadIdx.x][1],
                                                 s.rec[slot][threadIdx.x][2], s.cull2[threadIdx.x]);
        if (MODE == GS_BWD_SM)
            for (int e = threadIdx.x; e < kB * 9; e += L::kThreads) sm.acc[e] = 0.f;
        if (__syncthreads_or(!ok)) break;
        const int pos_limit = (int)wmax - b * kB;
        const int nl = compact_warp(s, n_in, pos_limit, wx0, wx1, wy0, wy1, warp, lane);
        for (int k = nl - 1; k >= 0; --k) {
            const int j = s.list[warp][k];
            const unsigned pos = (unsigned)(b * kB + j);
            const float4 r0 = s.rec[slot][j][0];   // (mean_x, mean_y, A, B)
            const float4 r1 = s.rec[slot][j][1];   // (D, o, r, g)
            const float4 r2 = s.rec[slot][j][2];   // (b, r, A', D')
            const float dx = r0.x - fpx;
            float dy[PX], u[PX], oG[PX], alpha[PX];
            bool c[PX];
            bool any = false;
#pragma unroll
            for (int q = 0; q < PX; ++q) {
                dy[q] = r0.y - fpy[q];
                u[q] = __fmaf_rn(r2.y, dy[q], dx);
                oG[q] = r1.y * ex2_approx(__fmaf_rn(r2.z * u[q], u[q], r2.w * dy[q] * dy[q]));  // o exp(power)
                alpha[q] = fminf(kAlphaMax, oG[q]);
                c[q] = pos < last[q] && alpha[q] >= kAlphaMin;
                any |= c[q];
            }
            const unsigned ballot = __ballot_sync(0xffffffffu, any);
            if (ballot == 0u) continue;
            // The lane's sums over its pixels. The geometric gradients are linear in dL/dpower
            // with pixel-dependent factors: d power / d mean = -(A u, B u + D dy), d power / d(A, B, C)
            // = -(dx^2 / 2, dx dy, dy^2 / 2), and the lane's pixels share dx, so the lane forms the
            // moments P = sum dp, M = sum dp u, F = sum dp dy, Q = sum dp dy^2 once and converts
            // them; dL/dopacity = sum G dL/dalpha = P / o.
            float P = 0.f, M = 0.f, F = 0.f, Q = 0.f, cg0 = 0.f, cg1 = 0.f, cg2 = 0.f;
#pragma unroll
            for (int q = 0; q < PX; ++q) {
                if (c[q]) {
                    float aT, dp;
                    pixel_step(alpha[q], oG[q], r1, r2, T[q], gS[q], ga[q][0], ga[q][1], ga[q][2], aT, dp);
                    P += dp;
                    M = __fmaf_rn(dp, u[q], M);
                    const float f = dp * dy[q];
                    F += f;
                    Q = __fmaf_rn(f, dy[q], Q);
                    cg0 = __fmaf_rn(aT, ga[q][0], cg0);
                    cg1 = __fmaf_rn(aT, ga[q][1], cg1);
                    cg2 = __fmaf_rn(aT, ga[q][2], cg2);
                }
            }
            float v[9];
            v[0] = -r0.z * M;
            v[1] = -__fmaf_rn(r0.w, M, r1.x * F);
            v[2] = (-0.5f * dx * dx) * P;
            v[3] = -dx * F;
            v[4] = -0.5f * Q;
            v[5] = P * rcp_approx(r1.y);
            v[6] = cg0;
            v[7] = cg1;
            v[8] = cg2;
            const int nact = __popc(ballot);
            if (MODE == GS_BWD_DIRECT || (MODE == GS_BWD_ADAPTIVE && nact < thr)) {
                if (any) {
                    float* gp = grad2d + 12 * (size_t)s.gidx[slot][j];
                    red_add_global_v4(gp, v[0], v[1], v[2], v[3]);
                    red_add_global_v4(gp + 4, v[4], v[5], v[6], v[7]);
                    red_add_global(gp + 8, v[8]);
                }
            } else if (MODE == GS_BWD_SM && nact < thr) {
                if (any) {
                    float* ap = sm.acc + 9 * j;
#pragma unroll
                    for (int e = 0; e < 9; ++e) red_add_shared(ap + e, v[e]);
                }
            } else {
                float v8;
                const float x = warp_reduce9(v, lane, v8);
                if (MODE == GS_BWD_SM) {
                    float* ap = sm.acc + 9 * j;
                    if ((lane & 3) == 0) red_add_shared(ap + (lane >> 2), x);
                    if (lane == 1) red_add_shared(ap + 8, v8);
                } else {
                    float* gp = grad2d + 12 * (size_t)s.gidx[slot][j];
                    if ((lane & 3) == 0) red_add_global(gp + (lane >> 2), x);
                    if (lane == 1) red_add_global(gp + 8, v8);
                }
            }
        }
        if (STAGING == GS_STAGE_LOADS) {
            pre[0] = nxt[0]; pre[1] = nxt[1]; pre[2] = nxt[2];
        }
        __syncthreads();
        if (MODE == GS_BWD_SM && threadIdx.x < n_in) {
            const float* a = sm.acc + 9 * threadIdx.x;
            const float e0 = a[0], e1 = a[1], e2 = a[2], e3 = a[3], e4 = a[4], e5 = a[5], e6 = a[6], e7 = a[7], e8 = a[8];
            if ((e0 != 0.f) | (e1 != 0.f) | (e2 != 0.f) | (e3 != 0.f) | (e4 != 0.f) | (e5 != 0.f) | (e6 != 0.f) |
                (e7 != 0.f) | (e8 != 0.f)) {
                float* gp = grad2d + 12 * (size_t)s.gidx[slot][threadIdx.x];
                red_add_global_v4(gp, e0, e1, e2, e3);
                red_add_global_v4(gp + 4, e4, e5, e6, e7);
                red_add_global(gp + 8, e8);
            }
        }
        if (threadIdx.x == 0 && b >= 2) stage_expect<STAGING>(s, slot, kB);
        __syncthreads();
    }
    // after a wait that gave up, bulk copies still in flight must land before the block exits
    if (STAGING == GS_STAGE_BULK)
        for (int k = consumed + 1; k <= issued; ++k) mbar_wait_bounded(&s.bar[k & 1], (unsigned)(k >> 1) & 1u, kDrainLimit, err);
}

// ---- host-side launchers ------------------------------------------------------------------------

cudaError_t launch_render_fwd(int staging, const gs_proj& proj, const unsigned* vals, const unsigned* ranges,
                              const KernelCamera& cam, float* image, float* t_final, unsigned* n_contrib,
                              unsigned spin_limit, unsigned* err, cudaStream_t st) {
    const int tiles = cam.tiles_x * cam.tiles_y;
    const float4* rec = reinterpret_cast<const float4*>(proj.rec);
    const uint2* rg = reinterpret_cast<const uint2*>(ranges);
    count_launches(1);
    return launch_pdl(staging == GS_STAGE_LOADS ? k_render_fwd<GS_STAGE_LOADS> : k_render_fwd<GS_STAGE_BULK>,
                      dim3(tiles), dim3(kFwdBlock), 0, st, rec, vals, rg, cam, (unsigned)proj.n, image, t_final,
                      n_contrib, spin_limit, err);
}

template <int MODE, int PX>
static cudaError_t launch_bwd_layout(int staging, int tiles, const float4* rec, const unsigned* vals, const uint2* rg,
                                     const KernelCamera& cam, unsigned n, const float* dl, const float* target,
                                     float* loss, const float* tf, const unsigned* nc, float* g2, int thr,
                                     unsigned spin, unsigned* err, cudaStream_t st) {
    return launch_pdl(staging == GS_STAGE_LOADS ? k_render_bwd<MODE, GS_STAGE_LOADS, PX>
                                                : k_render_bwd<MODE, GS_STAGE_BULK, PX>,
                      dim3(tiles), dim3(BwdLayout<PX>::kThreads), 0, st, rec, vals, rg, cam, n, dl, target, loss, tf, nc,
                      g2, thr, spin, err);
}

// The 16x8 warp blocks (two warps per tile) unless the image has fewer than two tiles per SM, where
// the 8x8 blocks (four warps per tile) keep more warps in flight.
template <int MODE>
static cudaError_t launch_bwd_mode(int staging, int tiles, const float4* rec, const unsigned* vals, const uint2* rg,
                                   const KernelCamera& cam, unsigned n, const float* dl, const float* target,
                                   float* loss, const float* tf, const unsigned* nc, float* g2, int thr, unsigned spin,
                                   unsigned* err, cudaStream_t st) {
    if (tiles < 2 * device_sm_count())
        return launch_bwd_layout<MODE, 2>(staging, tiles, rec, vals, rg, cam, n, dl, target, loss, tf, nc, g2, thr, spin,
                                          err, st);
    return launch_bwd_layout<MODE, 4>(staging, tiles, rec, vals, rg, cam, n, dl, target, loss, tf, nc, g2, thr, spin,
                                      err, st);
}

cudaError_t launch_render_bwd(int mode, int staging, int thr, const gs_proj& proj, const unsigned* vals,
                              const unsigned* ranges, const KernelCamera& cam, const float* dl_dimage,
                              const float* target, float* loss, const float* t_final, const unsigned* n_contrib,
                              float* grad2d, unsigned spin_limit, unsigned* err, cudaStream_t st) {
    const int tiles = cam.tiles_x * cam.tiles_y;
    const float4* rec = reinterpret_cast<const float4*>(proj.rec);
    const uint2* rg = reinterpret_cast<const uint2*>(ranges);
    const unsigned n = (unsigned)proj.n;
    count_launches(1);
    switch (mode) {
        case GS_BWD_DIRECT: return launch_bwd_mode<GS_BWD_DIRECT>(staging, tiles, rec, vals, rg, cam, n, dl_dimage, target, loss, t_final, n_contrib, grad2d, thr, spin_limit, err, st);
        case GS_BWD_WARP: return launch_bwd_mode<GS_BWD_WARP>(staging, tiles, rec, vals, rg, cam, n, dl_dimage, target, loss, t_final, n_contrib, grad2d, thr, spin_limit, err, st);
        case GS_BWD_ADAPTIVE: return launch_bwd_mode<GS_BWD_ADAPTIVE>(staging, tiles, rec, vals, rg, cam, n, dl_dimage, target, loss, t_final, n_contrib, grad2d, thr, spin_limit, err, st);
        default: return launch_bwd_mode<GS_BWD_SM>(staging, tiles, rec, vals, rg, cam, n, dl_dimage, target, loss, t_final, n_contrib, grad2d, thr, spin_limit, err, st);
    }
}

}  // namespace gs
