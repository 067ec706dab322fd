// Device-side helpers shared by the library's kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gs.h"

namespace gs {

constexpr int kTile = 16;          // tile side, pixels
constexpr int kRecFloats = 12;     // floats per projected record (48 bytes)

// Bits of the device error word (its address is passed to every kernel that can set it):
// bit 0 = a bounded wait gave up, bit 1 = a consistency check failed.
constexpr unsigned kErrTimeout = 1u;
constexpr unsigned kErrCheck = 2u;

struct KernelCamera {
    float R[9], t[3];
    float fx, fy, cx, cy;
    int width, height;
    int tiles_x, tiles_y;
    float bg[3];
    float campos[3];   // camera centre in world coordinates, -R^T t
    float limx, limy;  // clamp of x/z, y/z in the projection Jacobian (huge = no clamp)
    float near_z, lowpass;
};

struct Rect { int x0, y0, x1, y1; };  // inclusive tile bounds; empty when x0 > x1

// floor(v + 1/2) of a finite float, exactly: v - floor(v) is exact or rounds monotonically
// without crossing 1/2, so the comparison with 1/2 is exact.
__device__ __forceinline__ long long floor_half(float v) {
    const float f = floorf(v);
    return (long long)f + ((v - f) >= 0.5f ? 1 : 0);
}

// Tiles overlapped by the square of half-side r around the mean. In pixel-index coordinates
// (pixel i has its centre at i + 0.5, so xh = mean_x - 0.5) tile tx covers indices 16 tx .. 16 tx + 15
// and overlaps [xh - r, xh + r] iff ceil((xh - r - 15) / 16) <= tx <= floor((xh + r) / 16); likewise
// for y. With r an integer, floor(xh + r) = floor(mean_x + 1/2) - 1 + r and
// ceil(xh - r - 15) = -floor(-mean_x + 1/2) - r - 15, and the outer floor / ceil of a division by 16
// of an integer are shifts, so the bounds are computed exactly in integer arithmetic.
// Requires finite means and 0 < r < 2^24; means are clamped to +-2^26 first, which cannot change
// a rectangle of an image narrower than 2^25 pixels.
__device__ __forceinline__ Rect tile_rect(float mx, float my, int r, int tiles_x, int tiles_y) {
    const float lim = 67108864.0f;
    mx = fminf(fmaxf(mx, -lim), lim);
    my = fminf(fmaxf(my, -lim), lim);
    const long long x1 = (floor_half(mx) - 1 + r) >> 4;
    const long long y1 = (floor_half(my) - 1 + r) >> 4;
    const long long x0 = -((floor_half(-mx) + r + 15) >> 4);
    const long long y0 = -((floor_half(-my) + r + 15) >> 4);
    const long long cx0 = x0 > 0 ? x0 : 0, cy0 = y0 > 0 ? y0 : 0;
    const long long cx1 = x1 < tiles_x - 1 ? x1 : tiles_x - 1, cy1 = y1 < tiles_y - 1 ? y1 : tiles_y - 1;
    Rect R;
    if (cx0 <= cx1 && cy0 <= cy1) {
        R.x0 = (int)cx0; R.x1 = (int)cx1; R.y0 = (int)cy0; R.y1 = (int)cy1;
    } else {
        R.x0 = 1; R.x1 = 0; R.y0 = 1; R.y1 = 0;
    }
    return R;
}

__device__ __forceinline__ unsigned smem_u32(const void* p) {
    return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

// ---- programmatic dependent launch (inline PTX, sm_90+) ---------------------------------------
// A kernel launched with programmatic stream serialization (launch_pdl) may have its blocks
// dispatched while the kernel before it in the stream is still running. pdl_wait blocks until that
// kernel has completed and its memory operations are visible. Every kernel launched that way calls
// it before touching memory that kernel may write or read, normally as its first statement. Since
// each kernel lets its dependents launch only after its own wait, anything written two or more
// kernels back is complete when a block starts and may be read before the wait (the later
// depth-sort passes do so). Without a programmatic dependency it returns at once.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
// Allows the next kernel in the stream (when launched by launch_pdl) to start dispatching its
// blocks, which then wait in pdl_wait: its launch overlaps this kernel's last wave.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }
// Both, at kernel entry.
__device__ __forceinline__ void pdl_entry() {
    pdl_wait();
    pdl_launch_dependents();
}

// ---- mbarrier + bulk asynchronous copy (inline PTX, sm_90+) ----------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// One bulk copy global -> shared of `bytes` (multiple of 16, both addresses 16-byte aligned),
// completing `bytes` of transaction count on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Orders the calling thread's earlier shared-memory writes before its later bulk copies that read
// them (generic proxy -> async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One bulk copy shared -> global of `bytes` (multiple of 16, both addresses 16-byte aligned) in the
// calling thread's bulk group; the shared source may be reused after bulk_wait_read().
__device__ __forceinline__ void bulk_copy_s2g(void* dst, const void* src, unsigned bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
                 "r"(bytes)
                 : "memory");
}

// As bulk_copy_s2g, but adds the floats to global memory (one float32 addition per element,
// performed at the L2).
__device__ __forceinline__ void bulk_add_s2g(float* dst, const float* src, unsigned bytes) {
    asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_u32(src)), "r"(bytes)
                 : "memory");
}

// Closes the calling thread's bulk group and waits until its copies have read their shared sources.
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.commit_group;\n\tcp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Asynchronous 4-byte global -> shared copy (no register staging; completes at cp_async_wait_all,
// which waits for the calling thread's own copies).
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

// As cp_async4 for 8 bytes (both addresses 8-byte aligned).
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// Copies the SH coefficients of the warp's 32 Gaussians (contiguous K3 floats each) between global
// memory and a padded shared-memory tile (row stride K3 + 1: conflict-free per-thread rows) with
// coalesced accesses, for the rows whose bit is set in `rows` (lane order). LOAD: global -> shared
// (asynchronous copies, waited for before returning unless WAIT is false, in which case the
// caller waits with cp_async_wait_all; the caller then synchronises the warp); else shared ->
// global (ADD: added to global).
template <int K3, bool LOAD, bool ADD, bool WAIT = true>
__device__ __forceinline__ void sh_tile_copy(float* tile, float* g, int first, int n, int lane, unsigned rows) {
    const int cnt = min(32, n - first);
    if (cnt <= 0 || rows == 0u) return;
    const int total = cnt * K3;
    float* gw = g + (size_t)first * K3;
    // loads are asynchronous copies, all in flight at once; the caller synchronises the warp
#pragma unroll 4
    for (int e = lane; e < total; e += 32) {
        const int row = e / K3, col = e - row * K3;
        if (!((rows >> row) & 1u)) continue;
        if (LOAD) cp_async4(&tile[row * (K3 + 1) + col], gw + e);
        else if (ADD) gw[e] += tile[row * (K3 + 1) + col];
        else gw[e] = tile[row * (K3 + 1) + col];
    }
    if (LOAD && WAIT) cp_async_wait_all();
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bound of the waits that let in-flight bulk copies land before a block exits early; independent
// of the caller's spin limit so that a small limit cannot leave copies running into a dead block.
constexpr unsigned kDrainLimit = 1u << 22;

// Bounded wait for phase `parity` of `bar`; false (and the timeout bit set) when it gives up.
// Every 1024 polls it also gives up if another wait has already set the timeout bit, so that a
// systematic failure costs one wait bound in total rather than one per block.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, unsigned parity, unsigned limit, unsigned* err) {
    for (unsigned i = 0; i < limit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 1023u) == 1023u && (*(volatile unsigned*)err & kErrTimeout)) return false;
    }
    atomicOr(err, kErrTimeout);
    return false;
}

// ---- reductions (inline PTX) -----------------------------------------------------------------

__device__ __forceinline__ void red_add_global(float* p, float v) {
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

__device__ __forceinline__ void red_add_global_v4(float* p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

__device__ __forceinline__ void red_add_shared(float* p, float v) {
    asm volatile("red.shared.add.f32 [%0], %1;" ::"r"(smem_u32(p)), "f"(v) : "memory");
}

// 2^x with the hardware approximation (relative error about 2^-22).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Reciprocal with the hardware approximation (relative error within about one unit in the last place).
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---- packed float32 pairs (inline PTX, sm_100+) -----------------------------------------------
// Two floats in one 64-bit register pair; each packed operation rounds each half exactly as the
// scalar operation would (round to nearest even), and issues as one instruction.
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 f2_pack(float lo, float hi) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ float2 f2_unpack(f32x2 v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return make_float2(lo, hi);
}

__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

__device__ __forceinline__ f32x2 f2_sub(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ f32x2 f2_mul(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

}  // namespace gs
